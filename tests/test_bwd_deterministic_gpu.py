"""GPU: the deterministic backward (nc_attn_bwd_deterministic) through the C ABI.

Three things are checked:
  * parity with the fp64 oracle, at the tolerances of the plain backward
    (|dX - dX_ref| <= 3e-2 * max|dX_ref|, the scale floored at 1e-4);
  * bitwise reproducibility of dq, dk and dv over repeated calls whose
    workspaces start with different garbage;
  * dk and dv bitwise equal to those of nc_attn_bwd (the same products in the
    same order in both modes), dq equal to its dq up to summation order and
    the rounding of P (kept in fp32 by the dQ pass, bf16 in the main pass).
"""
import math

import numpy as np
import pytest
import torch

from causal_sliding_window_fwd_b300 import workloads

pytestmark = pytest.mark.gpu

G_TOL = 3e-2


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_sliding_window_fwd_b300 import nc_attn
    return nc_attn


def rel_err(got, ref):
    got = got.detach().float().cpu().numpy()
    ref = np.asarray(ref)
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-4))


def forward(nc, q, k, v, window, scale):
    B, T, H, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    nc.nc_attn_fwd(q, k, v, o, lse, window, scale)
    return o, lse


def backward(nc, q, k, v, o, dO, lse, window, scale, deterministic, fill=0xFF):
    B, T, H, D = q.shape
    ws = torch.full((nc.nc_attn_bwd_workspace_bytes(B, T, H, D),), fill, dtype=torch.uint8, device=q.device)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    fn = nc.nc_attn_bwd_deterministic if deterministic else nc.nc_attn_bwd
    fn(q, k, v, o, dO, lse, dq, dk, dv, window, scale, ws)
    assert nc.nc_get_device_error() == 0
    return dq, dk, dv


CASES = [
    # (B, T, H, D, window): single blocks, ragged tails, windows of 1, below, at and above a block,
    # full causal, and more (query block, head, batch) items than SMs
    (1, 1, 1, 64, 1), (1, 7, 1, 128, 3), (2, 128, 1, 64, 1), (1, 200, 2, 128, 127), (1, 257, 1, 128, 129),
    (1, 333, 2, 64, 332), (2, 384, 3, 128, -1), (1, 513, 2, 64, 100), (1, 700, 1, 128, 512),
    (2, 800, 48, 64, 300), (1, 1100, 40, 128, 200),
]


@pytest.mark.parametrize("B,T,H,D,window", CASES)
def test_deterministic_matches_oracle(nc, oracle_mod, B, T, H, D, window):
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=3000 + T + window, device="cuda")
    scale = 1.0 / math.sqrt(D)
    o, lse = forward(nc, q, k, v, window, scale)
    dq, dk, dv = backward(nc, q, k, v, o, dO, lse, window, scale, True)
    dq_r, dk_r, dv_r = oracle_mod.bwd(q.cpu(), k.cpu(), v.cpu(), dO.cpu(), window, scale)
    assert rel_err(dq, dq_r) <= G_TOL, "dq"
    assert rel_err(dk, dk_r) <= G_TOL, "dk"
    assert rel_err(dv, dv_r) <= G_TOL, "dv"
    # dK and dV come from the same products in the same order as in the plain backward
    dq2, dk2, dv2 = backward(nc, q, k, v, o, dO, lse, window, scale, False)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    # the two paths round dS differently (the dQ pass keeps P in fp32), so they agree to about one
    # bf16 unit of the largest entries
    assert (dq.float() - dq2.float()).abs().max().item() <= 1e-2 * dq2.float().abs().max().item()


def test_deterministic_is_bitwise_repeatable(nc):
    B, T, H, D, W = 2, 1000, 20, 128, 300
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=31, device="cuda")
    o, lse = forward(nc, q, k, v, W, 0.088)
    first = backward(nc, q, k, v, o, dO, lse, W, 0.088, True, fill=0x00)
    for fill in (0xFF, 0x7F):
        again = backward(nc, q, k, v, o, dO, lse, W, 0.088, True, fill=fill)
        for x, y in zip(first, again):
            assert torch.equal(x, y)


def test_deterministic_window_one(nc):
    """Window 1: o = v, dv = dO exactly, and dq = dk = 0 up to the rounding of dP - Delta."""
    q, k, v, dO = workloads.make_qkvdo_shape(2, 300, 3, 128, seed=77, device="cuda")
    o, lse = forward(nc, q, k, v, 1, 0.088)
    dq, dk, dv = backward(nc, q, k, v, o, dO, lse, 1, 0.088, True)
    assert torch.equal(dv, dO)
    assert dq.float().abs().max().item() < 1e-5 and dk.float().abs().max().item() < 1e-5


@pytest.mark.parametrize("wl_name,call_idx", [("D20_PAIR", 0), ("D20_PAIR", 1), ("D30_ALT", 0), ("LONG_SW", 0)])
def test_deterministic_full_size(nc, oracle_mod, wl_name, call_idx):
    """Training calls at full size (the depth-20 pair, the window-512 depth-30 call, the long-context
    call): one slice of every scheduling group against the oracle, repeatability, and agreement with
    the plain backward."""
    call = getattr(workloads, wl_name).calls[call_idx]
    q, k, v, dO = workloads.make_qkvdo(call, "cuda")
    o, lse = forward(nc, q, k, v, call.window, call.scale)
    dq, dk, dv = backward(nc, q, k, v, o, dO, lse, call.window, call.scale, True)
    dq1, dk1, dv1 = backward(nc, q, k, v, o, dO, lse, call.window, call.scale, True, fill=0x00)
    assert torch.equal(dq, dq1) and torch.equal(dk, dk1) and torch.equal(dv, dv1)
    dq2, dk2, dv2 = backward(nc, q, k, v, o, dO, lse, call.window, call.scale, False)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert (dq.float() - dq2.float()).abs().max().item() <= 2e-2 * dq2.float().abs().max().item()
    # the dQ pass hands out (query block, (b, h)) items in groups of about one wave of (b, h) pairs
    n_qb = (call.T + 127) // 128
    pairs = call.B * call.H
    group = min(pairs, (148 + n_qb - 1) // n_qb)
    picks = sorted({divmod(min(g0 + group, pairs) - 1, call.H) for g0 in range(0, pairs, group)} |
                   {(0, 0), (call.B - 1, call.H - 1)})
    sel = lambda x: torch.stack([x[b, :, h] for b, h in picks]).unsqueeze(2)
    dq_r, dk_r, dv_r = oracle_mod.bwd(*(sel(x).cpu() for x in (q, k, v, dO)), call.window, call.scale)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), (dq_r, dk_r, dv_r)):
        g = sel(g).float().cpu()
        for i, (b, h) in enumerate(picks):
            assert rel_err(g[i], r[i]) <= G_TOL, (name, b, h)


# ---------------------------------------------------------------- packed documents


def varlen_inputs(lens, H, D, seed, total=None):
    total = sum(lens) if total is None else total
    g = workloads.generator(seed, "cuda")
    q, k, v, dO = (workloads.randn_bf16((total, H, D), g, "cuda") for _ in range(4))
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    return q, k, v, dO, cu


def varlen_backward(nc, q, k, v, o, dO, lse, cu, max_len, window, scale, deterministic, fill=0xFF):
    total, H, D = q.shape
    ws = torch.full((nc.nc_attn_bwd_workspace_bytes(1, total, H, D),), fill, dtype=torch.uint8, device=q.device)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    nc.nc_attn_bwd_varlen(q, k, v, o, dO, lse, cu, dq, dk, dv, max_len, window, scale, ws,
                          deterministic=deterministic)
    return dq, dk, dv


@pytest.mark.parametrize("lens,H,D,window", [
    ([130, 1, 257, 64, 300], 2, 128, -1), ([130, 1, 257, 64, 300], 2, 128, 100), ([1000, 24, 512], 3, 64, 200),
    ([5, 3], 1, 128, 1), ([640], 2, 128, 256),
])
def test_varlen_deterministic_matches_oracle_and_repeats(nc, oracle_mod, lens, H, D, window):
    q, k, v, dO, cu = varlen_inputs(lens, H, D, 7600 + sum(lens) + D)
    scale = 1.0 / math.sqrt(D)
    o, lse = nc.attn_fwd_varlen(q, k, v, cu, max(lens), window, scale)
    runs = [varlen_backward(nc, q, k, v, o, dO, lse, cu, max(lens), window, scale, True, fill) for fill in (0xFF, 0x00)]
    assert nc.nc_get_device_error() == 0
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    dq, dk, dv = runs[0]
    pq, pk, pv = varlen_backward(nc, q, k, v, o, dO, lse, cu, max(lens), window, scale, False)
    assert torch.equal(dk, pk) and torch.equal(dv, pv)
    refs = oracle_mod.bwd_varlen(q.unsqueeze(0).cpu(), k.unsqueeze(0).cpu(), v.unsqueeze(0).cpu(),
                                 dO.unsqueeze(0).cpu(), cu.cpu(), window, scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_err(got, ref[0]) <= G_TOL, name


def test_varlen_deterministic_rows_outside_documents(nc):
    """Rows past the last document: dq is zero (as from nc_attn_bwd_varlen), dk and dv are not written."""
    lens, total, H, D = [100, 200], 400, 2, 128
    q, k, v, dO, cu = varlen_inputs(lens, H, D, 7700, total=total)
    o, lse = nc.attn_fwd_varlen(q, k, v, cu, 200, 64)
    dq, dk, dv = varlen_backward(nc, q, k, v, o, dO, lse, cu, 200, 64, 1.0 / math.sqrt(D), True)
    assert nc.nc_get_device_error() == 0
    assert (dq[300:].float() == 0).all()
    assert torch.isnan(dk[300:].float()).all() and torch.isnan(dv[300:].float()).all()
    pq, pk, pv = varlen_backward(nc, q, k, v, o, dO, lse, cu, 200, 64, 1.0 / math.sqrt(D), False)
    assert torch.equal(dk[:300], pk[:300]) and torch.equal(dv[:300], pv[:300])
    assert (pq[300:].float() == 0).all()


def test_varlen_deterministic_bad_document_reports(nc):
    lens = [100, 400, 50]  # the middle document is longer than max_seqlen below
    q, k, v, dO, cu = varlen_inputs(lens, 2, 128, 7800)
    o = torch.zeros_like(q)
    lse = torch.zeros((2, sum(lens)), dtype=torch.float32, device="cuda")
    varlen_backward(nc, q, k, v, o, dO, lse, cu, 256, -1, 0.1, True)
    assert nc.nc_get_device_error() == nc.NC_ERR_BAD_SEQLENS
    assert nc.nc_get_device_error() == 0
