"""GPU parity of the rotary entry points (q and k turned by one launch, then the attention; dq and dk
turned back in the backward's conversion pass) and of the standalone turn, against the fp64 oracle.

Tolerances as in test_parity_gpu: output <= 2e-2 max|ref|, lse <= 1e-3 absolute, gradients <= 3e-2
max|ref| (per (b, h) slice at full size).  The kernel turns q and k in float32 and rounds the turned rows to
bf16; the oracle takes that quantisation the same way (float32 turn, then round to nearest even) and is fp64
from there on, including its exact turn back of the gradients.
"""
import math

import numpy as np
import pytest
import torch

from causal_sliding_window_fwd_b300 import workloads

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, G_TOL = 2e-2, 1e-3, 3e-2


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_sliding_window_fwd_b300 import nc_attn
    return nc_attn


def rel_err(got, ref):
    got = got.detach().float().cpu().numpy() if torch.is_tensor(got) else np.asarray(got)
    ref = np.asarray(ref)
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-4))


def abs_err(got, ref):
    got = got.detach().float().cpu().numpy() if torch.is_tensor(got) else np.asarray(got)
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    return float(np.abs(got - np.asarray(ref)).max())


def run(nc, q, k, v, dO, c, s, window, scale):
    B, T, H, D = q.shape
    o, qr, kr = (torch.full_like(q, float("nan")) for _ in range(3))
    lse = torch.full((B, H, T), float("nan"), dtype=torch.float32, device=q.device)
    nc.nc_attn_fwd_rotary(q, k, v, c, s, qr, kr, o, lse, window, scale)
    ws = torch.full((nc.nc_attn_bwd_workspace_bytes(B, T, H, D),), 0xFF, dtype=torch.uint8, device=q.device)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    nc.nc_attn_bwd_rotary(qr, kr, v, c, s, o, dO, lse, dq, dk, dv, window, scale, ws)
    assert nc.nc_get_device_error() == 0
    return o, lse, dq, dk, dv


CASES = [
    # (B, T, H, D, window)
    (1, 128, 2, 64, 32), (1, 1, 1, 128, -1), (2, 200, 1, 128, 1), (1, 257, 2, 128, 129), (1, 333, 1, 64, 100),
    (2, 384, 3, 128, -1), (1, 700, 2, 128, 512), (2, 800, 40, 64, 300), (1, 1100, 24, 128, 200),
]


@pytest.mark.parametrize("B,T,H,D,window", CASES)
def test_rotary_matches_oracle(nc, oracle_mod, B, T, H, D, window):
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=4000 + T + window, device="cuda")
    c, s = workloads.rope_tables(T, D, device="cuda")
    scale = 1.0 / math.sqrt(D)
    o, lse, dq, dk, dv = run(nc, q, k, v, dO, c, s, window, scale)
    args = [x.cpu() for x in (q, k, v)]
    o_r, lse_r = oracle_mod.fwd_rotary(*args, c.cpu(), s.cpu(), window, scale)
    assert rel_err(o, o_r) <= O_TOL
    assert abs_err(lse, lse_r) <= LSE_TOL
    dq_r, dk_r, dv_r = oracle_mod.bwd_rotary(*args, dO.cpu(), c.cpu(), s.cpu(), window, scale)
    assert rel_err(dq, dq_r) <= G_TOL, "dq"
    assert rel_err(dk, dk_r) <= G_TOL, "dk"
    assert rel_err(dv, dv_r) <= G_TOL, "dv"


@pytest.mark.parametrize("D", [64, 128])
def test_identity_tables_give_the_plain_kernels(nc, D):
    """cos = 1, sin = 0 turns nothing: the turned rows are the inputs and every output equals the plain
    forward / backward (dq up to the order in which its fp32 partials are added)."""
    B, T, H, W = 2, 333, 3, 100
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=4100 + D, device="cuda")
    c = torch.ones((T, D // 2), dtype=torch.float32, device="cuda")
    s = torch.zeros((T, D // 2), dtype=torch.float32, device="cuda")
    o, lse, dq, dk, dv = run(nc, q, k, v, dO, c, s, W, 0.09)
    o2, lse2 = nc.attn_fwd(q, k, v, W, 0.09)
    dq2, dk2, dv2 = nc.attn_bwd(q, k, v, o2, dO, lse2, W, 0.09)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert (dq.float() - dq2.float()).abs().max().item() <= 1e-2 * dq2.float().abs().max().item()


@pytest.mark.parametrize("wl_name,call_idx", [("D20_PAIR", 0), ("D20_PAIR", 1), ("LONG_SW", 0)])
def test_rotary_full_size(nc, oracle_mod, wl_name, call_idx):
    """Training shapes at full size: the first and last (b, h) of every backward scheduling group."""
    call = getattr(workloads, wl_name).calls[call_idx]
    q, k, v, dO = workloads.make_qkvdo(call, "cuda")
    c, s = workloads.rope_tables(call.T, call.D, device="cuda")
    o, lse, dq, dk, dv = run(nc, q, k, v, dO, c, s, call.window, call.scale)
    n_kb = (call.T + 127) // 128
    pairs = call.B * call.H
    group = min(pairs, (148 + n_kb - 1) // n_kb)
    picks = sorted({divmod(bh, call.H) for g0 in range(0, pairs, group) for bh in (g0, min(g0 + group, pairs) - 1)})

    def sel(x):
        return torch.stack([x[b, :, h] for b, h in picks]).unsqueeze(2)

    qs, ks, vs, dos = (sel(x).cpu() for x in (q, k, v, dO))
    o_r, lse_r = oracle_mod.fwd_rotary(qs, ks, vs, c.cpu(), s.cpu(), call.window, call.scale)
    dq_r, dk_r, dv_r = oracle_mod.bwd_rotary(qs, ks, vs, dos, c.cpu(), s.cpu(), call.window, call.scale)
    got = [sel(x).float().cpu().numpy() for x in (o, dq, dk, dv)]
    got_lse = torch.stack([lse[b, h] for b, h in picks]).cpu().numpy()
    for i, (b, h) in enumerate(picks):
        assert rel_err(got[0][i], o_r[i]) <= O_TOL, ("o", b, h)
        assert abs_err(got_lse[i], lse_r[i, 0]) <= LSE_TOL, ("lse", b, h)
        for name, g, r in zip(("dq", "dk", "dv"), got[1:], (dq_r, dk_r, dv_r)):
            assert rel_err(g[i], r[i]) <= G_TOL, (name, b, h)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("inverse", [False, True])
def test_standalone_turn_matches_oracle(nc, oracle_mod, D, inverse):
    """The unfused turn: every element within one bf16 rounding of the fp64 turn (|err| <= 2^-8 |ref|,
    plus 1e-5 for the fp32 products), and in place equal to out of place."""
    B, T, H = 3, 301, 5
    x = workloads.make_qkvdo_shape(B, T, H, D, seed=4200 + D, device="cuda")[0]
    c, s = workloads.rope_tables(T, D, device="cuda")
    y = nc.rotary(x, c, s, inverse=inverse)
    ref = np.asarray(oracle_mod.rotary(x.cpu(), c.cpu(), s.cpu(), inverse=inverse))
    got = y.float().cpu().numpy()
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all()
    x2 = x.clone()
    nc.nc_rotary(x2, c, s, x2, inverse)
    assert torch.equal(x2, y)
    assert nc.nc_get_device_error() == 0


def test_turned_rows_and_the_standalone_turn_agree(nc, oracle_mod):
    """The turned q and k that the rotary forward writes are the standalone turn's, and they are the
    oracle's float32 turn rounded to bf16, bit for bit."""
    B, T, H, D, W = 2, 500, 3, 128, 200
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=4300, device="cuda")
    c, s = workloads.rope_tables(T, D, device="cuda")
    o, lse, qr, kr = nc.attn_fwd_rotary(q, k, v, c, s, W, 0.1)
    assert torch.equal(qr, nc.rotary(q, c, s)) and torch.equal(kr, nc.rotary(k, c, s))
    np.testing.assert_array_equal(qr.double().cpu().numpy(), oracle_mod.rotary_bf16(q.cpu(), c.cpu(), s.cpu()))
    o2, lse2 = nc.attn_fwd(qr, kr, v, W, 0.1)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_rotary_composes_with_packed_documents(nc, oracle_mod):
    """Packed documents with each row turned by its position inside its document: the standalone turn with
    per-row tables [total, D/2] (B = 1, T = total), the varlen forward and backward on the turned rows, and the
    turn back of dq and dk.  The oracle composes its own turn, its per-document attention and its exact
    transpose."""
    lens = [130, 1, 257, 64, 300, 128]
    H, D = 2, 128
    total = sum(lens)
    g = workloads.generator(4700, "cuda")
    q, k, v, dO = (workloads.randn_bf16((total, H, D), g, "cuda") for _ in range(4))
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    pos = torch.cat([torch.arange(n) for n in lens])
    c_all, s_all = workloads.rope_tables(max(lens), D)
    c, s = c_all[pos].contiguous().cuda(), s_all[pos].contiguous().cuda()
    scale = 1.0 / math.sqrt(D)
    for window in (-1, 100):
        qr = nc.rotary(q.unsqueeze(0), c, s)[0]
        kr = nc.rotary(k.unsqueeze(0), c, s)[0]
        o, lse = nc.attn_fwd_varlen(qr, kr, v, cu, max(lens), window, scale)
        dqr, dkr, dv = nc.attn_bwd_varlen(qr, kr, v, o, dO, lse, cu, max(lens), window, scale)
        dq = nc.rotary(dqr.unsqueeze(0), c, s, inverse=True)[0]
        dk = nc.rotary(dkr.unsqueeze(0), c, s, inverse=True)[0]
        assert nc.nc_get_device_error() == 0
        cc, ss = c.cpu(), s.cpu()
        qr_o = oracle_mod.rotary_bf16(q.cpu().unsqueeze(0), cc, ss)
        kr_o = oracle_mod.rotary_bf16(k.cpu().unsqueeze(0), cc, ss)
        # the turned rows are a quantisation decided in float32: bit-exact
        assert np.array_equal(qr.float().cpu().numpy(), qr_o[0]) and np.array_equal(kr.float().cpu().numpy(), kr_o[0])
        vv, gg = v.cpu().unsqueeze(0), dO.cpu().unsqueeze(0)
        o_r, lse_r = oracle_mod.fwd_varlen(qr_o, kr_o, vv, cu.cpu(), window, scale)
        dqr_r, dkr_r, dv_r = oracle_mod.bwd_varlen(qr_o, kr_o, vv, gg, cu.cpu(), window, scale)
        dq_r = oracle_mod.rotary(dqr_r, cc, ss, inverse=True)
        dk_r = oracle_mod.rotary(dkr_r, cc, ss, inverse=True)
        assert rel_err(o, o_r[0]) <= O_TOL
        assert abs_err(lse, lse_r[0]) <= LSE_TOL
        for got, ref in ((dq, dq_r[0]), (dk, dk_r[0]), (dv, dv_r[0])):
            assert rel_err(got, ref) <= G_TOL


def test_rotary_composes_with_the_deterministic_backward(nc):
    """Rotary q and k with a bitwise-reproducible backward: the deterministic backward on the turned rows, then
    the turn back of dq and dk.  Two runs are bitwise equal, and the result agrees with the fused rotary
    backward (which adds dQ with fp32 atomics) to its atomic-order noise."""
    B, T, H, D, W = 2, 520, 2, 128, 200
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=4800, device="cuda")
    c, s = workloads.rope_tables(T, D, device="cuda")
    o, lse, qr, kr = nc.attn_fwd_rotary(q, k, v, c, s, W)
    runs = []
    for _ in range(2):
        dqr, dkr, dv = nc.attn_bwd(qr, kr, v, o, dO, lse, W, deterministic=True)
        runs.append((nc.rotary(dqr, c, s, inverse=True), nc.rotary(dkr, c, s, inverse=True), dv))
    assert all(torch.equal(a, b) for a, b in zip(*runs))
    dq_f, dk_f, dv_f = nc.attn_bwd_rotary(qr, kr, v, c, s, o, dO, lse, W)
    dq, dk, dv = runs[0]
    assert torch.equal(dv, dv_f)
    for got, ref in ((dq, dq_f), (dk, dk_f)):
        err = (got.float() - ref.float()).abs().max().item()
        assert err <= 1e-2 * ref.float().abs().max().item()
    assert nc.nc_get_device_error() == 0
