"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances, max over all compared elements:
  output          |O - O_ref|   <= 2e-2 * max|O_ref|
  log-sum-exp     |L - L_ref|   <= 1e-3 (absolute)
  gradients       |dX - dX_ref| <= 3e-2 * max|dX_ref|   for X in q, k, v
The inputs are bf16 and the kernels accumulate in fp32; the oracle sees the
same bf16 tensors widened exactly to fp64.  Where the reference is identically
zero (dQ and dK for a window of 1) the scale max|ref| is floored at 1e-4: the
fp32 rounding noise of dP - Delta (two sums of D products in different
orders) then has to stay below 3e-6.  Gradients of every other case are of
order 0.1 to 1, so the floor never loosens them.
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
    got = got.detach().float().cpu().numpy() if torch.is_tensor(got) else got
    ref = np.asarray(ref)
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-4))


def abs_err(got, ref):
    got = got.detach().float().cpu().numpy() if torch.is_tensor(got) else got
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    return float(np.abs(got - np.asarray(ref)).max())


def run_fwd_bwd(nc, q, k, v, dO, window, scale):
    B, T, H, D = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, T), float("nan"), dtype=torch.float32, device=q.device)
    nc.nc_attn_fwd(q, k, v, o, lse, window, scale)
    ws = torch.full((nc.nc_attn_bwd_workspace_bytes(B, T, H, D),), 0xFF, dtype=torch.uint8, device=q.device)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    nc.nc_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, window, scale, ws)
    assert nc.nc_get_device_error() == 0
    return o, lse, dq, dk, dv


def check_against_oracle(oracle_mod, q, k, v, dO, window, scale, o, lse, dq, dk, dv, grads=True):
    o_ref, lse_ref = oracle_mod.fwd(q, k, v, window, scale)
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL
    if grads:
        dq_r, dk_r, dv_r = oracle_mod.bwd(q, k, v, dO, window, scale)
        assert rel_err(dq, dq_r) <= G_TOL, "dq"
        assert rel_err(dk, dk_r) <= G_TOL, "dk"
        assert rel_err(dv, dv_r) <= G_TOL, "dv"


# ---------------------------------------------------------------- small shapes, whole tensors


def test_tiny_workload(nc, oracle_mod):
    call = workloads.TINY.calls[0]
    q, k, v, dO = workloads.make_qkvdo(call, "cuda")
    outs = run_fwd_bwd(nc, q, k, v, dO, call.window, call.scale)
    check_against_oracle(oracle_mod, q, k, v, dO, call.window, call.scale, *outs)


SWEEP = [
    # (B, T, H, D, window)
    (1, 1, 1, 64, 1), (1, 1, 1, 128, -1), (1, 7, 1, 128, 3), (2, 128, 1, 64, 1), (1, 128, 2, 128, 2),
    (1, 200, 2, 128, 127), (1, 200, 1, 128, 128), (1, 257, 1, 128, 129), (1, 333, 2, 64, 332),
    (1, 333, 1, 128, 333), (1, 333, 1, 128, 338), (2, 384, 3, 128, -1), (1, 513, 2, 64, 100),
    (1, 640, 1, 128, 256), (1, 700, 1, 128, 512),
    # more (query-tile pair, head, batch) work items than SMs, so persistent CTAs run several
    # items each, including items whose second query tile lies past T
    (2, 800, 48, 64, 300), (1, 1100, 40, 128, 200),
]


@pytest.mark.parametrize("B,T,H,D,window", SWEEP)
def test_shape_sweep(nc, oracle_mod, B, T, H, D, window):
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=1000 + T + window, device="cuda")
    scale = 1.0 / math.sqrt(D)
    outs = run_fwd_bwd(nc, q, k, v, dO, window, scale)
    check_against_oracle(oracle_mod, q, k, v, dO, window, scale, *outs)


def test_window_one_is_exact_identity(nc):
    q, k, v, dO = workloads.make_qkvdo_shape(2, 300, 3, 128, seed=77, device="cuda")
    o, lse, dq, dk, dv = run_fwd_bwd(nc, q, k, v, dO, 1, 0.088)
    assert torch.equal(o, v)
    torch.testing.assert_close(dv, dO, rtol=0, atol=0)
    assert dq.float().abs().max().item() < 1e-5 and dk.float().abs().max().item() < 1e-5


def test_scale_other_than_default(nc, oracle_mod):
    q, k, v, dO = workloads.make_qkvdo_shape(1, 256, 2, 64, seed=5, device="cuda")
    outs = run_fwd_bwd(nc, q, k, v, dO, 100, 0.3)
    check_against_oracle(oracle_mod, q, k, v, dO, 100, 0.3, *outs)


def test_repeat_calls_agree(nc):
    q, k, v, dO = workloads.make_qkvdo_shape(2, 512, 2, 128, seed=9, device="cuda")
    a = run_fwd_bwd(nc, q, k, v, dO, 200, 0.088)
    b = run_fwd_bwd(nc, q, k, v, dO, 200, 0.088)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for x, y in zip(a[2:], b[2:]):
        assert rel_err(x, y.float().cpu().numpy()) <= 1e-2


def test_guard_bytes_untouched(nc):
    """Outputs live inside larger buffers; the bytes around them must not change."""
    B, T, H, D, W = 1, 300, 2, 128, 64
    n = B * T * H * D
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=11, device="cuda")
    pad = 4096
    big = [torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    o, dq, dk, dv = (b[pad:pad + n].view(B, T, H, D) for b in big)
    lbig = torch.full((B * H * T + 2 * pad,), 5.0, dtype=torch.float32, device="cuda")
    lse = lbig[pad:pad + B * H * T].view(B, H, T)
    nc.nc_attn_fwd(q, k, v, o, lse, W, 0.088)
    wsz = nc.nc_attn_bwd_workspace_bytes(B, T, H, D)
    wbig = torch.full((wsz + 2 * pad,), 0xAB, dtype=torch.uint8, device="cuda")
    nc.nc_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, W, 0.088, wbig[pad:pad + wsz])
    torch.cuda.synchronize()
    for b in big:
        assert (b[:pad] == 7.0).all() and (b[pad + n:] == 7.0).all()
    assert (lbig[:pad] == 5.0).all() and (lbig[pad + B * H * T:] == 5.0).all()
    assert (wbig[:pad] == 0xAB).all() and (wbig[pad + wsz:] == 0xAB).all()


# ---------------------------------------------------------------- full workload sizes, sampled slices


def _slice(x, b, h):
    return x[b:b + 1, :, h:h + 1, :]


def bwd_group_picks(call, n_sm=148):
    """(b, h) slices covering every scheduling group of the backward: its work items are (key block,
    (b, h)) taken in groups of about one wave of (b, h) pairs, the last group possibly short.  The
    first and last pair of every group, plus the very last pair."""
    n_kb = (call.T + 127) // 128
    pairs = call.B * call.H
    group = min(pairs, (n_sm + n_kb - 1) // n_kb)
    picks = set()
    for g0 in range(0, pairs, group):
        for bh in (g0, min(g0 + group, pairs) - 1):
            picks.add(divmod(bh, call.H))
    picks.add((call.B - 1, call.H - 1))
    return sorted(picks)


def check_slices(oracle_mod, call, q, k, v, dO, o, lse, dq, dk, dv, picks):
    """Every picked (b, h) slice against the oracle, with the tolerances applied per slice (the scale
    of each error bound is that slice's own largest reference value)."""
    def sel(x):  # [n, T, 1, D]
        return torch.stack([x[b, :, h] for b, h in picks]).unsqueeze(2)

    qs, ks, vs, dos = (sel(x).cpu() for x in (q, k, v, dO))
    o_ref, lse_ref = oracle_mod.fwd(qs, ks, vs, call.window, call.scale)
    dq_r, dk_r, dv_r = oracle_mod.bwd(qs, ks, vs, dos, call.window, call.scale)
    got = [sel(x).float().cpu().numpy() for x in (o, dq, dk, dv)]
    got_lse = torch.stack([lse[b, h] for b, h in picks]).cpu().numpy()
    for i, (b, h) in enumerate(picks):
        assert rel_err(got[0][i], o_ref[i]) <= O_TOL, ("o", b, h)
        assert abs_err(got_lse[i], lse_ref[i, 0]) <= LSE_TOL, ("lse", b, h)
        for name, g, r in zip(("dq", "dk", "dv"), got[1:], (dq_r, dk_r, dv_r)):
            assert rel_err(g[i], r[i]) <= G_TOL, (name, b, h)


# every training call at full size; the full-causal depth-20 call and the long-context call are
# checked on every (b, h) slice, the others on every backward scheduling group
FULL_SIZE = [("D20_PAIR", 0, "groups"), ("D20_PAIR", 1, "all"), ("D30_ALT", 0, "groups"), ("D30_ALT", 1, "groups"),
             ("D30_ALT", 2, "groups"), ("D30_ALT", 3, "groups"), ("LONG_SW", 0, "all")]


@pytest.mark.parametrize("wl_name,call_idx,which", FULL_SIZE)
def test_full_size(nc, oracle_mod, wl_name, call_idx, which):
    call = getattr(workloads, wl_name).calls[call_idx]
    q, k, v, dO = workloads.make_qkvdo(call, "cuda")
    o, lse, dq, dk, dv = run_fwd_bwd(nc, q, k, v, dO, call.window, call.scale)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t).all()
    # a property that holds for every (b, h): sum_j dV_j = sum_i dO_i
    sv = dv.float().sum(1)
    so = dO.float().sum(1)
    assert (sv - so).abs().max().item() <= 3e-2 * so.abs().max().item() + 0.5
    picks = ([(b, h) for b in range(call.B) for h in range(call.H)] if which == "all" else bwd_group_picks(call))
    check_slices(oracle_mod, call, q, k, v, dO, o, lse, dq, dk, dv, picks)


# ---------------------------------------------------------------- decode


def _decode_oracle_for(oracle_mod, q, kc, vc, lens, n_list, window, scale):
    Lmax = int(max(int(lens[n]) for n in n_list))
    qs = q[n_list].cpu()
    ks = kc[n_list, :Lmax].cpu()
    vs = vc[n_list, :Lmax].cpu()
    return oracle_mod.decode(qs, ks, vs, lens[n_list].cpu(), window, scale)


@pytest.mark.parametrize("window", [1024, -1])
def test_decode_full_size_poisoned(nc, oracle_mod, window):
    wl = workloads.DECODE
    q, kc, vc, lens = workloads.make_decode(wl, "cuda", poison_tail=True)
    if window > 0:  # rows before the window are never read either
        pos = torch.arange(wl.Tmax, device="cuda").view(1, -1)
        dead = (pos < (lens.view(-1, 1) - window)).view(wl.N, wl.Tmax, 1, 1)
        kc.masked_fill_(dead, float("nan"))
        vc.masked_fill_(dead, float("nan"))
    o, lse = nc.attn_decode(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    picks = [0, 1, int(torch.argmax(lens)), int(torch.argmin(lens)), 33, 63]
    o_ref, lse_ref, ok = _decode_oracle_for(oracle_mod, q, kc, vc, lens, picks, window, wl.scale)
    assert ok
    assert rel_err(o[picks], o_ref) <= O_TOL
    assert abs_err(lse[picks], lse_ref) <= LSE_TOL


@pytest.mark.parametrize("D,window", [(64, 1), (64, 100), (128, 5), (128, -1), (64, -1)])
def test_decode_small(nc, oracle_mod, D, window):
    wl = workloads.DecodeWorkload("small", 7, 700, 3, D, 1, 700, (window,), 4242 + D)
    q, kc, vc, lens = workloads.make_decode(wl, "cuda")
    lens[0] = 1
    lens[1] = 700
    dead = (torch.arange(wl.Tmax, device="cuda").view(1, -1) >= lens.view(-1, 1)).view(wl.N, wl.Tmax, 1, 1)
    kc.masked_fill_(dead, float("nan"))
    vc.masked_fill_(dead, float("nan"))
    o, lse = nc.attn_decode(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref, ok = oracle_mod.decode(q.cpu(), kc.nan_to_num().cpu(), vc.nan_to_num().cpu(), lens.cpu(),
                                           window, wl.scale)
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL


@pytest.mark.parametrize("window", [5000, -1])
def test_decode_one_long_sequence_over_many_ctas(nc, oracle_mod, window):
    """Few sequences take the balanced split: the visible rows of all of them are cut into one equal range
    per CTA, so the 8000-row sequence here is spread over a few hundred CTAs (its combine merges more than
    32 partials, in several rounds) while the two short ones sit inside one CTA's range."""
    wl = workloads.DecodeWorkload("uneven", 3, 8000, 3, 128, 1, 8000, (window,), 515)
    q, kc, vc, _ = workloads.make_decode(wl, "cuda")
    lens = torch.tensor([1, 8000, 5], dtype=torch.int32, device="cuda")
    dead = (torch.arange(wl.Tmax, device="cuda").view(1, -1) >= lens.view(-1, 1)).view(wl.N, wl.Tmax, 1, 1)
    kc.masked_fill_(dead, float("nan"))
    vc.masked_fill_(dead, float("nan"))
    o, lse = nc.attn_decode(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref, ok = oracle_mod.decode(q.cpu(), kc.nan_to_num().cpu(), vc.nan_to_num().cpu(), lens.cpu(),
                                           window, wl.scale)
    assert ok
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL


@pytest.mark.parametrize("window", [100, -1])
def test_decode_many_sequences_fixed_chunks(nc, oracle_mod, window):
    """More than 1024 sequences take fixed 128-row chunks (D = 64) per CTA instead of the balanced split."""
    wl = workloads.DecodeWorkload("many", 1100, 300, 2, 64, 1, 300, (window,), 616)
    q, kc, vc, lens = workloads.make_decode(wl, "cuda")
    dead = (torch.arange(wl.Tmax, device="cuda").view(1, -1) >= lens.view(-1, 1)).view(wl.N, wl.Tmax, 1, 1)
    kc.masked_fill_(dead, float("nan"))
    vc.masked_fill_(dead, float("nan"))
    o, lse = nc.attn_decode(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref, ok = oracle_mod.decode(q.cpu(), kc.nan_to_num().cpu(), vc.nan_to_num().cpu(), lens.cpu(),
                                           window, wl.scale)
    assert ok
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL


@pytest.mark.parametrize("window", [100, -1])
def test_decode_more_heads_than_the_bulk_path_takes(nc, oracle_mod, window):
    """More than 16 heads: the balanced split streams with plain loads (warps over heads) instead of the
    bulk-copy stage ring."""
    wl = workloads.DecodeWorkload("heads", 5, 700, 20, 64, 1, 700, (window,), 717)
    q, kc, vc, lens = workloads.make_decode(wl, "cuda", poison_tail=True)
    o, lse = nc.attn_decode(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref, ok = oracle_mod.decode(q.cpu(), kc.nan_to_num().cpu(), vc.nan_to_num().cpu(), lens.cpu(),
                                           window, wl.scale)
    assert ok
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL


@pytest.mark.parametrize("N,H,D,window,Tmax", [(3, 16, 128, -1, 900), (5, 1, 64, 77, 640), (2, 7, 128, 300, 1000),
                                                 (4, 16, 64, 129, 513)])
def test_decode_bulk_chunk_shapes(nc, oracle_mod, N, H, D, window, Tmax):
    """The bulk-copy split's chunk is as many whole cache rows (all heads) as fit a 24 KB stage, rounded to whole
    batches of four steps: 6 rows at 16 heads of 128, 192 rows at one head of 64; lengths cover 1 and Tmax."""
    wl = workloads.DecodeWorkload("bulk", N, Tmax, H, D, 1, Tmax, (window,), 818 + H + D)
    q, kc, vc, lens = workloads.make_decode(wl, "cuda")
    lens[0] = 1
    lens[-1] = Tmax
    dead = (torch.arange(wl.Tmax, device="cuda").view(1, -1) >= lens.view(-1, 1)).view(wl.N, wl.Tmax, 1, 1)
    kc.masked_fill_(dead, float("nan"))
    vc.masked_fill_(dead, float("nan"))
    o, lse = nc.attn_decode(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref, ok = oracle_mod.decode(q.cpu(), kc.nan_to_num().cpu(), vc.nan_to_num().cpu(), lens.cpu(),
                                           window, wl.scale)
    assert ok
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL


def test_decode_equals_last_forward_row(nc):
    B, T, H, D, W = 2, 600, 2, 128, 256
    q, k, v, _ = workloads.make_qkvdo_shape(B, T, H, D, seed=31, device="cuda")
    o, lse = nc.attn_fwd(q, k, v, W)
    lens = torch.tensor([T, 451], dtype=torch.int32, device="cuda")
    qd = torch.stack([q[0, T - 1], q[1, 450]]).contiguous()
    od, lsed = nc.attn_decode(qd, k, v, lens, W)
    # sequence 1 is a 451-row prefix: compare with a forward over that prefix alone
    o1, lse1 = nc.attn_fwd(q[1:2, :451].contiguous(), k[1:2, :451].contiguous(), v[1:2, :451].contiguous(), W)
    torch.testing.assert_close(od[0].float(), o[0, T - 1].float(), atol=2e-2, rtol=0)
    torch.testing.assert_close(od[1].float(), o1[0, 450].float(), atol=2e-2, rtol=0)
    assert (lsed[0] - lse[0, :, T - 1]).abs().max().item() < 1e-3
    assert (lsed[1] - lse1[0, :, 450]).abs().max().item() < 1e-3


def test_decode_bad_length_reports_and_nans(nc):
    wl = workloads.DecodeWorkload("bad", 4, 256, 2, 128, 1, 256, (-1,), 99)
    q, kc, vc, lens = workloads.make_decode(wl, "cuda")
    lens[1] = 0
    lens[2] = 257
    o, lse = nc.attn_decode(q, kc, vc, lens, -1, wl.scale)
    assert nc.nc_get_device_error() == nc.NC_ERR_BAD_CACHE_LEN
    assert torch.isnan(o[1].float()).all() and torch.isnan(o[2].float()).all()
    assert torch.isfinite(o[0].float()).all() and torch.isfinite(o[3].float()).all()
    assert nc.nc_get_device_error() == 0  # cleared by the read


# ---------------------------------------------------------------- prefill over a KV cache


def _prefill_inputs(N, Tq, Tmax, H, D, lens, seed):
    g = workloads.generator(seed, "cuda")
    q = workloads.randn_bf16((N, Tq, H, D), g, "cuda")
    kc = workloads.randn_bf16((N, Tmax, H, D), g, "cuda")
    vc = workloads.randn_bf16((N, Tmax, H, D), g, "cuda")
    return q, kc, vc, torch.tensor(lens, dtype=torch.int32, device="cuda")


def _poison_past_length(kc, vc, lens):
    """Every cache row at or beyond a sequence's length holds NaN: the rest of the 128-row block
    that holds its last row (loaded, masked out, and its value rows zeroed before the P*V product)
    as well as every later row (never read)."""
    for n, L in enumerate(int(x) for x in lens):
        kc[n, L:] = float("nan")
        vc[n, L:] = float("nan")


PREFILL_CASES = [
    # (N, Tq, Tmax, H, D, window, lens)
    (2, 1, 300, 2, 128, 100, [1, 300]),
    (2, 37, 400, 2, 64, -1, [37, 251]),
    (3, 128, 512, 2, 128, 64, [128, 300, 512]),
    (2, 200, 700, 1, 128, 129, [200, 650]),
    (2, 257, 1024, 2, 64, 1, [300, 1024]),
    (4, 90, 1000, 3, 128, 512, [90, 91, 513, 999]),
    (2, 600, 2048, 2, 128, 256, [600, 1999]),
]


@pytest.mark.parametrize("N,Tq,Tmax,H,D,window,lens", PREFILL_CASES)
def test_prefill_small(nc, oracle_mod, N, Tq, Tmax, H, D, window, lens):
    q, kc, vc, lens_t = _prefill_inputs(N, Tq, Tmax, H, D, lens, 5000 + Tq + Tmax)
    scale = 1.0 / math.sqrt(D)
    o_ref, lse_ref, ok = oracle_mod.prefill(q.cpu(), kc.cpu(), vc.cpu(), lens_t.cpu(), window, scale)
    assert ok
    _poison_past_length(kc, vc, lens)
    o, lse = nc.attn_prefill(q, kc, vc, lens_t, window, scale)
    assert nc.nc_get_device_error() == 0
    assert rel_err(o, o_ref) <= O_TOL
    assert abs_err(lse, lse_ref) <= LSE_TOL


def test_prefill_of_whole_sequence_is_the_forward(nc):
    """Every cache row new (L = Tq = Tmax): the same products in the same order as the forward."""
    B, T, H, D, W = 2, 333, 2, 128, 100
    q, k, v, _ = workloads.make_qkvdo_shape(B, T, H, D, seed=61, device="cuda")
    o, lse = nc.attn_fwd(q, k, v, W)
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    op, lsep = nc.attn_prefill(q, k, v, lens, W)
    assert nc.nc_get_device_error() == 0
    assert torch.equal(op, o) and torch.equal(lsep, lse)


def test_prefill_of_one_token_matches_decode(nc):
    N, Tmax, H, D, W = 5, 900, 2, 128, 300
    q, kc, vc, lens = _prefill_inputs(N, 1, Tmax, H, D, [1, 2, 129, 640, 900], 71)
    op, lsep = nc.attn_prefill(q, kc, vc, lens, W)
    od, lsed = nc.attn_decode(q[:, 0].contiguous(), kc, vc, lens, W)
    assert nc.nc_get_device_error() == 0
    torch.testing.assert_close(op[:, 0].float(), od.float(), atol=2e-2, rtol=0)
    assert (lsep[:, :, 0] - lsed).abs().max().item() < 1e-3


def test_prefill_bad_length_reports_and_nans(nc, oracle_mod):
    N, Tq, Tmax, H, D = 4, 50, 256, 2, 128
    q, kc, vc, lens = _prefill_inputs(N, Tq, Tmax, H, D, [50, 49, 257, 200], 83)
    o, lse = nc.attn_prefill(q, kc, vc, lens, -1)
    assert nc.nc_get_device_error() == nc.NC_ERR_BAD_CACHE_LEN
    for n in (1, 2):
        assert torch.isnan(o[n].float()).all() and torch.isnan(lse[n]).all()
    good = [0, 3]
    o_ref, lse_ref, ok = oracle_mod.prefill(q[good].cpu(), kc[good].cpu(), vc[good].cpu(), lens[good].cpu(), -1,
                                            1.0 / math.sqrt(D))
    assert ok
    assert rel_err(o[good], o_ref) <= O_TOL
    assert abs_err(lse[good], lse_ref) <= LSE_TOL
    assert nc.nc_get_device_error() == 0  # cleared by the read


@pytest.mark.parametrize("window", [1024, -1])
def test_prefill_full_size_sampled(nc, oracle_mod, window):
    """The benchmark's prefill workload; the oracle checks the last 256 new tokens of a few
    (sequence, head) slices, which sit at the same cache positions in a Tq = 256 prefill."""
    wl = workloads.PREFILL
    q, kc, vc, lens = workloads.make_prefill(wl, "cuda")
    o, lse = nc.attn_prefill(q, kc, vc, lens, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    seqs, heads, tail = [0, int(torch.argmax(lens)), int(torch.argmin(lens))], [0, 7], 256
    for hh in heads:
        qs = q[seqs, wl.Tq - tail:, hh:hh + 1].contiguous().cpu()
        ks = kc[seqs, :, hh:hh + 1].contiguous().cpu()
        vs = vc[seqs, :, hh:hh + 1].contiguous().cpu()
        o_ref, lse_ref, ok = oracle_mod.prefill(qs, ks, vs, lens[seqs].cpu(), window, wl.scale)
        assert ok
        assert rel_err(o[seqs, wl.Tq - tail:, hh:hh + 1], o_ref) <= O_TOL
        assert abs_err(lse[seqs, hh:hh + 1, wl.Tq - tail:], lse_ref) <= LSE_TOL


# ---------------------------------------------------------------- document-masked (varlen) attention


VARLEN_CASES = [
    # (doc lengths, H, D, window)
    ([7], 2, 128, 3),
    ([1, 1, 130, 0, 257, 5], 2, 128, -1),
    ([300, 64, 1, 700], 2, 64, 100),
    ([128, 128, 256, 511, 1], 3, 128, 128),
    ([1000, 999, 2], 1, 128, 1),
]


def _varlen_inputs(lens, H, D, seed):
    total = sum(lens)
    g = workloads.generator(seed, "cuda")
    q, k, v, dO = (workloads.randn_bf16((total, H, D), g, "cuda") for _ in range(4))
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    return q, k, v, dO, cu


@pytest.mark.parametrize("lens,H,D,window", VARLEN_CASES)
def test_fwd_varlen_small(nc, oracle_mod, lens, H, D, window):
    q, k, v, _, cu = _varlen_inputs(lens, H, D, 6000 + sum(lens))
    scale = 1.0 / math.sqrt(D)
    o, lse = nc.attn_fwd_varlen(q, k, v, cu, max(lens), window, scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref = oracle_mod.fwd_varlen(q.unsqueeze(0).cpu(), k.unsqueeze(0).cpu(), v.unsqueeze(0).cpu(),
                                           cu.cpu(), window, scale)
    assert rel_err(o, o_ref[0]) <= O_TOL
    assert abs_err(lse, lse_ref[0]) <= LSE_TOL


@pytest.mark.parametrize("lens,H,D,window", VARLEN_CASES)
def test_bwd_varlen_small(nc, oracle_mod, lens, H, D, window):
    q, k, v, dO, cu = _varlen_inputs(lens, H, D, 7000 + sum(lens))
    scale = 1.0 / math.sqrt(D)
    o, lse = nc.attn_fwd_varlen(q, k, v, cu, max(lens), window, scale)
    dq, dk, dv = nc.attn_bwd_varlen(q, k, v, o, dO, lse, cu, max(lens), window, scale)
    assert nc.nc_get_device_error() == 0
    refs = oracle_mod.bwd_varlen(q.unsqueeze(0).cpu(), k.unsqueeze(0).cpu(), v.unsqueeze(0).cpu(),
                                 dO.unsqueeze(0).cpu(), cu.cpu(), window, scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        assert rel_err(got, ref[0]) <= G_TOL, name


def test_bwd_varlen_single_document_is_the_backward(nc):
    T, H, D, W = 333, 2, 128, 100
    q, k, v, dO = workloads.make_qkvdo_shape(1, T, H, D, seed=93, device="cuda")
    o, lse, dq, dk, dv = run_fwd_bwd(nc, q, k, v, dO, W, 1.0 / math.sqrt(D))
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    dqv, dkv, dvv = nc.attn_bwd_varlen(q[0], k[0], v[0], o[0], dO[0], lse[0], cu, T, W, 1.0 / math.sqrt(D))
    assert nc.nc_get_device_error() == 0
    assert torch.equal(dkv, dk[0]) and torch.equal(dvv, dv[0])  # one key block per CTA: a fixed order
    torch.testing.assert_close(dqv.float(), dq[0].float(), atol=2e-2, rtol=0)  # dQ sums in any order


@pytest.mark.parametrize("window", [1024, -1])
def test_varlen_full_size_sampled(nc, oracle_mod, window):
    """The packed-documents workload; the oracle checks a few documents on two heads."""
    wl = workloads.VARLEN
    q, k, v, dO, cu, max_len = workloads.make_varlen(wl, "cuda")
    o, lse = nc.attn_fwd_varlen(q, k, v, cu, max_len, window, wl.scale)
    dq, dk, dv = nc.attn_bwd_varlen(q, k, v, o, dO, lse, cu, max_len, window, wl.scale)
    assert nc.nc_get_device_error() == 0
    lens = (cu[1:] - cu[:-1]).tolist()
    for d in (0, int(np.argmax(lens)), int(np.argmin(lens)), len(lens) - 1):
        a, b = int(cu[d]), int(cu[d + 1])
        for hh in (0, 9):
            sl = lambda x: x[a:b, hh:hh + 1].unsqueeze(0).cpu()
            o_ref, lse_ref = oracle_mod.fwd(sl(q), sl(k), sl(v), window, wl.scale)
            assert rel_err(o[a:b, hh:hh + 1], o_ref[0]) <= O_TOL
            assert abs_err(lse[hh:hh + 1, a:b], lse_ref[0]) <= LSE_TOL
            refs = oracle_mod.bwd(sl(q), sl(k), sl(v), sl(dO), window, wl.scale)
            for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
                assert rel_err(got[a:b, hh:hh + 1], ref[0]) <= G_TOL, name


def test_fwd_varlen_single_document_is_the_forward(nc):
    T, H, D, W = 333, 2, 128, 100
    q, k, v, _ = workloads.make_qkvdo_shape(1, T, H, D, seed=91, device="cuda")
    o, lse = nc.attn_fwd(q, k, v, W)
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    ov, lsev = nc.attn_fwd_varlen(q[0], k[0], v[0], cu, T, W)
    assert nc.nc_get_device_error() == 0
    assert torch.equal(ov, o[0]) and torch.equal(lsev, lse[0])


def test_fwd_varlen_bad_document_reports(nc, oracle_mod):
    lens = [100, 400, 50]  # the middle document is longer than max_seqlen below
    q, k, v, _, cu = _varlen_inputs(lens, 2, 128, 97)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((2, sum(lens)), float("nan"), dtype=torch.float32, device="cuda")
    nc.nc_attn_fwd_varlen(q, k, v, cu, o, lse, 256, -1, 0.1)
    assert nc.nc_get_device_error() == nc.NC_ERR_BAD_SEQLENS
    assert torch.isnan(o[100:500].float()).all()  # not written
    o_ref, lse_ref = oracle_mod.fwd_varlen(q.unsqueeze(0).cpu(), k.unsqueeze(0).cpu(), v.unsqueeze(0).cpu(),
                                           cu.cpu(), -1, 0.1)
    for sl in (slice(0, 100), slice(500, 550)):
        assert rel_err(o[sl], o_ref[0, sl]) <= O_TOL
        assert abs_err(lse[:, sl], lse_ref[0][:, sl]) <= LSE_TOL
    assert nc.nc_get_device_error() == 0


# ---------------------------------------------------------------- failure detection


def test_bounded_wait_reports_timeout_and_context_survives(nc):
    """A wait on a barrier nothing completes runs out (about 1 ms), sets the error word, and returns."""
    nc.nc_debug_watchdog_selftest(2_000_000)
    assert nc.nc_get_device_error() == nc.NC_ERR_DEVICE_TIMEOUT
    assert nc.nc_get_device_error() == 0
    q, k, v, dO = workloads.make_qkvdo_shape(1, 128, 1, 64, seed=3, device="cuda")
    o, lse = nc.attn_fwd(q, k, v, 16)
    assert nc.nc_get_device_error() == 0 and torch.isfinite(o.float()).all()
