"""The library's calls inside CUDA graphs: captured once, replayed, and equal to the same calls run eagerly.

Every launch goes to the caller's stream and the host does no synchronisation, so a torch CUDA graph can
capture a training step (forward + backward), a packed-document step, or an engine step (append + prefill,
append + decode).  Replays must give the eager results: bitwise where the kernels are deterministic (forward,
dk, dv, decode, prefill), within the fp32 atomic-order noise for dq.
"""
import numpy as np
import pytest
import torch

from causal_sliding_window_fwd_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_sliding_window_fwd_b300 import nc_attn
    return nc_attn


def capture(fn):
    """Runs fn once eagerly on a side stream (first-call setup happens outside the capture), then captures it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def close_dq(a, b):
    return (a.float() - b.float()).abs().max().item() <= 1e-2 * b.float().abs().max().item()


def test_training_step_in_a_graph(nc):
    B, T, H, D, W = 2, 640, 3, 128, 256
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=6100, device="cuda")
    o_e, lse_e = nc.attn_fwd(q, k, v, W)
    dq_e, dk_e, dv_e = nc.attn_bwd(q, k, v, o_e, dO, lse_e, W)
    o, lse = torch.empty_like(q), torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(nc.nc_attn_bwd_workspace_bytes(B, T, H, D), dtype=torch.uint8, device="cuda")
    scale = nc.default_scale(D)

    def step():
        nc.nc_attn_fwd(q, k, v, o, lse, W, scale)
        nc.nc_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, W, scale, ws)

    g = capture(step)
    for _ in range(3):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_e) and torch.equal(lse, lse_e)
        assert torch.equal(dk, dk_e) and torch.equal(dv, dv_e) and close_dq(dq, dq_e)
    assert nc.nc_get_device_error() == 0


def test_packed_documents_step_in_a_graph(nc):
    lens = [300, 1, 129, 511]
    total, H, D, W = sum(lens), 2, 128, 128
    g0 = workloads.generator(6200, "cuda")
    q, k, v, dO = (workloads.randn_bf16((total, H, D), g0, "cuda") for _ in range(4))
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    o_e, lse_e = nc.attn_fwd_varlen(q, k, v, cu, max(lens), W)
    dq_e, dk_e, dv_e = nc.attn_bwd_varlen(q, k, v, o_e, dO, lse_e, cu, max(lens), W)
    o, lse = torch.empty_like(q), torch.empty((H, total), dtype=torch.float32, device="cuda")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(nc.nc_attn_bwd_workspace_bytes(1, total, H, D), dtype=torch.uint8, device="cuda")
    scale = nc.default_scale(D)

    def step():
        nc.nc_attn_fwd_varlen(q, k, v, cu, o, lse, max(lens), W, scale)
        nc.nc_attn_bwd_varlen(q, k, v, o, dO, lse, cu, dq, dk, dv, max(lens), W, scale, ws)

    g = capture(step)
    for _ in range(3):
        for t in (o, lse, dq, dk, dv):
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_e) and torch.equal(lse, lse_e)
        assert torch.equal(dk, dk_e) and torch.equal(dv, dv_e) and close_dq(dq, dq_e)
    assert nc.nc_get_device_error() == 0


@pytest.mark.parametrize("Tq", [1, 160])
def test_engine_step_in_a_graph(nc, Tq):
    """Append the new tokens' keys and values, then prefill (Tq > 1) or decode (Tq = 1)."""
    N, Tmax, H, D, W = 3, 600, 2, 128, 256
    g0 = workloads.generator(6300 + Tq, "cuda")
    kc0, vc0 = (workloads.randn_bf16((N, Tmax, H, D), g0, "cuda") for _ in range(2))
    kn, vn, q = (workloads.randn_bf16((N, Tq, H, D), g0, "cuda") for _ in range(3))
    lens = torch.tensor([Tq, 600, 333], dtype=torch.int32, device="cuda")
    scale = nc.default_scale(D)
    kc, vc = kc0.clone(), vc0.clone()
    ws = torch.empty(nc.nc_attn_decode_workspace_bytes(N, Tmax, H, D), dtype=torch.uint8, device="cuda")
    q1 = q[:, 0].contiguous()  # the decode query [N, H, D]
    if Tq == 1:
        o, lse = torch.empty((N, H, D), dtype=torch.bfloat16, device="cuda"), torch.empty((N, H), device="cuda")
    else:
        o, lse = torch.empty_like(q), torch.empty((N, H, Tq), dtype=torch.float32, device="cuda")

    def step():
        nc.nc_kv_append(kn, vn, kc, vc, lens)
        if Tq == 1:
            nc.nc_attn_decode(q1, kc, vc, lens, o, lse, W, scale, ws)
        else:
            nc.nc_attn_prefill(q, kc, vc, lens, o, lse, W, scale)

    step()
    torch.cuda.synchronize()
    o_e, lse_e, kc_e = o.clone(), lse.clone(), kc.clone()
    g = capture(step)
    for _ in range(3):
        kc.copy_(kc0)
        vc.copy_(vc0)
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(kc, kc_e) and torch.equal(o, o_e) and torch.equal(lse, lse_e)
    assert nc.nc_get_device_error() == 0
