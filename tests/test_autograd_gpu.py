"""The autograd nodes of the Python binding (sliding_window_attention, varlen_attention, rotary_attention).

They only route the library's forward and backward calls through torch.autograd, so their gradients must be
the direct calls' gradients: bitwise where the backward is deterministic (dk, dv always; dq with the
deterministic backward), within the fp32 atomic-order noise of dq otherwise.  One small case also goes to the
oracle, with the tolerances of test_parity_gpu.
"""
import math

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


def leaves(*ts):
    return [t.detach().clone().requires_grad_(True) for t in ts]


def backprop(o, dO):
    # d/d(o) of sum(o * dO) is dO: the node's backward receives exactly the bf16 dO
    (o.float() * dO.float()).sum().backward()


@pytest.mark.parametrize("window", [-1, 300])
@pytest.mark.parametrize("deterministic", [False, True])
def test_attention_node_equals_direct_calls(nc, window, deterministic):
    q, k, v, dO = workloads.make_qkvdo_shape(2, 700, 3, 128, seed=5100 + window, device="cuda")
    o_ref, lse = nc.attn_fwd(q, k, v, window)
    dq_ref, dk_ref, dv_ref = nc.attn_bwd(q, k, v, o_ref, dO, lse, window, deterministic=True)
    ql, kl, vl = leaves(q, k, v)
    o = nc.sliding_window_attention(ql, kl, vl, window, deterministic=deterministic)
    assert torch.equal(o, o_ref)
    backprop(o, dO)
    assert torch.equal(kl.grad, dk_ref) and torch.equal(vl.grad, dv_ref)
    if deterministic:
        assert torch.equal(ql.grad, dq_ref)
    else:
        err = (ql.grad.float() - dq_ref.float()).abs().max().item()
        assert err <= 1e-2 * dq_ref.float().abs().max().item()
    assert nc.nc_get_device_error() == 0


def test_attention_node_takes_views_of_a_fused_projection(nc):
    B, T, H, D = 1, 520, 2, 64
    g = workloads.generator(5200, "cuda")
    qkv = workloads.randn_bf16((B, T, 3, H, D), g, "cuda").requires_grad_(True)
    dO = workloads.randn_bf16((B, T, H, D), g, "cuda")
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]  # strided views
    assert not q.is_contiguous()
    o = nc.sliding_window_attention(q, k, v, 128, deterministic=True)
    backprop(o, dO)
    qc, kc, vc = (t.detach().contiguous() for t in (q, k, v))
    o_ref, lse = nc.attn_fwd(qc, kc, vc, 128)
    grads = nc.attn_bwd(qc, kc, vc, o_ref, dO, lse, 128, deterministic=True)
    assert torch.equal(o, o_ref)
    for i in range(3):
        assert torch.equal(qkv.grad[:, :, i], grads[i])


def test_attention_node_against_the_oracle(nc, oracle_mod):
    q, k, v, dO = workloads.make_qkvdo_shape(1, 333, 2, 128, seed=5300, device="cuda")
    ql, kl, vl = leaves(q, k, v)
    o = nc.sliding_window_attention(ql, kl, vl, 100)
    backprop(o, dO)
    scale = 1.0 / math.sqrt(128)
    o_r, _ = oracle_mod.fwd(*(t.cpu() for t in (q, k, v)), 100, scale)
    g_r = oracle_mod.bwd(*(t.cpu() for t in (q, k, v, dO)), 100, scale)
    rel = lambda a, r: float(np.abs(a.detach().float().cpu().numpy() - r).max() / max(np.abs(r).max(), 1e-4))
    assert rel(o, o_r) <= 2e-2
    for got, ref in zip((ql.grad, kl.grad, vl.grad), g_r):
        assert rel(got, ref) <= 3e-2


def test_varlen_node_equals_direct_calls(nc):
    lens = [130, 1, 257, 64, 300]
    total, H, D = sum(lens), 2, 128
    g = workloads.generator(5400, "cuda")
    q, k, v, dO = (workloads.randn_bf16((total, H, D), g, "cuda") for _ in range(4))
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
    o_ref, lse = nc.attn_fwd_varlen(q, k, v, cu, max(lens), 100)
    dq_ref, dk_ref, dv_ref = nc.attn_bwd_varlen(q, k, v, o_ref, dO, lse, cu, max(lens), 100)
    ql, kl, vl = leaves(q, k, v)
    o = nc.varlen_attention(ql, kl, vl, cu, max(lens), 100)
    assert torch.equal(o, o_ref)
    backprop(o, dO)
    assert torch.equal(kl.grad, dk_ref) and torch.equal(vl.grad, dv_ref)
    err = (ql.grad.float() - dq_ref.float()).abs().max().item()
    assert err <= 1e-2 * dq_ref.float().abs().max().item()


def test_rotary_node_equals_direct_calls(nc):
    B, T, H, D = 2, 384, 2, 128
    q, k, v, dO = workloads.make_qkvdo_shape(B, T, H, D, seed=5500, device="cuda")
    c, s = workloads.rope_tables(T, D, device="cuda")
    o_ref, lse, qr, kr = nc.attn_fwd_rotary(q, k, v, c, s, 256)
    dq_ref, dk_ref, dv_ref = nc.attn_bwd_rotary(qr, kr, v, c, s, o_ref, dO, lse, 256)
    ql, kl, vl = leaves(q, k, v)
    o = nc.rotary_attention(ql, kl, vl, c, s, 256)
    assert torch.equal(o, o_ref)
    backprop(o, dO)
    assert torch.equal(kl.grad, dk_ref) and torch.equal(vl.grad, dv_ref)
    err = (ql.grad.float() - dq_ref.float()).abs().max().item()
    assert err <= 1e-2 * dq_ref.float().abs().max().item()
