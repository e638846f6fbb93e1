"""The forward's stale-maximum softmax on inputs that make it work: against the fp64 oracle.

The forward keeps one reference maximum per row and raises it (rescaling O and l in place) only when a key
block's maximum exceeds it by more than 2^8 in exp2 units; a row that has seen no visible key yet (its window
starts past the item's first key block) takes the next block's maximum directly.  Random inputs of unit scale
almost never raise the maximum after the first block, so these cases build the scores on purpose:

- growing scores: every query has a large first coordinate and the keys' first coordinate grows with the
  position, so each key block's maximum is above the previous one by more than 2^8 and every block rescales;
- shrinking scores: the same with the keys reversed, so the first block holds the maximum and later blocks
  underflow towards zero weight;
- large random scores: inputs scaled up so that rescales happen at scattered blocks and rows.

Windows that are multiples of the 128-key block leave the last row of every query tile with nothing visible in
its first block.  Tolerances are those of the parity tests.  On the ramps only dV of the gradients is compared:
there one key dominates each row, dP - Delta cancels for it, and Delta = rowsum(dO * O) comes from the forward's
bf16 O while the oracle's comes from its exact O.  That rounding, times keys and queries of norm 34, moves dQ
and dK by up to about 12% of their largest value, a property of the method's precision (the backward has no running
maximum to test), not of the forward.
"""
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
    got = got.detach().float().cpu().numpy()
    assert np.isfinite(got).all(), "non-finite values in GPU output"
    ref = np.asarray(ref)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-4))


def ramp_inputs(B, T, H, D, amp, reverse, seed):
    """q = amp * e_0 + small noise; k_t = amp * (t / T) * e_0 + small noise (reversed: (T - 1 - t) / T)."""
    g = workloads.generator(seed, "cuda")
    q, k, v, dO = (0.25 * workloads.randn_bf16((B, T, H, D), g, "cuda").float() for _ in range(4))
    pos = torch.arange(T, device="cuda", dtype=torch.float32)
    if reverse:
        pos = T - 1 - pos
    q[..., 0] = amp
    k[..., 0] = amp * (pos / T)[None, :, None]
    return tuple(x.to(torch.bfloat16).contiguous() for x in (q, k, v, dO))


def check(nc, oracle_mod, q, k, v, dO, window, grads=("dq", "dk", "dv")):
    B, T, H, D = q.shape
    scale = nc.default_scale(D)
    o, lse = nc.attn_fwd(q, k, v, window, scale)
    assert nc.nc_get_device_error() == 0
    o_ref, lse_ref = oracle_mod.fwd(q, k, v, window, scale)
    assert rel_err(o, o_ref) <= O_TOL
    assert float(np.abs(lse.cpu().numpy() - np.asarray(lse_ref)).max()) <= LSE_TOL
    if grads:
        dq, dk, dv = nc.attn_bwd(q, k, v, o, dO, lse, window, scale)
        assert nc.nc_get_device_error() == 0
        dq_r, dk_r, dv_r = oracle_mod.bwd(q, k, v, dO, window, scale)
        for name, got, ref in (("dq", dq, dq_r), ("dk", dk, dk_r), ("dv", dv, dv_r)):
            if name in grads:
                assert rel_err(got, ref) <= G_TOL, name
    return lse


@pytest.mark.parametrize("window", [1024, 2048, 384])
def test_growing_scores_rescale_every_block(nc, oracle_mod, window):
    # per key block the score rises by 34 * 34 * 128 / 2048 / sqrt(128) = 6.4 (natural units), 9.2 in exp2
    # units: above the 2^8 threshold, so every block of every row raises its maximum
    B, T, H, D = 1, 2048, 2, 128
    q, k, v, dO = ramp_inputs(B, T, H, D, 34.0, reverse=False, seed=7100 + window)
    lse = check(nc, oracle_mod, q, k, v, dO, window, grads=("dv",))
    # the log-sum-exp grows with the row, far beyond what a single unscaled block could hold
    assert float(lse[..., -1].min()) > 80.0


@pytest.mark.parametrize("window", [1024, 2048])
def test_shrinking_scores(nc, oracle_mod, window):
    B, T, H, D = 1, 2048, 2, 128
    q, k, v, dO = ramp_inputs(B, T, H, D, 34.0, reverse=True, seed=7200 + window)
    check(nc, oracle_mod, q, k, v, dO, window, grads=("dv",))


@pytest.mark.parametrize("shape", [(2, 1024, 3, 128, 256), (1, 1536, 2, 128, 640), (2, 1000, 2, 64, 512)])
def test_large_random_scores(nc, oracle_mod, shape):
    B, T, H, D, W = shape
    g = workloads.generator(7300 + T + W, "cuda")
    q = (3.0 * workloads.randn_bf16((B, T, H, D), g, "cuda").float()).to(torch.bfloat16)
    k = (3.0 * workloads.randn_bf16((B, T, H, D), g, "cuda").float()).to(torch.bfloat16)
    v, dO = (workloads.randn_bf16((B, T, H, D), g, "cuda") for _ in range(2))
    check(nc, oracle_mod, q, k, v, dO, W)
