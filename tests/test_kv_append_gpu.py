"""KV-cache append (nc_kv_append): new rows land at positions L - Tq .. L - 1 of each sequence, nothing else
changes, and prefill over the appended cache matches the oracle.

The append is a byte copy, so the check is bit-exact against the definition written out on the host (numpy
indexing of the cache as it was before the call).
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


def inputs(N, Tq, Tmax, H, D, seed):
    g = workloads.generator(seed, "cuda")
    kc, vc = (workloads.randn_bf16((N, Tmax, H, D), g, "cuda") for _ in range(2))
    kn, vn = (workloads.randn_bf16((N, Tq, H, D), g, "cuda") for _ in range(2))
    return kc, vc, kn, vn


def expected(cache, new, lens):
    """The cache as the definition gives it: rows L - Tq .. L - 1 of sequence n replaced by its new rows
    (sequences with L outside [Tq, Tmax] left alone); on the host, as int16 bit patterns."""
    out = cache.cpu().view(torch.int16).numpy().copy()
    nw = new.cpu().view(torch.int16).numpy()
    Tq, Tmax = nw.shape[1], out.shape[1]
    for n, L in enumerate(lens):
        if Tq <= L <= Tmax:
            out[n, L - Tq:L] = nw[n]
    return out


@pytest.mark.parametrize("D", [64, 128])
def test_kv_append_writes_only_the_new_rows(nc, D):
    N, Tq, Tmax, H = 5, 37, 300, 3
    kc, vc, kn, vn = inputs(N, Tq, Tmax, H, D, 5600 + D)
    lens = [37, 300, 100, 256, 129]
    ek, ev = expected(kc, kn, lens), expected(vc, vn, lens)
    nc.nc_kv_append(kn, vn, kc, vc, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert nc.nc_get_device_error() == 0
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), ek)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy(), ev)


def test_kv_append_bad_length_reports_and_leaves_the_sequence(nc):
    N, Tq, Tmax, H, D = 3, 40, 128, 2, 128
    kc, vc, kn, vn = inputs(N, Tq, Tmax, H, D, 5700)
    lens = [39, 129, 90]  # too short for the new rows, past Tmax, good
    ek, ev = expected(kc, kn, lens), expected(vc, vn, lens)
    nc.nc_kv_append(kn, vn, kc, vc, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert nc.nc_get_device_error() == nc.NC_ERR_BAD_CACHE_LEN
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), ek)
    assert np.array_equal(vc.cpu().view(torch.int16).numpy(), ev)
    assert nc.nc_get_device_error() == 0


@pytest.mark.parametrize("Tq", [1, 200])
def test_append_then_prefill_matches_the_oracle(nc, oracle_mod, Tq):
    """The engine's step: append the new tokens' keys and values, then attend (Tq = 1 is a decode step).  The
    new-token rows of the cache hold NaN before the append, so a missed row would show."""
    N, Tmax, H, D, W = 4, 700, 2, 128, 256
    kc, vc, kn, vn = inputs(N, Tq, Tmax, H, D, 5800 + Tq)
    lens = [Tq, 700, 300, 453]
    for n, L in enumerate(lens):
        kc[n, L - Tq:L] = float("nan")
        vc[n, L - Tq:L] = float("nan")
    ek, ev = expected(kc, kn, lens), expected(vc, vn, lens)
    q = workloads.randn_bf16((N, Tq, H, D), workloads.generator(5900 + Tq, "cuda"), "cuda")
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    nc.nc_kv_append(kn, vn, kc, vc, lens_d)
    o, lse = nc.attn_prefill(q, kc, vc, lens_d, W)
    assert nc.nc_get_device_error() == 0
    assert np.array_equal(kc.cpu().view(torch.int16).numpy(), ek)
    # the oracle takes the cache as the definition gives it, not the GPU's copy
    kc_e = torch.from_numpy(ek).view(torch.bfloat16)
    vc_e = torch.from_numpy(ev).view(torch.bfloat16)
    o_ref, lse_ref, ok = oracle_mod.prefill(q.cpu(), kc_e, vc_e, torch.tensor(lens, dtype=torch.int32), W,
                                            1.0 / math.sqrt(D))
    assert ok
    o_np = o.float().cpu().numpy()
    assert np.isfinite(o_np).all()
    assert float(np.abs(o_np - o_ref).max() / max(np.abs(o_ref).max(), 1e-4)) <= 2e-2
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= 1e-3
