"""The decode entry point for callers that cannot allocate device memory.

nc_attn_decode_noalloc takes no workspace and allocates nothing; its split-K
partials live in a fixed scratch array inside the library.  It must give the
same results as nc_attn_decode (which uses a caller-provided workspace), call
after call, even though every call reuses the same scratch.  This file is
collected last so that a failure here never hides the other tests.
"""
import ctypes

import pytest
import torch

from causal_sliding_window_fwd_b300 import workloads

O_TOL, LSE_TOL = 2e-2, 1e-3


@pytest.fixture(scope="module")
def nc():
    from causal_sliding_window_fwd_b300 import build_lib
    build_lib.build()
    from causal_sliding_window_fwd_b300 import nc_attn
    return nc_attn


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes fake device addresses; run on a host without a GPU")
def test_scratch_limit_is_enforced_before_any_launch(nc):
    # 1024 sequences of 40 heads over a 256-row cache: 43 MB of partial slots (one per sequence and per
    # CTA of the balanced split, times 40 heads), above the 16 MiB scratch
    need = nc.nc_attn_decode_noalloc_scratch_bytes(1024, 256, 40, 128, -1)
    assert need > nc.NC_DECODE_NOALLOC_SCRATCH_BYTES
    fake = [ctypes.c_void_p(0x400000000 * (i + 1)) for i in range(6)]  # 16 GiB apart: no two ranges overlap
    launches = nc.nc_launch_count()
    rc = nc.lib.nc_attn_decode_noalloc(*fake, 1024, 256, 40, 128, -1, ctypes.c_float(0.088), None)
    assert rc == nc.NC_ERR_WORKSPACE
    assert nc.nc_launch_count() == launches  # refused before any launch
    # many sequences take fixed chunks: 2048 sequences, full window over 8192 rows needs far more
    assert nc.nc_attn_decode_noalloc_scratch_bytes(2048, 8192, 10, 128, -1) > nc.NC_DECODE_NOALLOC_SCRATCH_BYTES
    assert nc.nc_attn_decode_noalloc_scratch_bytes(64, 8192, 10, 128, 1024) <= nc.NC_DECODE_NOALLOC_SCRATCH_BYTES


def _via_workspace(nc, q, kc, vc, lens, window, scale):
    o, lse = nc.attn_decode(q, kc, vc, lens, window, scale)
    return o, lse


def _via_noalloc(nc, q, kc, vc, lens, window, scale):
    N, Tmax, H, D = kc.shape
    o = torch.full((N, H, D), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((N, H), float("nan"), dtype=torch.float32, device=q.device)
    rc = nc.lib.nc_attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(lens.data_ptr()), ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        N, Tmax, H, D, int(window), ctypes.c_float(scale),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == nc.NC_OK, nc.status_string(rc)
    return o, lse


def _close(a, b, tol):
    a, b = a.float(), b.float()
    assert torch.isfinite(a).all()
    return (a - b).abs().max().item() <= tol


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_twice(nc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = workloads.DECODE
    q, kc, vc, lens = workloads.make_decode(wl, "cuda", poison_tail=True)
    small = workloads.DecodeWorkload("small", 5, 600, 3, 64, 1, 600, (-1,), 17)
    q2, kc2, vc2, lens2 = workloads.make_decode(small, "cuda", poison_tail=True)
    # two calls in a row on different problems; the second reuses the scratch the first left behind
    for (qq, kk, vv, ll, w, sc) in ((q, kc, vc, lens, 1024, wl.scale), (q2, kc2, vc2, lens2, -1, small.scale)):
        o_ref, lse_ref = _via_workspace(nc, qq, kk, vv, ll, w, sc)
        o, lse = _via_noalloc(nc, qq, kk, vv, ll, w, sc)
        assert nc.nc_get_device_error() == 0
        assert _close(o, o_ref, O_TOL * o_ref.float().abs().max().item())
        assert _close(lse, lse_ref, LSE_TOL)
