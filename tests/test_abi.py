"""Host-side checks of the C ABI: the library loads, exports every declared
entry point, sizes its workspaces, and rejects bad arguments before touching
the GPU (these calls pass fake pointers, which validation refuses first)."""
import ctypes
import math
import os
import re
import threading

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from causal_sliding_window_fwd_b300 import build_lib
    build_lib.build()
    from causal_sliding_window_fwd_b300 import nc_attn
    return nc_attn


def _declared():
    txt = open(os.path.join(ROOT, "include", "nc_attn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const char\*|nc_status|size_t|unsigned long long)\s+(nc_\w+)\s*\(",
                                 txt, re.M)))


def test_header_declares_the_abi():
    assert {"nc_attn_fwd", "nc_attn_bwd", "nc_attn_bwd_deterministic", "nc_attn_decode", "nc_attn_prefill", "nc_attn_fwd_varlen",
            "nc_attn_bwd_workspace_bytes",
            "nc_attn_decode_workspace_bytes", "nc_get_device_error", "nc_status_string",
            "nc_launch_count"} <= set(_declared())


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name
    assert set(lib.EXPORTED) <= set(_declared())


def test_status_strings(lib):
    assert lib.status_string(0) == "NC_OK"
    assert lib.status_string(6) == "NC_ERR_BAD_CACHE_LEN"


def test_workspace_sizes(lib):
    B, T, H, D = 16, 2048, 10, 128
    need = lib.nc_attn_bwd_workspace_bytes(B, T, H, D)
    assert need >= B * T * H * D * 4 + B * H * T * 4
    assert need < B * T * H * D * 4 + B * H * T * 4 + 1024
    assert lib.nc_attn_bwd_workspace_bytes(0, T, H, D) == 0
    dec = lib.nc_attn_decode_workspace_bytes(64, 8192, 10, 128)
    assert 0 < dec < 64 * 1024 * 1024
    assert lib.nc_attn_decode_workspace_bytes(64, 8192, 10, 96) == 0


# Fake, 16-byte aligned and non-overlapping "device" addresses: validation must
# reject each call below before any CUDA call is made.  These tests run only where
# no GPU is present, so a change in the order of the checks can never hand a fake
# address to a kernel on a real device.
A = [0x10000000 + i * 0x10000000 for i in range(12)]
host_only = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="passes fake device addresses; run on a host without a GPU")
GOOD = dict(B=2, T=64, H=2, D=64, window=16, scale=0.125)


def _fwd(lib, ptrs=None, **kw):
    a = dict(GOOD, **kw)
    p = list(A[:5]) if ptrs is None else ptrs
    return lib.lib.nc_attn_fwd(*[ctypes.c_void_p(x) for x in p], a["B"], a["T"], a["H"], a["D"], a["window"],
                               ctypes.c_float(a["scale"]), None)


@host_only
@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(T=-1), 1), (dict(H=0), 1),
    (dict(D=96), 2), (dict(D=256), 2),
    (dict(window=0), 1), (dict(window=-2), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=math.nan), 1), (dict(scale=math.inf), 1),
])
def test_fwd_rejects_bad_sizes(lib, kw, code):
    assert _fwd(lib, **kw) == code


@host_only
def test_fwd_rejects_null_misaligned_and_aliased(lib):
    for i in range(5):
        p = list(A[:5]); p[i] = 0
        assert _fwd(lib, p) == lib.NC_ERR_INVALID
        p = list(A[:5]); p[i] += 8
        assert _fwd(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:5]); p[3] = p[0]            # o aliases q
    assert _fwd(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:5]); p[4] = p[3] + 64       # lse inside o
    assert _fwd(lib, p) == lib.NC_ERR_INVALID


def _bwd(lib, ptrs=None, ws=None, ws_bytes=None, fn="nc_attn_bwd", **kw):
    a = dict(GOOD, **kw)
    p = list(A[:9]) if ptrs is None else ptrs
    need = lib.nc_attn_bwd_workspace_bytes(a["B"], a["T"], a["H"], a["D"])
    ws = A[9] if ws is None else ws
    ws_bytes = need if ws_bytes is None else ws_bytes
    return getattr(lib.lib, fn)(*[ctypes.c_void_p(x) for x in p], a["B"], a["T"], a["H"], a["D"], a["window"],
                                ctypes.c_float(a["scale"]), ctypes.c_void_p(ws), ws_bytes, None)


@host_only
@pytest.mark.parametrize("fn", ["nc_attn_bwd", "nc_attn_bwd_deterministic"])
def test_bwd_rejects_bad_arguments(lib, fn):
    assert _bwd(lib, D=80, fn=fn) == lib.NC_ERR_UNSUPPORTED
    assert _bwd(lib, window=0, fn=fn) == lib.NC_ERR_INVALID
    need = lib.nc_attn_bwd_workspace_bytes(2, 64, 2, 64)
    assert _bwd(lib, ws_bytes=need - 1, fn=fn) == lib.NC_ERR_WORKSPACE
    assert _bwd(lib, ws=0, fn=fn) == lib.NC_ERR_WORKSPACE
    assert _bwd(lib, ws=A[9] + 4, fn=fn) == lib.NC_ERR_INVALID
    for i in range(9):
        p = list(A[:9]); p[i] = 0
        assert _bwd(lib, p, fn=fn) == lib.NC_ERR_INVALID
    p = list(A[:9]); p[6] = p[0]            # dq aliases q
    assert _bwd(lib, p, fn=fn) == lib.NC_ERR_INVALID
    p = list(A[:9]); p[7] = p[6]            # dk aliases dq
    assert _bwd(lib, p, fn=fn) == lib.NC_ERR_INVALID
    assert _bwd(lib, ws=A[1], fn=fn) == lib.NC_ERR_INVALID  # workspace over k


def _dec(lib, ptrs=None, ws_bytes=None, **kw):
    a = dict(N=4, Tmax=256, H=2, D=128, window=64, scale=0.1)
    a.update(kw)
    p = list(A[:6]) if ptrs is None else ptrs
    need = lib.nc_attn_decode_workspace_bytes(a["N"], a["Tmax"], a["H"], a["D"])
    ws_bytes = need if ws_bytes is None else ws_bytes
    return lib.lib.nc_attn_decode(*[ctypes.c_void_p(x) if x is not None else None for x in p],
                                  a["N"], a["Tmax"], a["H"], a["D"], a["window"], ctypes.c_float(a["scale"]),
                                  ctypes.c_void_p(A[10]), ws_bytes, None)


@host_only
def test_decode_rejects_bad_arguments(lib):
    assert _dec(lib, N=0) == lib.NC_ERR_INVALID
    assert _dec(lib, D=32) == lib.NC_ERR_UNSUPPORTED
    assert _dec(lib, window=0) == lib.NC_ERR_INVALID
    assert _dec(lib, scale=-0.5) == lib.NC_ERR_INVALID
    need = lib.nc_attn_decode_workspace_bytes(4, 256, 2, 128)
    assert _dec(lib, ws_bytes=need - 4) == lib.NC_ERR_WORKSPACE
    for i in range(5):
        p = list(A[:6]); p[i] = 0
        assert _dec(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[4] = p[1]            # o aliases the key cache
    assert _dec(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[3] = p[3] + 2        # lens misaligned
    assert _dec(lib, p) == lib.NC_ERR_INVALID


def _pre(lib, ptrs=None, **kw):
    a = dict(N=4, Tq=16, Tmax=256, H=2, D=128, window=64, scale=0.1)
    a.update(kw)
    p = list(A[:6]) if ptrs is None else ptrs
    return lib.lib.nc_attn_prefill(*[ctypes.c_void_p(x) if x is not None else None for x in p],
                                   a["N"], a["Tq"], a["Tmax"], a["H"], a["D"], a["window"],
                                   ctypes.c_float(a["scale"]), None)


@host_only
def test_prefill_rejects_bad_arguments(lib):
    assert _pre(lib, N=0) == lib.NC_ERR_INVALID
    assert _pre(lib, Tq=0) == lib.NC_ERR_INVALID
    assert _pre(lib, Tq=257) == lib.NC_ERR_INVALID  # more new tokens than cache rows
    assert _pre(lib, D=96) == lib.NC_ERR_UNSUPPORTED
    assert _pre(lib, window=0) == lib.NC_ERR_INVALID
    assert _pre(lib, scale=float("nan")) == lib.NC_ERR_INVALID
    for i in range(6):
        p = list(A[:6]); p[i] = 0
        assert _pre(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[4] = p[2]            # o aliases the value cache
    assert _pre(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[0] = p[0] + 8        # q not 16-byte aligned
    assert _pre(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[3] = p[3] + 2        # lens misaligned
    assert _pre(lib, p) == lib.NC_ERR_INVALID


def _fvl(lib, ptrs=None, **kw):
    a = dict(n_docs=3, total=512, max_seqlen=300, H=2, D=128, window=64, scale=0.1)
    a.update(kw)
    p = list(A[:6]) if ptrs is None else ptrs
    return lib.lib.nc_attn_fwd_varlen(*[ctypes.c_void_p(x) if x is not None else None for x in p],
                                      a["n_docs"], a["total"], a["max_seqlen"], a["H"], a["D"], a["window"],
                                      ctypes.c_float(a["scale"]), None)


@host_only
def test_fwd_varlen_rejects_bad_arguments(lib):
    assert lib.status_string(7) == "NC_ERR_BAD_SEQLENS"
    assert _fvl(lib, n_docs=0) == lib.NC_ERR_INVALID
    assert _fvl(lib, total=0) == lib.NC_ERR_INVALID
    assert _fvl(lib, max_seqlen=0) == lib.NC_ERR_INVALID
    assert _fvl(lib, max_seqlen=513) == lib.NC_ERR_INVALID  # longer than the packed rows
    assert _fvl(lib, D=32) == lib.NC_ERR_UNSUPPORTED
    assert _fvl(lib, window=-2) == lib.NC_ERR_INVALID
    for i in range(6):
        p = list(A[:6]); p[i] = 0
        assert _fvl(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[4] = p[0]            # o aliases q
    assert _fvl(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[3] = p[3] + 2        # cu_seqlens misaligned
    assert _fvl(lib, p) == lib.NC_ERR_INVALID


@host_only
@pytest.mark.parametrize("entry", ["nc_attn_bwd_varlen", "nc_attn_bwd_varlen_deterministic"])
def test_bwd_varlen_rejects_bad_arguments(lib, entry):
    def call(ptrs=None, ws_bytes=None, **kw):
        a = dict(n_docs=3, total=512, max_seqlen=300, H=2, D=128, window=64, scale=0.1)
        a.update(kw)
        p = list(A[:10]) if ptrs is None else ptrs
        need = lib.nc_attn_bwd_workspace_bytes(1, a["total"], a["H"], a["D"])
        return getattr(lib.lib, entry)(*[ctypes.c_void_p(x) if x is not None else None for x in p],
                                       a["n_docs"], a["total"], a["max_seqlen"], a["H"], a["D"], a["window"],
                                       ctypes.c_float(a["scale"]), ctypes.c_void_p(A[11]),
                                       need if ws_bytes is None else ws_bytes, None)
    assert call(n_docs=0) == lib.NC_ERR_INVALID
    assert call(max_seqlen=600) == lib.NC_ERR_INVALID
    assert call(D=80) == lib.NC_ERR_UNSUPPORTED
    assert call(ws_bytes=64) == lib.NC_ERR_WORKSPACE
    for i in range(10):
        p = list(A[:10]); p[i] = 0
        assert call(p) == lib.NC_ERR_INVALID
    p = list(A[:10]); p[7] = p[1]            # dq aliases k
    assert call(p) == lib.NC_ERR_INVALID


def _noalloc(lib, ptrs, N=4, Tmax=256, H=2, D=128, window=64):
    return lib.lib.nc_attn_decode_noalloc(*[ctypes.c_void_p(x) if x is not None else None for x in ptrs],
                                          N, Tmax, H, D, window, ctypes.c_float(0.1), None)


@host_only
def test_decode_noalloc_rejects_the_overlaps_decode_rejects(lib):
    """Byte ranges, not just pointer equality: no output may overlap an input or the other output."""
    N, Tmax, H, D = 4, 256, 2, 128
    p = list(A[:6]); p[4] = p[1] + 4096          # o inside the key cache
    assert _noalloc(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[5] = p[0] + 16            # lse overlapping q
    assert _noalloc(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[5] = p[3]                 # lse over cache_lens
    assert _noalloc(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[5] = p[4] + 32            # lse inside o
    assert _noalloc(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:6]); p[4] = p[2] + 2 * N * Tmax * H * D - 16   # o straddling the end of the value cache
    assert _noalloc(lib, p) == lib.NC_ERR_INVALID
    # the same placements are refused by the workspace decode
    p = list(A[:6]); p[4] = p[1] + 4096
    assert _dec(lib, p) == lib.NC_ERR_INVALID


def test_noalloc_scratch_bytes_follow_the_call_limits(lib):
    assert lib.nc_attn_decode_noalloc_scratch_bytes(64, 8192, 10, 128, 1024) > 0
    assert lib.nc_attn_decode_noalloc_scratch_bytes(0, 8192, 10, 128, 1024) == 0
    assert lib.nc_attn_decode_noalloc_scratch_bytes(64, 8192, 10, 96, 1024) == 0
    assert lib.nc_attn_decode_noalloc_scratch_bytes(64, 8192, 10, 128, 0) == 0
    # sizes the call refuses as unsupported (N*H >= 2^31, Tmax*H*D >= 2^40) get 0, not a size
    assert lib.nc_attn_decode_noalloc_scratch_bytes(1 << 22, 256, 1 << 9, 64, 64) == 0
    assert lib.nc_attn_decode_noalloc_scratch_bytes(1, 1 << 30, 1 << 4, 128, 64) == 0


@host_only
def test_abi_calls_from_many_threads(lib):
    """Entry points called from many host threads at once give each caller its own answer (the
    library keeps no per-device host state that first calls could race on)."""
    errors = []

    def worker(k):
        try:
            for i in range(200):
                assert _fwd(lib, D=96) == lib.NC_ERR_UNSUPPORTED
                assert _fwd(lib, window=0) == lib.NC_ERR_INVALID
                p = list(A[:5]); p[3] = p[0]
                assert _fwd(lib, p) == lib.NC_ERR_INVALID
                assert _bwd(lib, ws_bytes=16) == lib.NC_ERR_WORKSPACE
                assert lib.nc_attn_bwd_workspace_bytes(2, 64 + i, 2, 64) > 0
                assert lib.status_string((i + k) % 8).startswith("NC_")
        except AssertionError as e:  # pragma: no cover - reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(16)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:3]


def _fwd_rot(lib, ptrs=None, **kw):
    a = dict(GOOD, **kw)
    p = list(A[:9]) if ptrs is None else ptrs
    return lib.lib.nc_attn_fwd_rotary(*[ctypes.c_void_p(x) for x in p], a["B"], a["T"], a["H"], a["D"],
                                      a["window"], ctypes.c_float(a["scale"]), None)


def _rot(lib, ptrs=None, inverse=0, **kw):
    a = dict(GOOD, **kw)
    p = list(A[:4]) if ptrs is None else ptrs
    return lib.lib.nc_rotary(*[ctypes.c_void_p(x) for x in p], a["B"], a["T"], a["H"], a["D"], inverse, None)


@host_only
def test_rotary_entries_reject_bad_arguments(lib):
    # forward: q k v cos sin qr kr o lse
    assert _fwd_rot(lib, D=96) == lib.NC_ERR_UNSUPPORTED
    assert _fwd_rot(lib, window=0) == lib.NC_ERR_INVALID
    for i in range(9):
        p = list(A[:9]); p[i] = 0
        assert _fwd_rot(lib, p) == lib.NC_ERR_INVALID
        p = list(A[:9]); p[i] += 8
        assert _fwd_rot(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:9]); p[7] = p[3] + 256       # o over the cosine table
    assert _fwd_rot(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:9]); p[8] = p[4]             # lse over the sine table
    assert _fwd_rot(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:9]); p[5] = p[0]             # qr over q (the turn is not in place here)
    assert _fwd_rot(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:9]); p[6] = p[5] + 64        # kr overlapping qr
    assert _fwd_rot(lib, p) == lib.NC_ERR_INVALID
    # backward: qr kr v cos sin o dO lse dq dk dv, workspace
    need = lib.nc_attn_bwd_workspace_bytes(2, 64, 2, 64)

    def bwd_rot(p, ws=A[11], ws_bytes=need, **kw):
        a = dict(GOOD, **kw)
        return lib.lib.nc_attn_bwd_rotary(*[ctypes.c_void_p(x) for x in p], a["B"], a["T"], a["H"], a["D"],
                                          a["window"], ctypes.c_float(a["scale"]), ctypes.c_void_p(ws), ws_bytes,
                                          None)
    assert bwd_rot(list(A[:11]), D=96) == lib.NC_ERR_UNSUPPORTED
    assert bwd_rot(list(A[:11]), ws_bytes=need - 1) == lib.NC_ERR_WORKSPACE
    for i in range(11):
        p = list(A[:11]); p[i] = 0
        assert bwd_rot(p) == lib.NC_ERR_INVALID
    p = list(A[:11]); p[8] = p[3]            # dq over the cosine table
    assert bwd_rot(p) == lib.NC_ERR_INVALID
    assert bwd_rot(list(A[:11]), ws=A[4]) == lib.NC_ERR_INVALID   # workspace over the sine table
    # the standalone turn: x cos sin y
    assert _rot(lib, D=96) == lib.NC_ERR_UNSUPPORTED
    assert _rot(lib, B=0) == lib.NC_ERR_INVALID
    assert _rot(lib, B=1 << 16, T=1 << 15, H=1) == lib.NC_ERR_UNSUPPORTED   # B * T * H = 2^31 rows
    for i in range(4):
        p = list(A[:4]); p[i] = 0
        assert _rot(lib, p) == lib.NC_ERR_INVALID
        p = list(A[:4]); p[i] += 8
        assert _rot(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:4]); p[3] = p[0] + 128       # y partly over x (in place means y == x exactly)
    assert _rot(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:4]); p[3] = p[1]             # y over the cosine table
    assert _rot(lib, p) == lib.NC_ERR_INVALID


def _append(lib, ptrs=None, N=2, Tq=4, Tmax=64, H=2, D=64):
    p = list(A[:5]) if ptrs is None else ptrs
    return lib.lib.nc_kv_append(*[ctypes.c_void_p(x) for x in p], N, Tq, Tmax, H, D, None)


@host_only
def test_kv_append_rejects_bad_arguments(lib):
    # k_new v_new kcache vcache cache_lens
    assert _append(lib, D=96) == lib.NC_ERR_UNSUPPORTED
    assert _append(lib, N=0) == lib.NC_ERR_INVALID
    assert _append(lib, Tq=0) == lib.NC_ERR_INVALID
    assert _append(lib, Tq=65) == lib.NC_ERR_INVALID
    for i in range(5):
        p = list(A[:5]); p[i] = 0
        assert _append(lib, p) == lib.NC_ERR_INVALID
    for i in range(4):
        p = list(A[:5]); p[i] += 8           # rows must be 16-byte aligned
        assert _append(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:5]); p[4] += 2               # lengths must be 4-byte aligned
    assert _append(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:5]); p[3] = p[2] + 256       # vcache overlapping kcache
    assert _append(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:5]); p[2] = p[0]             # kcache over k_new
    assert _append(lib, p) == lib.NC_ERR_INVALID
    p = list(A[:5]); p[3] = p[4] - 64        # vcache over the lengths
    assert _append(lib, p) == lib.NC_ERR_INVALID
