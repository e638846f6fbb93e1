"""Python binding of the nc_attn C ABI (``include/nc_attn.h``).

Argument marshalling only: torch tensors are checked for dtype, device,
shape and contiguity, and their device pointers and the current CUDA stream
are handed to ``libnc_attn.so``.  Every step of the computation runs in the
library's CUDA kernels; there is no other implementation behind these calls,
and importing this module fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnc_attn.so")

NC_OK = 0
NC_ERR_INVALID = 1
NC_ERR_UNSUPPORTED = 2
NC_ERR_WORKSPACE = 3
NC_ERR_CUDA = 4
NC_ERR_DEVICE_TIMEOUT = 5
NC_ERR_BAD_CACHE_LEN = 6
NC_ERR_BAD_SEQLENS = 7
NC_WINDOW_FULL = -1

# Entry points declared in include/nc_attn.h.
EXPORTED = ("nc_status_string", "nc_attn_fwd", "nc_attn_bwd_workspace_bytes", "nc_attn_bwd",
            "nc_attn_bwd_deterministic",
            "nc_attn_decode_workspace_bytes", "nc_attn_decode", "nc_attn_prefill", "nc_attn_fwd_varlen",
            "nc_attn_bwd_varlen", "nc_attn_fwd_rotary", "nc_attn_bwd_rotary", "nc_rotary",
            "nc_get_device_error",
            "nc_launch_count",
            "nc_attn_decode_noalloc_scratch_bytes", "nc_attn_decode_noalloc", "nc_debug_watchdog_selftest",
            "nc_kv_append", "nc_attn_bwd_varlen_deterministic")

# Size of the library's fixed decode scratch array (NC_DECODE_NOALLOC_SCRATCH_BYTES).
NC_DECODE_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class NcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {status_string(code)} ({code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libnc_attn.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                          "or python causal_sliding_window_fwd_b300/build_lib.py")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.nc_status_string.argtypes = [i]
    lib.nc_status_string.restype = ctypes.c_char_p
    lib.nc_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.nc_attn_fwd.restype = i
    lib.nc_attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.nc_attn_bwd_workspace_bytes.restype = sz
    lib.nc_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.nc_attn_bwd.restype = i
    lib.nc_attn_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.nc_attn_bwd_deterministic.restype = i
    lib.nc_attn_decode_workspace_bytes.argtypes = [i, i, i, i]
    lib.nc_attn_decode_workspace_bytes.restype = sz
    lib.nc_attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.nc_attn_decode.restype = i
    lib.nc_attn_prefill.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.nc_attn_prefill.restype = i
    lib.nc_kv_append.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.nc_kv_append.restype = i
    lib.nc_attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    lib.nc_attn_fwd_varlen.restype = i
    lib.nc_attn_bwd_varlen.argtypes = [vp] * 10 + [i, i, i, i, i, i, f, vp, sz, vp]
    lib.nc_attn_bwd_varlen.restype = i
    lib.nc_attn_bwd_varlen_deterministic.argtypes = [vp] * 10 + [i, i, i, i, i, i, f, vp, sz, vp]
    lib.nc_attn_bwd_varlen_deterministic.restype = i
    lib.nc_attn_fwd_rotary.argtypes = [vp] * 9 + [i, i, i, i, i, f, vp]
    lib.nc_attn_fwd_rotary.restype = i
    lib.nc_attn_bwd_rotary.argtypes = [vp] * 11 + [i, i, i, i, i, f, vp, sz, vp]
    lib.nc_attn_bwd_rotary.restype = i
    lib.nc_rotary.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.nc_rotary.restype = i
    lib.nc_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int), vp]
    lib.nc_get_device_error.restype = i
    lib.nc_launch_count.argtypes = []
    lib.nc_launch_count.restype = ctypes.c_ulonglong
    lib.nc_attn_decode_noalloc_scratch_bytes.argtypes = [i, i, i, i, i]
    lib.nc_attn_decode_noalloc_scratch_bytes.restype = sz
    lib.nc_attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.nc_attn_decode_noalloc.restype = i
    lib.nc_debug_watchdog_selftest.argtypes = [ctypes.c_ulonglong, vp]
    lib.nc_debug_watchdog_selftest.restype = i
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.nc_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != NC_OK:
        raise NcError(code, where)


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


# ---------------------------------------------------------------- raw C-ABI mirrors


def nc_attn_bwd_workspace_bytes(B: int, T: int, H: int, D: int) -> int:
    return int(lib.nc_attn_bwd_workspace_bytes(B, T, H, D))


def nc_attn_decode_workspace_bytes(N: int, Tmax: int, H: int, D: int) -> int:
    return int(lib.nc_attn_decode_workspace_bytes(N, Tmax, H, D))


def nc_attn_fwd(q, k, v, o, lse, window: int, scale: float, stream=None) -> None:
    """Forward into caller-owned o [B,T,H,D] bf16 and lse [B,H,T] fp32."""
    B, T, H, D = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(t, n, torch.bfloat16, (B, T, H, D))
    _need(lse, "lse", torch.float32, (B, H, T))
    _check(lib.nc_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, H, D, int(window), float(scale),
                           _stream(q.device, stream)), "nc_attn_fwd")


def nc_attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, window: int, scale: float, workspace, stream=None) -> None:
    """Backward into caller-owned dq, dk, dv; ``workspace`` is a uint8 device tensor."""
    _bwd_call("nc_attn_bwd", q, k, v, o, dO, lse, dq, dk, dv, window, scale, workspace, stream)


def nc_attn_bwd_deterministic(q, k, v, o, dO, lse, dq, dk, dv, window: int, scale: float, workspace,
                              stream=None) -> None:
    """Bitwise-reproducible backward into caller-owned dq, dk, dv (same arguments as nc_attn_bwd)."""
    _bwd_call("nc_attn_bwd_deterministic", q, k, v, o, dO, lse, dq, dk, dv, window, scale, workspace, stream)


def _bwd_call(name, q, k, v, o, dO, lse, dq, dk, dv, window, scale, workspace, stream):
    B, T, H, D = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, n, torch.bfloat16, (B, T, H, D))
    _need(lse, "lse", torch.float32, (B, H, T))
    _need(workspace, "workspace", torch.uint8)
    _check(getattr(lib, name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                              B, T, H, D, int(window), float(scale), _ptr(workspace), workspace.numel(),
                              _stream(q.device, stream)), name)


def _rope_tables(rope_cos, rope_sin, T, D):
    _need(rope_cos, "rope_cos", torch.float32, (T, D // 2))
    _need(rope_sin, "rope_sin", torch.float32, (T, D // 2))


def nc_attn_fwd_rotary(q, k, v, rope_cos, rope_sin, qr, kr, o, lse, window: int, scale: float, stream=None) -> None:
    """Attention over the rotary-embedded q and k (tables fp32 [T, D/2]); the turned q, k go to qr, kr."""
    B, T, H, D = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("qr", qr), ("kr", kr), ("o", o)):
        _need(t, n, torch.bfloat16, (B, T, H, D))
    _need(lse, "lse", torch.float32, (B, H, T))
    _rope_tables(rope_cos, rope_sin, T, D)
    _check(lib.nc_attn_fwd_rotary(_ptr(q), _ptr(k), _ptr(v), _ptr(rope_cos), _ptr(rope_sin), _ptr(qr), _ptr(kr),
                                  _ptr(o), _ptr(lse), B, T, H, D, int(window), float(scale),
                                  _stream(q.device, stream)), "nc_attn_fwd_rotary")


def nc_attn_bwd_rotary(qr, kr, v, rope_cos, rope_sin, o, dO, lse, dq, dk, dv, window: int, scale: float, workspace,
                       stream=None) -> None:
    """Backward of nc_attn_fwd_rotary from the turned rows qr, kr: dq, dk with respect to the unturned q, k."""
    B, T, H, D = qr.shape
    for n, t in (("qr", qr), ("kr", kr), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        _need(t, n, torch.bfloat16, (B, T, H, D))
    _need(lse, "lse", torch.float32, (B, H, T))
    _rope_tables(rope_cos, rope_sin, T, D)
    _need(workspace, "workspace", torch.uint8)
    _check(lib.nc_attn_bwd_rotary(_ptr(qr), _ptr(kr), _ptr(v), _ptr(rope_cos), _ptr(rope_sin), _ptr(o), _ptr(dO),
                                  _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, T, H, D, int(window), float(scale),
                                  _ptr(workspace), workspace.numel(), _stream(qr.device, stream)),
           "nc_attn_bwd_rotary")


def nc_rotary(x, rope_cos, rope_sin, y, inverse: bool = False, stream=None) -> None:
    """The rotary turn of x [B, T, H, D] bf16 into y (x itself for in place); the transpose with inverse."""
    B, T, H, D = x.shape
    _need(x, "x", torch.bfloat16, (B, T, H, D))
    _need(y, "y", torch.bfloat16, (B, T, H, D))
    _rope_tables(rope_cos, rope_sin, T, D)
    _check(lib.nc_rotary(_ptr(x), _ptr(rope_cos), _ptr(rope_sin), _ptr(y), B, T, H, D, int(bool(inverse)),
                         _stream(x.device, stream)), "nc_rotary")


def rotary(x, rope_cos, rope_sin, inverse: bool = False, stream=None):
    """Returns the rotary turn of x (a new tensor)."""
    y = torch.empty_like(x)
    nc_rotary(x, rope_cos, rope_sin, y, inverse, stream)
    return y


def attn_fwd_rotary(q, k, v, rope_cos, rope_sin, window: int, scale: float | None = None, stream=None):
    """Returns (o, lse, qr, kr): attention over the rotary-embedded q and k, and the turned q, k (which
    attn_bwd_rotary takes)."""
    B, T, H, D = q.shape
    scale = default_scale(D) if scale is None else scale
    qr, kr, o = torch.empty_like(q), torch.empty_like(k), torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    nc_attn_fwd_rotary(q, k, v, rope_cos, rope_sin, qr, kr, o, lse, window, scale, stream)
    return o, lse, qr, kr


def attn_bwd_rotary(qr, kr, v, rope_cos, rope_sin, o, dO, lse, window: int, scale: float | None = None,
                    workspace=None, stream=None):
    """Returns (dq, dk, dv) of the rotary forward, dq and dk with respect to the unturned q and k."""
    B, T, H, D = qr.shape
    scale = default_scale(D) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nc_attn_bwd_workspace_bytes(B, T, H, D), dtype=torch.uint8, device=qr.device)
    dq, dk, dv = torch.empty_like(qr), torch.empty_like(qr), torch.empty_like(qr)
    nc_attn_bwd_rotary(qr, kr, v, rope_cos, rope_sin, o, dO, lse, dq, dk, dv, window, scale, workspace, stream)
    return dq, dk, dv


def nc_attn_decode(q, kcache, vcache, cache_lens, o, lse, window: int, scale: float, workspace, stream=None) -> None:
    """Decode into caller-owned o [N,H,D] bf16 and lse [N,H] fp32 (or None)."""
    N, Tmax, H, D = kcache.shape
    _need(q, "q", torch.bfloat16, (N, H, D))
    _need(kcache, "kcache", torch.bfloat16)
    _need(vcache, "vcache", torch.bfloat16, (N, Tmax, H, D))
    _need(cache_lens, "cache_lens", torch.int32, (N,))
    _need(o, "o", torch.bfloat16, (N, H, D))
    if lse is not None:
        _need(lse, "lse", torch.float32, (N, H))
    _need(workspace, "workspace", torch.uint8)
    _check(lib.nc_attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_lens), _ptr(o), _ptr(lse),
                              N, Tmax, H, D, int(window), float(scale), _ptr(workspace), workspace.numel(),
                              _stream(q.device, stream)), "nc_attn_decode")


def nc_attn_fwd_varlen(q, k, v, cu_seqlens, o, lse, max_seqlen: int, window: int, scale: float,
                       stream=None) -> None:
    """Document-masked forward over packed rows q, k, v, o [total,H,D] bf16; lse [H,total] fp32;
    cu_seqlens int32 [n_docs+1] on the device."""
    total, H, D = q.shape
    n_docs = cu_seqlens.shape[0] - 1
    for name, x in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need(x, name, torch.bfloat16, (total, H, D))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (n_docs + 1,))
    _need(lse, "lse", torch.float32, (H, total))
    _check(lib.nc_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(o), _ptr(lse), n_docs, total,
                                  int(max_seqlen), H, D, int(window), float(scale), _stream(q.device, stream)),
           "nc_attn_fwd_varlen")


def nc_attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, dq, dk, dv, max_seqlen: int, window: int, scale: float,
                       workspace, stream=None, deterministic: bool = False) -> None:
    """Backward of the document-masked forward into caller-owned dq, dk, dv [total,H,D]; ``deterministic``
    calls nc_attn_bwd_varlen_deterministic (bitwise-reproducible)."""
    total, H, D = q.shape
    n_docs = cu_seqlens.shape[0] - 1
    for name, x in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO), ("dq", dq), ("dk", dk), ("dv", dv)):
        _need(x, name, torch.bfloat16, (total, H, D))
    _need(lse, "lse", torch.float32, (H, total))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (n_docs + 1,))
    _need(workspace, "workspace", torch.uint8)
    fn, name = ((lib.nc_attn_bwd_varlen_deterministic, "nc_attn_bwd_varlen_deterministic") if deterministic
                else (lib.nc_attn_bwd_varlen, "nc_attn_bwd_varlen"))
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(cu_seqlens), _ptr(dq), _ptr(dk), _ptr(dv),
              n_docs, total, int(max_seqlen), H, D, int(window), float(scale), _ptr(workspace), workspace.numel(),
              _stream(q.device, stream)), name)


def nc_attn_bwd_varlen_deterministic(q, k, v, o, dO, lse, cu_seqlens, dq, dk, dv, max_seqlen: int, window: int,
                                     scale: float, workspace, stream=None) -> None:
    """The bitwise-reproducible backward of the document-masked forward."""
    nc_attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, dq, dk, dv, max_seqlen, window, scale, workspace, stream,
                       deterministic=True)


def attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, max_seqlen: int, window: int, scale: float | None = None,
                    workspace=None, stream=None, deterministic: bool = False):
    """Returns (dq, dk, dv), each [total,H,D] bf16; ``deterministic`` selects the bitwise-reproducible backward."""
    total, H, D = q.shape
    scale = default_scale(D) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nc_attn_bwd_workspace_bytes(1, total, H, D), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    nc_attn_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens, dq, dk, dv, max_seqlen, window, scale, workspace, stream,
                       deterministic)
    return dq, dk, dv


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, window: int, scale: float | None = None, stream=None):
    """Returns (o [total,H,D], lse [H,total])."""
    total, H, D = q.shape
    scale = default_scale(D) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device)
    nc_attn_fwd_varlen(q, k, v, cu_seqlens, o, lse, max_seqlen, window, scale, stream)
    return o, lse


def nc_attn_prefill(q, kcache, vcache, cache_lens, o, lse, window: int, scale: float, stream=None) -> None:
    """Prefill into caller-owned o [N,Tq,H,D] bf16 and lse [N,H,Tq] fp32; cache_lens count the new tokens."""
    N, Tmax, H, D = kcache.shape
    Tq = q.shape[1]
    _need(q, "q", torch.bfloat16, (N, Tq, H, D))
    _need(kcache, "kcache", torch.bfloat16)
    _need(vcache, "vcache", torch.bfloat16, (N, Tmax, H, D))
    _need(cache_lens, "cache_lens", torch.int32, (N,))
    _need(o, "o", torch.bfloat16, (N, Tq, H, D))
    _need(lse, "lse", torch.float32, (N, H, Tq))
    _check(lib.nc_attn_prefill(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_lens), _ptr(o), _ptr(lse),
                               N, Tq, Tmax, H, D, int(window), float(scale), _stream(q.device, stream)),
           "nc_attn_prefill")


def nc_kv_append(k_new, v_new, kcache, vcache, cache_lens, stream=None) -> None:
    """Writes the new rows k_new, v_new [N,Tq,H,D] bf16 into the caches [N,Tmax,H,D] at positions
    cache_lens[n] - Tq .. cache_lens[n] - 1 (the lengths count the new tokens, as prefill and decode take them)."""
    N, Tmax, H, D = kcache.shape
    Tq = k_new.shape[1]
    _need(k_new, "k_new", torch.bfloat16, (N, Tq, H, D))
    _need(v_new, "v_new", torch.bfloat16, (N, Tq, H, D))
    _need(kcache, "kcache", torch.bfloat16)
    _need(vcache, "vcache", torch.bfloat16, (N, Tmax, H, D))
    _need(cache_lens, "cache_lens", torch.int32, (N,))
    _check(lib.nc_kv_append(_ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache), _ptr(cache_lens),
                            N, Tq, Tmax, H, D, _stream(kcache.device, stream)), "nc_kv_append")


def nc_attn_decode_noalloc_scratch_bytes(N: int, Tmax: int, H: int, D: int, window: int) -> int:
    return int(lib.nc_attn_decode_noalloc_scratch_bytes(N, Tmax, H, D, int(window)))


def nc_attn_decode_noalloc(q, kcache, vcache, cache_lens, o, lse, window: int, scale: float, stream=None) -> None:
    """Decode for callers that cannot allocate: no workspace argument, nothing allocated.

    The partial results go to a fixed scratch array inside the library (see
    NC_DECODE_NOALLOC_SCRATCH_BYTES); calls that would need more raise NcError
    with NC_ERR_WORKSPACE.  Calls whose GPU work overlaps share that array and
    race; keep them ordered (one stream).
    """
    N, Tmax, H, D = kcache.shape
    _need(q, "q", torch.bfloat16, (N, H, D))
    _need(kcache, "kcache", torch.bfloat16)
    _need(vcache, "vcache", torch.bfloat16, (N, Tmax, H, D))
    _need(cache_lens, "cache_lens", torch.int32, (N,))
    _need(o, "o", torch.bfloat16, (N, H, D))
    if lse is not None:
        _need(lse, "lse", torch.float32, (N, H))
    _check(lib.nc_attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(cache_lens), _ptr(o), _ptr(lse),
                                      N, Tmax, H, D, int(window), float(scale), _stream(q.device, stream)),
           "nc_attn_decode_noalloc")


def nc_get_device_error(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the library's device error code."""
    code = ctypes.c_int(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib.nc_get_device_error(ctypes.byref(code), _stream(dev, stream)), "nc_get_device_error")
    return code.value


def nc_debug_watchdog_selftest(limit_cycles: int, stream=None, device=None) -> None:
    """Run the bounded-wait self-test kernel; afterwards nc_get_device_error() reports the timeout."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib.nc_debug_watchdog_selftest(int(limit_cycles), _stream(dev, stream)), "nc_debug_watchdog_selftest")


def nc_launch_count() -> int:
    """Kernels the library has enqueued since it was loaded."""
    return int(lib.nc_launch_count())


# ---------------------------------------------------------------- allocating conveniences


def attn_fwd(q, k, v, window: int, scale: float | None = None, stream=None):
    """Returns (o, lse) for bf16 q, k, v [B, T, H, D]."""
    B, T, H, D = q.shape
    scale = default_scale(D) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    nc_attn_fwd(q, k, v, o, lse, window, scale, stream)
    return o, lse


def attn_bwd(q, k, v, o, dO, lse, window: int, scale: float | None = None, workspace=None, stream=None,
             deterministic: bool = False):
    """Returns (dq, dk, dv); ``deterministic`` selects the bitwise-reproducible backward."""
    B, T, H, D = q.shape
    scale = default_scale(D) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nc_attn_bwd_workspace_bytes(B, T, H, D), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    (nc_attn_bwd_deterministic if deterministic else nc_attn_bwd)(q, k, v, o, dO, lse, dq, dk, dv, window, scale,
                                                                  workspace, stream)
    return dq, dk, dv


def attn_prefill(q, kcache, vcache, cache_lens, window: int, scale: float | None = None, stream=None):
    """Returns (o [N,Tq,H,D], lse [N,H,Tq]) for the new tokens q [N,Tq,H,D]."""
    N, Tmax, H, D = kcache.shape
    Tq = q.shape[1]
    scale = default_scale(D) if scale is None else scale
    o = torch.empty((N, Tq, H, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((N, H, Tq), dtype=torch.float32, device=q.device)
    nc_attn_prefill(q, kcache, vcache, cache_lens, o, lse, window, scale, stream)
    return o, lse


def attn_decode(q, kcache, vcache, cache_lens, window: int, scale: float | None = None, workspace=None,
                with_lse: bool = True, stream=None):
    """Returns (o [N,H,D], lse [N,H] or None)."""
    N, Tmax, H, D = kcache.shape
    scale = default_scale(D) if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nc_attn_decode_workspace_bytes(N, Tmax, H, D), dtype=torch.uint8, device=q.device)
    o = torch.empty((N, H, D), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((N, H), dtype=torch.float32, device=q.device) if with_lse else None
    nc_attn_decode(q, kcache, vcache, cache_lens, o, lse, window, scale, workspace, stream)
    return o, lse


# ---------------------------------------------------------------- autograd nodes (training)
# Each node calls the library's forward, keeps what its backward call needs, and calls that backward:
# no arithmetic here.  Non-contiguous inputs (views of a fused projection) are copied to contiguous ones,
# since the kernels take dense [B, T, H, D] rows.


class _SlidingWindowAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, window: int, scale: float, deterministic: bool):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse = attn_fwd(q, k, v, window, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.window, ctx.scale, ctx.deterministic = window, scale, deterministic
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = attn_bwd(q, k, v, o, dO.contiguous(), lse, ctx.window, ctx.scale,
                              deterministic=ctx.deterministic)
        return dq, dk, dv, None, None, None


class _VarlenAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, max_seqlen: int, window: int, scale: float, deterministic: bool):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse = attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, window, scale)
        ctx.save_for_backward(q, k, v, o, lse, cu_seqlens)
        ctx.max_seqlen, ctx.window, ctx.scale, ctx.deterministic = max_seqlen, window, scale, deterministic
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, o, lse, cu = ctx.saved_tensors
        dq, dk, dv = attn_bwd_varlen(q, k, v, o, dO.contiguous(), lse, cu, ctx.max_seqlen, ctx.window, ctx.scale,
                                     deterministic=ctx.deterministic)
        return dq, dk, dv, None, None, None, None, None


class _RotaryAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, rope_cos, rope_sin, window: int, scale: float):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse, qr, kr = attn_fwd_rotary(q, k, v, rope_cos, rope_sin, window, scale)
        ctx.save_for_backward(qr, kr, v, rope_cos, rope_sin, o, lse)
        ctx.window, ctx.scale = window, scale
        return o

    @staticmethod
    def backward(ctx, dO):
        qr, kr, v, c, s, o, lse = ctx.saved_tensors
        dq, dk, dv = attn_bwd_rotary(qr, kr, v, c, s, o, dO.contiguous(), lse, ctx.window, ctx.scale)
        return dq, dk, dv, None, None, None, None


def sliding_window_attention(q, k, v, window: int, scale: float | None = None, deterministic: bool = False):
    """o for bf16 q, k, v [B, T, H, D] (D = 64 or 128), with a backward for autograd: causal attention in
    which each query sees its own position and the window - 1 before it (window <= 0: full causal).
    ``deterministic`` selects the bitwise-reproducible backward."""
    scale = default_scale(q.shape[-1]) if scale is None else scale
    return _SlidingWindowAttention.apply(q, k, v, int(window), float(scale), bool(deterministic))


def varlen_attention(q, k, v, cu_seqlens, max_seqlen: int, window: int, scale: float | None = None,
                     deterministic: bool = False):
    """o for packed documents q, k, v [total, H, D] (document d is rows cu_seqlens[d] .. cu_seqlens[d+1]-1,
    each attending only within itself), with a backward for autograd (``deterministic``: bitwise-reproducible)."""
    scale = default_scale(q.shape[-1]) if scale is None else scale
    return _VarlenAttention.apply(q, k, v, cu_seqlens, int(max_seqlen), int(window), float(scale), bool(deterministic))


def rotary_attention(q, k, v, rope_cos, rope_sin, window: int, scale: float | None = None):
    """o for q and k turned by the rotary tables (fp32 [T, D/2]) before the attention, with a backward for
    autograd whose q and k gradients are with respect to the unturned q and k."""
    scale = default_scale(q.shape[-1]) if scale is None else scale
    return _RotaryAttention.apply(q, k, v, rope_cos, rope_sin, int(window), float(scale))
