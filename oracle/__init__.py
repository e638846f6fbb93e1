"""fp64 CPU oracle for causal sliding-window softmax attention (test infrastructure).

Only the test suite, the package's ``smoke()`` check and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library and its Python binding
never do; the two implementations share no code.

The arithmetic lives in ``nc_oracle.c`` (plain loops, double precision, OpenMP
over independent (batch, head) slices).  This module only compiles it on
demand, converts inputs to contiguous float64 arrays and calls it through
ctypes.  See ``nc_oracle.c`` for the definition, the pages it follows and the
readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

WINDOW_FULL = -1


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, OpenMP, no fast-math, no contraction of a*b+c)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """ctypes view of one compiled oracle library (the default one, or a test's mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, ctypes.c_double]
        lib.oracle_fwd.restype = None
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, L, L, L, ctypes.c_double]
        lib.oracle_bwd.restype = None
        lib.oracle_decode.argtypes = [dp, dp, dp, ctypes.POINTER(ctypes.c_int), dp, dp,
                                      L, L, L, L, L, ctypes.c_double]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [dp, dp, dp, ctypes.POINTER(ctypes.c_int), dp, dp,
                                       L, L, L, L, L, L, ctypes.c_double]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_rotary.argtypes = [dp, dp, dp, dp, L, L, L, L, ctypes.c_int]
        lib.oracle_rotary.restype = None
        lib.oracle_rotary_f32.argtypes = [dp, dp, dp, dp, L, L, L, L]
        lib.oracle_rotary_f32.restype = None
        lib.oracle_round_bf16.argtypes = [dp, L]
        lib.oracle_round_bf16.restype = None
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        self.lib = lib

    def fwd(self, q, k, v, window: int, scale: float):
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, T, H, D = q.shape
        assert k.shape == q.shape and v.shape == q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, T), dtype=np.float64)
        self.lib.oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, H, D,
                            int(window), float(scale))
        return o, lse

    def bwd(self, q, k, v, dO, window: int, scale: float):
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        B, T, H, D = q.shape
        dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
        self.lib.oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                            B, T, H, D, int(window), float(scale))
        return dq, dk, dv

    def rotary(self, x, cos, sin, inverse: bool = False):
        x = _f64(x)
        c, s = _f64(cos), _f64(sin)
        B, T, H, D = x.shape
        assert c.shape == (T, D // 2) and s.shape == c.shape and D % 2 == 0
        y = np.empty_like(x)
        self.lib.oracle_rotary(_ptr(x), _ptr(c), _ptr(s), _ptr(y), B, T, H, D, 1 if inverse else 0)
        return y

    def rotary_f32(self, x, cos, sin):
        x = _f64(x)
        c, s = _f64(cos), _f64(sin)
        B, T, H, D = x.shape
        assert c.shape == (T, D // 2) and s.shape == c.shape and D % 2 == 0
        y = np.empty_like(x)
        self.lib.oracle_rotary_f32(_ptr(x), _ptr(c), _ptr(s), _ptr(y), B, T, H, D)
        return y

    def round_bf16(self, x):
        y = _f64(x).copy()
        self.lib.oracle_round_bf16(_ptr(y), y.size)
        return y

    def decode(self, q, kcache, vcache, cache_lens, window: int, scale: float):
        q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
        if hasattr(cache_lens, "detach"):
            cache_lens = cache_lens.detach().to("cpu").numpy()
        lens = np.ascontiguousarray(cache_lens, dtype=np.int32)
        N, H, D = q.shape
        Tmax = kc.shape[1]
        assert kc.shape == (N, Tmax, H, D) and vc.shape == kc.shape and lens.shape == (N,)
        o = np.empty_like(q)
        lse = np.empty((N, H), dtype=np.float64)
        rc = self.lib.oracle_decode(_ptr(q), _ptr(kc), _ptr(vc),
                                    lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                    _ptr(o), _ptr(lse), N, Tmax, H, D, int(window), float(scale))
        return o, lse, rc == 0

    def prefill(self, q, kcache, vcache, cache_lens, window: int, scale: float):
        q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
        if hasattr(cache_lens, "detach"):
            cache_lens = cache_lens.detach().to("cpu").numpy()
        lens = np.ascontiguousarray(cache_lens, dtype=np.int32)
        N, Tq, H, D = q.shape
        Tmax = kc.shape[1]
        assert kc.shape == (N, Tmax, H, D) and vc.shape == kc.shape and lens.shape == (N,)
        o = np.empty_like(q)
        lse = np.empty((N, H, Tq), dtype=np.float64)
        rc = self.lib.oracle_prefill(_ptr(q), _ptr(kc), _ptr(vc),
                                     lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                     _ptr(o), _ptr(lse), N, Tq, Tmax, H, D, int(window), float(scale))
        return o, lse, rc == 0


def _load() -> OracleLib:
    global _lib
    if _lib is None:
        _lib = OracleLib(build())
    return _lib


def _f64(x) -> np.ndarray:
    """Widen a torch tensor (any float dtype, any device) or array to contiguous float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return int(_load().lib.oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().lib.oracle_set_num_threads(int(n))


def fwd(q, k, v, window: int, scale: float):
    """Exact attention forward.  q, k, v: [B, T, H, D].  Returns (o [B,T,H,D], lse [B,H,T])."""
    return _load().fwd(q, k, v, window, scale)


def bwd(q, k, v, dO, window: int, scale: float):
    """Exact gradients of sum(O * dO) w.r.t. q, k, v.  Returns (dq, dk, dv), each [B, T, H, D]."""
    return _load().bwd(q, k, v, dO, window, scale)


def prefill(q, kcache, vcache, cache_lens, window: int, scale: float):
    """Prefill (append) over a KV cache.  q [N,Tq,H,D]; caches [N,Tmax,H,D]; cache_lens [N] (int),
    each counting the Tq new tokens, whose keys/values are already in the cache.

    Returns (o [N,Tq,H,D], lse [N,H,Tq], ok).  ok is False when some length is outside
    [Tq, Tmax]; that sequence's rows are NaN.
    """
    return _load().prefill(q, kcache, vcache, cache_lens, window, scale)


def _doc_bounds(cu_seqlens):
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
    cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
    assert cu[0] == 0 and all(b >= a for a, b in zip(cu, cu[1:])), "cu_seqlens must start at 0 and not decrease"
    return cu


def fwd_varlen(q, k, v, cu_seqlens, window: int, scale: float):
    """Document-masked (varlen) forward over packed rows.  q, k, v: [1, total, H, D]; document d is rows
    cu_seqlens[d] .. cu_seqlens[d+1]-1 and attends only within itself (the window counts positions inside
    the document).  Each document is an independent problem, so this is the forward applied per slice.
    Returns (o [1, total, H, D], lse [1, H, total])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = _doc_bounds(cu_seqlens)
    _, total, H, D = q.shape
    assert cu[-1] == total
    o = np.empty_like(q)
    lse = np.empty((1, H, total), dtype=np.float64)
    for a, b in zip(cu, cu[1:]):
        if b > a:
            od, ld = _load().fwd(q[:, a:b], k[:, a:b], v[:, a:b], window, scale)
            o[:, a:b] = od
            lse[:, :, a:b] = ld
    return o, lse


def bwd_varlen(q, k, v, dO, cu_seqlens, window: int, scale: float):
    """Gradients of the document-masked forward: the backward applied per document slice."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    cu = _doc_bounds(cu_seqlens)
    dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
    for a, b in zip(cu, cu[1:]):
        if b > a:
            g = _load().bwd(q[:, a:b], k[:, a:b], v[:, a:b], dO[:, a:b], window, scale)
            dq[:, a:b], dk[:, a:b], dv[:, a:b] = g
    return dq, dk, dv


def decode(q, kcache, vcache, cache_lens, window: int, scale: float):
    """One-token decode.  q [N,H,D]; caches [N,Tmax,H,D]; cache_lens [N] (int).

    Returns (o [N,H,D], lse [N,H], ok).  ok is False when some length is outside
    [1, Tmax]; that sequence's rows are NaN.
    """
    return _load().decode(q, kcache, vcache, cache_lens, window, scale)


def rotary(x, cos, sin, inverse: bool = False):
    """Rotary position embedding of x [B, T, H, D] (rotate-half pairing, see ``oracle_rotary``);
    cos, sin: [T, D/2], row t for position t.  ``inverse`` applies the transpose."""
    return _load().rotary(x, cos, sin, inverse)


def round_bf16(x):
    """x rounded to the nearest bfloat16 value (ties to even), as float64."""
    return _load().round_bf16(x)


def rotary_f32(x, cos, sin):
    """The rotary turn evaluated in float32 as the CUDA kernels evaluate it (see ``oracle_rotary_f32``)."""
    return _load().rotary_f32(x, cos, sin)


def rotary_bf16(x, cos, sin):
    """The turned rows as the attention receives them: the float32 turn rounded to bf16."""
    return round_bf16(rotary_f32(x, cos, sin))


def fwd_rotary(q, k, v, cos, sin, window: int, scale: float):
    """Attention with the rotary embedding applied to q and k first (positions 0 .. T-1).  The turned
    q and k are bf16 values (the model's dtype) when the attention takes them.
    Returns (o [B,T,H,D], lse [B,H,T])."""
    return _load().fwd(rotary_bf16(q, cos, sin), rotary_bf16(k, cos, sin), v, window, scale)


def bwd_rotary(q, k, v, dO, cos, sin, window: int, scale: float):
    """Gradients of sum(O * dO) for the rotary forward with respect to the unrotated q, k and to v:
    the attention gradients at the (bf16) turned q and k, turned back by the exact transpose.  The
    rounding is a change of dtype, not of the function: its gradient is taken as the identity."""
    dqr, dkr, dv = _load().bwd(rotary_bf16(q, cos, sin), rotary_bf16(k, cos, sin), v, dO, window, scale)
    return rotary(dqr, cos, sin, inverse=True), rotary(dkr, cos, sin, inverse=True), dv
