"""Pins for the fp64 CPU oracle, checked against things other than itself.

Each test ties the oracle to something the definition of windowed causal
softmax attention fixes on its own: a hand-worked example, closed forms,
invariants, brute-force dense enumeration, a library routine for the same
definition (torch SDPA in fp64 with an explicit band mask) and finite
differences of the forward.  A mistake in the oracle (a dropped term, a wrong
sign, an off-by-one window, a transposed operand) fails at least one of them;
``test_oracle_mutants.py`` plants such mistakes to show it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from causal_sliding_window_fwd_b300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _val(x):
    if isinstance(x, str):
        return eval(x, {"ln3": math.log(3.0), "ln4": math.log(4.0), "ln5": math.log(5.0)})
    return float(x)


def _arr(rows):
    return np.array([[_val(c) for c in r] for r in rows], dtype=np.float64)


def _bthd(rows):
    a = _arr(rows)
    return a.reshape(1, a.shape[0], 1, a.shape[1])


# ---------------------------------------------------------------- golden


def test_hand_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "hand_window2.json")))
    q, k, v, dO = (_bthd(g[n]) for n in ("q", "k", "v", "dO"))
    o, lse = oracle_mod.fwd(q, k, v, g["window"], g["scale"])
    np.testing.assert_allclose(o[0, :, 0, :], _arr(g["o"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], [_val(x) for x in g["lse"]], rtol=0, atol=1e-12)
    dq, dk, dv = oracle_mod.bwd(q, k, v, dO, g["window"], g["scale"])
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        np.testing.assert_allclose(got[0, :, 0, :], _arr(g[name]), rtol=0, atol=1e-12, err_msg=name)
    # decode over a cache of the same three rows, length 3, query q2
    od, lsed, ok = oracle_mod.decode(q[:, 2], k, v, np.array([3]), g["window"], g["scale"])
    assert ok
    np.testing.assert_allclose(od[0, 0], _arr(g["o"])[2], rtol=0, atol=1e-12)
    assert abs(lsed[0, 0] - math.log(5.0)) < 1e-12


# ---------------------------------------------------------------- closed forms


def test_window_one_is_identity(oracle_mod):
    B, T, H, D = 2, 9, 3, 5
    q, k, v, dO = (_rand((B, T, H, D), s) for s in range(4))
    o, lse = oracle_mod.fwd(q, k, v, 1, 0.7)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, 0.7 * np.einsum("bthd,bthd->bht", q, k), rtol=1e-14, atol=1e-14)
    dq, dk, dv = oracle_mod.bwd(q, k, v, dO, 1, 0.7)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_array_equal(dv, dO)


@pytest.mark.parametrize("window", [2, 7, 40, -1])
def test_first_query_sees_only_itself(oracle_mod, window):
    B, T, H, D = 1, 12, 2, 6
    q, k, v = (_rand((B, T, H, D), 10 + s) for s in range(3))
    o, lse = oracle_mod.fwd(q, k, v, window, 0.3)
    np.testing.assert_array_equal(o[:, 0], v[:, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]), atol=1e-14)


@pytest.mark.parametrize("window", [1, 3, 8, 100])
def test_identical_keys_give_uniform_weights(oracle_mod, window):
    B, T, H, D = 1, 11, 2, 4
    q, v = _rand((B, T, H, D), 20), _rand((B, T, H, D), 21)
    c = _rand((H, D), 22)
    k = np.broadcast_to(c, (B, T, H, D)).copy()
    o, lse = oracle_mod.fwd(q, k, v, window, 0.5)
    for i in range(T):
        lo = max(0, i - window + 1)
        n = i - lo + 1
        np.testing.assert_allclose(o[:, i], v[:, lo:i + 1].mean(axis=1), atol=1e-13)
        expect = 0.5 * np.einsum("bhd,hd->bh", q[:, i], c) + math.log(n)
        np.testing.assert_allclose(lse[:, :, i], expect, atol=1e-13)


# ---------------------------------------------------------------- invariants


@pytest.mark.parametrize("window", [1, 4, 13, -1])
def test_rows_sum_to_one(oracle_mod, window):
    B, T, H, D = 2, 13, 2, 3
    q, k = _rand((B, T, H, D), 30), _rand((B, T, H, D), 31)
    o, _ = oracle_mod.fwd(q, k, np.ones((B, T, H, D)), window, 1.3)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)


def test_window_at_least_T_is_full_causal(oracle_mod):
    B, T, H, D = 1, 10, 2, 4
    q, k, v, dO = (_rand((B, T, H, D), 40 + s) for s in range(4))
    ref_o, ref_l = oracle_mod.fwd(q, k, v, -1, 0.5)
    ref_g = oracle_mod.bwd(q, k, v, dO, -1, 0.5)
    for w in (T, T + 5, 10 ** 6):
        o, l = oracle_mod.fwd(q, k, v, w, 0.5)
        np.testing.assert_array_equal(o, ref_o)
        np.testing.assert_array_equal(l, ref_l)
        for a, b in zip(oracle_mod.bwd(q, k, v, dO, w, 0.5), ref_g):
            np.testing.assert_array_equal(a, b)
    # and a window of T-1 differs (the last row loses key 0)
    o, _ = oracle_mod.fwd(q, k, v, T - 1, 0.5)
    assert not np.allclose(o[:, T - 1], ref_o[:, T - 1])
    np.testing.assert_array_equal(o[:, :T - 1], ref_o[:, :T - 1])


def test_key_shift_invariance(oracle_mod):
    B, T, H, D = 1, 9, 2, 5
    q, k, v = (_rand((B, T, H, D), 50 + s) for s in range(3))
    c = _rand((H, D), 53)
    o1, l1 = oracle_mod.fwd(q, k, v, 4, 0.8)
    o2, l2 = oracle_mod.fwd(q, k + c, v, 4, 0.8)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.8 * np.einsum("bthd,hd->bht", q, c), atol=1e-12)


def test_window_edge_is_exact(oracle_mod):
    """Key i-W+1 is seen by query i and key i-W is not."""
    B, T, H, D, W = 1, 12, 1, 3, 4
    q, k, v = (_rand((B, T, H, D), 60 + s) for s in range(3))
    i = 9
    o0, _ = oracle_mod.fwd(q, k, v, W, 1.0)
    v_out = v.copy(); v_out[:, i - W] += 100.0
    o1, _ = oracle_mod.fwd(q, k, v_out, W, 1.0)
    np.testing.assert_array_equal(o1[:, i], o0[:, i])
    v_in = v.copy(); v_in[:, i - W + 1] += 100.0
    o2, _ = oracle_mod.fwd(q, k, v_in, W, 1.0)
    assert np.abs(o2[:, i] - o0[:, i]).max() > 1e-3
    v_fut = v.copy(); v_fut[:, i + 1] += 100.0
    o3, _ = oracle_mod.fwd(q, k, v_fut, W, 1.0)
    np.testing.assert_array_equal(o3[:, i], o0[:, i])


@pytest.mark.parametrize("window", [1, 3, 6, -1])
def test_gradient_sums(oracle_mod, window):
    B, T, H, D = 2, 10, 2, 4
    q, k, v, dO = (_rand((B, T, H, D), 70 + s) for s in range(4))
    dq, dk, dv = oracle_mod.bwd(q, k, v, dO, window, 0.6)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=1), dO.sum(axis=1), atol=1e-12)


@pytest.mark.parametrize("window", [1, 5, 64, -1])
def test_decode_equals_last_forward_row(oracle_mod, window):
    N, Tmax, H, D = 3, 20, 2, 8
    kc, vc = _rand((N, Tmax, H, D), 80), _rand((N, Tmax, H, D), 81)
    qs = _rand((N, Tmax, H, D), 82)
    lens = np.array([1, 7, 20], dtype=np.int32)
    q_dec = np.stack([qs[n, lens[n] - 1] for n in range(N)])
    o, lse, ok = oracle_mod.decode(q_dec, kc, vc, lens, window, 0.35)
    assert ok
    for n in range(N):
        L = lens[n]
        of, lf = oracle_mod.fwd(qs[n:n + 1, :L], kc[n:n + 1, :L], vc[n:n + 1, :L], window, 0.35)
        np.testing.assert_allclose(o[n], of[0, L - 1], atol=1e-13)
        np.testing.assert_allclose(lse[n], lf[0, :, L - 1], atol=1e-13)


def test_decode_ignores_slots_outside_window_and_length(oracle_mod):
    N, Tmax, H, D, W = 2, 16, 1, 4, 5
    q = _rand((N, H, D), 90)
    kc, vc = _rand((N, Tmax, H, D), 91), _rand((N, Tmax, H, D), 92)
    lens = np.array([9, 16], dtype=np.int32)
    o0, l0, _ = oracle_mod.decode(q, kc, vc, lens, W, 0.5)
    kp, vp = kc.copy(), vc.copy()
    for n, L in enumerate(lens):
        kp[n, L:] = np.nan; vp[n, L:] = np.nan
        kp[n, :L - W] = np.nan; vp[n, :L - W] = np.nan
    o1, l1, _ = oracle_mod.decode(q, kp, vp, lens, W, 0.5)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_decode_bad_length_is_reported(oracle_mod):
    q = _rand((2, 1, 4), 95)
    kc, vc = _rand((2, 8, 1, 4), 96), _rand((2, 8, 1, 4), 97)
    o, lse, ok = oracle_mod.decode(q, kc, vc, np.array([0, 8], dtype=np.int32), -1, 0.5)
    assert not ok
    assert np.isnan(o[0]).all() and np.isnan(lse[0]).all()
    assert np.isfinite(o[1]).all()


# ---------------------------------------------------------------- brute force


def _dense_masked_reference(q, k, v, window, scale):
    """Dense T x T enumeration with an explicit 0/1 visibility matrix (pure Python loops)."""
    B, T, H, D = q.shape
    W = T if window <= 0 else min(window, T)
    mask = [[1 if (j <= i and i - j < W) else 0 for j in range(T)] for i in range(T)]
    o = np.zeros_like(q)
    lse = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            for i in range(T):
                logits = [scale * sum(q[b, i, h, d] * k[b, j, h, d] for d in range(D)) if mask[i][j] else -math.inf
                          for j in range(T)]
                m = max(logits)
                z = sum(math.exp(x - m) for x in logits)
                lse[b, h, i] = m + math.log(z)
                for d in range(D):
                    o[b, i, h, d] = sum(math.exp(logits[j] - m) / z * v[b, j, h, d] for j in range(T))
    return o, lse


@pytest.mark.parametrize("T,D,window", [(1, 1, 1), (5, 3, 2), (8, 4, 3), (8, 2, 8), (7, 4, -1)])
def test_brute_force_tiny(oracle_mod, T, D, window):
    B, H = 2, 2
    q, k, v = (_rand((B, T, H, D), 100 + s) for s in range(3))
    o, lse = oracle_mod.fwd(q, k, v, window, 0.9)
    ob, lb = _dense_masked_reference(q, k, v, window, 0.9)
    np.testing.assert_allclose(o, ob, atol=1e-13)
    np.testing.assert_allclose(lse, lb, atol=1e-13)


# ---------------------------------------------------------------- library routine


def _band_mask(T, window):
    W = T if window <= 0 else min(window, T)
    i = torch.arange(T).view(T, 1)
    j = torch.arange(T).view(1, T)
    return (j <= i) & (i - j < W)


@pytest.mark.parametrize("T,D,window", [(16, 8, 1), (33, 16, 5), (40, 8, 40), (64, 16, 17), (29, 8, -1)])
def test_matches_torch_sdpa_fp64(oracle_mod, T, D, window):
    B, H = 2, 3
    scale = 1.0 / math.sqrt(D)
    q, k, v, dO = (torch.from_numpy(_rand((B, T, H, D), 110 + s)) for s in range(4))
    qt, kt, vt = (x.transpose(1, 2).clone().requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=_band_mask(T, window), scale=scale)
    out.backward(dO.transpose(1, 2))
    logits = scale * qt.detach() @ kt.detach().transpose(-1, -2)
    lse_ref = torch.logsumexp(logits.masked_fill(~_band_mask(T, window), -math.inf), dim=-1)

    o, lse = oracle_mod.fwd(q, k, v, window, scale)
    np.testing.assert_allclose(o, out.detach().transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), atol=1e-12)
    dq, dk, dv = oracle_mod.bwd(q, k, v, dO, window, scale)
    np.testing.assert_allclose(dq, qt.grad.transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.transpose(1, 2).numpy(), atol=1e-12)


def test_matches_torch_sdpa_on_bf16_workload(oracle_mod):
    """The tiny workload's own bf16 tensors, widened exactly to fp64."""
    call = workloads.TINY.calls[0]
    q, k, v, dO = workloads.make_qkvdo(call, "cpu")
    q64, k64, v64 = (x.double().transpose(1, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q64, k64, v64, attn_mask=_band_mask(call.T, call.window), scale=call.scale)
    o, _ = oracle_mod.fwd(q, k, v, call.window, call.scale)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), atol=1e-12)


# ---------------------------------------------------------------- finite differences


@pytest.mark.parametrize("window", [1, 3, 8])
def test_backward_matches_finite_differences(oracle_mod, window):
    """Central differences of L = sum(O * G) from the oracle's own forward."""
    B, T, H, D = 1, 8, 1, 4
    scale = 0.5
    base = [_rand((B, T, H, D), 120 + s) for s in range(3)]
    G = _rand((B, T, H, D), 123)
    grads = oracle_mod.bwd(*base, G, window, scale)
    eps = 1e-6
    rng = np.random.default_rng(7)
    for which in range(3):
        for _ in range(12):
            idx = (0, int(rng.integers(T)), 0, int(rng.integers(D)))
            plus = [x.copy() for x in base]; plus[which][idx] += eps
            minus = [x.copy() for x in base]; minus[which][idx] -= eps
            lp = (oracle_mod.fwd(*plus, window, scale)[0] * G).sum()
            lm = (oracle_mod.fwd(*minus, window, scale)[0] * G).sum()
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grads[which][idx]) < 1e-7, (which, idx, fd, grads[which][idx])


# ---------------------------------------------------------------- prefill over a KV cache


@pytest.mark.parametrize("window", [1, 4, 9, -1])
def test_prefill_rows_equal_forward_rows(oracle_mod, window):
    """Appending Tq tokens to a cache equals the last Tq rows of the forward over the whole sequence."""
    N, Tq, Tmax, H, D = 3, 5, 24, 2, 8
    kc, vc = _rand((N, Tmax, H, D), 300), _rand((N, Tmax, H, D), 301)
    qs = _rand((N, Tmax, H, D), 302)
    lens = np.array([5, 13, 24], dtype=np.int32)
    q = np.stack([qs[n, lens[n] - Tq:lens[n]] for n in range(N)])
    o, lse, ok = oracle_mod.prefill(q, kc, vc, lens, window, 0.4)
    assert ok
    for n in range(N):
        L = lens[n]
        of, lf = oracle_mod.fwd(qs[n:n + 1, :L], kc[n:n + 1, :L], vc[n:n + 1, :L], window, 0.4)
        np.testing.assert_allclose(o[n], of[0, L - Tq:L], atol=1e-13)
        np.testing.assert_allclose(lse[n], lf[0, :, L - Tq:L], atol=1e-13)


@pytest.mark.parametrize("window", [1, 6, -1])
def test_prefill_of_one_token_is_decode(oracle_mod, window):
    N, Tmax, H, D = 4, 16, 2, 4
    kc, vc = _rand((N, Tmax, H, D), 310), _rand((N, Tmax, H, D), 311)
    q = _rand((N, 1, H, D), 312)
    lens = np.array([1, 2, 9, 16], dtype=np.int32)
    o, lse, ok = oracle_mod.prefill(q, kc, vc, lens, window, 0.7)
    od, ld, okd = oracle_mod.decode(q[:, 0], kc, vc, lens, window, 0.7)
    assert ok and okd
    np.testing.assert_allclose(o[:, 0], od, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], ld, atol=1e-14)


def _dense_prefill_reference(q, kc, lens, vc, window, scale):
    """Explicit (query, cache row) visibility matrix per sequence, pure Python loops."""
    N, Tq, H, D = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((N, H, Tq))
    for n in range(N):
        L = int(lens[n])
        for h in range(H):
            for t in range(Tq):
                i = L - Tq + t
                vis = [1 if (j <= i and (window <= 0 or i - j < window)) else 0 for j in range(kc.shape[1])]
                logits = [scale * sum(q[n, t, h, d] * kc[n, j, h, d] for d in range(D)) if vis[j] else -math.inf
                          for j in range(kc.shape[1])]
                m = max(logits)
                z = sum(math.exp(x - m) for x in logits)
                lse[n, h, t] = m + math.log(z)
                for d in range(D):
                    o[n, t, h, d] = sum(math.exp(logits[j] - m) / z * vc[n, j, h, d] for j in range(kc.shape[1])
                                        if vis[j])
    return o, lse


@pytest.mark.parametrize("Tq,window", [(1, 2), (3, 2), (4, -1), (6, 3)])
def test_prefill_brute_force_tiny(oracle_mod, Tq, window):
    N, Tmax, H, D = 2, 9, 2, 3
    q = _rand((N, Tq, H, D), 320)
    kc, vc = _rand((N, Tmax, H, D), 321), _rand((N, Tmax, H, D), 322)
    lens = np.array([Tq, Tmax], dtype=np.int32)
    o, lse, ok = oracle_mod.prefill(q, kc, vc, lens, window, 0.8)
    ob, lb = _dense_prefill_reference(q, kc, lens, vc, window, 0.8)
    assert ok
    np.testing.assert_allclose(o, ob, atol=1e-13)
    np.testing.assert_allclose(lse, lb, atol=1e-13)


@pytest.mark.parametrize("Tq,L,window", [(8, 8, -1), (7, 30, 5), (16, 40, 16), (1, 33, -1)])
def test_prefill_matches_torch_sdpa_fp64(oracle_mod, Tq, L, window):
    """torch SDPA with a band mask offset to the queries' cache positions."""
    H, D = 3, 8
    scale = 1.0 / math.sqrt(D)
    q = torch.from_numpy(_rand((1, Tq, H, D), 330))
    kc, vc = (torch.from_numpy(_rand((1, L, H, D), 331 + s)) for s in range(2))
    i = torch.arange(L - Tq, L).view(Tq, 1)
    j = torch.arange(L).view(1, L)
    mask = (j <= i) & ((i - j < window) if window > 0 else torch.ones_like(j, dtype=torch.bool))
    out = torch.nn.functional.scaled_dot_product_attention(q.transpose(1, 2), kc.transpose(1, 2), vc.transpose(1, 2),
                                                           attn_mask=mask, scale=scale)
    logits = scale * q.transpose(1, 2) @ kc.transpose(1, 2).transpose(-1, -2)
    lse_ref = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
    o, lse, ok = oracle_mod.prefill(q, kc, vc, np.array([L], dtype=np.int32), window, scale)
    assert ok
    np.testing.assert_allclose(o, out.transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), atol=1e-12)


def test_prefill_ignores_slots_outside_window_and_length(oracle_mod):
    N, Tq, Tmax, H, D, W = 2, 4, 20, 1, 4, 6
    q = _rand((N, Tq, H, D), 340)
    kc, vc = _rand((N, Tmax, H, D), 341), _rand((N, Tmax, H, D), 342)
    lens = np.array([11, 20], dtype=np.int32)
    o0, l0, _ = oracle_mod.prefill(q, kc, vc, lens, W, 0.5)
    kp, vp = kc.copy(), vc.copy()
    for n, L in enumerate(lens):
        kp[n, L:] = np.nan; vp[n, L:] = np.nan
        first = L - Tq - W + 1  # the first query's earliest visible row
        kp[n, :first] = np.nan; vp[n, :first] = np.nan
    o1, l1, _ = oracle_mod.prefill(q, kp, vp, lens, W, 0.5)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_prefill_bad_length_is_reported(oracle_mod):
    q = _rand((2, 3, 1, 4), 350)
    kc, vc = _rand((2, 8, 1, 4), 351), _rand((2, 8, 1, 4), 352)
    o, lse, ok = oracle_mod.prefill(q, kc, vc, np.array([2, 8], dtype=np.int32), -1, 0.5)
    assert not ok
    assert np.isnan(o[0]).all() and np.isnan(lse[0]).all()
    assert np.isfinite(o[1]).all()


# ---------------------------------------------------------------- document-masked (varlen) attention


def _packed_mask(cu, window):
    """Explicit (query, key) visibility over packed rows: same document, causal, inside the window."""
    total = cu[-1]
    doc = np.zeros(total, dtype=np.int64)
    start = np.zeros(total, dtype=np.int64)
    for d, (a, b) in enumerate(zip(cu, cu[1:])):
        doc[a:b] = d
        start[a:b] = a
    i = np.arange(total).reshape(-1, 1)
    j = np.arange(total).reshape(1, -1)
    m = (doc.reshape(-1, 1) == doc.reshape(1, -1)) & (j <= i)
    if window > 0:
        m &= (i - j) < window
    return m


@pytest.mark.parametrize("cu,window", [([0, 7], 3), ([0, 3, 3, 10, 16], 4), ([0, 1, 2, 9], -1), ([0, 5, 12], 1)])
def test_varlen_matches_torch_sdpa_with_packed_mask(oracle_mod, cu, window):
    """torch SDPA in fp64 with an explicit block-diagonal band mask, and its autograd."""
    total, H, D = cu[-1], 2, 8
    scale = 1.0 / math.sqrt(D)
    q, k, v, dO = (torch.from_numpy(_rand((1, total, H, D), 400 + s)) for s in range(4))
    mask = torch.from_numpy(_packed_mask(cu, window))
    qt, kt, vt = (x.transpose(1, 2).clone().requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    out.backward(dO.transpose(1, 2))
    logits = scale * qt.detach() @ kt.detach().transpose(-1, -2)
    lse_ref = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
    o, lse = oracle_mod.fwd_varlen(q, k, v, cu, window, scale)
    np.testing.assert_allclose(o, out.detach().transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref.numpy(), atol=1e-12)
    dq, dk, dv = oracle_mod.bwd_varlen(q, k, v, dO, cu, window, scale)
    np.testing.assert_allclose(dq, qt.grad.transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.transpose(1, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.transpose(1, 2).numpy(), atol=1e-12)


def test_varlen_documents_do_not_interact(oracle_mod):
    cu = [0, 6, 6, 15, 20]
    total, H, D = cu[-1], 2, 4
    q, k, v, dO = (_rand((1, total, H, D), 410 + s) for s in range(4))
    o0, l0 = oracle_mod.fwd_varlen(q, k, v, cu, 5, 0.6)
    g0 = oracle_mod.bwd_varlen(q, k, v, dO, cu, 5, 0.6)
    q2, k2, v2, dO2 = (x.copy() for x in (q, k, v, dO))
    for x in (q2, k2, v2, dO2):
        x[:, 6:15] = _rand((1, 9, H, D), 420)  # replace the third document only
    o1, l1 = oracle_mod.fwd_varlen(q2, k2, v2, cu, 5, 0.6)
    g1 = oracle_mod.bwd_varlen(q2, k2, v2, dO2, cu, 5, 0.6)
    for sl in (slice(0, 6), slice(15, 20)):
        np.testing.assert_array_equal(o1[:, sl], o0[:, sl])
        np.testing.assert_array_equal(l1[:, :, sl], l0[:, :, sl])
        for a, b in zip(g1, g0):
            np.testing.assert_array_equal(a[:, sl], b[:, sl])


def test_varlen_single_document_is_the_forward(oracle_mod):
    q, k, v = (_rand((1, 13, 2, 4), 430 + s) for s in range(3))
    o, lse = oracle_mod.fwd_varlen(q, k, v, [0, 13], 4, 0.5)
    of, lf = oracle_mod.fwd(q, k, v, 4, 0.5)
    np.testing.assert_array_equal(o, of)
    np.testing.assert_array_equal(lse, lf)


# ---------------------------------------------------------------- rotary embedding (fused prologue)
# The oracle's rotary is the rotate-half pairing of Llama-like models: the pair (x_i, x_{i+D/2}) of
# position t is turned by the angle whose cosine and sine the tables hold at (t, i).


def _tables(T, D, base=10000.0):
    c, s = workloads.rope_tables(T, D, base)
    return c.double().numpy(), s.double().numpy()


def test_rotary_matches_complex_rotation(oracle_mod):
    """The same turn written as complex multiplication: z = x_i + i x_{i+D/2}, z' = z (c + i s)."""
    B, T, H, D = 2, 9, 3, 8
    x = _rand((B, T, H, D), 700)
    c, s = _tables(T, D)
    y = oracle_mod.rotary(x, c, s)
    xt = torch.from_numpy(x)
    z = torch.complex(xt[..., : D // 2], xt[..., D // 2:])
    e = torch.complex(torch.from_numpy(c), torch.from_numpy(s)).view(1, T, 1, D // 2)
    zr = z * e
    expect = torch.cat([zr.real, zr.imag], dim=-1).numpy()
    np.testing.assert_allclose(y, expect, rtol=0, atol=1e-12)


def test_rotary_position_zero_is_identity(oracle_mod):
    B, T, H, D = 1, 5, 2, 8
    x = _rand((B, T, H, D), 701)
    c, s = _tables(T, D)
    y = oracle_mod.rotary(x, c, s)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    assert np.abs(y[:, 1:] - x[:, 1:]).max() > 1e-3  # later positions do turn


def test_rotary_preserves_norms_and_the_transpose_turns_back(oracle_mod):
    B, T, H, D = 2, 7, 2, 16
    x = _rand((B, T, H, D), 702)
    c, s = _tables(T, D)
    y = oracle_mod.rotary(x, c, s)
    half = D // 2
    pair_x = x[..., :half] ** 2 + x[..., half:] ** 2
    pair_y = y[..., :half] ** 2 + y[..., half:] ** 2
    r2 = (c ** 2 + s ** 2).reshape(1, T, 1, half)  # 1 up to the float32 rounding of the tables
    np.testing.assert_allclose(pair_y, pair_x * r2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle_mod.rotary(y, c, s, inverse=True), x * np.concatenate([r2, r2], -1),
                               rtol=1e-12, atol=1e-12)


def test_rotary_scores_depend_on_relative_position(oracle_mod):
    """With angles t * f_i, the score of a rotated query at position p and a rotated key at p' depends
    only on p - p'."""
    T, D = 12, 8
    a, b = _rand((D,), 703), _rand((D,), 704)
    c, s = workloads.rope_tables(T, D)
    # exact angles in float64 (the float32 tables are only used for the layout)
    ang = np.arange(T)[:, None] * (10000.0 ** (-np.arange(0, D, 2) / D))[None, :]
    c, s = np.cos(ang), np.sin(ang)
    qa = oracle_mod.rotary(np.broadcast_to(a, (1, T, 1, D)).copy(), c, s)[0, :, 0]
    kb = oracle_mod.rotary(np.broadcast_to(b, (1, T, 1, D)).copy(), c, s)[0, :, 0]
    S = qa @ kb.T  # S[p, p']
    for dlt in range(-(T - 1), T):
        diag = np.diagonal(S, offset=dlt)
        np.testing.assert_allclose(diag, diag[0], rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("window", [1, 3, -1])
def test_rotary_attention_gradients_match_finite_differences(oracle_mod, window):
    """Gradients of L = sum(O * G) for O = attention(rotary(q), rotary(k), v) with respect to the
    unrotated q, k and v: the attention gradients turned back by the transpose."""
    B, T, H, D = 1, 7, 1, 4
    scale = 0.5
    c, s = _tables(T, D)
    base = [_rand((B, T, H, D), 710 + i) for i in range(3)]
    G = _rand((B, T, H, D), 713)

    def fwd(q, k, v):
        return oracle_mod.fwd(oracle_mod.rotary(q, c, s), oracle_mod.rotary(k, c, s), v, window, scale)[0]

    dqr, dkr, dv = oracle_mod.bwd(oracle_mod.rotary(base[0], c, s), oracle_mod.rotary(base[1], c, s), base[2],
                                  G, window, scale)
    grads = [oracle_mod.rotary(dqr, c, s, inverse=True), oracle_mod.rotary(dkr, c, s, inverse=True), dv]
    eps = 1e-6
    rng = np.random.default_rng(9)
    for which in range(3):
        for _ in range(10):
            idx = (0, int(rng.integers(T)), 0, int(rng.integers(D)))
            plus = [x.copy() for x in base]; plus[which][idx] += eps
            minus = [x.copy() for x in base]; minus[which][idx] -= eps
            fd = ((fwd(*plus) * G).sum() - (fwd(*minus) * G).sum()) / (2 * eps)
            assert abs(fd - grads[which][idx]) < 1e-7, (which, idx, fd, grads[which][idx])


def test_rotary_module_functions_compose_as_stated(oracle_mod):
    """fwd_rotary / bwd_rotary (used by the GPU tests) are the attention of the rotated q, k (the float32
    turn rounded to bf16) and the gradients turned back."""
    import oracle
    B, T, H, D = 1, 6, 2, 8
    c, s = workloads.rope_tables(T, D)
    q, k, v, dO = (torch.from_numpy(_rand((B, T, H, D), 720 + i)) for i in range(4))
    # the turned q and k are rounded to bf16 (values a bf16 tensor can hold) before the attention
    rq = oracle_mod.round_bf16(oracle_mod.rotary_f32(q, c, s))
    rk = oracle_mod.round_bf16(oracle_mod.rotary_f32(k, c, s))
    for r in (rq, rk):
        np.testing.assert_array_equal(torch.from_numpy(r).to(torch.bfloat16).double().numpy(), r)
    o, lse = oracle.fwd_rotary(q, k, v, c, s, 3, 0.3)
    o2, lse2 = oracle_mod.fwd(rq, rk, v, 3, 0.3)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    g = oracle.bwd_rotary(q, k, v, dO, c, s, 3, 0.3)
    gr = oracle_mod.bwd(rq, rk, v, dO, 3, 0.3)
    np.testing.assert_array_equal(g[0], oracle_mod.rotary(gr[0], c, s, inverse=True))
    np.testing.assert_array_equal(g[1], oracle_mod.rotary(gr[1], c, s, inverse=True))
    np.testing.assert_array_equal(g[2], gr[2])


def test_round_bf16_hand_values(oracle_mod):
    """Nearest bf16 value (8 significant bits), ties to even, worked by hand."""
    u = 2.0 ** -7  # spacing of bf16 values in [1, 2)
    cases = [
        (1.0, 1.0), (1 + u / 2, 1.0), (1 + 3 * u / 2, 1 + 2 * u), (1 + u / 2 + 2.0 ** -30, 1 + u),
        (-(1 + u / 2 + 2.0 ** -30), -(1 + u)), (1 + u / 2 - 2.0 ** -30, 1.0), (3.0, 3.0),
        (2 + u, 2.0), (2 + 3 * u, 2 + 4 * u), (0.0, 0.0), (1.0 / 3.0, 0.333984375),
        (2.0 ** -130 + 2.0 ** -134, 2.0 ** -130), (2.0 ** -130 + 3 * 2.0 ** -134, 2.0 ** -130 + 2.0 ** -132),
    ]
    got = oracle_mod.round_bf16(np.array([a for a, _ in cases]))
    np.testing.assert_array_equal(got, np.array([b for _, b in cases]))


def test_round_bf16_matches_torch_float32(oracle_mod):
    """For values a float32 holds, torch's float32 -> bfloat16 conversion is the same single rounding."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(20000) * 2.0 ** rng.integers(-30, 30, 20000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = oracle_mod.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(oracle_mod.round_bf16(got), got)  # already bf16 values stay put


def _bf16_rows(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16).double().numpy()


def test_rotary_f32_matches_a_numpy_restatement(oracle_mod):
    """The float32 turn: each product of a bf16 value and a float32 table entry is exact in float64, so
    fmaf(x1, c, -fl(x2 s)) is x1 c - fl(x2 s) rounded once to float32 (numpy float32 ops round per op)."""
    B, T, H, D = 2, 50, 3, 64
    x = _bf16_rows((B, T, H, D), 730)
    c32, s32 = workloads.rope_tables(T, D)
    c = c32.numpy().reshape(1, T, 1, D // 2).astype(np.float64)
    s = s32.numpy().reshape(1, T, 1, D // 2).astype(np.float64)
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    p2s = (x2.astype(np.float32) * s.astype(np.float32)).astype(np.float64)
    p2c = (x2.astype(np.float32) * c.astype(np.float32)).astype(np.float64)
    y1 = (x1 * c - p2s).astype(np.float32).astype(np.float64)
    y2 = (x1 * s + p2c).astype(np.float32).astype(np.float64)
    got = oracle_mod.rotary_f32(x, c32.numpy(), s32.numpy())
    np.testing.assert_array_equal(got, np.concatenate([y1, y2], axis=-1))


def test_rotary_f32_is_the_turn_to_float_precision(oracle_mod):
    B, T, H, D = 1, 40, 2, 32
    x = _bf16_rows((B, T, H, D), 731)
    c, s = workloads.rope_tables(T, D)
    exact = oracle_mod.rotary(x, c, s)
    got = oracle_mod.rotary_f32(x, c, s)
    half = D // 2
    mag = np.abs(x[..., :half]) + np.abs(x[..., half:])
    bound = 2.0 ** -22 * np.concatenate([mag, mag], axis=-1) + 1e-30
    assert (np.abs(got - exact) <= bound).all()
