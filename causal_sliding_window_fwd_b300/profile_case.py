"""Run one attention call a few times on seeded inputs, for profilers (ncu).

    python -m causal_sliding_window_fwd_b300.profile_case --op fwd --B 16 --T 2048 --H 10 --D 128 --window 2048
    python -m causal_sliding_window_fwd_b300.profile_case --op bwd ...
    python -m causal_sliding_window_fwd_b300.profile_case --op bwd_det ...   (nc_attn_bwd_deterministic)
    python -m causal_sliding_window_fwd_b300.profile_case --op decode --window 1024
    python -m causal_sliding_window_fwd_b300.profile_case --op prefill --window 1024   (prefill workload)
    python -m causal_sliding_window_fwd_b300.profile_case --op varlen_bwd --window 1024 (packed documents)
    python -m causal_sliding_window_fwd_b300.profile_case --op rope_fwd / rope_bwd ...  (rotary variants)

The inputs are made and the forward (needed by the backward) is run before
the profiled launches; ``--iters`` calls of the chosen op follow.
"""
from __future__ import annotations

import argparse
import math

import torch

from causal_sliding_window_fwd_b300 import nc_attn, workloads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", choices=["fwd", "bwd", "bwd_det", "decode", "prefill", "varlen_fwd", "varlen_bwd",
                                     "rope_fwd", "rope_bwd", "append"], default="fwd")
    ap.add_argument("--B", type=int, default=16)
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--H", type=int, default=10)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--window", type=int, default=2048)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--seed", type=int, default=101)
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    if a.op == "decode":
        wl = workloads.DECODE
        q, kc, vc, lens = workloads.make_decode(wl, dev)
        ws = torch.empty(nc_attn.nc_attn_decode_workspace_bytes(wl.N, wl.Tmax, wl.H, wl.D), dtype=torch.uint8,
                         device=dev)
        o = torch.empty((wl.N, wl.H, wl.D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.N, wl.H), dtype=torch.float32, device=dev)
        for _ in range(a.iters):
            nc_attn.nc_attn_decode(q, kc, vc, lens, o, lse, a.window, wl.scale, ws)
    elif a.op == "prefill":
        wl = workloads.PREFILL
        q, kc, vc, lens = workloads.make_prefill(wl, dev)
        o = torch.empty_like(q)
        lse = torch.empty((wl.N, wl.H, wl.Tq), dtype=torch.float32, device=dev)
        for _ in range(a.iters):
            nc_attn.nc_attn_prefill(q, kc, vc, lens, o, lse, a.window, wl.scale)
    elif a.op == "append":
        # the prefill workload's new tokens' keys and values into its caches
        wl = workloads.PREFILL
        q, kc, vc, lens = workloads.make_prefill(wl, dev)
        v_new = torch.empty_like(q).copy_(q)
        for _ in range(a.iters):
            nc_attn.nc_kv_append(q, v_new, kc, vc, lens)
    elif a.op in ("varlen_fwd", "varlen_bwd"):
        wl = workloads.VARLEN
        q, k, v, dO, cu, max_len = workloads.make_varlen(wl, dev)
        scale = 1.0 / math.sqrt(wl.D)
        o, lse = nc_attn.attn_fwd_varlen(q, k, v, cu, max_len, a.window, scale)
        if a.op == "varlen_fwd":
            for _ in range(a.iters):
                nc_attn.nc_attn_fwd_varlen(q, k, v, cu, o, lse, max_len, a.window, scale)
        else:
            total = q.shape[0]
            ws = torch.empty(nc_attn.nc_attn_bwd_workspace_bytes(1, total, wl.H, wl.D), dtype=torch.uint8, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            for _ in range(a.iters):
                nc_attn.nc_attn_bwd_varlen(q, k, v, o, dO, lse, cu, dq, dk, dv, max_len, a.window, scale, ws)
    elif a.op in ("rope_fwd", "rope_bwd"):
        scale = 1.0 / math.sqrt(a.D)
        q, k, v, dO = workloads.make_qkvdo_shape(a.B, a.T, a.H, a.D, a.seed, dev)
        c, s = workloads.rope_tables(a.T, a.D, device=dev)
        o, lse, qr, kr = nc_attn.attn_fwd_rotary(q, k, v, c, s, a.window, scale)
        if a.op == "rope_fwd":
            for _ in range(a.iters):
                nc_attn.nc_attn_fwd_rotary(q, k, v, c, s, qr, kr, o, lse, a.window, scale)
        else:
            ws = torch.empty(nc_attn.nc_attn_bwd_workspace_bytes(a.B, a.T, a.H, a.D), dtype=torch.uint8, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            for _ in range(a.iters):
                nc_attn.nc_attn_bwd_rotary(qr, kr, v, c, s, o, dO, lse, dq, dk, dv, a.window, scale, ws)
    else:
        scale = 1.0 / math.sqrt(a.D)
        q, k, v, dO = workloads.make_qkvdo_shape(a.B, a.T, a.H, a.D, a.seed, dev)
        o, lse = nc_attn.attn_fwd(q, k, v, a.window, scale)
        if a.op == "fwd":
            for _ in range(a.iters):
                nc_attn.nc_attn_fwd(q, k, v, o, lse, a.window, scale)
        else:
            ws = torch.empty(nc_attn.nc_attn_bwd_workspace_bytes(a.B, a.T, a.H, a.D), dtype=torch.uint8, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            fn = nc_attn.nc_attn_bwd_deterministic if a.op == "bwd_det" else nc_attn.nc_attn_bwd
            for _ in range(a.iters):
                fn(q, k, v, o, dO, lse, dq, dk, dv, a.window, scale, ws)
    torch.cuda.synchronize()
    assert nc_attn.nc_get_device_error() == 0
    print("done", a.op)


if __name__ == "__main__":
    main()
