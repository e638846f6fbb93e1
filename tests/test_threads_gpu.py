"""First calls from several host threads at once, in a fresh process.

The library keeps no per-device host state that a first call would set up: every
call looks up the kernel attribute, the SM count and the device addresses it needs.
Eight threads, each with its own CUDA stream, make the process's very first calls
into the library at the same time; each must get the result that a later call from a
single thread gets.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading, torch
sys.path.insert(0, sys.argv[1])
from causal_sliding_window_fwd_b300 import nc_attn, workloads
torch.cuda.set_device(0)
cases = [(1, 384, 2, 128, w) for w in (1, 64, 200, -1)] + [(2, 300, 1, 64, w) for w in (7, 129, 300, -1)]
inputs = [workloads.make_qkvdo_shape(B, T, H, D, seed=900 + i, device="cuda") for i, (B, T, H, D, w) in enumerate(cases)]
torch.cuda.synchronize()
outs = [None] * len(cases)
barrier = threading.Barrier(len(cases))
def run(i):
    B, T, H, D, w = cases[i]
    q, k, v, dO = inputs[i]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        barrier.wait()
        o, lse = nc_attn.attn_fwd(q, k, v, w, 1.0 / D ** 0.5, s)
        dq, dk, dv = nc_attn.attn_bwd(q, k, v, o, dO, lse, w, 1.0 / D ** 0.5, stream=s)
        s.synchronize()
    outs[i] = (o, lse, dq, dk, dv)
threads = [threading.Thread(target=run, args=(i,)) for i in range(len(cases))]
for t in threads: t.start()
for t in threads: t.join()
assert nc_attn.nc_get_device_error() == 0
for i, (B, T, H, D, w) in enumerate(cases):
    q, k, v, dO = inputs[i]
    o, lse = nc_attn.attn_fwd(q, k, v, w, 1.0 / D ** 0.5)
    dq, dk, dv = nc_attn.attn_bwd(q, k, v, o, dO, lse, w, 1.0 / D ** 0.5)
    torch.cuda.synchronize()
    got = outs[i]
    assert torch.equal(got[0], o) and torch.equal(got[1], lse), i
    assert torch.equal(got[3], dk) and torch.equal(got[4], dv), i
    assert (got[2].float() - dq.float()).abs().max().item() <= 1e-2 * dq.float().abs().max().item() + 1e-6, i
print("threads ok")
'''


@pytest.mark.gpu
def test_first_calls_from_eight_threads():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
