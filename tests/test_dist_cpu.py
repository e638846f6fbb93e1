"""The benchmark's multi-process plumbing on CPU: two gloo ranks on 127.0.0.1.

Every rank runs its own replica of the workload; the ranks only meet at a
barrier and a max-reduction of their step times (no collective touches the
attention data).  This exercises that code path without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    t = d.max(10.0 + rank)           # each rank's "step time"; the job time is the slowest rank's
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{d.rank} {d.world} {t}\n")
    d.close()


def test_two_rank_barrier_and_max(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    rows = sorted(open(tmp_path / f"rank{r}.txt").read().split() for r in range(world))
    assert [r[0] for r in rows] == ["0", "1"]
    assert all(r[1] == "2" for r in rows)
    assert all(float(r[2]) == 11.0 for r in rows)


def test_reference_arm_is_rank0_only(tmp_path, monkeypatch):
    """Under torchrun the reference arm prints on rank 0 and other ranks exit without work."""
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.main() == 0
