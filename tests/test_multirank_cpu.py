"""The multi-process (N > 1) path of bench.py on the CPU: two gloo ranks on
127.0.0.1.  Each rank draws its own batch (weak scaling: the path shards by
independent sequences, with no data-path collective), and the timing is the
maximum over the ranks (the only collective)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import bench
    from linear_recurrence_sequence_gb300 import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 1.0 + 1.5 * rank                 # a per-rank "step time"
        total = bench.reduce_max(local_ms, world)   # max over ranks
        seed = bench.shard_seed(0, rank)
        inp = synth.samu_inputs(1, 8, 16, seed, h0=False)
        np.save(os.path.join(out_dir, f"x{rank}.npy"), inp["x_sel"])
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{total} {seed}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_independent_batches(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    vals = [open(tmp_path / f"r{r}.txt").read().split() for r in range(world)]
    totals = [float(v[0]) for v in vals]
    seeds = [int(v[1]) for v in vals]
    assert totals == [2.5, 2.5]                      # every rank sees the max over ranks
    assert seeds[0] != seeds[1]
    x0, x1 = np.load(tmp_path / "x0.npy"), np.load(tmp_path / "x1.npy")
    assert not np.array_equal(x0, x1)                # independent batches per rank


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0


def test_reduce_max_is_identity_on_one_process():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
