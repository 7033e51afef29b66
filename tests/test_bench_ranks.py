"""The replica path of bench.py (torchrun, N > 1) on CPU: two gloo ranks.
Every rank runs its own block (rank-offset prompt and embedding seeds, the
same weights), the job's clock is the max over ranks and its token count
sums the ranks; the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int) -> None:
    import bench
    import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # the job's clock: element-wise max of the ranks' times
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        got = bench.max_over_ranks(mine, world, "cpu")
        assert got == [float(world), 5.0, 0.25 * world], got
        # tokens of the whole job
        w = synth.WORKLOADS["tiny"]
        assert bench.job_tokens(w, 3, world) == w.b * w.n * 3 * world
        # each replica has its own inputs, and the same weights
        x = synth.prompt(w, device="cpu", seed_offset=rank)
        t = synth.decode_inputs(w, device="cpu", seed_offset=rank)
        wq = synth.layer_weights(w, 0, "cpu")["wq"]
        xs = [torch.zeros_like(x) for _ in range(world)]
        ts = [torch.zeros_like(t) for _ in range(world)]
        ws = [torch.zeros_like(wq) for _ in range(world)]
        dist.all_gather(xs, x)
        dist.all_gather(ts, t)
        dist.all_gather(ws, wq)
        assert not torch.equal(xs[0], xs[1]) and not torch.equal(ts[0], ts[1])
        assert torch.equal(ws[0], ws[1])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    port = _free_port()
    ctx = mp.start_processes(_rank_main, args=(2, port), nprocs=2, join=False, start_method="spawn")
    while not ctx.join(timeout=120):
        pass
    for p in ctx.processes:
        assert p.exitcode == 0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import argparse
    import bench
    import synth
    args = argparse.Namespace(gpus=2, steps=1, warmup=1)
    assert bench.run_reference(args, synth.WORKLOADS["tiny"], 1, 2) is None
    assert capsys.readouterr().out == ""
