"""The benchmark's multi-rank path on CPU: two gloo ranks on this host.

On GPUs every rank is an independent replica (weak scaling: the decode has no
exchange step), so the only cross-rank work is the timing protocol: a barrier
on both sides of the timed region, the max of the elapsed times over ranks,
and the whole-job microseconds per call computed from it.  These tests run
that protocol with world size 2 over gloo.
"""
import os
import socket
import time

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # max over ranks of a per-rank value
        got = bench.reduce_max(1.5 + rank, world)
        assert got == 1.5 + world - 1
        # the timed-region protocol: ranks that take different times report the slowest one
        bench.barrier(world)
        t0 = time.perf_counter()
        time.sleep(0.05 * (rank + 1))
        el = time.perf_counter() - t0
        bench.barrier(world)
        slowest = bench.reduce_max(el, world)
        assert slowest >= el
        assert slowest >= 0.05 * world
        # replicas draw different inputs with the same recipe
        from sparse_mla_decode_paged_gb300 import workloads as wl
        spec = bench.replica_spec("tiny", rank)
        wk = wl.make_workload(spec, device="cpu")
        sig = torch.tensor([float(wk.topk_idx.to(torch.float64).sum()), float(wk.q.float().sum())],
                           dtype=torch.float64)
        sigs = [torch.zeros_like(sig) for _ in range(world)]
        dist.all_gather(sigs, sig)
        assert not torch.equal(sigs[0], sigs[1])
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{slowest!r} {wk.B} {wk.H} {wk.topk}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_timing_protocol(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    lines = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    # every rank saw the same max
    assert lines[0][0] == lines[1][0]
    # and the same shape of work (weak scaling: per-rank work is fixed)
    assert lines[0][1:] == lines[1][1:]


def test_aggregate_us_per_call_counts_all_ranks():
    # 2 ranks, 1000 calls each, slowest rank 10 ms: 2000 calls in 10 ms, 5 us per call for the whole job
    assert bench.aggregate_us_per_call(0.010, 1000, 2) == pytest.approx(5.0)
    assert bench.aggregate_us_per_call(0.010, 1000, 1) == pytest.approx(10.0)
    # doubling ranks with per-rank work fixed halves the whole-job time per call at equal elapsed time
    for n in (1, 2, 4, 8):
        assert bench.aggregate_us_per_call(0.020, 500, n) * n == pytest.approx(40.0)


def test_single_rank_helpers_are_identity():
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)   # no process group: must not need one


def test_replica_spec_rank0_keeps_configuration():
    from sparse_mla_decode_paged_gb300 import workloads as wl
    for name in bench.ALL_CONFIGS:
        assert bench.replica_spec(name, 0) == wl.CONFIGS[name]
        s1 = bench.replica_spec(name, 1)
        assert s1.seed != wl.CONFIGS[name].seed
        assert (s1.B, s1.H, s1.topk) == (wl.CONFIGS[name].B, wl.CONFIGS[name].H, wl.CONFIGS[name].topk)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        workload, steps, warmup = "tiny", 1, 3
    bench.main_reference(A())
    assert capsys.readouterr().out == ""
