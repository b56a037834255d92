"""Host-side logic of the benchmark's multi-rank path, on CPU with gloo ranks:
the timing of a step is the slowest rank's, and the throughput counts every
rank's tokens (independent replicas, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 30.0 - 5 * rank]            # rank 0: (10, 30), rank 1: (11, 25)
    got = bench.max_over_ranks(mine, world, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == [11.0, 30.0] and out[1] == [11.0, 30.0]


def test_single_rank_and_throughput():
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    # 2 ranks x 64 tokens x 100 steps in 20 ms
    assert bench.tokens_per_s(2, 64, 100, 20.0) == pytest.approx(640000.0)
    assert bench.stage1_bytes(64, 6144, 8) == 8282112
    assert bench.stage2_bytes(64, 6144, 151552) == 931768576


def test_traffic_hash_ignores_comments_only():
    """The ncu traffic stays attached to a kernel through comment edits and is
    dropped by any code edit: the hash is over the code without comments."""
    src = 'asm("mov.b32 %0, %1; // not a comment");  // note\n/* block\n note */ int a = 1;\n\n'
    code = bench.strip_comments(src)
    assert code == 'asm("mov.b32 %0, %1; // not a comment");\n int a = 1;'
    assert bench.strip_comments(src.replace("note", "other words")) == code
    assert bench.strip_comments(src.replace("a = 1", "a = 2")) != code
    assert bench.strip_comments('s = "a\\"/*b*/"; /* c */') == 's = "a\\"/*b*/";'



def test_reference_arm_times_the_whole_workload_and_shares_the_config():
    """The reference arm (the oracle on the host's cores) computes the whole
    workload every step, so ms_per_step x steps is time it actually ran, and it
    prints the same config object as the GPU arm."""
    import argparse
    import time

    import synth
    args = argparse.Namespace(workload="tiny", variant="fp8", steps=2, warmup=1, mtp=1)
    t0 = time.perf_counter()
    r = bench.run_reference(args, 0, 1)
    wall = time.perf_counter() - t0
    w = synth.workload("tiny")
    assert r["impl"] == "reference" and r["steps"] == 2
    assert r["config"] == bench.bench_config(args, w, 1)
    assert set(r["config"]) >= {"workload", "variant", "l2", "parallelism", "weight_layout"}
    assert r["ms_per_step"] * r["steps"] <= wall * 1e3
    assert r["value"] == pytest.approx(w.T / (r["ms_per_step"] * 1e-3), rel=1e-3)
    assert "all 4096 vocab rows" in r["cpu_baseline"]["sample"]
