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

