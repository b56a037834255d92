"""Sequence-parallel rows on the host: every token row is
owned by exactly one rank, and stage 1 run by each rank on its own rows
composes, across gloo ranks, to stage 1 on all rows (the oracle on CPU)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import norm_fp8_quant_gb300 as nfq


def test_row_ranges_partition_every_row():
    for T in (0, 1, 5, 64, 151, 8192):
        for world in (1, 2, 3, 8):
            ranges = [nfq.sp_row_range(T, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [r1 - r0 for r0, r1 in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        nfq.sp_row_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import oracle
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.workload("tiny", T=9, H=512, k=3, seed=2)
    r0, r1 = nfq.sp_row_range(w.T, rank, world)
    inp = synth.stage1_inputs(w, rows=list(range(r0, r1)))
    mine = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"], w.eps)
    gathered = [None] * world
    dist.all_gather_object(gathered, (r0, r1, mine))
    if rank == 0:
        out["parts"] = gathered
    dist.barrier()
    dist.destroy_process_group()


def test_stage1_on_sequence_parallel_ranks_composes():
    import oracle
    import synth
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
    w = synth.workload("tiny", T=9, H=512, k=3, seed=2)
    inp = synth.stage1_inputs(w)
    full = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"], w.eps)
    parts = sorted(out["parts"], key=lambda x: x[0])
    for key in ("hidden", "codes", "scales"):
        assert np.array_equal(np.concatenate([p[2][key] for p in parts]), full[key])
