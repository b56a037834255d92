"""Benchmark of the MTP draft-layer tail on GB300.

One step = one pass of the whole hot path over one batch of the decode c=64
draft step (GLM-5.2 shapes): T=64 tokens, hidden 6144, k=8 BF16 partials with
1% outlier channels x20, residual, RMSNorm, packed FP8 activation, then the
FP8 LM head over vocab 151552 in 8 shards with the fused greedy argmax.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is draft tokens/s of K steps run one
after another on one stream with inputs resident in HBM, timed by CUDA events
at the two ends; the K-step run is repeated (`repeats`: by default enough
repeats for about 0.4 s of timed steps, 5 to 200) and `value` is the median,
with the spread in `repeats`.  The per-kernel durations behind
`norm_quant`, `lm_head` and `roofline` come from a further run of the K steps
with CUDA events around every launch (`instrumented_ms_per_step`);
`norm_quant.graph_us` times stage 1 alone from a CUDA graph of back-to-back
launches over the rotating inputs.  `e2e` repeats the measurement through the public API
with each step's stage-1 inputs copied from pinned host memory (on a copy
stream, overlapping the previous step's kernels) and its tokens read back.  Each step reads the
932 MB FP8 LM-head weight (> L2) and a different one of 40 rotating stage-1
input sets (283 MB in all), so no step is served from L2.  --workload picks
another of the five workloads (prefill runs the norm + quant stage alone).
With N > 1 (torchrun) every rank runs the same workload on its own GPU
(independent replicas, weak scaling; the only collectives are the timing
barrier and the max over ranks).

--impl reference times the CPU oracle instead (rank 0 only): each step is the
whole workload (stage 1 on every row, the LM head for every token over the
full vocabulary), its independent outputs split over the host's cores.

--stage1-sweep times stage 1 alone from CUDA graphs at T = 1 .. 8192 rows of
the decode c=64 shape and prints one JSON line with GB/s and the fraction of
the measured HBM peak per batch size.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "decode_c64"
METRIC = "norm+FP8-quant GB/s; LM-head+argmax draft tokens/s; % of GB300 roofline"
ROTATION_BYTES = 280_000_000   # stage-1 input sets rotated per step: > 2 x L2
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mtp", type=int, default=1,
                    help="draft positions per step (the hidden of each feeds the next)")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["decode_c64", "decode_c1", "prefill", "tie_stress", "tiny"])
    ap.add_argument("--variant", choices=["fp8", "nvfp4", "unfused"], default="fp8",
                    help="packed FP8 path (default), its NVFP4 form, or the unfused "
                         "reference arm (separate kernels, BF16 logits, full-vocab argmax)")
    ap.add_argument("--repeats", type=int, default=0,
                    help="times the K-step run is repeated, value being the median "
                         "(0: enough repeats for about 0.4 s of timed steps, 5 to 200)")
    ap.add_argument("--stage1-sweep", action="store_true",
                    help="stage 1 alone, CUDA-graph timed, at T = 1 .. 8192 (c=64 shape)")
    ap.add_argument("--probe-mma", action="store_true",
                    help="FP8 tcgen05 MMA rate from shared memory (the tensor roofline)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------ bytes & peaks --

def stage1_bytes(T, H, k):
    """Algorithmic HBM bytes of one stage-1 launch: k partials + residual +
    norm weight read; BF16 hidden, e4m3 codes and fp32 group scales written."""
    return k * T * H * 2 + T * H * 2 + H * 2 + T * H * 2 + T * H + T * (H // 128) * 4


def stage2_bytes(T, H, V):
    """Algorithmic HBM bytes of one LM-head launch: FP8 weight + block scales,
    activation codes + scales read; int32 tokens written."""
    G = H // 128
    return V * H + ((V + 127) // 128) * G * 4 + T * H + T * G * 4 + T * 4


def stage1_bytes_nvfp4(T, H, k):
    """Stage 1 with the NVFP4 activation: the same reads; BF16 hidden, e2m1
    codes (H/2 bytes a row), e4m3 block scales (H/16) and fp32 row scales written."""
    return k * T * H * 2 + T * H * 2 + H * 2 + T * H * 2 + T * H // 2 + T * H // 16 + T * 4


def stage2_bytes_nvfp4(T, H, V):
    """NVFP4 LM head: e2m1 weight codes and e4m3 block scales (9/16 byte per
    weight), the activation's codes, block scales and row scales read; int32
    tokens written."""
    return V * H // 2 + V * H // 16 + T * H // 2 + T * H // 16 + T * 4 + T * 4


def stage1_bytes_unfused(T, H, k):
    """The unfused stage 1: BF16 all-reduce (k partials in, sum out), add +
    RMSNorm (sum and residual in, hidden out), group quantisation (hidden in,
    codes and scales out)."""
    return (k * T * H * 2 + T * H * 2) + (3 * T * H * 2 + H * 2) + \
        (T * H * 2 + T * H + T * (H // 128) * 4)


def stage2_bytes_unfused(T, H, V):
    """The unfused LM head: the FP8 LM head's reads plus BF16 logits written and
    read back by the full-vocab argmax."""
    return stage2_bytes(T, H, V) + 2 * T * V * 2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def strip_comments(text):
    """C/C++/CUDA source without its comments, trailing blanks and blank lines
    (string literals kept as they are)."""
    out, i, n, in_str = [], 0, len(text), False
    while i < n:
        c = text[i]
        if in_str:
            out.append(text[i:i + 2] if c == "\\" else c)
            i += 2 if c == "\\" else 1
            in_str = c != '"'
            continue
        if c == '"':
            in_str = True
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(files):
    """Hash of the kernel sources' code: a change to comments alone keeps it."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "norm_fp8_quant_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu capture, if it was taken on
    the kernel source as it stands (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)[kernel]
        srcs = d["sources"]
        if d["source_hash"] != kernel_source_hash(srcs):
            return None
        return d["dram_bytes_per_launch"]
    except Exception:
        return None


# ------------------------------------------------------------- aggregation --

def max_over_ranks(values, world, device):
    """Element-wise max of per-rank floats (timings) across the process group."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def tokens_per_s(world, T, K, ms):
    """Whole-job draft tokens per second: every rank processed T tokens per step."""
    return world * T * K / (ms * 1e-3)


# ------------------------------------------------------------------ clocks --

REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 100 ms."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 5:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[3], int(parts[4], 16)))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside and rows:   # timed region shorter than the sampling period
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        mhz = sorted(r[1] for r in inside)
        mask = 0
        for r in inside:
            mask |= r[4]
        reasons = [n for b, n in REASON_BITS.items() if mask & b and b != 0x1]
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": inside[0][2], "reasons": reasons,
                "samples": len(inside)}


# -------------------------------------------------------------- our impl --

WORKLOAD_TEXT = {
    "decode_c64": "decode c=64 draft step (GLM-5.2 shapes): T=64, hidden=6144, k=8 BF16 partials "
                  "N(0,0.5) with 1% outlier channels x20, vocab=151552 in 8 shards, "
                  "128x128-block FP8 LM head",
    "decode_c1": "decode c=1 draft step (DeepSeek-V3.2 shapes): T=1, hidden=7168, k=8, "
                 "vocab=129280 in 8 shards",
    "prefill": "prefill bandwidth: T=8192, hidden=7168, k=8, norm + quant only",
    "tie_stress": "tie stress: T=256, hidden=6144, k=4, vocab=151552 in 8 shards",
    "tiny": "tiny: T=4, hidden=1024, k=2, vocab=4096 in 2 shards",
}


def rotation_sets(w):
    """Stage-1 input sets rotated over the timed steps (> 2 x L2 in all)."""
    set_bytes = (w.k + 1) * w.T * w.H * 2
    return int(min(64, max(2, -(-ROTATION_BYTES // set_bytes)))), set_bytes


def bench_config(args, w, world):
    """The `config` object of the JSON line; both arms print the same one."""
    fp4 = args.variant == "nvfp4"
    unfused = args.variant == "unfused"
    nsets, set_bytes = rotation_sets(w)
    cfg = {"workload": WORKLOAD_TEXT.get(args.workload, args.workload)
                       + ("; NVFP4 activation and LM head" if fp4 else
                          "; unfused reference arm: BF16 all-reduce, add+RMSNorm, "
                          "quant, BF16 logits, full-vocab argmax" if unfused else ""),
           "variant": args.variant,
           "draft_positions_per_step": max(1, args.mtp) if w.V > 0 and not unfused else 1,
           "l2": f"inputs larger than L2: {nsets} rotating stage-1 input sets "
                 f"({nsets * set_bytes / 1e6:.0f} MB)"
                 + (f", {(stage2_bytes_nvfp4(w.T, w.H, w.V) if fp4 else stage2_bytes(w.T, w.H, w.V)) / 1e6:.0f}"
                    f" MB {'NVFP4' if fp4 else 'FP8'} weight read every step" if w.V > 0 else ""),
           "parallelism": f"replicas x{world}"}
    if w.V > 0:
        cfg["weight_layout"] = ("packed once at load: tile-contiguous, pre-swizzled 16 KB blocks "
                                "of 128 rows x 128 bytes" + (" + 2 KB block-scale blocks" if fp4 else ""))
    return cfg


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import norm_fp8_quant_gb300 as nfq
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = synth.workload(args.workload)
    T, H, k, V, S = w.T, w.H, w.k, w.V, w.S
    has_lm = V > 0

    # inputs: stage-1 tensors in rotating device copies (more than twice L2 in
    # all), and the LM head weight packed once into the streaming layout
    inp = synth.stage1_inputs(w)
    to_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    host_parts = [to_bf16(p).pin_memory() for p in inp["partials"]]
    host_res = to_bf16(inp["residual"]).pin_memory()
    norm_w = to_bf16(inp["norm_w"]).to(dev)
    nsets, set_bytes = rotation_sets(w)
    sets = [([p.to(dev) for p in host_parts], host_res.to(dev)) for _ in range(nsets)]
    fp4 = args.variant == "nvfp4"
    unfused = args.variant == "unfused"
    if has_lm and not fp4:
        qw, sw = synth.lm_head_weights(w)
        qw_rowmajor = torch.from_numpy(qw).to(dev)
        sw_d = torch.from_numpy(sw).to(dev)
        del qw
        qw_d = nfq.pack_lm_head_weights(qw_rowmajor)
        torch.cuda.synchronize()
        del qw_rowmajor
    if has_lm and fp4:
        qw, sw, gw = synth.lm_head_weights_nvfp4(w)
        qw_d = nfq.pack_lm_head_weights_nvfp4(torch.from_numpy(qw).to(dev),
                                              torch.from_numpy(sw).to(dev), gw)
        torch.cuda.synchronize()
        del qw, sw
    if has_lm:
        ws = nfq.lm_head_workspace(T, S, dev)
    hidden = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    codes = torch.empty((T, H // 2 if fp4 else H), dtype=torch.uint8, device=dev)
    scales = torch.empty((T, H // 128), dtype=torch.float32, device=dev)
    bscales = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)
    gscales = torch.empty(T, dtype=torch.float32, device=dev)
    tokens = torch.empty(T, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    # every call of the timed loops goes through the public API as a prepared
    # call (arguments checked and marshalled once, per buffer set)
    def prepare_stage1(parts, res):
        if fp4:
            return nfq.prepare_reduce_norm_quant_nvfp4(parts, res, norm_w, w.eps, hidden, codes,
                                                       bscales, gscales)
        return nfq.prepare_reduce_norm_quant(parts, res, norm_w, w.eps, hidden, codes, scales)

    stage1_calls = {}

    def stage1(parts, res):
        key = id(res)
        if key not in stage1_calls:
            stage1_calls[key] = prepare_stage1(parts, res)
        stage1_calls[key]()

    if has_lm:
        stage2 = (nfq.prepare_lm_head_nvfp4_argmax(codes, bscales, gscales, qw_d, S, ws, tokens)
                  if fp4 else nfq.prepare_lm_head_fp8_argmax(codes, scales, qw_d, sw_d, S, ws,
                                                             tokens))
    if unfused:
        # the unfused reference arm: five separate kernels a step
        s_sum = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        logits = torch.empty((T, V), dtype=torch.bfloat16, device=dev) if has_lm else None

        def stage1(parts, res):
            nfq.unfused_allreduce_bf16(parts, out=s_sum)
            nfq.unfused_add_rmsnorm(s_sum, res, norm_w, w.eps, hidden_out=hidden)
            nfq.unfused_quant_fp8(hidden, codes_out=codes, scales_out=scales)

        def stage2():
            nfq.unfused_lm_head_logits(codes, scales, qw_d, sw_d, logits_out=logits)
            nfq.unfused_argmax_bf16(logits, tokens_out=tokens)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        stage1(*sets[i % nsets])
        if has_lm:
            stage2()
    barrier()
    if nfq.device_error() != nfq.NFQ_OK:
        raise RuntimeError("a kernel reported an expired wait during warm-up")

    K = args.steps
    for i in range(args.warmup):
        stage1(*sets[i % nsets])
        if has_lm:
            stage2()
    barrier()
    if nfq.device_error() != nfq.NFQ_OK:
        raise RuntimeError("a kernel reported an expired wait during warm-up")

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    t_wall0 = time.time()

    # (1) K steps one after another on one stream, events only at the two ends
    # (an event between two kernels would stop the second one's launch from
    # overlapping the first one's tail): the reported rate.  With --mtp P a
    # step is P chained draft positions: position p's hidden is the residual
    # of position p+1 (nfq_mtp_draft_chain), each position with its own partials.
    P = max(1, args.mtp) if has_lm and not unfused else 1
    if P > 1:
        chain_hidden = [torch.empty_like(hidden) for _ in range(2)]
        chain_tokens = torch.empty((P, T), dtype=torch.int32, device=dev)

        def chain(i):
            parts = [sets[(i * P + p) % nsets][0] for p in range(P)]
            if fp4:
                nfq.mtp_draft_chain_nvfp4(parts, sets[(i * P) % nsets][1], norm_w, qw_d, S, w.eps,
                                          hidden_bufs=chain_hidden, codes=codes,
                                          block_scales=bscales, row_scales=gscales,
                                          tokens_out=chain_tokens, workspace=ws)
            else:
                nfq.mtp_draft_chain(parts, sets[(i * P) % nsets][1], norm_w, qw_d, sw_d, S,
                                    w.eps, hidden_bufs=chain_hidden, codes=codes, scales=scales,
                                    tokens_out=chain_tokens, workspace=ws)
        for i in range(max(1, args.warmup // P)):
            chain(i)
    # the K-step run, repeated: each repeat times exactly K steps between
    # barriers; the reported value is the median repeat
    rep_ms = []
    n_rep = max(1, args.repeats) if args.repeats > 0 else 200
    while len(rep_ms) < n_rep:
        barrier()
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        for i in range(K):
            if P > 1:
                chain(i)
            else:
                stage1(*sets[i % nsets])
                if has_lm:
                    stage2()
        e_end.record(stream)
        barrier()
        rep_ms.append(e_start.elapsed_time(e_end))
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("a kernel reported an expired wait during the timed steps")
        if args.repeats <= 0 and len(rep_ms) == 1:   # about 0.4 s of timed steps in all
            n_rep = int(min(200, max(5, -(-400.0 // max(rep_ms[0], 1e-3)))))
            if world > 1:                            # every rank runs the same count
                n_rep = int(max_over_ranks([float(n_rep)], world, dev)[0])
    total_ms = sorted(rep_ms)[len(rep_ms) // 2]

    # (2) the same K steps with CUDA events around every launch: per-kernel
    # durations for the roofline
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier()
    for i in range(K):
        ev[i][0].record(stream)
        stage1(*sets[i % nsets])
        ev[i][1].record(stream)
        if has_lm:
            stage2()
        ev[i][2].record(stream)
    barrier()
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None
    if nfq.device_error() != nfq.NFQ_OK:
        raise RuntimeError("a kernel reported an expired wait during the timed steps")
    instrumented_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    s1_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    s2_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K

    # (3) the same steps replayed from one CUDA graph (one step per rotating
    # input set; with --mtp P one chained P-position step per capture): the
    # step time without host launch overhead
    launches_per_step = ((5 if has_lm else 3) if unfused else (2 if has_lm else 1)) * P

    def graph_time(body, n_bodies):
        """ms per body of a CUDA graph holding n_bodies calls, replayed."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(n_bodies):
                body(j)
        g.replay()
        barrier()
        reps = max(3, -(-K // n_bodies))
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        barrier()
        del g
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("a kernel reported an expired wait in a graph replay")
        return g0.elapsed_time(g1) / (reps * n_bodies), reps * n_bodies

    def one_step(j):
        if P > 1:
            chain(j)
        else:
            stage1(*sets[j])
            if has_lm:
                stage2()
    n_graph = nsets if P == 1 else max(1, nsets // P)
    graph_ms, graph_steps = graph_time(one_step, n_graph)
    gpu_launches_graph = launches_per_step * graph_steps
    # stage 1 alone from a graph of back-to-back launches
    s1_graph_ms, _ = graph_time(lambda j: stage1(*sets[j]), nsets)
    gpu_launches = launches_per_step * K

    # end to end through the public API: every step copies its stage-1 inputs
    # (one pinned host batch holding the k partials and the residual) to the
    # device, runs both stages and reads its result back (tokens, or the group
    # scales when there is no LM head).  The copy of step i+1 runs on a copy
    # stream while step i's kernels run on the compute stream (three input
    # buffers in rotation); kernels of different steps never overlap.  The
    # host reads step i's result after enqueuing step i+1.
    h_in = torch.empty((k + 1, T, H), dtype=torch.bfloat16).pin_memory()
    for i in range(k):
        h_in[i].copy_(host_parts[i])
    h_in[k].copy_(host_res)
    copy_stream = torch.cuda.Stream(device=dev)
    NB = 3                                     # input buffers / result slots in rotation
    bufs = [torch.empty((k + 1, T, H), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    copied = [torch.cuda.Event() for _ in range(NB)]
    result_dev = tokens if has_lm else (gscales if fp4 else scales)
    result_host = [torch.empty(result_dev.shape, dtype=result_dev.dtype).pin_memory()
                   for _ in range(NB)]
    # the LM head writes each step's tokens straight into that step's pinned
    # host slot (the device addresses pinned memory directly), so no copy node
    # sits between the kernels of consecutive steps
    direct = has_lm and not unfused
    if direct:
        stage2_direct = [
            (nfq.prepare_lm_head_nvfp4_argmax(codes, bscales, gscales, qw_d, S, ws, result_host[b])
             if fp4 else nfq.prepare_lm_head_fp8_argmax(codes, scales, qw_d, sw_d, S, ws,
                                                        result_host[b]))
            for b in range(NB)]
    done = [torch.cuda.Event() for _ in range(NB)]
    h2d = h_in.numel() * h_in.element_size()
    d2h = result_dev.numel() * result_dev.element_size()

    def e2e_copy(i):
        b = i % NB
        with torch.cuda.stream(copy_stream):
            if i >= NB:
                copy_stream.wait_event(done[b])    # step i-NB is finished with the buffer
            bufs[b].copy_(h_in, non_blocking=True)
            copied[b].record()

    buf_views = [([bufs[b][j] for j in range(k)], bufs[b][k]) for b in range(NB)]

    def e2e_compute(i):
        b = i % NB
        stream.wait_event(copied[b])
        stage1(*buf_views[b])
        if direct:
            stage2_direct[b]()
        else:
            if has_lm:
                stage2()
            result_host[b].copy_(result_dev, non_blocking=True)
        done[b].record(stream)

    def e2e_read(i):
        done[i % NB].synchronize()
        return int(result_host[i % NB].view(-1)[0].item())

    def e2e_run(n):
        e2e_copy(0)
        for i in range(n):
            if i + 1 < n:
                e2e_copy(i + 1)
            e2e_compute(i)
            if i >= 1:
                e2e_read(i - 1)
        e2e_read(n - 1)

    e2e_steps = K if set_bytes < (1 << 28) else max(3, min(K, 20))
    e2e_run(max(3, min(args.warmup, 20)))
    barrier()
    c0 = time.perf_counter()
    e2e_run(e2e_steps)
    e2e_ms = (time.perf_counter() - c0) * 1e3
    barrier()

    total_ms, e2e_ms, graph_ms, s1_graph_ms = max_over_ranks(
        [total_ms, e2e_ms, graph_ms, s1_graph_ms], world, dev)
    rep_ms = max_over_ranks(rep_ms, world, dev)

    result = None
    if rank == 0:
        peak, peak_kind = load_peaks()
        b1 = (stage1_bytes_nvfp4(T, H, k) if fp4 else
              stage1_bytes_unfused(T, H, k) if unfused else stage1_bytes(T, H, k))
        gbs1 = b1 / (s1_ms * 1e-3) / 1e9
        value = tokens_per_s(world, T * P, K, total_ms)
        gbs1g = b1 / (s1_graph_ms * 1e-3) / 1e9
        rep_steps = sorted(x / K for x in rep_ms)
        result = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "draft tokens/s" if has_lm else "tokens/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(total_ms / K, 5),
            "repeats": {"n": len(rep_ms), "ms_per_step_median": round(total_ms / K, 5),
                        "ms_per_step_min": round(rep_steps[0], 5),
                        "ms_per_step_max": round(rep_steps[-1], 5),
                        "value_min": round(tokens_per_s(world, T * P, K, rep_steps[-1] * K), 1),
                        "value_max": round(tokens_per_s(world, T * P, K, rep_steps[0] * K), 1)},
            "draft_positions_per_step": P,
            "instrumented_ms_per_step": round(instrumented_ms / K, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("e2m1 MMA with e4m3 block-16 scales (NVFP4), fp32 accumulate; bf16 in, "
                      "fp32 norm" if fp4 else "e4m3 MMA, fp32 accumulate; bf16 in, fp32 norm"),
            "data": "synthetic",
            "config": bench_config(args, w, world),
            "norm_quant": {"us": round(s1_ms * 1e3, 3), "GB/s": round(gbs1, 1),
                           "frac": round(gbs1 / peak, 4), "bytes": b1,
                           "graph_us": round(s1_graph_ms * 1e3, 3),
                           "graph_GB/s": round(gbs1g, 1), "graph_frac": round(gbs1g / peak, 4),
                           "traffic": (ncu_traffic("norm_quant_nvfp4" if fp4 else "norm_quant")
                                       if args.workload == WORKLOAD and not unfused else None)},
            "e2e": {"value": round(tokens_per_s(world, T, e2e_steps, e2e_ms), 1),
                    "unit": "draft tokens/s" if has_lm else "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": gpu_launches,
            "clocks": clocks,
        }
        result["graph"] = {"ms_per_step": round(graph_ms, 5),
                           "value": round(tokens_per_s(world, T * P, 1, graph_ms), 1),
                           # positive: what host launches cost over a graph replay
                           "stream_minus_graph_us_per_step": round((total_ms / K - graph_ms) * 1e3, 2),
                           "gpu_launches": gpu_launches_graph}
        if has_lm:
            b2 = (stage2_bytes_nvfp4(T, H, V) if fp4 else
                  stage2_bytes_unfused(T, H, V) if unfused else stage2_bytes(T, H, V))
            gbs2 = b2 / (s2_ms * 1e-3) / 1e9
            result["lm_head"] = {"us": round(s2_ms * 1e3, 3), "GB/s": round(gbs2, 1),
                                 "frac": round(gbs2 / peak, 4), "bytes": b2,
                                 "draft_tokens_per_s": round(T / (s2_ms * 1e-3), 1)}
            result["roofline"] = {"bound": "hbm", "achieved": round(gbs2, 1), "peak": peak,
                                  "unit": "GB/s", "frac": round(gbs2 / peak, 4),
                                  "traffic": (ncu_traffic("lm_head_nvfp4" if fp4 else "lm_head")
                                              if args.workload == WORKLOAD and not unfused
                                              else ncu_traffic("lm_head_nvfp4_tie_stress"
                                                               if fp4 else "lm_head_tie_stress")
                                              if args.workload == "tie_stress" and not unfused
                                              else ncu_traffic("lm_head_decode_c1")
                                              if args.workload == "decode_c1" and not fp4
                                              and not unfused else None),
                                  "kernel": ("lm_head_fp4_kernel" if fp4 and T <= 128 else
                                             "lm_head_fp4_pair_kernel (CTA pairs, cta_group::2)"
                                             if fp4 and T <= 256 else
                                             f"lm_head_fp4 x {(T + 255) // 256}" if fp4 else
                                             "lm_head_small_kernel (BF16 logits) + "
                                             "unfused_argmax_kernel" if unfused else
                                             "lm_head_small_kernel" if T <= 128 else
                                             "lm_head_pair_kernel (CTA pairs, cta_group::2)"
                                             if T <= 256 else
                                             f"lm_head_small_kernel x {(T + 255) // 256}"),
                                  "peak_source": peak_kind}
        else:
            result["roofline"] = {"bound": "hbm", "achieved": round(gbs1, 1), "peak": peak,
                                  "unit": "GB/s", "frac": round(gbs1 / peak, 4),
                                  "traffic": (ncu_traffic("norm_quant_prefill")
                                              if args.workload == "prefill" and not fp4
                                              and not unfused else None),
                                  "kernel": ("reduce_norm_quant_kernel (persistent)" if T > 512
                                             else "stage1_split_kernel"),
                                  "peak_source": peak_kind}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


# ------------------------------------------------------------ CPU oracle --

def oracle_threads():
    return max(1, min(64, os.cpu_count() or 1))


def _split(n, parts):
    """[0, n) as up to `parts` contiguous non-empty ranges."""
    parts = max(1, min(parts, n))
    return [(i * n // parts, (i + 1) * n // parts) for i in range(parts)]


def oracle_sample(w, inp, qw, sw, rows, tokens, threads=1, gw=None):
    """Oracle time of stage 1 on the sampled rows plus the LM head for `tokens`
    over `rows` vocab rows; returns (seconds, seconds for the whole step).

    With threads > 1 the independent outputs are split over host threads: the
    token rows of stage 1, then the vocab rows of the LM head.  Every output keeps its own fixed order, so
    the results are the same; the oracle's C calls release the interpreter lock."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    fp4 = gw is not None                           # the NVFP4 variant of both stages
    stage1 = oracle.reduce_norm_quant_nvfp4 if fp4 else oracle.reduce_norm_quant
    R = inp["partials"].shape[1]
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        outs = list(pool.map(
            lambda ab: stage1(inp["partials"][:, ab[0]:ab[1]], inp["residual"][ab[0]:ab[1]],
                              inp["norm_w"], w.eps),
            _split(R, threads)))
        t1 = time.perf_counter()
        if qw is None:
            return t1 - t0, (t1 - t0) * w.T / R
        cat = lambda key: np.concatenate([o[key] for o in outs])
        tok = np.asarray(tokens, np.int32)
        jobs = [(tok, a, b) for a, b in _split(rows, threads)]
        if fp4:
            codes, bs, gs = cat("codes"), cat("block_scales"), cat("global_scales")
            head = lambda j: oracle.lm_head_logits_nvfp4(codes, bs, gs, qw[:rows], sw[:rows], gw,
                                                         tokens=j[0], v0=j[1], v1=j[2])
        else:
            codes, scales = cat("codes"), cat("scales")
            head = lambda j: oracle.lm_head_logits(codes, scales, qw[:rows],
                                                   sw[: (rows + 127) // 128],
                                                   tokens=j[0], v0=j[1], v1=j[2])
        list(pool.map(head, jobs))
        t2 = time.perf_counter()
    full = (t1 - t0) + (t2 - t1) * (w.V / rows)     # whole step, all T tokens
    return t2 - t0, full


def sample_weights(name, rows, fp4):
    """The first `rows` vocab rows of the workload's LM-head weight (the
    generator draws rows in order), FP8 (codes, scales, None) or NVFP4
    (codes, block scales, tensor scale of the sample)."""
    import synth
    ww = synth.workload(name, V=rows, S=1)
    if fp4:
        return synth.lm_head_weights_nvfp4(ww)
    qw, sw = synth.lm_head_weights(ww)
    return qw, sw, None


def cpu_baseline(name, variant="fp8"):
    import synth
    w = synth.workload(name)
    n = oracle_threads()
    fp4 = variant == "nvfp4"
    g1 = 1.0 if fp4 else None
    if w.V == 0:
        rows = list(range(min(w.T, 2048)))
        inp = synth.stage1_inputs(w, rows=rows)
        _, full1 = oracle_sample(w, inp, None, None, 0, None, threads=1, gw=g1)
        secs, full = oracle_sample(w, inp, None, None, 0, None, threads=n, gw=g1)
        return {"value": round(w.T / full, 2), "unit": "tokens/s", "cores": n, "kind": "oracle",
                "single_thread_value": round(w.T / full1, 2),
                "sample": f"stage 1 on {len(rows)} of {w.T} rows, rows split over {n} host "
                          f"threads ({secs:.1f} s), scaled to all rows"}
    inp = synth.stage1_inputs(w)
    rows = min(w.V, 8 * (w.V // w.S)) if w.V >= 4096 else w.V
    qw, sw, gw = sample_weights(name, rows, fp4)
    toks = list(range(w.T))
    secs, full = oracle_sample(w, inp, qw, sw, rows, toks, threads=n, gw=gw)
    rows1 = max(128, rows // 32)
    secs1, full1 = oracle_sample(w, inp, qw, sw, rows1, toks, threads=1, gw=gw)
    return {"value": round(w.T / full, 4), "unit": "draft tokens/s", "cores": n,
            "kind": "oracle",
            "single_thread_value": round(w.T / full1, 4),
            "sample": f"stage 1 on all {w.T} rows + LM head for all {w.T} tokens over "
                      f"{rows} of {w.V} vocab rows, outputs split over {n} host threads "
                      f"({secs:.1f} s; single thread: {rows1} rows, {secs1:.1f} s), "
                      f"scaled to the full vocab"}


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host's cores over the whole
    workload every step: stage 1 on every row, then the LM head for every token
    over the full vocabulary (outputs split over threads, each in its fixed
    order), so that ms_per_step x steps is the time the arm ran."""
    if rank != 0:
        return None
    import synth
    w = synth.workload(args.workload)
    has_lm = w.V > 0
    fp4 = args.variant == "nvfp4"
    n = oracle_threads()
    inp = synth.stage1_inputs(w)
    if has_lm:
        qw, sw, gw = sample_weights(args.workload, w.V, fp4)
        rows, toks = w.V, list(range(w.T))
        sample = (f"per step: stage 1 on all {w.T} rows + LM head for all {w.T} tokens over all "
                  f"{w.V} vocab rows")
    else:
        qw = sw = None
        gw = 1.0 if fp4 else None
        rows, toks = 0, None
        sample = f"per step: stage 1 on all {w.T} rows"
    for _ in range(args.warmup):
        oracle_sample(w, inp, qw, sw, rows, toks, threads=n, gw=gw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(w, inp, qw, sw, rows, toks, threads=n, gw=gw)
    elapsed = time.perf_counter() - t0
    full = elapsed / max(1, args.steps)
    value = w.T / full                    # one draft position per step: T tokens
    unit = "draft tokens/s" if has_lm else "tokens/s"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4),
            "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(full * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp32 (fp64 norm)", "data": "synthetic",
            "config": bench_config(args, w, world),
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": n,
                             "kind": "oracle",
                             "sample": f"{sample}; outputs split over {n} host threads; "
                                       f"{args.steps} steps in {elapsed:.1f} s"},
            "e2e": {"value": round(value, 4), "unit": unit,
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


SWEEP_T = [1, 16, 64, 128, 256, 512, 1024, 2048, 4096, 8192]


def run_stage1_sweep(args, local):
    """Stage 1 alone at T = 1 .. 8192 rows of the decode c=64 shape (H = 6144,
    k = 8 partials with the outlier channels), each batch size timed from a
    CUDA graph of back-to-back launches over rotating input sets (> 2 x L2).
    `read_floor_us` times the small-batch kernel's loads alone (the same grid,
    no arithmetic, no stores: nfq_probe_stage1_reads) the same way."""
    import numpy as np
    import torch

    import norm_fp8_quant_gb300 as nfq
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peak, peak_kind = load_peaks()
    wmax = synth.workload(WORKLOAD, T=max(SWEEP_T))
    inp = synth.stage1_inputs(wmax)
    to_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    norm_w = to_bf16(inp["norm_w"]).to(dev)
    H, k = wmax.H, wmax.k
    rows = []
    for T in SWEEP_T:
        w = synth.workload(WORKLOAD, T=T)
        nsets, _ = rotation_sets(w)
        host = [to_bf16(inp["partials"][i, :T]) for i in range(k)] + [to_bf16(inp["residual"][:T])]
        sets = [[h.to(dev) for h in host] for _ in range(nsets)]
        hidden = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        codes = torch.empty((T, H), dtype=torch.uint8, device=dev)
        scales = torch.empty((T, H // 128), dtype=torch.float32, device=dev)
        calls = [nfq.prepare_reduce_norm_quant(st[:k], st[k], norm_w, w.eps, hidden, codes, scales)
                 for st in sets]
        for c in calls[:3]:
            c()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for c in calls:
                c()
        g.replay()
        torch.cuda.synchronize()
        reps = max(3, -(-max(args.steps, 400) // nsets)) if T <= 1024 else max(3, args.steps // 100)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("a kernel reported an expired wait in the stage-1 sweep")
        us = e0.elapsed_time(e1) * 1e3 / (reps * nsets)
        # the floor: the small-batch kernel's loads alone, same grid, same graph
        reads = [nfq.prepare_probe_stage1_reads(st[:k], st[k]) for st in sets]
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            for c in reads:
                c()
        g2.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            g2.replay()
        e1.record()
        torch.cuda.synchronize()
        floor_us = e0.elapsed_time(e1) * 1e3 / (reps * nsets)
        del g2, reads
        gbs = stage1_bytes(T, H, k) / (us * 1e-6) / 1e9
        plan = nfq.stage1_split_plan(T, H, k,
                                     torch.cuda.get_device_properties(dev).multi_processor_count)
        rows.append({"T": T, "us": round(us, 3), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "read_floor_us": round(floor_us, 3),
                     "kernel": (f"stage1_split_kernel, {plan['ctas_per_row']} CTAs per row, "
                                f"{plan['vpt']} vectors per thread, inputs "
                                + ("copied into shared memory" if plan["tma"] else
                                   "loaded into registers") if plan["ctas_per_row"]
                                else "reduce_norm_quant_kernel (persistent)"),
                     "launches": reps * nsets})
        del g, calls, sets
        torch.cuda.empty_cache()
    reach = [r["T"] for r in rows if r["frac"] >= 0.75]
    return {"metric": "norm+FP8-quant GB/s by batch size (stage 1 alone, CUDA-graph timed)",
            "unit": "GB/s", "peak": peak, "peak_source": peak_kind,
            "config": {"workload": f"decode c=64 shape: H={H}, k={k} BF16 partials N(0,0.5) with "
                                   "1% outlier channels x20, residual N(0,1); first T rows",
                       "l2": "inputs larger than L2: rotating input sets (> 280 MB per batch size)"},
            "rows": rows, "smallest_T_at_frac_0.75": reach[0] if reach else None}


def run_probe_mma(args, local):
    """The FP8 dense tensor rate on this GPU: every SM (or SM pair) issuing
    back-to-back tcgen05.mma kind::f8f6f4 from shared memory in the LM head's
    shapes, timed with CUDA events (the measurement kernel of nfq_probe_fp8_mma)."""
    import torch

    import norm_fp8_quant_gb300 as nfq

    torch.cuda.set_device(local)
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    rows = []
    for pair, stages in ((False, 1), (True, 1), (False, 4), (True, 4), (False, 0)):
        ctas = sms // 2 if pair else sms
        iters = 2048
        for _ in range(3):
            nfq.probe_fp8_mma(pair, ctas, iters, stages)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n = max(5, min(50, args.steps))
        flops = 0.0
        e0.record()
        for _ in range(n):
            flops += nfq.probe_fp8_mma(pair, ctas, iters, stages)
        e1.record()
        torch.cuda.synchronize()
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("the MMA probe reported an expired wait")
        ms = e0.elapsed_time(e1)
        mma_ns = ms * 1e6 / (n * iters * 4)
        rows.append({"shape": ("cta_group::2, M=256 x N=256 x K=32 per CTA pair" if pair else
                               "cta_group::1, M=128 x N=256 x K=32 per CTA"),
                     "operand_sets": max(1, stages),
                     "tmem_readers": ("16 warps reading TMEM meanwhile (the epilogue's pattern)"
                                      if stages == 0 else None),
                     "ctas": 2 * ctas if pair else ctas, "launches": n,
                     "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1),
                     "ns_per_mma": round(mma_ns, 2)})
    for pair in (False, True):
        # the NVFP4 LM head's block-scaled MMA (K = 64 e2m1 elements each)
        ctas = sms // 2 if pair else sms
        iters = 2048
        for _ in range(3):
            nfq.probe_nvfp4_mma(pair, ctas, iters)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n = max(5, min(50, args.steps))
        flops = 0.0
        e0.record()
        for _ in range(n):
            flops += nfq.probe_nvfp4_mma(pair, ctas, iters)
        e1.record()
        torch.cuda.synchronize()
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("the MMA probe reported an expired wait")
        ms = e0.elapsed_time(e1)
        rows.append({"shape": ("NVFP4 block-scaled, cta_group::2, M=256 x N=256 x K=64 per CTA pair"
                               if pair else
                               "NVFP4 block-scaled, cta_group::1, M=128 x N=256 x K=64 per CTA"),
                     "operand_sets": 1, "tmem_readers": None,
                     "ctas": 2 * ctas if pair else ctas, "launches": n,
                     "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1),
                     "ns_per_mma": round(ms * 1e6 / (n * iters * 4), 2)})
    tmem = []
    for batched in (False, True):
        iters = 4096
        for _ in range(3):
            nfq.probe_tmem_ld(batched, sms, iters)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n = max(5, min(50, args.steps))
        nbytes = 0.0
        e0.record()
        for _ in range(n):
            nbytes += nfq.probe_tmem_ld(batched, sms, iters)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        tmem.append({"pattern": ("four 16-column loads, one wait" if batched else
                                 "16-column loads, a wait after each (the LM head epilogue)"),
                     "ctas": sms, "launches": n,
                     "TB/s": round(nbytes / (ms * 1e-3) / 1e12, 2)})
    hand = []
    for pair, buffers, mode in ((False, 2, 2), (False, 2, 0), (False, 2, 1), (True, 2, 2),
                                (True, 2, 0), (True, 2, 1), (False, 4, 1), (False, 8, 1),
                                (False, 4, 3), (True, 4, 1), (True, 4, 3)):
        ctas = sms // 2 if pair else sms
        iters = 2048
        for _ in range(3):
            nfq.probe_handshake(pair, buffers, mode, ctas, iters)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n = max(5, min(50, args.steps))
        e0.record()
        for _ in range(n):
            nfq.probe_handshake(pair, buffers, mode, ctas, iters)
        e1.record()
        torch.cuda.synchronize()
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("the hand-off probe reported an expired wait")
        ms = e0.elapsed_time(e1)
        hand.append({"shape": ("CTA pairs, M=256" if pair else "single CTAs, M=128"),
                     "buffers": buffers, "N": 512 // buffers,
                     "epilogue": {0: "16 warps release each buffer unread",
                                  1: "16 warps read their columns (16 at a time), then release",
                                  2: "none: each group of MMAs waited for before the next",
                                  3: "each buffer its own 8 warps, 64 columns each, then release"}[mode],
                     "ctas": 2 * ctas if pair else ctas, "launches": n,
                     "ns_per_k_block": round(ms * 1e6 / (n * iters), 1)})
    shapes = []
    for m, n in ((128, 256), (128, 128), (128, 64), (128, 16), (64, 256), (64, 64)):
        # the time of one K = 32 FP8 MMA by shape: why the weight is the N = 256 operand
        iters = 2048
        for _ in range(2):
            nfq.probe_fp8_mma_shape(m, n, sms, iters)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n_l = max(5, min(50, args.steps))
        e0.record()
        for _ in range(n_l):
            nfq.probe_fp8_mma_shape(m, n, sms, iters)
        e1.record()
        torch.cuda.synchronize()
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("the MMA shape probe reported an expired wait")
        shapes.append({"M": m, "N": n, "ctas": sms, "launches": n_l,
                       "ns_per_mma": round(e0.elapsed_time(e1) * 1e6 / (n_l * iters * 4), 2)})
    latency = []
    for mode, what in ((0, "two warps of one CTA, local arrivals"),
                       (1, "the two CTAs of a cluster, remote arrivals at CTA scope"),
                       (2, "the two CTAs of a cluster, remote arrivals with cluster-scope release"),
                       (3, "the two CTAs of a cluster, st.async counted on the peer's barrier")):
        iters = 20000
        for _ in range(2):
            nfq.probe_handoff(mode, iters)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        n = 5
        e0.record()
        hops = 0
        for _ in range(n):
            hops += nfq.probe_handoff(mode, iters)
        e1.record()
        torch.cuda.synchronize()
        if nfq.device_error() != nfq.NFQ_OK:
            raise RuntimeError("the hand-off latency probe reported an expired wait")
        latency.append({"between": what, "launches": n,
                        "ns_one_way": round(e0.elapsed_time(e1) * 1e6 / hops, 1)})
    return {"metric": "FP8 dense tensor rate (tcgen05.mma kind::f8f6f4 from shared memory)",
            "unit": "TFLOP/s", "rows": rows, "mma_shapes": shapes, "tmem_read": tmem,
            "handoff_latency": latency,
            "handshake": {"rows": hand,
                          "what": "the LM head's accumulator hand-off without data: per K block "
                                  "(128 deep, 256 weight columns) four MMAs per N-column group, "
                                  "one TMEM buffer per group"},
            "config": {"workload": "every SM issues 2048 K blocks of four back-to-back MMAs into "
                                   "one TMEM accumulator from zeroed shared-memory tiles"}}


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.probe_mma:
        from norm_fp8_quant_gb300 import build
        if rank == 0:
            build.build()
            print(json.dumps(run_probe_mma(args, local)), flush=True)
        return
    if args.stage1_sweep:
        from norm_fp8_quant_gb300 import build
        if rank == 0:
            build.build()
            print(json.dumps(run_stage1_sweep(args, local)), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    from norm_fp8_quant_gb300 import build
    if rank == 0:
        build.build()
    else:
        while not os.path.exists(build.LIB):
            time.sleep(0.5)
    res = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            import synth
            res["cpu_baseline"] = cpu_baseline(args.workload, args.variant)
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
