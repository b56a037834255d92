"""Seeded synthetic inputs for the MTP draft-layer tail (both sides use these).

This module draws random numbers and stores them in the formats the path
consumes.  It holds none of the path's arithmetic: the only conversions are
torch library casts (fp32 -> bfloat16, fp32 -> float8_e4m3fn) and the offline
128x128 block quantisation of the LM-head weight, which the path receives
already quantised.  Draws come from the counter-based generator in gen.c, so
any row can be regenerated on its own (used for sampled checks at full size).

Workloads (shapes of the DeepSeek-V3.2 / GLM-5.2 MTP draft tail; N(0, s) means
standard deviation s):

  tiny        T=4    H=1024 k=2 partials N(0,1)   V=4096   S=2
  decode_c1   T=1    H=7168 k=8 partials N(0,0.5) V=129280 S=8
  decode_c64  T=64   H=6144 k=8 partials N(0,0.5), 1% outlier channels x20,
              V=151552 S=8
  prefill     T=8192 H=7168 k=8 partials N(0,0.5) (norm + quant only)
  tie_stress  T=256  H=6144 k=4 partials N(0,0.5) V=151552 S=8, 30% of tokens
              get an exact duplicate maximum logit across a shard boundary

Every workload: residual N(0,1), norm weight 1+N(0,0.1), LM-head weight
N(0,0.02) block-quantised to e4m3 with one fp32 scale per 128x128 block,
seed 0.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_libsynth.so")

# stream ids of the counter-based generator
STREAM_RESIDUAL = 1
STREAM_NORM_W = 2
STREAM_LM_W = 3
STREAM_OUTLIER = 4
STREAM_TIES = 5
STREAM_PARTIAL0 = 100


def build(force: bool = False) -> str:
    """Compile gen.c into _libsynth.so next to it (host C, no GPU)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_f32.argtypes = [
            ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
            ctypes.c_double, ctypes.c_double, ctypes.c_void_p, ctypes.c_uint64,
            ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal_f32.restype = None
        lib.synth_choose.argtypes = [ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        lib.synth_choose.restype = None
        lib.synth_bits.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_bits.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, count: int, mean: float = 0.0,
               std: float = 1.0, start: int = 0,
               colmult: np.ndarray | None = None) -> np.ndarray:
    """Elements start..start+count-1 of normal stream (seed, stream) as fp32."""
    out = np.empty(int(count), dtype=np.float32)
    if count == 0:
        return out
    cm = None
    ncols = 0
    if colmult is not None:
        cm = np.ascontiguousarray(colmult, dtype=np.float32)
        ncols = cm.size
    _load().synth_normal_f32(seed, stream, start, count, mean, std,
                             None if cm is None else cm.ctypes.data, ncols,
                             out.ctypes.data, _threads())
    return out


def choose(seed: int, stream: int, length: int, n: int) -> np.ndarray:
    out = np.empty(max(n, 1), dtype=np.int64)
    _load().synth_choose(seed, stream, length, n, out.ctypes.data)
    return out[:n]


def bits(seed: int, stream: int, j: int) -> int:
    return int(_load().synth_bits(seed, stream, j))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16) via torch's round-to-nearest-even cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    k: int
    partial_std: float
    V: int = 0            # 0: norm + quant only
    S: int = 1
    outlier_frac: float = 0.0
    outlier_mult: float = 20.0
    tie_frac: float = 0.0
    residual_std: float = 1.0
    norm_w_std: float = 0.1
    weight_std: float = 0.02
    eps: float = 1e-6
    seed: int = 0

    @property
    def G(self) -> int:
        return self.H // 128

    @property
    def n_vblocks(self) -> int:
        return (self.V + 127) // 128


WORKLOADS = {
    "tiny": Workload("tiny", T=4, H=1024, k=2, partial_std=1.0, V=4096, S=2),
    "decode_c1": Workload("decode_c1", T=1, H=7168, k=8, partial_std=0.5,
                          V=129280, S=8),
    "decode_c64": Workload("decode_c64", T=64, H=6144, k=8, partial_std=0.5,
                           V=151552, S=8, outlier_frac=0.01),
    "prefill": Workload("prefill", T=8192, H=7168, k=8, partial_std=0.5),
    "tie_stress": Workload("tie_stress", T=256, H=6144, k=4, partial_std=0.5,
                           V=151552, S=8, tie_frac=0.3),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


def outlier_channels(w: Workload) -> np.ndarray:
    n = int(round(w.outlier_frac * w.H))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    return np.sort(choose(w.seed, STREAM_OUTLIER, w.H, n))


def _colmult(w: Workload):
    ch = outlier_channels(w)
    if ch.size == 0:
        return None
    m = np.ones(w.H, dtype=np.float32)
    m[ch] = w.outlier_mult
    return m


def stage1_inputs(w: Workload, rows=None) -> dict:
    """BF16 inputs of the reduce + residual + RMSNorm + quant stage.

    rows: None for all T rows, else an iterable of token indices (the returned
    arrays then hold those rows in that order).
    Returns uint16 bit patterns: partials [k][R][H], residual [R][H], norm_w [H].
    """
    H = w.H
    rows = list(range(w.T)) if rows is None else [int(r) for r in rows]
    cm = _colmult(w)
    R = len(rows)
    contiguous = rows == list(range(rows[0], rows[0] + R)) if R else True

    def draw(stream, std, colmult):
        if contiguous:
            start = rows[0] * H if R else 0
            f = normal_f32(w.seed, stream, R * H, 0.0, std, start, colmult)
        else:
            f = np.concatenate([normal_f32(w.seed, stream, H, 0.0, std, r * H, colmult)
                                for r in rows]) if R else np.zeros(0, np.float32)
        return to_bf16_bits(f).reshape(R, H)

    partials = np.stack([draw(STREAM_PARTIAL0 + i, w.partial_std, cm)
                         for i in range(w.k)]) if w.k else np.zeros((0, R, H), np.uint16)
    residual = draw(STREAM_RESIDUAL, w.residual_std, None)
    norm_w = to_bf16_bits(normal_f32(w.seed, STREAM_NORM_W, H, 1.0, w.norm_w_std))
    return {"partials": partials, "residual": residual, "norm_w": norm_w, "rows": rows}


def lm_head_weights(w: Workload, chunk_blocks: int = 64):
    """LM-head weight: fp32 N(0, weight_std) draws [V][H], block-quantised.

    Per 128x128 block (rows v//128, columns k//128): scale = amax / 448 in fp32,
    codes = float8_e4m3fn(W / scale) by torch's cast (|W/scale| <= 448 so the
    cast never leaves the finite range); an all-zero block gets scale 0 and
    codes 0.  Returns (codes uint8 [V][H], scales float32 [ceil(V/128)][H/128]).
    """
    import torch
    V, H, G = w.V, w.H, w.G
    nvb = w.n_vblocks
    codes = np.empty((V, H), dtype=np.uint8)
    scales = np.empty((nvb, G), dtype=np.float32)
    for b0 in range(0, nvb, chunk_blocks):
        b1 = min(nvb, b0 + chunk_blocks)
        r0, r1 = b0 * 128, min(V, b1 * 128)
        f = normal_f32(w.seed, STREAM_LM_W, (r1 - r0) * H, 0.0, w.weight_std, r0 * H)
        Wt = torch.zeros(((b1 - b0) * 128, H), dtype=torch.float32)
        Wt[: r1 - r0] = torch.from_numpy(f).view(r1 - r0, H)
        Wb = Wt.view(b1 - b0, 128, G, 128)
        amax = Wb.abs().amax(dim=(1, 3))
        sc = amax / 448.0
        safe = torch.where(sc > 0, sc, torch.ones_like(sc))
        q = (Wb / safe[:, None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        q = torch.where((sc > 0)[:, None, :, None], q, torch.zeros_like(q))
        codes[r0:r1] = q.reshape((b1 - b0) * 128, H)[: r1 - r0].numpy()
        scales[b0:b1] = sc.numpy()
    return codes, scales


def nvfp4_quantise_rows(x, g):
    """NVFP4 form of fp32 rows x [R][H] (H a multiple of 16) with the fp32 row
    scales g [R] (or one scalar for a whole tensor): per 16 consecutive values
    the block scale is e4m3(amax / (6 g)) (torch's round-to-nearest-even cast,
    clamped at 448), the effective scale dec(block scale) * g, and the codes
    are the e2m1 values nearest to x / effective scale (ties to the even code,
    saturating at 6; codes 0 where the effective scale is 0), packed two to a
    byte with element 2i in the low nibble.  Returns (codes uint8 [R][H/2],
    block scales uint8 [R][H/16])."""
    import torch
    xt = torch.as_tensor(np.ascontiguousarray(x, np.float32))
    R, H = xt.shape
    gt = torch.as_tensor(np.asarray(g, np.float32)).reshape(-1, 1)
    gt = gt.expand(R, 1) if gt.shape[0] == 1 else gt
    xb = xt.view(R, H // 16, 16)
    amax = xb.abs().amax(dim=2)
    d = gt * np.float32(6.0)
    u = torch.where(d > 0, amax / torch.where(d > 0, d, torch.ones_like(d)), torch.zeros_like(amax))
    sb = u.clamp(max=448.0).to(torch.float8_e4m3fn)
    eff = sb.float() * gt
    q = xb / torch.where(eff > 0, eff, torch.ones_like(eff))[:, :, None]
    a = q.abs().clamp(max=6.0)
    step = torch.where(a < 2, 0.5, torch.where(a < 4, 1.0, 2.0))
    r = (torch.round(a / step) * step).clamp(max=6.0)      # torch.round: half to even
    lut = torch.tensor([0, 1, 2, 3, 4, 0, 5, 0, 6, 0, 0, 0, 7], dtype=torch.uint8)
    code = lut[(r * 2).long()] | (torch.signbit(q).to(torch.uint8) << 3)
    code = torch.where((eff > 0)[:, :, None], code, torch.zeros_like(code)).view(R, H)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed.numpy(), sb.view(torch.uint8).numpy()


def lm_head_weights_nvfp4(w: Workload, chunk_rows: int = 8192):
    """NVFP4 LM-head weight from the same fp32 N(0, weight_std) draws as
    lm_head_weights: one fp32 scale for the whole tensor, amax / (448 * 6),
    then nvfp4_quantise_rows.  Returns (codes uint8 [V][H/2], block scales
    uint8 [V][H/16], tensor scale float)."""
    V, H = w.V, w.H
    amax = np.float32(0.0)
    for r0 in range(0, V, chunk_rows):
        r1 = min(V, r0 + chunk_rows)
        f = normal_f32(w.seed, STREAM_LM_W, (r1 - r0) * H, 0.0, w.weight_std, r0 * H)
        amax = max(amax, np.float32(np.abs(f).max()))
    gw = np.float32(amax / np.float32(2688.0))
    codes = np.empty((V, H // 2), np.uint8)
    bs = np.empty((V, H // 16), np.uint8)
    for r0 in range(0, V, chunk_rows):
        r1 = min(V, r0 + chunk_rows)
        f = normal_f32(w.seed, STREAM_LM_W, (r1 - r0) * H, 0.0, w.weight_std, r0 * H)
        codes[r0:r1], bs[r0:r1] = nvfp4_quantise_rows(f.reshape(r1 - r0, H), gw)
    return codes, bs, float(gw)


# planted e4m3 codes: +448 and -448
_PLUS_MAX, _MINUS_MAX = 0x7E, 0xFE


def plant_ties(w: Workload, codes: np.ndarray, scales: np.ndarray,
               act_codes: np.ndarray) -> dict:
    """Tie-stress construction on an already generated LM-head weight (in place).

    For every internal shard boundary b (shard width V/S, a multiple of 128):
    the first 128-row block of the upper shard takes over the scale row of the
    last block of the lower shard, so rows of the two blocks with equal codes
    dequantise identically.  A planted row for token t has code +448 where the
    activation code of t is positive, -448 where negative and 0 where zero; it
    is written into one row of each of the two blocks, so token t meets two
    exactly equal maxima on either side of the boundary.  round(tie_frac * T)
    tokens are planted, spread round-robin over the boundaries; the first token
    of each boundary uses the adjacent pair (last row of the lower shard, first
    row of the upper shard).  Returns {token: lowest planted global row}.
    Only byte copies happen here.
    """
    V, S, T = w.V, w.S, act_codes.shape[0]
    width = V // S
    assert V % S == 0 and width % 128 == 0 and width >= 128
    n_tie = int(round(w.tie_frac * T))
    bounds = [s * width for s in range(1, S)]
    tokens = choose(w.seed, STREAM_TIES, T, n_tie)
    expected = {}
    for b in bounds:
        scales[b // 128] = scales[b // 128 - 1]
    per_bound_count = {b: 0 for b in bounds}
    for j, t in enumerate(tokens):
        b = bounds[j % len(bounds)]
        c = per_bound_count[b]
        per_bound_count[b] += 1
        if c >= 128:
            raise ValueError("too many planted rows for one boundary")
        lo = b - 1 - c          # rows b-1, b-2, ... in the lower shard's last block
        hi = b + c              # rows b, b+1, ... in the upper shard's first block
        a = act_codes[t]
        mag_zero = (a & 0x7F) == 0
        neg = (a & 0x80) != 0
        row = np.where(mag_zero, 0, np.where(neg, _MINUS_MAX, _PLUS_MAX)).astype(np.uint8)
        codes[lo] = row
        codes[hi] = row
        expected[int(t)] = lo
    return expected
