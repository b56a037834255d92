"""CPU oracle for the MTP draft-layer tail — TEST INFRASTRUCTURE.

Only tests/, the smoke check in __graft_entry__ and the benchmark's CPU-baseline
and reference legs may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or runs anything here,
and this package imports nothing from the product.

The arithmetic lives in oracle.c (plain single-threaded C, fp32 where the
method fixes fp32, fp64 for the norm); this file builds it with gcc and passes
numpy arrays to it.  Every function here is pinned by tests/test_oracle_pins.py
to closed forms, library routines, brute force and hand-built cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")

EPS = 1e-6
GROUP = 128


def build(force: bool = False) -> str:
    """Compile oracle.c (no fast-math, no FMA contraction) into _liboracle.so."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None
_P = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_f32.restype = ctypes.c_float
        lib.or_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.or_f64_to_bf16.restype = ctypes.c_uint16
        lib.or_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.or_f32_to_bf16.restype = ctypes.c_uint16
        lib.or_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_to_f32.restype = ctypes.c_float
        lib.or_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.or_f32_to_e4m3.restype = ctypes.c_uint8
        lib.or_reduce_norm_quant.argtypes = [_P, ctypes.c_int, _P, _P, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P]
        lib.or_reduce_norm_quant.restype = None
        lib.or_lm_head_logits.argtypes = [_P, _P, ctypes.c_int, _P, ctypes.c_int, _P, _P,
                                          ctypes.c_int, ctypes.c_int, _P]
        lib.or_lm_head_logits.restype = None
        lib.or_argmax.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  _P, _P, _P, _P, _P]
        lib.or_argmax.restype = None
        lib.or_e2m1_to_f32.argtypes = [ctypes.c_uint8]
        lib.or_e2m1_to_f32.restype = ctypes.c_float
        lib.or_f32_to_e2m1.argtypes = [ctypes.c_float]
        lib.or_f32_to_e2m1.restype = ctypes.c_uint8
        lib.or_nvfp4_quant.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P, _P]
        lib.or_nvfp4_quant.restype = None
        lib.or_lm_head_logits_nvfp4.argtypes = [_P, _P, _P, ctypes.c_int, _P, ctypes.c_int,
                                                _P, _P, ctypes.c_float, ctypes.c_int,
                                                ctypes.c_int, _P]
        lib.or_lm_head_logits_nvfp4.restype = None
        lib.or_unfused_reduce_bf16.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
        lib.or_unfused_reduce_bf16.restype = None
        lib.or_unfused_add_rmsnorm.argtypes = [_P, _P, _P, ctypes.c_double, ctypes.c_int,
                                               ctypes.c_int, _P]
        lib.or_unfused_add_rmsnorm.restype = None
        lib.or_quant_fp8_rows.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P]
        lib.or_quant_fp8_rows.restype = None
        lib.or_argmax_bf16.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P]
        lib.or_argmax_bf16.restype = None
        lib.or_f32_to_bf16_array.argtypes = [_P, ctypes.c_size_t, _P]
        lib.or_f32_to_bf16_array.restype = None
        _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ codecs --

def bf16_to_f32(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, np.uint16)
    _load().or_f32_to_bf16_array(x.ctypes.data, x.size, out.ctypes.data)
    return out


def f64_to_bf16(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float64).ravel()
    return np.array([lib.or_f64_to_bf16(float(v)) for v in x], dtype=np.uint16)


def e4m3_to_f32(codes) -> np.ndarray:
    lib = _load()
    c = _c(codes, np.uint8).ravel()
    return np.array([lib.or_e4m3_to_f32(int(v)) for v in c], dtype=np.float32)


def f32_to_e4m3(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32).ravel()
    return np.array([lib.or_f32_to_e4m3(float(v)) for v in x], dtype=np.uint8)


# ----------------------------------------------------------------- stage 1 --

def reduce_norm_quant(partials, residual, norm_w, eps: float = EPS, want_x: bool = False):
    """Stage 1 on rows [R][H]: returns dict(hidden uint16, codes uint8,
    scales float32 [R][H/128], and x float32 / rr float64 when want_x)."""
    p = _c(partials, np.uint16)
    k, R, H = p.shape
    assert H % GROUP == 0
    res = _c(residual, np.uint16)
    w = _c(norm_w, np.uint16)
    assert res.shape == (R, H) and w.shape == (H,)
    hidden = np.empty((R, H), np.uint16)
    codes = np.empty((R, H), np.uint8)
    scales = np.empty((R, H // GROUP), np.float32)
    x = np.empty((R, H), np.float32) if want_x else None
    rr = np.empty(R, np.float64) if want_x else None
    _load().or_reduce_norm_quant(p.ctypes.data, k, res.ctypes.data, w.ctypes.data, eps, R, H,
                                 hidden.ctypes.data, codes.ctypes.data, scales.ctypes.data,
                                 None if x is None else x.ctypes.data,
                                 None if rr is None else rr.ctypes.data)
    out = {"hidden": hidden, "codes": codes, "scales": scales}
    if want_x:
        out["x"], out["rr"] = x, rr
    return out


# ----------------------------------------------------------------- stage 2 --

def lm_head_logits(qa, sa, qw, sw, tokens=None, v0: int = 0, v1: int | None = None):
    """fp32 logits [len(tokens)][v1-v0] of the block-scaled FP8 LM head."""
    qa = _c(qa, np.uint8)
    T, H = qa.shape
    sa = _c(sa, np.float32)
    qw = _c(qw, np.uint8)
    sw = _c(sw, np.float32)
    V = qw.shape[0]
    v1 = V if v1 is None else v1
    tok = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    out = np.empty((tok.size, v1 - v0), np.float32)
    _load().or_lm_head_logits(qa.ctypes.data, sa.ctypes.data, H, tok.ctypes.data, tok.size,
                              qw.ctypes.data, sw.ctypes.data, v0, v1, out.ctypes.data)
    return out


def argmax(logits, S: int):
    """Per-row greedy token, per-shard results and relative top-2 gap."""
    L = _c(logits, np.float32)
    n, V = L.shape
    assert V % S == 0
    tok = np.empty(n, np.int32)
    val = np.empty(n, np.float32)
    sidx = np.empty((n, S), np.int32)
    sval = np.empty((n, S), np.float32)
    gap = np.empty(n, np.float64)
    _load().or_argmax(L.ctypes.data, n, V, S, tok.ctypes.data, val.ctypes.data,
                      sidx.ctypes.data, sval.ctypes.data, gap.ctypes.data)
    return {"tokens": tok, "values": val, "shard_idx": sidx, "shard_val": sval, "gap": gap}


def shard_gaps(logits, S: int) -> np.ndarray:
    """Relative top-2 gap inside each shard, [n][S] (for per-shard id checks)."""
    L = np.asarray(logits, np.float32)
    n, V = L.shape
    w = V // S
    out = np.empty((n, S))
    for s in range(S):
        r = argmax(L[:, s * w:(s + 1) * w], 1)
        out[:, s] = r["gap"]
    return out


# ---------------------------------------------------------- NVFP4 variant --

NVFP4_BLOCK = 16


def e2m1_to_f32(codes) -> np.ndarray:
    """Decode 4-bit e2m1 codes (one per array element, 0..15)."""
    lib = _load()
    c = _c(codes, np.uint8).ravel()
    return np.array([lib.or_e2m1_to_f32(int(v)) for v in c], dtype=np.float32).reshape(np.shape(codes))


def f32_to_e2m1(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32).ravel()
    return np.array([lib.or_f32_to_e2m1(float(v)) for v in x], dtype=np.uint8)


def nvfp4_quant(hidden):
    """NVFP4 codes [R][H/2] (packed), block scales [R][H/16], row scales [R] of
    BF16 rows [R][H]."""
    h = _c(hidden, np.uint16)
    R, H = h.shape
    assert H % NVFP4_BLOCK == 0
    codes = np.empty((R, H // 2), np.uint8)
    bs = np.empty((R, H // NVFP4_BLOCK), np.uint8)
    gs = np.empty(R, np.float32)
    _load().or_nvfp4_quant(h.ctypes.data, R, H, codes.ctypes.data, bs.ctypes.data, gs.ctypes.data)
    return {"codes": codes, "block_scales": bs, "global_scales": gs}


def reduce_norm_quant_nvfp4(partials, residual, norm_w, eps: float = EPS):
    """Stage 1 with the NVFP4 activation: the BF16 hidden of reduce_norm_quant,
    quantised by nvfp4_quant."""
    o = reduce_norm_quant(partials, residual, norm_w, eps)
    q = nvfp4_quant(o["hidden"])
    return {"hidden": o["hidden"], **q}


def lm_head_logits_nvfp4(qa, sa, ga, qw, sw, gw: float, tokens=None, v0: int = 0,
                         v1: int | None = None):
    """fp32 logits [len(tokens)][v1-v0] of the NVFP4 LM head."""
    qa = _c(qa, np.uint8)
    T, H2 = qa.shape
    H = 2 * H2
    sa = _c(sa, np.uint8)
    ga = _c(ga, np.float32)
    qw = _c(qw, np.uint8)
    sw = _c(sw, np.uint8)
    V = qw.shape[0]
    v1 = V if v1 is None else v1
    tok = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    out = np.empty((tok.size, v1 - v0), np.float32)
    _load().or_lm_head_logits_nvfp4(qa.ctypes.data, sa.ctypes.data, ga.ctypes.data, H,
                                    tok.ctypes.data, tok.size, qw.ctypes.data, sw.ctypes.data,
                                    float(gw), v0, v1, out.ctypes.data)
    return out


# ------------------------------------------------------ unfused reference arm --

def unfused_reduce_bf16(partials):
    """bf16(sum of the k BF16 partials in fp32), the separate all-reduce's output."""
    p = _c(partials, np.uint16)
    k, R, H = p.shape
    out = np.empty((R, H), np.uint16)
    _load().or_unfused_reduce_bf16(p.ctypes.data, k, R, H, out.ctypes.data)
    return out


def unfused_add_rmsnorm(x, residual, norm_w, eps: float = EPS):
    x = _c(x, np.uint16)
    R, H = x.shape
    res = _c(residual, np.uint16)
    w = _c(norm_w, np.uint16)
    out = np.empty((R, H), np.uint16)
    _load().or_unfused_add_rmsnorm(x.ctypes.data, res.ctypes.data, w.ctypes.data, eps, R, H,
                                   out.ctypes.data)
    return out


def quant_fp8_rows(hidden):
    h = _c(hidden, np.uint16)
    R, H = h.shape
    codes = np.empty((R, H), np.uint8)
    scales = np.empty((R, H // GROUP), np.float32)
    _load().or_quant_fp8_rows(h.ctypes.data, R, H, codes.ctypes.data, scales.ctypes.data)
    return {"codes": codes, "scales": scales}


def argmax_bf16(logits_bits):
    L = _c(logits_bits, np.uint16)
    n, V = L.shape
    tok = np.empty(n, np.int32)
    _load().or_argmax_bf16(L.ctypes.data, n, V, tok.ctypes.data)
    return tok


def unfused_step(partials, residual, norm_w, qw, sw, eps: float = EPS, tokens=None):
    """The unfused path end to end: BF16 all-reduce, add + RMSNorm, group quant,
    BF16 logits, full-vocab argmax.  Returns its intermediate results."""
    s = unfused_reduce_bf16(partials)
    hidden = unfused_add_rmsnorm(s, residual, norm_w, eps)
    q = quant_fp8_rows(hidden)
    L = lm_head_logits(q["codes"], q["scales"], qw, sw, tokens=tokens)
    Lb = f32_to_bf16(L.ravel()).reshape(L.shape)
    return {"sum": s, "hidden": hidden, **q, "logits": Lb, "tokens": argmax_bf16(Lb)}
