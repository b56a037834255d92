"""Shared helpers of the parity tests: GPU upload, acceptance checks.

Acceptance rules (the method's stated tolerances, with the readings noted):
  hidden  BF16 within 1 ulp in sign-magnitude order (+0 == -0)
  scales  within 1e-6 relative in every group whose 128 BF16 hidden values
          agree exactly with the oracle; elsewhere the GPU scale must equal
          max|GPU hidden| / 448 in fp32 (self-consistency)
  codes   bit-exact in groups whose hidden agrees; elsewhere at most one e4m3
          step apart, and such differences on at most 0.1% of all elements
  tokens  exact wherever the oracle's top-2 relative gap is >= 1e-3 and for
          exact ties (gap 0); in between a near tie is counted, and the GPU's
          pick must still be within the logit tolerance of the maximum
  logits  |GPU - oracle| <= 2 * gamma_H * sum_k |a_k w_k| (fp32 accumulation
          bound applied to both sides), gamma_n = n u / (1 - n u), u = 2^-24
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle

U = 2.0 ** -24


def oracle_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _vocab_ranges(V: int, parts: int):
    parts = max(1, min(parts, V))
    return [(i * V // parts, (i + 1) * V // parts) for i in range(parts)]


def oracle_logits(qa, sa, qw, sw, tokens):
    """The oracle's fp32 logits [len(tokens)][V], the vocab rows split over host
    threads.  Every logit is one call's fixed-order sum, so the result is the
    single-threaded one; the oracle's C calls release the interpreter lock."""
    V = qw.shape[0]
    tok = np.asarray(tokens, np.int32)
    out = np.empty((tok.size, V), np.float32)

    def job(r):
        out[:, r[0]:r[1]] = oracle.lm_head_logits(qa, sa, qw, sw, tokens=tok, v0=r[0], v1=r[1])
    with ThreadPoolExecutor(oracle_threads()) as pool:
        list(pool.map(job, _vocab_ranges(V, 4 * oracle_threads())))
    return out


def oracle_logits_nvfp4(qa, sa, ga, qw, sw, gw, tokens):
    """As oracle_logits, for the NVFP4 LM head."""
    V = qw.shape[0]
    tok = np.asarray(tokens, np.int32)
    out = np.empty((tok.size, V), np.float32)

    def job(r):
        out[:, r[0]:r[1]] = oracle.lm_head_logits_nvfp4(qa, sa, ga, qw, sw, gw, tokens=tok,
                                                        v0=r[0], v1=r[1])
    with ThreadPoolExecutor(oracle_threads()) as pool:
        list(pool.map(job, _vocab_ranges(V, 4 * oracle_threads())))
    return out


_E4M3 = None


def e4m3_table() -> np.ndarray:
    """The oracle's decoding of all 256 e4m3 codes (fp64), for vectorised lookups."""
    global _E4M3
    if _E4M3 is None:
        _E4M3 = oracle.e4m3_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    return _E4M3


def to_dev_bf16(bits: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_dev(a: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bf16_host(t) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _ordered_bf16(bits):
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _ordered_e4m3(codes):
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def check_stage1(hidden, codes, scales, ref, max_code_frac=1e-3):
    """hidden/codes/scales: host arrays from the GPU; ref: oracle dict.
    Returns a dict of counts for reporting."""
    R, H = ref["hidden"].shape
    G = H // 128
    dh = np.abs(_ordered_bf16(hidden) - _ordered_bf16(ref["hidden"]))
    assert dh.max(initial=0) <= 1, f"hidden differs by {dh.max()} bf16 ulps"
    group_same = (dh.reshape(R, G, 128) == 0).all(axis=2)
    # scales: rel 1e-6 where the group's hidden agrees
    so, sg = ref["scales"], scales
    rel = np.abs(sg.astype(np.float64) - so) / np.maximum(np.abs(so).astype(np.float64), 1e-30)
    bad = group_same & (rel > 1e-6) & ~((sg == 0) & (so == 0))
    assert not bad.any(), f"{bad.sum()} scales off in agreeing groups"
    # self-consistency everywhere
    yg = np.abs(oracle.bf16_to_f32(hidden).reshape(R, G, 128)).max(axis=2)
    assert np.array_equal(sg, (yg / np.float32(448)).astype(np.float32)), "scale != amax/448"
    # codes: identical (zero sign ignored) in agreeing groups
    cg = np.where((codes & 0x7F) == 0, 0, codes).reshape(R, G, 128)
    co = np.where((ref["codes"] & 0x7F) == 0, 0, ref["codes"]).reshape(R, G, 128)
    diff = cg != co
    assert not (diff & group_same[:, :, None]).any(), "codes differ in a group whose hidden agrees"
    step = np.abs(_ordered_e4m3(cg) - _ordered_e4m3(co))
    assert step.max(initial=0) <= 1, f"codes differ by {step.max()} steps"
    frac = diff.sum() / diff.size
    assert frac <= max_code_frac, f"{frac:.2e} of codes differ"
    return {"hidden_ulp_diffs": int((dh > 0).sum()), "groups_differing": int((~group_same).sum()),
            "codes_differing": int(diff.sum())}


def dequant_rows(codes, scales):
    """fp64 dequantised rows of a [R][H] code block with [R][G] or [Rb][G] scales."""
    return e4m3_table()[np.asarray(codes, np.uint8)] * \
        np.repeat(scales.astype(np.float64), 128, axis=1)


def abs_dot(qa_row, sa_row, qw, sw, rows):
    """sum_k |a_k w_k| for one activation row against weight rows `rows`."""
    a = np.abs(dequant_rows(qa_row[None, :], sa_row[None, :]))[0]
    out = []
    for v in rows:
        w = np.abs(dequant_rows(qw[v][None, :], sw[v // 128][None, :]))[0]
        out.append(float(a @ w))
    return np.array(out)


_LOGITS_CACHE = {}


def check_stage2(tokens, qa, sa, qw, sw, S, sample, max_logit=None, shard_idx=None,
                 shard_val=None, expected=None, cache_key=None):
    """Compare GPU draft tokens (and optional outputs) on the token rows
    `sample` with the oracle's full-vocab logits; expected: {token: id} known by
    construction.  cache_key: reuse the oracle's logits of an earlier call with
    the same key (the same activation, weight and sample).  Returns (#near
    ties, #checked)."""
    H = qa.shape[1]
    gamma = (H + 2) * U / (1 - (H + 2) * U)
    if cache_key is not None and cache_key in _LOGITS_CACHE:
        L = _LOGITS_CACHE[cache_key]
    else:
        L = oracle_logits(qa, sa, qw, sw, sample)
        if cache_key is not None:
            _LOGITS_CACHE.clear()
            _LOGITS_CACHE[cache_key] = L
    r = oracle.argmax(L, S)
    near = 0
    V = qw.shape[0]
    width = V // S
    for i, t in enumerate(sample):
        gap = r["gap"][i]
        tol = 2 * gamma * abs_dot(qa[t], sa[t], qw, sw, [int(r["tokens"][i])])[0]
        if expected is not None and t in expected:
            assert r["tokens"][i] == expected[t], "oracle misses a planted tie"
        if gap >= 1e-3 or gap == 0.0:
            assert tokens[t] == r["tokens"][i], f"token {t}: gpu {tokens[t]} oracle {r['tokens'][i]} gap {gap}"
        else:
            near += 1
            assert L[i, tokens[t]] >= r["values"][i] - 2 * tol
        if max_logit is not None:
            assert abs(float(max_logit[t]) - float(r["values"][i])) <= tol + 1e-30
        if shard_idx is not None:
            sg = oracle.shard_gaps(L[i:i + 1], S)[0]
            for s in range(S):
                oi = int(r["shard_idx"][i, s])
                gi = int(shard_idx[s, t])
                assert s * width <= gi < (s + 1) * width
                stol = 2 * gamma * abs_dot(qa[t], sa[t], qw, sw, [oi])[0]
                if sg[s] >= 1e-3 or sg[s] == 0.0:
                    assert gi == oi, f"token {t} shard {s}: gpu {gi} oracle {oi}"
                else:
                    assert L[i, gi] >= r["shard_val"][i, s] - 2 * stol
                if shard_val is not None:
                    assert abs(float(shard_val[s, t]) - float(r["shard_val"][i, s])) <= stol + 1e-30
    return near, len(sample)


# ------------------------------------------------------------------ NVFP4 --

def _nib(c):
    """unpacked e2m1 codes [R][2*B] of packed bytes [R][B], -0 written as +0"""
    c = np.asarray(c, np.uint8)
    u = np.stack([c & 15, c >> 4], axis=-1).reshape(c.shape[0], -1)
    return np.where((u & 7) == 0, 0, u)


def check_stage1_fp4(hidden, codes, bscales, gscales, ref_hidden):
    """hidden within 1 BF16 ulp of the oracle; the oracle's NVFP4 quantiser
    applied to the GPU's own hidden reproduces the GPU's codes, block scales and
    row scales bit for bit (zero codes compared without their sign).  Returns
    the number of rows whose hidden differs from the oracle's."""
    dh = np.abs(_ordered_bf16(hidden) - _ordered_bf16(ref_hidden))
    assert dh.max(initial=0) <= 1, f"hidden differs by {dh.max()} bf16 ulps"
    q = oracle.nvfp4_quant(hidden)
    assert np.array_equal(np.asarray(gscales, np.float32).view(np.uint32),
                          q["global_scales"].view(np.uint32)), "row scales"
    assert np.array_equal(bscales, q["block_scales"]), "block scales"
    assert np.array_equal(_nib(codes), _nib(q["codes"])), "e2m1 codes"
    return int((dh.max(axis=1) > 0).sum())


def _nvfp4_dequant(codes, bs):
    u = np.asarray(codes, np.uint8)
    u = np.stack([u & 15, u >> 4], axis=-1).reshape(u.shape[0], -1)
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])[u & 7]
    v = np.where(u & 8, -mag, mag)
    s = e4m3_table()[np.asarray(bs, np.uint8)]
    return v * np.repeat(s, 16, axis=1)


def check_stage2_fp4(tokens, qa, sa, ga, qw, sw, gw, S, sample, max_logit=None,
                     shard_idx=None, shard_val=None, expected=None, cache_key=None):
    """As check_stage2, for the NVFP4 LM head: the logit bound is
    2 gamma_n sum_b |c_b| |ga gw| with n = H/16 + 2 (the block-scaled products
    are exact; only their fp32 sum and the final scaling round)."""
    H = qa.shape[1] * 2
    n = H // 16 + 2
    gamma = n * U / (1 - n * U)
    if cache_key is not None and cache_key in _LOGITS_CACHE:
        L = _LOGITS_CACHE[cache_key]
    else:
        L = oracle_logits_nvfp4(qa, sa, ga, qw, sw, gw, sample)
        if cache_key is not None:
            _LOGITS_CACHE.clear()
            _LOGITS_CACHE[cache_key] = L
    r = oracle.argmax(L, S)
    V = qw.shape[0]
    width = V // S
    near = 0
    for i, t in enumerate(sample):
        a = np.abs(_nvfp4_dequant(qa[t:t + 1], sa[t:t + 1]))[0]
        scale = abs(float(np.float32(ga[t]) * np.float32(gw)))

        def tol_of(v):
            w = np.abs(_nvfp4_dequant(qw[v:v + 1], sw[v:v + 1]))[0]
            return 2 * gamma * float(a @ w) * scale + 4 * U * abs(float(L[i, v])) + 1e-30
        gap = r["gap"][i]
        tol = tol_of(int(r["tokens"][i]))
        if expected is not None and t in expected:
            assert r["tokens"][i] == expected[t], "oracle misses a planted tie"
        if gap >= 1e-3 or gap == 0.0:
            assert tokens[t] == r["tokens"][i], f"token {t}: gpu {tokens[t]} oracle {r['tokens'][i]} gap {gap}"
        else:
            near += 1
            assert L[i, tokens[t]] >= r["values"][i] - 2 * tol
        if max_logit is not None:
            assert abs(float(max_logit[t]) - float(r["values"][i])) <= tol
        if shard_idx is not None:
            sg = oracle.shard_gaps(L[i:i + 1], S)[0]
            for s in range(S):
                oi = int(r["shard_idx"][i, s])
                gi = int(shard_idx[s, t])
                assert s * width <= gi < (s + 1) * width
                stol = tol_of(oi)
                if sg[s] >= 1e-3 or sg[s] == 0.0:
                    assert gi == oi, f"token {t} shard {s}: gpu {gi} oracle {oi}"
                else:
                    assert L[i, gi] >= r["shard_val"][i, s] - 2 * stol
                if shard_val is not None:
                    assert abs(float(shard_val[s, t]) - float(r["shard_val"][i, s])) <= stol
    return near, len(sample)
