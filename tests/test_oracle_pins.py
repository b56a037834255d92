"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one oracle function to a library routine, a closed form, an
invariant, brute force or a hand-derived case, chosen so that a plausible slip
(a dropped term, a wrong sign or index, a transposed operand, a wrong rounding
rule) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def torch_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_e4m3_codes(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_e4m3_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def bf16_bits_of(x):
    """bits of an fp32 value that is exactly representable in bf16"""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------------- BF16 --

def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # the C decoder agrees with the vectorised one on a sample
    lib = oracle._load()
    for b in [0x0000, 0x8000, 0x3F80, 0xC000, 0x7F80, 0x0001, 0x7F7F, 0x0080]:
        assert np.float32(lib.or_bf16_to_f32(b)).view(np.uint32) == ours[b].view(np.uint32)


def test_bf16_encode_matches_torch_on_random_and_midpoints():
    mags = np.exp2(rng.uniform(-140, 127.9, 20000)).astype(np.float32)
    x = np.where(rng.random(20000) < 0.5, -mags, mags).astype(np.float32)
    assert np.array_equal(oracle.f32_to_bf16(x), torch_bf16_bits(x))
    # every midpoint between two consecutive positive finite bf16 values in a
    # spread of binades: ties go to the even pattern (torch agrees)
    lo = np.arange(0x0001, 0x7F7F, 37, dtype=np.uint32)
    a = (lo << 16).view(np.float32).astype(np.float64)
    b = ((lo + 1) << 16).view(np.float32).astype(np.float64)
    mid = ((a + b) / 2).astype(np.float32)
    got = oracle.f32_to_bf16(mid)
    assert np.array_equal(got, torch_bf16_bits(mid))
    assert np.all(got % 2 == 0)
    # overflow: the midpoint above the largest finite value rounds to infinity
    big = np.float32((2 - 2**-8) * 2.0**127)
    assert oracle.f32_to_bf16([big])[0] == 0x7F80


def test_bf16_from_double_rounds_once():
    # 1 + 2^-8 + 2^-40 lies just above the midpoint of 1 and 1 + 2^-7: a direct
    # rounding gives 1 + 2^-7 (0x3F81); rounding through fp32 first would lose
    # the 2^-40 and give the even neighbour 1.0 (0x3F80).
    assert oracle.f64_to_bf16([1 + 2**-8 + 2**-40])[0] == 0x3F81
    assert oracle.f64_to_bf16([1 + 2**-8])[0] == 0x3F80
    assert oracle.f64_to_bf16([-(1 + 3 * 2**-8)])[0] == 0xBF82
    # nearest by brute force against the two neighbours
    d = rng.normal(0, 3, 5000)
    c = oracle.f64_to_bf16(d).astype(np.int64)
    val = oracle.bf16_to_f32(c.astype(np.uint16)).astype(np.float64)
    for delta in (-1, 1):
        nb = oracle.bf16_to_f32((c + delta).astype(np.uint16)).astype(np.float64)
        assert np.all(np.abs(d - val) <= np.abs(d - nb))


# ------------------------------------------------------------------- e4m3 --

def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    ref = torch_e4m3_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448 and ours[0x01] == 2.0**-9 and ours[0x08] == 2.0**-6


def test_e4m3_encode_matches_torch_in_range_and_at_midpoints():
    mags = np.exp2(rng.uniform(-14, math.log2(448), 20000)).astype(np.float32)
    x = np.where(rng.random(20000) < 0.5, -mags, mags).astype(np.float32)
    assert np.array_equal(oracle.f32_to_e4m3(x), torch_e4m3_codes(x))
    pos = np.arange(0, 0x7E, dtype=np.uint8)
    a = oracle.e4m3_to_f32(pos).astype(np.float64)
    b = oracle.e4m3_to_f32(pos + 1).astype(np.float64)
    mid = ((a + b) / 2).astype(np.float32)
    got = oracle.f32_to_e4m3(mid)
    assert np.array_equal(got, torch_e4m3_codes(mid))
    assert np.all(got % 2 == 0)           # ties to the even mantissa
    # round-trip of every finite code
    fin = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    back = oracle.f32_to_e4m3(oracle.e4m3_to_f32(fin))
    assert np.array_equal(back, fin)


def test_e4m3_saturation_sign_and_nan():
    over = np.array([448.0, 449.0, 463.9, 464.0, 479.0, 480.0, 1e6, np.inf], np.float32)
    assert np.all(oracle.f32_to_e4m3(over) == 0x7E)
    assert np.all(oracle.f32_to_e4m3(-over) == 0xFE)
    assert oracle.f32_to_e4m3([np.nan])[0] == 0x7F
    # a negative value that rounds to zero keeps the sign bit, as torch does
    tiny = np.array([-1e-10, -2.0**-11], np.float32)
    assert np.all(oracle.f32_to_e4m3(tiny) == 0x80)
    assert np.array_equal(oracle.f32_to_e4m3(tiny), torch_e4m3_codes(tiny))
    assert oracle.f32_to_e4m3([2.0**-10])[0] == 0x00     # half of 2^-9 ties to 0
    assert oracle.f32_to_e4m3([3 * 2.0**-10])[0] == 0x02  # 1.5 * 2^-9 ties to 2 * 2^-9


# ------------------------------------------------------- stage 1: reduce --

def _rows(vals_per_partial, residual, w, H, R=1):
    k = len(vals_per_partial)
    p = np.stack([np.full((R, H), bf16_bits_of(v), np.uint16) for v in vals_per_partial])
    r = np.full((R, H), bf16_bits_of(residual), np.uint16)
    wv = np.full(H, bf16_bits_of(w), np.uint16)
    return p, r, wv


def test_reduce_integer_inputs_sum_exactly():
    k, R, H = 5, 3, 256
    ints = rng.integers(-100, 101, (k + 1, R, H)).astype(np.float32)
    p = np.stack([bf16_bits_of(ints[i]) for i in range(k)])
    r = bf16_bits_of(ints[k])
    w = bf16_bits_of(np.ones(H, np.float32))
    o = oracle.reduce_norm_quant(p, r, w, want_x=True)
    assert np.array_equal(o["x"], ints.sum(axis=0))
    # k = 1 with a zero residual is the identity on x
    o1 = oracle.reduce_norm_quant(p[:1], np.zeros_like(r), w, want_x=True)
    assert np.array_equal(o1["x"], ints[0])


def test_reduce_is_fp32_in_partial_order_without_bf16_rounding():
    H = 128
    # (2^24 + 1) + -2^24 in fp32 is 0: the sum is taken left to right in fp32
    p, r, w = _rows([2.0**24, 1.0, -(2.0**24)], 0.0, 1.0, H)
    assert np.all(oracle.reduce_norm_quant(p, r, w, want_x=True)["x"] == 0.0)
    # 1 + 2^-8 is exact in fp32 but would round to 1.0 in bf16: no
    # intermediate bf16 rounding of the partial sum
    p, r, w = _rows([1.0, 2.0**-8], 0.0, 1.0, H)
    assert np.all(oracle.reduce_norm_quant(p, r, w, want_x=True)["x"] == np.float32(1 + 2**-8))
    # the residual is added after the partials: (2^24 + 1) - 2^24 + 1 = 1
    p, r, w = _rows([2.0**24, 1.0, -(2.0**24)], 1.0, 1.0, H)
    assert np.all(oracle.reduce_norm_quant(p, r, w, want_x=True)["x"] == 1.0)


# --------------------------------------------------------- stage 1: norm --

def _load_golden():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "norm_quant_constant_rows.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(None, 1)
            if key == "case":
                cur = {"name": val}
                cases.append(cur)
            else:
                cur[key] = val
    return cases


@pytest.mark.parametrize("case", _load_golden(), ids=lambda c: c["name"])
def test_golden_hand_derived_rows(case):
    H = int(case["H"])
    pv = [float(v) for v in case["p"].split(",")]
    p, r, w = _rows(pv, float(case["r"]), float(case["w"]), H, R=2)
    o = oracle.reduce_norm_quant(p, r, w)
    assert np.all(o["hidden"] == int(case["hidden"], 16))
    assert np.all(o["scales"].view(np.uint32) == int(case["scale"], 16))
    assert np.all(o["codes"] == int(case["code"], 16))


def test_rmsnorm_unit_weight_has_rms_one():
    R, H, k = 6, 1024, 3
    p = bf16_bits_of(torch.randn(k, R, H, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).float().numpy())
    r = np.zeros((R, H), np.uint16)
    w = bf16_bits_of(np.ones(H, np.float32))
    o = oracle.reduce_norm_quant(p, r, w, want_x=True)
    y = oracle.bf16_to_f32(o["hidden"]).astype(np.float64)
    x = o["x"].astype(np.float64)
    ms = (x * x).mean(axis=1)
    rms_exact = np.sqrt(ms / (ms + 1e-6))          # closed form of RMS(x * rsqrt(ms+eps))
    rms = np.sqrt((y * y).mean(axis=1))
    assert np.allclose(rms, rms_exact, rtol=2**-8, atol=0)
    assert np.allclose(rms, 1.0, rtol=2**-8)
    # the rounding is to the nearest bf16 of the exact fp64 value, element-wise
    exact = x * (1.0 / np.sqrt(ms + 1e-6))[:, None]
    assert np.array_equal(o["hidden"].ravel(), oracle.f64_to_bf16(exact.ravel()))


def test_rmsnorm_weight_scales_output_and_sign():
    R, H = 2, 256
    g = torch.Generator().manual_seed(7)
    p = bf16_bits_of(torch.randn(2, R, H, generator=g).to(torch.bfloat16).float().numpy())
    r = bf16_bits_of(torch.randn(R, H, generator=g).to(torch.bfloat16).float().numpy())
    wf = torch.randn(H, generator=g).to(torch.bfloat16).float().numpy()
    a = oracle.reduce_norm_quant(p, r, bf16_bits_of(wf))
    b = oracle.reduce_norm_quant(p, r, bf16_bits_of(-2 * wf))
    ya = oracle.bf16_to_f32(a["hidden"])
    yb = oracle.bf16_to_f32(b["hidden"])
    assert np.array_equal(yb, -2 * ya)               # power-of-two scaling is exact
    assert np.array_equal(b["scales"], 2 * a["scales"])
    # per-element weight: a weight that is zero on one column zeroes that column only
    wz = wf.copy()
    wz[17] = 0.0
    c = oracle.reduce_norm_quant(p, r, bf16_bits_of(wz))
    yc = oracle.bf16_to_f32(c["hidden"])
    assert np.all(yc[:, 17] == 0) and np.array_equal(np.delete(yc, 17, 1), np.delete(ya, 17, 1))


# -------------------------------------------------------- stage 1: quant --

def _random_stage1(R=8, H=1024, k=4, seed=3):
    g = torch.Generator().manual_seed(seed)
    p = bf16_bits_of(torch.randn(k, R, H, generator=g).mul(0.5).to(torch.bfloat16).float().numpy())
    r = bf16_bits_of(torch.randn(R, H, generator=g).to(torch.bfloat16).float().numpy())
    w = bf16_bits_of((1 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16).float().numpy())
    return p, r, w


def test_quant_error_bound_amax_code_and_monotone():
    p, r, w = _random_stage1()
    o = oracle.reduce_norm_quant(p, r, w)
    R, H = o["hidden"].shape
    y = oracle.bf16_to_f32(o["hidden"]).reshape(R, H // 128, 128).astype(np.float64)
    s = o["scales"].astype(np.float64)[:, :, None]
    q = oracle.e4m3_to_f32(o["codes"]).reshape(R, H // 128, 128).astype(np.float64)
    amax = np.abs(y).max(axis=2)
    assert np.array_equal(o["scales"], (amax.astype(np.float32) / np.float32(448)))
    # half an e4m3 step of |y/scale| times the scale (plus the fp32 division's rounding)
    v = np.abs(y / s)
    e = np.floor(np.log2(np.maximum(v, 2.0**-6)))
    ulp = np.where(v < 2.0**-6, 2.0**-9, 2.0**(e - 3))
    assert np.all(np.abs(y - q * s) <= (0.5 * ulp * (1 + 2**-20) + 2**-22 * v) * s)
    # the group's largest magnitude maps to +-448
    codes = o["codes"].reshape(R, H // 128, 128)
    at = np.abs(y).argmax(axis=2)
    top = np.take_along_axis(codes, at[:, :, None], 2)[:, :, 0]
    assert np.all((top & 0x7F) == 0x7E)
    # codes are monotone in the hidden value inside a group
    order = np.argsort(y, axis=2, kind="stable")
    qs = np.take_along_axis(q, order, 2)
    assert np.all(np.diff(qs, axis=2) >= 0)


def test_quant_reads_the_emitted_bf16_hidden():
    """The packed FP8 equals quantising the BF16 hidden that is returned, so a
    consumer can rely on the pair without requantising."""
    p, r, w = _random_stage1(R=3, H=512, k=2, seed=11)
    o = oracle.reduce_norm_quant(p, r, w)
    y = oracle.bf16_to_f32(o["hidden"])
    R, H = y.shape
    sc = np.abs(y.reshape(R, H // 128, 128)).max(axis=2) / np.float32(448)
    v = (y.reshape(R, H // 128, 128) / sc[:, :, None]).astype(np.float32)
    assert np.array_equal(o["codes"].ravel(), torch_e4m3_codes(v.ravel()))


# -------------------------------------------------------------- LM head --

def _rand_codes(shape, g):
    c = torch.randint(0, 256, shape, generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C        # no NaN codes
    return c


def test_lm_head_one_hot_activation_gives_dequantised_column():
    g = torch.Generator().manual_seed(2)
    T, H, V = 3, 384, 300
    qw = _rand_codes((V, H), g)
    sw = torch.rand(((V + 127) // 128, H // 128), generator=g).numpy().astype(np.float32) + 0.5
    qa = np.zeros((T, H), np.uint8)
    ks = [5, 130, 383]
    for t, k0 in enumerate(ks):
        qa[t, k0] = 0x38                  # e4m3 1.0
    sa = np.ones((T, H // 128), np.float32)
    L = oracle.lm_head_logits(qa, sa, qw, sw)
    for t, k0 in enumerate(ks):
        col = oracle.e4m3_to_f32(qw[:, k0]) * sw[np.arange(V) // 128, k0 // 128]
        assert np.array_equal(L[t], col.astype(np.float32))


def test_lm_head_within_higham_bound_of_fp64_gemm():
    g = torch.Generator().manual_seed(4)
    T, H, V = 4, 512, 257
    qa = _rand_codes((T, H), g)
    qw = _rand_codes((V, H), g)
    sa = (torch.rand((T, H // 128), generator=g) * 0.01).numpy().astype(np.float32)
    sw = (torch.rand(((V + 127) // 128, H // 128), generator=g) * 0.001).numpy().astype(np.float32)
    L = oracle.lm_head_logits(qa, sa, qw, sw).astype(np.float64)
    A = torch_e4m3_decode(qa).astype(np.float64) * np.repeat(sa, 128, axis=1)
    W = torch_e4m3_decode(qw).astype(np.float64) * np.repeat(sw, 128, axis=1)[np.arange(V) // 128]
    L64 = A @ W.T
    absL = np.abs(A) @ np.abs(W).T
    u = 2.0**-24
    gamma = (H + 2) * u / (1 - (H + 2) * u)          # products of three roundings + H-term sum
    assert np.all(np.abs(L - L64) <= gamma * absL)
    # sub-range and token selection agree with the full computation
    part = oracle.lm_head_logits(qa, sa, qw, sw, tokens=[3, 1], v0=100, v1=140)
    assert np.array_equal(part, L[[3, 1], 100:140].astype(np.float32))


# --------------------------------------------------------------- argmax --

def _brute(L, S):
    n, V = L.shape
    tok = np.empty(n, np.int64)
    for i in range(n):
        order = np.lexsort((np.arange(V), -L[i].astype(np.float64)))
        tok[i] = order[0]
    w = V // S
    sidx = np.empty((n, S), np.int64)
    for s in range(S):
        for i in range(n):
            seg = L[i, s * w:(s + 1) * w].astype(np.float64)
            sidx[i, s] = s * w + np.lexsort((np.arange(w), -seg))[0]
    return tok, sidx


def test_argmax_matches_sort_based_brute_force_with_many_ties():
    L = rng.integers(-3, 4, (50, 24)).astype(np.float32)
    for S in (1, 2, 3, 4, 6, 8):
        r = oracle.argmax(L, S)
        tok, sidx = _brute(L, S)
        assert np.array_equal(r["tokens"], tok)
        assert np.array_equal(r["shard_idx"], sidx)
        assert np.array_equal(r["values"], L[np.arange(50), tok])


def test_argmax_planted_ties_across_shard_boundaries_and_signed_zero():
    V, S = 32, 4
    L = np.full((6, V), -1.0, np.float32)
    L[0, [7, 8]] = 5.0                 # straddles the shard 0 / shard 1 boundary
    L[1, [8, 7]] = 5.0
    L[2, [0, V - 1]] = 2.0             # first and last index
    L[3, :] = -0.0
    L[3, 9] = 0.0                      # -0 == +0: lowest index wins
    L[4, [31, 24, 23]] = 3.0
    L[5, 15] = np.float32(1.0)
    L[5, 16] = np.nextafter(np.float32(1.0), np.float32(2.0))
    r = oracle.argmax(L, S)
    assert list(r["tokens"]) == [7, 7, 0, 0, 23, 16]
    assert list(r["shard_idx"][0]) == [7, 8, 16, 24]
    assert list(r["shard_idx"][4]) == [0, 8, 23, 24]
    assert r["gap"][0] == 0 and r["gap"][2] == 0 and r["gap"][5] > 0


# The relative top-2 gap decides which draft ids must match exactly (gap >= 1e-3
# or gap == 0) and which are near ties, so its value is pinned, not only its
# sign: gap = (L1 - L2) / |L1| with L2 the best logit at another index, and
# L1 - L2 when L1 == 0.  Each row below is built so that one plausible slip
# gives a different value: dividing by L2 ([4, 2] -> 1.0), dropping the
# absolute value ([-2, -3] -> -0.5), taking L2 as the second-largest distinct
# value ([3, 3, 1] -> 2/3), or dividing by zero when L1 == 0.
GAP_ROWS = [
    ([4.0, 3.0, -1.0, 0.0], 0.25),
    ([4.0, 2.0], 0.5),
    ([-2.0, -3.0, -7.0], 0.5),
    ([0.0, -0.5, -4.0], 0.5),
    ([-0.0, -0.25], 0.25),
    ([3.0, 3.0, 1.0], 0.0),
    ([1.0, 5.0, 2.0, 5.0, 4.0], 0.0),
    ([-1.0, 0.5, 0.25, -3.0], 0.5),
    ([8.0, 6.0, 7.0, 1.0], 0.125),
]


@pytest.mark.parametrize("row,gap", GAP_ROWS)
def test_argmax_gap_value_hand_computed(row, gap):
    L = np.array([row], np.float32)
    r = oracle.argmax(L, 1)
    assert r["gap"][0] == gap


def test_argmax_gap_value_is_placed_by_row_not_shard():
    """The gap is taken over the whole vocabulary; the runner-up may sit in
    another shard than the maximum."""
    L = np.full((1, 16), -9.0, np.float32)
    L[0, 2] = 10.0
    L[0, 13] = 8.0                     # shard 3 of 4
    assert oracle.argmax(L, 4)["gap"][0] == 0.2


def test_argmax_gap_value_matches_a_sorted_copy():
    """Brute force on random rows with repeated values: sort a copy in
    descending order, L1 the first element and L2 the second (which equals L1
    when the maximum is repeated), gap in fp64 from the fp32 values."""
    for n, V, lo, hi in ((40, 9, -4, 5), (40, 33, -2, 3), (20, 200, -50, 50)):
        L = (rng.integers(lo, hi, (n, V)) / 4.0).astype(np.float32)
        L[:5] += rng.normal(0, 1, (5, V)).astype(np.float32)
        r = oracle.argmax(L, 1)
        for i in range(n):
            s = np.sort(L[i].astype(np.float64))[::-1]
            want = (s[0] - s[1]) if s[0] == 0 else (s[0] - s[1]) / abs(s[0])
            assert r["gap"][i] == want, (i, L[i], r["gap"][i], want)


# ----------------------------------------------------------- tie stress --

def test_tie_stress_construction_is_reproduced_by_the_oracle():
    import synth
    w = synth.workload("tie_stress", T=24, H=512, k=2, V=4096, S=8)
    inp = synth.stage1_inputs(w)
    o = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"])
    qw, sw = synth.lm_head_weights(w)
    expected = synth.plant_ties(w, qw, sw, o["codes"])
    assert len(expected) == round(0.3 * 24)
    L = oracle.lm_head_logits(o["codes"], o["scales"], qw, sw)
    r = oracle.argmax(L, w.S)
    width = w.V // w.S
    for t, row in expected.items():
        assert r["tokens"][t] == row
        assert r["gap"][t] == 0.0                       # an exact duplicate maximum
        twin = [v for v in range(w.V) if v != row and L[t, v] == L[t, row]]
        assert len(twin) == 1 and twin[0] // width == row // width + 1


# ------------------------------------------------------------------ NVFP4 --
# OCP Microscaling Formats v1.0, FP4 E2M1: the eight magnitudes of the format.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_matches_the_format_table():
    got = oracle.e2m1_to_f32(np.arange(16))
    for c in range(16):
        want = -E2M1_TABLE[c & 7] if c & 8 else E2M1_TABLE[c & 7]
        assert got[c] == want and (math.copysign(1, got[c]) < 0) == bool(c & 8)


def _e2m1_brute(x):
    """nearest of the eight magnitudes, ties to the even code (mantissa bit 0),
    saturating at 6; the sign is kept."""
    a = min(abs(float(x)), 6.0)
    d = [abs(a - v) for v in E2M1_TABLE]
    best = min(d)
    cands = [i for i in range(8) if d[i] == best]
    c = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
    return c | (8 if math.copysign(1, x) < 0 else 0)


def test_e2m1_encode_is_nearest_even_by_brute_force():
    xs = list(rng.uniform(-8, 8, 4000).astype(np.float32))
    mids = [(E2M1_TABLE[i] + E2M1_TABLE[i + 1]) / 2 for i in range(7)]
    xs += mids + [-m for m in mids] + [6.0, 6.5, 7.0, 1e9, -1e9, 0.0, -0.0, 1e-30, -1e-30]
    got = oracle.f32_to_e2m1(np.array(xs, np.float32))
    for x, g in zip(xs, got):
        assert g == _e2m1_brute(np.float32(x)), (x, g)
    # every code survives a round trip
    assert np.array_equal(oracle.f32_to_e2m1(oracle.e2m1_to_f32(np.arange(16))), np.arange(16))


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def _unpack(codes):
    c = np.asarray(codes, np.uint8)
    return np.stack([c & 15, c >> 4], axis=-1).reshape(c.shape[0], -1)


def test_nvfp4_quant_hand_derived_two_blocks():
    g = _read_golden("nvfp4_two_blocks.txt")
    vals = np.array([float(v) for v in g["values"]], np.float32)
    q = oracle.nvfp4_quant(bf16_bits_of(vals)[None, :])
    assert q["global_scales"][0] == np.float32(g["row_scale"][0])
    assert q["block_scales"][0].tolist() == [int(v, 16) for v in g["block_scales"]]
    assert _unpack(q["codes"])[0].tolist() == [int(v) for v in g["codes"]]


def _random_rows(R, H, seed):
    r = np.random.default_rng(seed)
    x = r.normal(0, 1, (R, H)).astype(np.float32) * np.exp2(r.integers(-6, 6, (R, 1))).astype(np.float32)
    x[:, r.integers(0, H, 3)] *= 30.0     # a few outlier channels
    return torch_bf16_bits(x)


def test_nvfp4_quant_invariants():
    R, H = 24, 512
    hid = _random_rows(R, H, 7)
    hid[3] = 0                      # an all-zero row
    hid[5, 32:48] = 0               # an all-zero block
    q = oracle.nvfp4_quant(hid)
    y = oracle.bf16_to_f32(hid).reshape(R, H)
    codes = _unpack(q["codes"])
    vals = np.where(codes & 8, -1.0, 1.0) * np.array(E2M1_TABLE)[codes & 7]
    sb = torch_e4m3_decode(q["block_scales"]).astype(np.float64)
    gs = q["global_scales"].astype(np.float64)
    for r in range(R):
        amax = np.abs(y[r]).max()
        if amax == 0:
            assert gs[r] == 0 and not q["block_scales"][r].any() and not codes[r].any()
            continue
        # the row scale is amax / (448 * 6) and the row's largest block scale is 448
        assert gs[r] == np.float32(np.float32(amax) / np.float32(2688.0))
        assert q["block_scales"][r].max() == 0x7E
        for b in range(H // 16):
            blk = y[r, 16 * b:16 * b + 16].astype(np.float64)
            eff = np.float32(np.float32(sb[r, b]) * np.float32(gs[r]))
            cb = codes[r, 16 * b:16 * b + 16]
            if eff == 0:
                assert not cb.any()
                continue
            # each code is the nearest e2m1 value of y / eff (brute force)
            for j in range(16):
                assert cb[j] == _e2m1_brute(np.float32(np.float32(blk[j]) / eff))
            # a block whose scale is a normal e4m3 value maps its maximum to +-6
            if sb[r, b] >= 2.0 ** -6:
                jm = int(np.argmax(np.abs(blk)))
                assert abs(vals[r, 16 * b + jm]) == 6.0
            # reconstruction within half an e2m1 step of the scaled value
            step = np.where(np.abs(blk) / eff < 2, 0.5, np.where(np.abs(blk) / eff < 4, 1.0, 2.0))
            err = np.abs(blk - vals[r, 16 * b:16 * b + 16] * eff)
            assert np.all(err <= 0.5 * step * eff * (1 + 1e-6) + 1e-30)


def test_nvfp4_quant_is_invariant_to_power_of_two_row_scaling():
    hid = _random_rows(6, 256, 11)
    y = oracle.bf16_to_f32(hid).reshape(6, 256)
    q1 = oracle.nvfp4_quant(hid)
    q2 = oracle.nvfp4_quant(bf16_bits_of(y * np.float32(8.0)))
    assert np.array_equal(q1["codes"], q2["codes"])
    assert np.array_equal(q1["block_scales"], q2["block_scales"])
    assert np.array_equal(q2["global_scales"], q1["global_scales"] * np.float32(8.0))


def _nvfp4_dequant(codes, bs, gs):
    c = _unpack(codes)
    v = np.where(c & 8, -1.0, 1.0) * np.array(E2M1_TABLE)[c & 7]
    s = torch_e4m3_decode(bs).astype(np.float64)
    return v * np.repeat(s, 16, axis=1) * np.asarray(gs, np.float64)[:, None]


def test_nvfp4_lm_head_one_hot_activation_gives_a_weight_column():
    H, V = 256, 40
    w = oracle.nvfp4_quant(_random_rows(V, H, 3))
    gw = np.float32(0.75)
    for k in (0, 1, 17, 255):
        codes = np.zeros((1, H // 2), np.uint8)
        codes[0, k // 2] = 0x2 << (4 * (k % 2))            # e2m1 1.0 at element k
        sa = np.zeros((1, H // 16), np.uint8)
        sa[0, k // 16] = 0x38                               # block scale 1.0
        L = oracle.lm_head_logits_nvfp4(codes, sa, np.ones(1, np.float32), w["codes"],
                                        w["block_scales"], gw)
        wd = _nvfp4_dequant(w["codes"], w["block_scales"], np.ones(V))
        want = (wd[:, k].astype(np.float32) * gw).astype(np.float32)
        assert np.array_equal(L[0], want)


def test_nvfp4_lm_head_matches_fp64_within_the_summation_bound():
    H, V, T = 512, 96, 5
    a = oracle.nvfp4_quant(_random_rows(T, H, 21))
    w = oracle.nvfp4_quant(_random_rows(V, H, 22))
    gw = np.float32(0.01)
    L = oracle.lm_head_logits_nvfp4(a["codes"], a["block_scales"], a["global_scales"],
                                    w["codes"], w["block_scales"], gw)
    ad = _nvfp4_dequant(a["codes"], a["block_scales"], np.ones(T))
    wd = _nvfp4_dequant(w["codes"], w["block_scales"], np.ones(V))
    exact = ad @ wd.T
    absd = np.abs(ad) @ np.abs(wd).T
    n = H // 16 + 2
    gam = n * 2.0 ** -24 / (1 - n * 2.0 ** -24)
    scale = a["global_scales"].astype(np.float64)[:, None] * float(gw)
    assert np.all(np.abs(L - exact * scale) <= gam * absd * scale + 1e-30)
    # the activation row scale and the weight scale enter as plain factors
    L2 = oracle.lm_head_logits_nvfp4(a["codes"], a["block_scales"], a["global_scales"] * 2,
                                     w["codes"], w["block_scales"], gw)
    assert np.array_equal(L2, L * 2)
    # transposing the roles of tokens and rows gives the transposed logits
    Lt = oracle.lm_head_logits_nvfp4(w["codes"], w["block_scales"], np.ones(V, np.float32),
                                     a["codes"], a["block_scales"], np.float32(1.0))
    assert np.allclose(Lt.T * scale, L, rtol=1e-5, atol=0)


# --------------------------------------------------- unfused reference arm --

def test_unfused_reduce_rounds_the_sum_once_to_bf16():
    # 1 + 2^-8 + 2^-9: the fp32 sum is exact, its BF16 rounding goes up to
    # 1 + 2^-7 (above the midpoint); the fused path would keep the fp32 value
    p = np.array([[[1.0, 3.0]], [[2.0 ** -8, -1.0]], [[2.0 ** -9, 0.5]]], np.float32)
    bits = np.stack([bf16_bits_of(p[i]) for i in range(3)])
    s = oracle.unfused_reduce_bf16(bits)
    assert oracle.bf16_to_f32(s).tolist() == [[1.0 + 2.0 ** -7, 2.5]]
    # k = 1 is the identity; integer partials sum exactly
    x = torch_bf16_bits(rng.normal(0, 3, (3, 64)).astype(np.float32))
    assert np.array_equal(oracle.unfused_reduce_bf16(x[None]), x)
    ints = rng.integers(-50, 50, (4, 2, 32)).astype(np.float32)
    got = oracle.bf16_to_f32(oracle.unfused_reduce_bf16(np.stack([bf16_bits_of(v) for v in ints])))
    assert np.array_equal(got, ints.sum(axis=0))


def test_unfused_norm_and_quant_equal_the_fused_ones_on_the_same_sum():
    """With k = 1 and a zero partial the unfused chain reduces to the fused
    stage 1 (no rounding is added): a cross-check of the two oracle paths."""
    R, H = 5, 384
    x = torch_bf16_bits(rng.normal(0, 1, (R, H)).astype(np.float32))
    res = torch_bf16_bits(rng.normal(0, 1, (R, H)).astype(np.float32))
    w = torch_bf16_bits((1 + rng.normal(0, 0.1, H)).astype(np.float32))
    fused = oracle.reduce_norm_quant(x[None], res, w)
    hid = oracle.unfused_add_rmsnorm(x, res, w)
    assert np.array_equal(hid, fused["hidden"])
    q = oracle.quant_fp8_rows(hid)
    assert np.array_equal(q["codes"], fused["codes"]) and np.array_equal(q["scales"], fused["scales"])
    # the group quantiser equals torch's e4m3 cast of hidden / (amax / 448)
    y = oracle.bf16_to_f32(hid).reshape(R, H // 128, 128)
    sc = (np.abs(y).max(axis=2) / np.float32(448)).astype(np.float32)
    want = torch_e4m3_codes((y / sc[:, :, None]).astype(np.float32)).reshape(R, H)
    assert np.array_equal(q["codes"], want)


def test_bf16_argmax_is_lowest_index_by_brute_force():
    for trial in range(20):
        r = np.random.default_rng(trial)
        L = r.integers(-3, 4, (3, 37)).astype(np.float32)   # many exact ties
        L[0, 5] = -0.0
        bits = bf16_bits_of(L)
        tok = oracle.argmax_bf16(bits)
        for i in range(3):
            m = L[i].max()
            assert tok[i] == min(v for v in range(37) if L[i, v] == m)


# ------------------------------------------------------------- end to end --

def e2e_golden_inputs():
    """The inputs of tests/golden/e2e_two_tokens.txt, as the arrays both sides
    take: partials [k][T][H], residual [T][H], norm weight [H] (BF16 bits), the
    weight codes [V][H] and block scales [1][H/128]."""
    g = _read_golden("e2e_two_tokens.txt")
    H = int(g["H"][0])
    T = 2
    k = len(g["partials_t0"])
    p = np.zeros((k, T, H), np.float32)
    r = np.zeros((T, H), np.float32)
    for t in range(T):
        for j, v in enumerate(g[f"partials_t{t}"]):
            p[j, t, :] = float(v)
        r[t, :] = float(g[f"residual_t{t}"][0])
    w = np.empty(H, np.float32)
    w[:128] = float(g["w_group0"][0])
    w[128::2] = float(g["w_group1_even"][0])
    w[129::2] = float(g["w_group1_odd"][0])
    qw = np.zeros((4, H), np.uint8)
    qw[0, :] = 0x38
    qw[1, :128], qw[1, 128:] = 0x38, 0xB8
    qw[2, :64] = 0x40
    qw[3, 255] = 0x38
    sw = np.array([[float(v) for v in g["wsc"]]], np.float32)
    return g, bf16_bits_of(p), bf16_bits_of(r), bf16_bits_of(w), qw, sw


def test_end_to_end_hand_derived_two_tokens():
    """Stage 1 into the LM head and the sharded argmax on a case worked by hand
    (tests/golden/e2e_two_tokens.txt): pins how the packed activation, its
    scales and the weight block scales compose, and the argmax outputs."""
    g, p, r, w, qw, sw = e2e_golden_inputs()
    H = p.shape[2]
    o = oracle.reduce_norm_quant(p, r, w)
    for t in range(2):
        h0, h1e, h1o = (int(v, 16) for v in g[f"hidden_t{t}"])
        assert np.all(o["hidden"][t, :128] == h0)
        assert np.all(o["hidden"][t, 128::2] == h1e) and np.all(o["hidden"][t, 129::2] == h1o)
        c0, c1e, c1o = (int(v, 16) for v in g[f"codes_t{t}"])
        assert np.all(o["codes"][t, :128] == c0)
        assert np.all(o["codes"][t, 128::2] == c1e) and np.all(o["codes"][t, 129::2] == c1o)
        assert o["scales"][t].view(np.uint32).tolist() == [int(v, 16) for v in g["scales"]]
    L = oracle.lm_head_logits(o["codes"], o["scales"], qw, sw)
    assert L.shape == (2, 4)
    for t in range(2):
        assert L[t].tolist() == [float(v) for v in g[f"logits_t{t}"]]
    a = oracle.argmax(L, 2)
    assert a["tokens"].tolist() == [int(v) for v in g["tokens"]]
    for t in range(2):
        assert a["shard_idx"][t].tolist() == [int(v) for v in g[f"shard_idx_t{t}"]]
        assert a["shard_val"][t].tolist() == [float(v) for v in g[f"shard_val_t{t}"]]
    assert H == 256


def nvfp4_e2e_golden_inputs():
    """The inputs of tests/golden/nvfp4_e2e_two_tokens.txt: partials [k][T][H],
    residual [T][H], norm weight [H] (BF16 bits), the NVFP4 weight codes
    [V][H/2] (packed), block scales [V][H/16] and its tensor scale."""
    g = _read_golden("nvfp4_e2e_two_tokens.txt")
    H, T = int(g["H"][0]), 2
    k = len(g["partials_t0"])
    p = np.zeros((k, T, H), np.float32)
    r = np.zeros((T, H), np.float32)
    for t in range(T):
        for j, v in enumerate(g[f"partials_t{t}"]):
            p[j, t, :] = float(v)
        r[t, :] = float(g[f"residual_t{t}"][0])
    w = np.empty(H, np.float32)
    w[:16] = np.tile([float(v) for v in g["w_block0"]], 4)
    w[16:] = np.tile([float(v) for v in g["w_rest"]], (H - 16) // 2)
    qw = np.zeros((4, H // 2), np.uint8)
    sw = np.full((4, H // 16), 0x38, np.uint8)
    qw[0, :] = 0x22
    qw[1, :8] = 0x22
    sw[1, 0] = 0x40
    qw[2, :] = 0x99
    qw[3, H // 2 - 1] = 0x70
    sw[3, H // 16 - 1] = 0x30
    return g, bf16_bits_of(p), bf16_bits_of(r), bf16_bits_of(w), qw, sw, float(g["gw"][0])


def check_nvfp4_e2e_stage1(g, hidden, codes, block_scales, row_scales):
    """Stage 1 of the NVFP4 hand-derived case against its expected bytes."""
    for t in range(2):
        h = [int(v, 16) for v in g[f"hidden_t{t}"]]
        assert hidden[t, :16].tolist() == h[:4] * 4
        assert hidden[t, 16:].tolist() == h[4:6] * 120
        c = [int(v, 16) for v in g[f"codes_t{t}"]]
        assert codes[t, :8].tolist() == c[:2] * 4
        assert np.all(codes[t, 8:] == c[2])
        b0, b1 = (int(v, 16) for v in g["block_scales"])
        assert block_scales[t, 0] == b0 and np.all(block_scales[t, 1:] == b1)
        assert np.float32(row_scales[t]).view(np.uint32) == int(g["row_scale"][0], 16)


def test_nvfp4_end_to_end_hand_derived_two_tokens():
    """The NVFP4 stage 1 into the NVFP4 LM head and the sharded argmax on a case
    worked by hand (tests/golden/nvfp4_e2e_two_tokens.txt): pins the packing
    order, which block scale meets which, the row and tensor scales, and the
    argmax outputs."""
    g, p, r, w, qw, sw, gw = nvfp4_e2e_golden_inputs()
    o = oracle.reduce_norm_quant_nvfp4(p, r, w)
    check_nvfp4_e2e_stage1(g, o["hidden"], o["codes"], o["block_scales"], o["global_scales"])
    L = oracle.lm_head_logits_nvfp4(o["codes"], o["block_scales"], o["global_scales"], qw, sw, gw)
    for t in range(2):
        assert L[t].tolist() == [float(v) for v in g[f"logits_t{t}"]]
    a = oracle.argmax(L, 2)
    assert a["tokens"].tolist() == [int(v) for v in g["tokens"]]
    for t in range(2):
        assert a["shard_idx"][t].tolist() == [int(v) for v in g[f"shard_idx_t{t}"]]
        assert a["shard_val"][t].tolist() == [float(v) for v in g[f"shard_val_t{t}"]]


def test_unfused_end_to_end_hand_derived_two_tokens():
    """The unfused path on the hand-derived case: the BF16 all-reduce output,
    the hidden, the activation, the BF16 logits and the tokens are the values
    worked by hand in tests/golden/e2e_two_tokens.txt."""
    g, p, r, w, qw, sw = e2e_golden_inputs()
    u = oracle.unfused_step(p, r, w, qw, sw)
    s0, s1 = (int(v, 16) for v in g["unfused_sum"])
    assert np.all(u["sum"][0] == s0) and np.all(u["sum"][1] == s1)
    fused = oracle.reduce_norm_quant(p, r, w)
    for key in ("hidden", "codes", "scales"):
        assert np.array_equal(u[key], fused[key])
    for t in range(2):
        assert u["logits"][t].tolist() == [int(v, 16) for v in g[f"unfused_logits_t{t}"]]
    assert u["tokens"].tolist() == [int(v) for v in g["tokens"]]
