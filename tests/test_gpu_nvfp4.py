"""GPU parity of the NVFP4 variant — stage 1 with the NVFP4 activation and the
block-scaled NVFP4 LM head with the fused argmax — against the CPU oracle,
through the C ABI (via the Python binding)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import (bf16_host, check_stage1_fp4, check_stage2_fp4, to_dev,
                           to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def run_stage1(nfq, inp, eps=1e-6):
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    res = to_dev_bf16(inp["residual"])
    w = to_dev_bf16(inp["norm_w"])
    h, c, bs, gs = nfq.mtp_reduce_norm_quant_nvfp4(parts, res, w, eps)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    return bf16_host(h), c.cpu().numpy(), bs.cpu().numpy(), gs.cpu().numpy()


def oracle_stage1(inp, eps=1e-6):
    return oracle.reduce_norm_quant_nvfp4(inp["partials"], inp["residual"], inp["norm_w"], eps)


# ----------------------------------------------------------------- stage 1 --

@pytest.mark.parametrize("name", ["tiny", "decode_c1", "decode_c64", "tie_stress"])
def test_nvfp4_stage1_full_workloads(nfq, name):
    inp = synth.stage1_inputs(synth.workload(name))
    h, c, bs, gs = run_stage1(nfq, inp)
    check_stage1_fp4(h, c, bs, gs, oracle_stage1(inp)["hidden"])


@pytest.mark.parametrize("T,H,k", [(1, 256, 1), (3, 768, 3), (17, 1024, 16), (153, 2048, 2),
                                   (2, 16384, 4), (5, 7168, 8), (40, 1280, 5)])
def test_nvfp4_stage1_edge_shapes(nfq, T, H, k):
    inp = synth.stage1_inputs(synth.workload("tiny", T=T, H=H, k=k, seed=3 * T + H + k))
    h, c, bs, gs = run_stage1(nfq, inp)
    check_stage1_fp4(h, c, bs, gs, oracle_stage1(inp)["hidden"])


def test_nvfp4_stage1_prefill_sampled_rows(nfq):
    """T = 8192, H = 7168, k = 8: rows spread over the persistent grid."""
    w = synth.workload("prefill")
    inp = synth.stage1_inputs(w)
    h, c, bs, gs = run_stage1(nfq, inp)
    rows = sorted(set([0, 1, 151, 152, 4095, 8190, 8191] +
                      list(np.random.default_rng(1).integers(0, w.T, 13))))
    sub = synth.stage1_inputs(w, rows=rows)
    check_stage1_fp4(h[rows], c[rows], bs[rows], gs[rows], oracle_stage1(sub)["hidden"])


def test_nvfp4_stage1_degenerate_rows(nfq):
    """An all-zero row (row scale 0), a row with one huge channel (most block
    scales underflow to subnormal e4m3 or zero), tiny magnitudes, negative
    zeros and cancelling partials."""
    T, H, k = 5, 512, 2
    p = np.zeros((k, T, H), np.float32)
    r = np.zeros((T, H), np.float32)
    p[0, 1] = np.random.default_rng(2).normal(0, 1e-3, H)
    p[0, 1, 77] = 3.0e4
    p[0, 2] = np.random.default_rng(3).normal(0, 1, H) * 1e-25
    p[:, 3] = -0.0
    p[0, 4] = 5.0
    p[1, 4] = -5.0
    r[4] = np.linspace(-3, 3, H)
    bits = synth.to_bf16_bits
    inp = {"partials": np.stack([bits(p[i]) for i in range(k)]), "residual": bits(r),
           "norm_w": bits(np.linspace(0.5, 1.5, H).astype(np.float32))}
    h, c, bs, gs = run_stage1(nfq, inp)
    check_stage1_fp4(h, c, bs, gs, oracle_stage1(inp)["hidden"])
    assert gs[0] == 0 and not bs[0].any() and not (c[0] & 0x77).any()
    assert gs[3] == 0


# ------------------------------------------------------------- LM head --

_weights = {}


def fp4_weights(w):
    key = (w.V, w.H, w.seed, w.weight_std)
    if key not in _weights:
        _weights.clear()
        _weights[key] = synth.lm_head_weights_nvfp4(w)
    return _weights[key]


def run_lm(nfq, act, qw, sw, gw, S, ws=None):
    wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
    out = nfq.lm_head_nvfp4_argmax(to_dev(act["codes"]), to_dev(act["block_scales"]),
                                   to_dev(act["global_scales"]), wp, S, workspace=ws,
                                   want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    return [x.cpu().numpy() for x in out]


def check(tok, mx, sidx, sval, act, qw, sw, gw, S, sample, expected=None, cache_key=None):
    return check_stage2_fp4(tok, act["codes"], act["block_scales"], act["global_scales"], qw,
                            sw, gw, S, sample, mx, sidx, sval, expected, cache_key=cache_key)


def test_nvfp4_lm_head_tiny_all_tokens(nfq):
    w = synth.workload("tiny")
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = fp4_weights(w)
    out = run_lm(nfq, act, qw, sw, gw, w.S)
    check(*out, act, qw, sw, gw, w.S, list(range(w.T)))


def test_nvfp4_lm_head_decode_c1_full_vocab(nfq):
    """T = 1, V = 129280: shard boundaries fall inside 128-row blocks."""
    w = synth.workload("decode_c1")
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = fp4_weights(w)
    out = run_lm(nfq, act, qw, sw, gw, w.S)
    check(*out, act, qw, sw, gw, w.S, [0])


def test_nvfp4_lm_head_decode_c64_all_tokens(nfq):
    w = synth.workload("decode_c64")
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = fp4_weights(w)
    tok, mx, sidx, sval = run_lm(nfq, act, qw, sw, gw, w.S)
    assert tok.shape == (64,) and np.all((0 <= tok) & (tok < w.V))
    check(tok, mx, sidx, sval, act, qw, sw, gw, w.S, list(range(w.T)))


@pytest.mark.parametrize("T,H,V,S", [(1, 256, 128, 1), (2, 512, 200, 2), (31, 1024, 1000, 5),
                                     (33, 256, 4100, 4), (64, 768, 2048, 64),
                                     (100, 512, 3000, 3), (128, 256, 1536, 6),
                                     (129, 256, 1024, 8), (250, 512, 640, 5),
                                     (256, 256, 128, 1), (300, 512, 2000, 4),
                                     (513, 256, 1024, 2), (7, 16384, 1000, 4),
                                     (200, 16384, 700, 7)])
def test_nvfp4_lm_head_edge_shapes(nfq, T, H, V, S):
    """Ragged vocab tails, one-block tiles, shards narrower than a warp's
    columns, every lane quadrant, two token groups in one launch (129..256
    tokens, ragged second group) and several launches (300, 513 tokens)."""
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=T + H + V + S)
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = fp4_weights(w)
    out = run_lm(nfq, act, qw, sw, gw, S)
    check(*out, act, qw, sw, gw, S, list(range(T)))


def test_nvfp4_lm_head_planted_ties_and_zero_logits(nfq):
    """Exact duplicate rows (codes and block scales) inside a column group,
    across groups, across the two blocks of a tile, across tiles and shards
    and at the last row; an all-zero activation row gives every logit +-0 and
    token 0."""
    T, H, V, S = 6, 512, 1024, 4
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=8)
    act = oracle_stage1(synth.stage1_inputs(w))
    act = {k_: v.copy() for k_, v in act.items()}
    act["codes"][5] = 0
    act["block_scales"][5] = 0
    qw, sw, gw = (x.copy() if isinstance(x, np.ndarray) else x for x in fp4_weights(w))
    pairs = {0: (3, 17), 1: (40, 100), 2: (127, 128), 3: (255, 256), 4: (700, 1023)}
    for t, (a, b) in pairs.items():
        # e2m1 +-6 where the activation is positive / negative, 0 where it is 0;
        # the largest block scale everywhere: this row wins for token t
        u = np.stack([act["codes"][t] & 15, act["codes"][t] >> 4], axis=-1).reshape(-1)
        pat = np.where((u & 7) == 0, 0, np.where(u & 8, 0xF, 0x7)).astype(np.uint8)
        row = (pat[0::2] | (pat[1::2] << 4)).astype(np.uint8)
        for v in (a, b):
            qw[v] = row
            sw[v] = 0x7E
    tok, mx, sidx, sval = run_lm(nfq, act, qw, sw, gw, S)
    for t, (a, b) in pairs.items():
        assert tok[t] == a
    assert tok[5] == 0 and mx[5] == 0.0 and not np.signbit(mx[5])
    assert list(sidx[:, 5]) == [0, 256, 512, 768]
    check(tok, mx, sidx, sval, act, qw, sw, gw, S, list(range(T)),
          expected={t: a for t, (a, b) in pairs.items()})


def test_nvfp4_pair_planted_ties(nfq):
    """200 tokens on CTA pairs, tokens of both CTAs (0..127 and 128..199), with
    exact duplicate rows (codes and block scales).  With 256 blocks over 76
    pairs the first pair holds blocks 0..2: a one-block tile (rows 0..63 in the
    even CTA, 64..127 in the odd one), then blocks 1 and 2 as one tile (128..255
    even, 256..383 odd).  The duplicates sit across the halves of a one-block
    tile (63 | 64) and of a two-block tile (255 | 256), inside one half, across
    tiles (127 | 128), across pairs (383 | 384), across shards (8191 | 8192) and
    at the last row.  The lowest index wins, and the pair form matches two token
    groups byte for byte."""
    T, H, V, S = 200, 512, 32768, 4
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=21)
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = (x.copy() if isinstance(x, np.ndarray) else x for x in fp4_weights(w))
    pairs = {0: (63, 64), 5: (255, 256), 64: (3, 17), 127: (127, 128), 128: (383, 384),
             150: (8191, 8192), 190: (20000, 32767), 199: (300, 301)}
    for t, (a, b) in pairs.items():
        # e2m1 +-6 where the activation is positive / negative, 0 where it is 0;
        # the largest block scale everywhere: this row wins for token t
        u = np.stack([act["codes"][t] & 15, act["codes"][t] >> 4], axis=-1).reshape(-1)
        pat = np.where((u & 7) == 0, 0, np.where(u & 8, 0xF, 0x7)).astype(np.uint8)
        row = (pat[0::2] | (pat[1::2] << 4)).astype(np.uint8)
        for v in (a, b):
            qw[v] = row
            sw[v] = 0x7E
    pair = run_lm(nfq, act, qw, sw, gw, S)
    nfq.lm_head_pair(False)
    try:
        groups = run_lm(nfq, act, qw, sw, gw, S)
    finally:
        nfq.lm_head_pair(True)
    for x, y in zip(pair, groups):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    tok = pair[0]
    for t, (a, b) in pairs.items():
        assert tok[t] == a
    check(*pair, act, qw, sw, gw, S, list(range(T)),
          expected={t: a for t, (a, b) in pairs.items()})


def test_nvfp4_gpu_stage1_feeds_the_lm_head(nfq):
    """The two NVFP4 stages chained on the GPU: the LM head on the GPU's own
    activation agrees with the oracle's LM head on that activation."""
    w = synth.workload("tiny", T=40, H=1024, V=8192, S=8, seed=12)
    inp = synth.stage1_inputs(w)
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    h, c, bs, gs = nfq.mtp_reduce_norm_quant_nvfp4(parts, to_dev_bf16(inp["residual"]),
                                                   to_dev_bf16(inp["norm_w"]))
    qw, sw, gw = fp4_weights(w)
    wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
    tok, mx, sidx, sval = nfq.lm_head_nvfp4_argmax(c, bs, gs, wp, w.S, want_max=True,
                                                   want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    act = {"codes": c.cpu().numpy(), "block_scales": bs.cpu().numpy(),
           "global_scales": gs.cpu().numpy()}
    check_stage1_fp4(bf16_host(h), act["codes"], act["block_scales"], act["global_scales"],
                     oracle_stage1(inp)["hidden"])
    check(tok.cpu().numpy(), mx.cpu().numpy(), sidx.cpu().numpy(), sval.cpu().numpy(), act,
          qw, sw, gw, w.S, list(range(w.T)))


def test_nvfp4_workspace_stays_zero_and_results_repeat(nfq):
    w = synth.workload("tiny", T=20, H=512, V=2048, S=4, seed=9)
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = fp4_weights(w)
    ws = nfq.lm_head_workspace(w.T, w.S, "cuda")
    first = None
    for _ in range(3):
        out = run_lm(nfq, act, qw, sw, gw, w.S, ws=ws)
        assert torch.count_nonzero(ws).item() == 0
        first = out if first is None else first
        for a, b in zip(first, out):
            assert np.array_equal(a, b)


@pytest.mark.parametrize("V,H", [(128, 256), (300, 512), (1000, 1024)])
def test_nvfp4_pack_layout(nfq, V, H):
    """Code blocks as the FP8 packing of the [V][H/2] bytes; scale block
    (vt, s) word (kk * 32 + i) * 4 + c = scales 4kk .. 4kk+3 of step s for row
    vt * 128 + 32c + i; zero past V."""
    rng = np.random.default_rng(V + H)
    codes = rng.integers(0, 256, (V, H // 2), dtype=np.uint8)
    bs = rng.integers(0, 0x7F, (V, H // 16), dtype=np.uint8)
    packed = nfq.pack_lm_head_weights_nvfp4(to_dev(codes), to_dev(bs), 1.0).data.cpu().numpy()
    nvt, G = (V + 127) // 128, H // 256
    assert packed.size == nvt * G * (16384 + 2048)
    cp = np.zeros((nvt * 128, H // 2), np.uint8)
    cp[:V] = codes
    blocks = cp.reshape(nvt, 128, G, 8, 16).transpose(0, 2, 1, 3, 4)
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    expect = np.empty_like(blocks)
    expect[:, :, r, c ^ (r % 8)] = blocks[:, :, r, c]
    assert np.array_equal(packed[:nvt * G * 16384], expect.reshape(-1))
    sp = np.zeros((nvt * 128, H // 16), np.uint8)
    sp[:V] = bs
    words = sp.reshape(nvt, 4, 32, G, 4, 4)            # vt, c, i, s, kk, byte
    want = words.transpose(0, 3, 4, 2, 1, 5)           # vt, s, kk, i, c, byte
    assert np.array_equal(packed[nvt * G * 16384:], want.reshape(-1))


@pytest.mark.parametrize("T", [136, 256])
def test_nvfp4_two_token_groups_full_vocab(nfq, T):
    """129..256 tokens in one launch over a full-size vocabulary, on CTA pairs
    (the default form): every token against the oracle."""
    w = synth.workload("tiny", T=T, H=1024, k=2, V=151552, S=8, seed=T + 3)
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = synth.lm_head_weights_nvfp4(w)
    out = run_lm(nfq, act, qw, sw, gw, w.S)
    check(*out, act, qw, sw, gw, w.S, list(range(T)), cache_key=("nvfp4_two", T))


@pytest.mark.parametrize("T,H,V,S", [(129, 256, 1024, 8), (200, 1024, 5000, 5),
                                     (256, 512, 128, 1), (160, 16384, 3000, 3),
                                     (255, 1024, 151552, 8)])
def test_nvfp4_cta_pairs_equal_two_token_groups(nfq, T, H, V, S):
    """129..256 tokens: the CTA-pair kernel (cta_group::2 block-scaled MMAs,
    each CTA holding half of every weight tile and the scales of all of it)
    and two independent 128-token groups give the same bytes; both match the
    oracle on every token.  Ragged second halves, one-block tiles (64 weight
    rows per CTA, N = 128), a single block, the widest rows and a full
    vocabulary are covered."""
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=T * 5 + V)
    act = oracle_stage1(synth.stage1_inputs(w))
    qw, sw, gw = fp4_weights(w)
    pair = run_lm(nfq, act, qw, sw, gw, S)
    nfq.lm_head_pair(False)
    try:
        groups = run_lm(nfq, act, qw, sw, gw, S)
    finally:
        nfq.lm_head_pair(True)
    for a, b in zip(pair, groups):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    check(*pair, act, qw, sw, gw, S, list(range(T)), cache_key=("nvfp4_pair", T, H, V, S))


def test_nvfp4_stage_tuning_keeps_the_bytes(nfq):
    """The pipeline-depth hook: the single-CTA kernel (64 tokens) and the
    CTA-pair kernel (200 tokens) give the same bytes at every depth they
    accept, and depths the pair kernel must refuse (a weight ring shallower
    than its 4-slot activation ring) fall back to the default."""
    outs = {}
    for T in (64, 200):
        w = synth.workload("tiny", T=T, H=1024, k=2, V=40000, S=4, seed=T + 7)
        act = oracle_stage1(synth.stage1_inputs(w))
        qw, sw, gw = fp4_weights(w)
        try:
            for stages in (0, 2, 3, 4, 5):
                nfq.lm_head_nvfp4_tune(stages)
                outs[(T, stages)] = run_lm(nfq, act, qw, sw, gw, w.S)
        finally:
            nfq.lm_head_nvfp4_tune(0)
        for stages in (2, 3, 4, 5):
            for a, b in zip(outs[(T, 0)], outs[(T, stages)]):
                assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (T, stages)
        check(*outs[(T, 0)], act, qw, sw, gw, w.S, list(range(T)))


def test_fp4_quotients_match_ieee_division_exhaustively(nfq):
    """The NVFP4 stage 1 forms each block-scale code and each e2m1 code without
    IEEE divisions.  Over every bf16 row maximum and every finite e4m3 block
    scale, the reciprocals equal the IEEE reciprocals, and for every bf16 block
    maximum and value the row can hold (and every NaN) both codes equal the
    ones IEEE division gives."""
    counts, first = nfq.check_fp4_quotient()
    assert counts == [0, 0, 0, 0], (
        f"mismatches (rcp d, scale code, rcp eff, e2m1 code) {counts}, first {first:#014x}")
