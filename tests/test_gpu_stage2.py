"""GPU parity of the FP8 LM head with the fused vocab-sharded argmax against
the CPU oracle, through the C ABI (via the Python binding)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import check_stage2, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def stage1_ref(w):
    inp = synth.stage1_inputs(w)
    return oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"])


@pytest.fixture(params=["rowmajor", "packed"])
def layout(request):
    return request.param


@pytest.fixture(params=["small", "wide"])
def family(request, nfq):
    """Kernel family for T <= 64: token-major small-batch or weight-major wide."""
    nfq.lm_head_small_batch(request.param == "small")
    yield request.param
    nfq.lm_head_small_batch(True)


def run_gpu(nfq, qa, sa, qw, sw, S, ws=None, layout="rowmajor"):
    w = to_dev(qw)
    if layout == "packed":
        w = nfq.pack_lm_head_weights(w)
    out = nfq.lm_head_fp8_argmax(to_dev(qa), to_dev(sa), w, to_dev(sw), S,
                                 workspace=ws, want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    return [None if x is None else x.cpu().numpy() for x in out]


def test_stage2_tiny_all_tokens(nfq, layout):
    w = synth.workload("tiny")
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, layout=layout)
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, w.S, list(range(w.T)),
                 mx, sidx, sval)


def test_stage2_decode_c1_full_vocab(nfq, layout):
    """T = 1, V = 129280 in 8 shards of 16160 rows: shard boundaries fall inside
    128-row scale blocks and tiles."""
    w = synth.workload("decode_c1")
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, layout=layout)
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, w.S, [0], mx, sidx, sval)


def test_stage2_decode_c64_all_tokens(nfq, layout, family):
    """Every one of the 64 tokens against the oracle's full-vocab logits: the
    M = 64 accumulator spreads the tokens over all four TMEM lane quadrants."""
    w = synth.workload("decode_c64")
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, layout=layout)
    assert tok.shape == (64,) and np.all((0 <= tok) & (tok < w.V))
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, w.S, list(range(w.T)), mx, sidx, sval,
                 cache_key="decode_c64")


def test_stage2_tie_stress(nfq, layout):
    """T = 256, V = 151552, S = 8; 30% of tokens have an exact duplicate maximum
    on either side of a shard boundary: the lower global index must win."""
    w = synth.workload("tie_stress")
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    expected = synth.plant_ties(w, qw, sw, ref["codes"])
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, layout=layout)
    width = w.V // w.S
    for t, row in expected.items():
        assert tok[t] == row, f"token {t}: {tok[t]} != {row}"
        s = row // width
        assert sidx[s, t] == row and sidx[s + 1, t] == row + 2 * ((s + 1) * width - 1 - row) + 1
        assert sval[s, t] == sval[s + 1, t] == mx[t]
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, w.S, list(range(w.T)), mx, sidx, sval,
                 expected=expected, cache_key="tie_stress")


@pytest.mark.parametrize("T", [136, 255])
def test_stage2_two_token_groups_full_grid(nfq, layout, T):
    """129..256 tokens run as two token groups over one weight stream: with a
    full-size vocab every CTA pair is busy, and the second group holds a ragged
    8 or 127 tokens.  Every token is checked against the oracle."""
    w = synth.workload("tiny", T=T, H=1024, k=2, V=151552, S=8, seed=T)
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, layout=layout)
    assert tok.shape == (T,) and np.all((0 <= tok) & (tok < w.V))
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, w.S, list(range(T)), mx, sidx, sval,
                 cache_key=("two_groups", T))


@pytest.mark.parametrize("T,H,V,S", [(1, 128, 128, 1), (3, 256, 200, 2), (16, 512, 1000, 5),
                                     (17, 384, 4100, 4), (33, 256, 2048, 64),
                                     (64, 1024, 3000, 3), (100, 512, 1536, 6),
                                     (129, 256, 1024, 8), (256, 256, 640, 5),
                                     (300, 256, 512, 2), (5, 16384, 1000, 4),
                                     (200, 16384, 384, 3)])
def test_stage2_edge_shapes(nfq, T, H, V, S, layout, family):
    """Ragged vocab tails, shard widths below a tile or a warp, every token
    count class (padding inside the MMA N, two warpgroups, 256-token chunks)."""
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=T + H + V + S)
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, S, layout=layout)
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, S, list(range(T)), mx, sidx, sval)


def test_stage2_planted_ties_and_zero_logits(nfq, layout, family):
    """Exact duplicates inside one warp, across warps of a tile, across tiles and
    at the last row; an all-zero activation row makes every logit +-0 and must
    give token 0."""
    T, H, V, S = 6, 256, 1024, 4
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=5)
    ref = stage1_ref(w)
    qa, sa = ref["codes"].copy(), ref["scales"].copy()
    qw, sw = synth.lm_head_weights(w)
    sw[:] = sw[0]                      # one scale row: equal codes give equal logits
    qa[5] = 0
    sa[5] = 0
    pairs = {0: (3, 17), 1: (40, 100), 2: (127, 128), 3: (255, 256), 4: (700, 1023)}
    for t, (a, b) in pairs.items():
        row = np.where((qa[t] & 0x7F) == 0, 0, np.where(qa[t] & 0x80, 0xFE, 0x7E)).astype(np.uint8)
        qw[a] = row
        qw[b] = row
    tok, mx, sidx, sval = run_gpu(nfq, qa, sa, qw, sw, S, layout=layout)
    for t, (a, b) in pairs.items():
        assert tok[t] == a
    assert tok[5] == 0 and mx[5] == 0.0 and not np.signbit(mx[5])
    assert list(sidx[:, 5]) == [0, 256, 512, 768]
    check_stage2(tok, qa, sa, qw, sw, S, list(range(T)), mx, sidx, sval,
                 expected={t: a for t, (a, b) in pairs.items()})


def test_stage2_workspace_stays_zero_across_calls(nfq):
    w = synth.workload("tiny", T=20, H=512, V=2048, S=4, seed=9)
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    ws = nfq.lm_head_workspace(w.T, w.S, "cuda")
    first = None
    for _ in range(3):
        out = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, ws=ws)
        assert torch.count_nonzero(ws).item() == 0
        if first is None:
            first = out
        for a, b in zip(first, out):
            assert np.array_equal(a, b)


@pytest.mark.parametrize("V,H", [(128, 128), (300, 256), (4096, 1024), (1000, 384)])
def test_pack_weights_layout(nfq, V, H):
    """The packed layout: block (vt, kb) at (vt * H/128 + kb) * 16 KB, row r at
    r * 128, 16-byte chunk c of the row at chunk c ^ (r % 8), zero rows past V."""
    rng = np.random.default_rng(V + H)
    w = rng.integers(0, 256, (V, H), dtype=np.uint8)
    packed = nfq.pack_lm_head_weights(to_dev(w)).data.cpu().numpy()
    nvt, G = (V + 127) // 128, H // 128
    assert packed.size == nvt * G * 16384
    wp = np.zeros((nvt * 128, H), np.uint8)
    wp[:V] = w
    blocks = wp.reshape(nvt, 128, G, 8, 16).transpose(0, 2, 1, 3, 4)      # vt, kb, r, c, 16
    r = np.arange(128)[:, None]
    c = np.arange(8)[None, :]
    expect = np.empty_like(blocks)
    expect[:, :, r, c ^ (r % 8)] = blocks[:, :, r, c]
    assert np.array_equal(packed, expect.reshape(-1))


@pytest.mark.parametrize("T,H,V,S", [(129, 256, 1024, 8), (200, 1024, 5000, 5),
                                     (256, 512, 128, 1), (160, 16384, 3000, 3),
                                     (255, 1024, 151552, 8)])
def test_stage2_cta_pairs_equal_two_token_groups(nfq, T, H, V, S, layout):
    """129..256 tokens: the CTA-pair kernel (cta_group::2 MMAs, each CTA
    holding half of every weight tile) and two independent 128-token groups
    give the same bytes; both match the oracle on every token.  Ragged second
    halves, a single 128-row block (one-block tiles, 64 weight rows per CTA),
    the widest rows and a full vocabulary are covered."""
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=T * 3 + V)
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    pair = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, S, layout=layout)
    nfq.lm_head_pair(False)
    try:
        groups = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, S, layout=layout)
    finally:
        nfq.lm_head_pair(True)
    for a, b in zip(pair, groups):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    check_stage2(pair[0], ref["codes"], ref["scales"], qw, sw, S, list(range(T)), *pair[1:],
                 cache_key=("pair", T, H, V, S))


@pytest.mark.parametrize("T", [64, 200])
def test_stage2_large_vocab_max_shards(nfq, T, layout):
    """A 262144-row vocabulary in the largest shard count (64 shards of 4096
    rows, boundaries inside CTA ranges and tiles): every token, every shard's
    result and the maxima against the oracle; 200 tokens run on CTA pairs."""
    w = synth.workload("tiny", T=T, H=256, k=2, V=262144, S=64, seed=T + 7)
    ref = stage1_ref(w)
    qw, sw = synth.lm_head_weights(w)
    tok, mx, sidx, sval = run_gpu(nfq, ref["codes"], ref["scales"], qw, sw, w.S, layout=layout)
    check_stage2(tok, ref["codes"], ref["scales"], qw, sw, w.S, list(range(T)), mx, sidx, sval,
                 cache_key=("large_vocab", T))
