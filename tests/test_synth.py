"""The seeded input generator: determinism, row sampling and distributions (CPU)."""
import numpy as np

import synth


def test_counter_based_rows_match_full_generation():
    w = synth.workload("decode_c64", T=6, H=768)
    full = synth.stage1_inputs(w)
    some = synth.stage1_inputs(w, rows=[5, 0, 3])
    assert np.array_equal(some["partials"], full["partials"][:, [5, 0, 3]])
    assert np.array_equal(some["residual"], full["residual"][[5, 0, 3]])
    assert np.array_equal(some["norm_w"], full["norm_w"])
    assert np.array_equal(synth.stage1_inputs(w)["partials"], full["partials"])


def test_thread_count_does_not_change_draws():
    a = synth.normal_f32(0, 7, 200000)
    lib = synth._load()
    b = np.empty_like(a)
    lib.synth_normal_f32(0, 7, 0, a.size, 0.0, 1.0, None, 0, b.ctypes.data, 1)
    assert np.array_equal(a, b)


def test_distributions_and_outlier_channels():
    x = synth.normal_f32(0, 9, 1 << 20, mean=1.0, std=0.1).astype(np.float64)
    assert abs(x.mean() - 1.0) < 1e-3 and abs(x.std() - 0.1) < 1e-3
    w = synth.workload("decode_c64")
    ch = synth.outlier_channels(w)
    assert ch.size == round(0.01 * 6144) == 61 and np.unique(ch).size == 61
    sub = synth.workload("decode_c64", T=2)
    p = synth.stage1_inputs(sub)["partials"]
    f = (p.astype(np.uint32) << 16).view(np.float32)
    out_std = f[:, :, ch].std()
    other = np.delete(f, ch, axis=2).std()
    assert 15 < out_std / other < 25           # outlier channels carry x20


def test_lm_head_weight_block_quantisation():
    w = synth.workload("tiny", V=384, H=256)
    qw, sw = synth.lm_head_weights(w)
    assert qw.shape == (384, 256) and sw.shape == (3, 2)
    assert np.all((qw & 0x7F) != 0x7F)
    blocks = qw.reshape(3, 128, 2, 128)
    # each block holds its amax at +-448
    assert np.all(((blocks & 0x7F) == 0x7E).any(axis=(1, 3)))
    assert 0.02 * 3 / 448 < sw.mean() < 0.02 * 6 / 448


def test_nvfp4_weight_quantiser_matches_the_oracle_on_bf16_rows():
    """The input generator's vectorised NVFP4 quantiser agrees with the
    oracle's row quantiser when both see the same BF16 rows and row scales."""
    import oracle
    rng = np.random.default_rng(5)
    x = (rng.normal(0, 1, (32, 256)) * np.exp2(rng.integers(-8, 8, (32, 1)))).astype(np.float32)
    x[4] = 0
    x[7, 16:32] = 0
    bits = synth.to_bf16_bits(x)
    xb = (bits.astype(np.uint32) << 16).view(np.float32)
    ref = oracle.nvfp4_quant(bits)
    codes, bs = synth.nvfp4_quantise_rows(xb, ref["global_scales"])
    assert np.array_equal(bs, ref["block_scales"])
    # +-0 codes are the same value
    zero = lambda c: np.where((c & 7) == 0, 0, c)
    lo = lambda c: zero(c & 15)
    hi = lambda c: zero(c >> 4)
    assert np.array_equal(lo(codes), lo(ref["codes"])) and np.array_equal(hi(codes), hi(ref["codes"]))


def test_nvfp4_weights_shape_and_scale():
    w = synth.workload("tiny")
    codes, bs, gw = synth.lm_head_weights_nvfp4(w)
    assert codes.shape == (w.V, w.H // 2) and bs.shape == (w.V, w.H // 16)
    f = synth.normal_f32(w.seed, synth.STREAM_LM_W, w.V * w.H, 0.0, w.weight_std)
    assert gw == np.float32(np.float32(np.abs(f).max()) / np.float32(2688.0))
    assert bs.max() == 0x7E            # the tensor's largest block reaches 448
