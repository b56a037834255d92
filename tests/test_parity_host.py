"""The parity helpers on the host (CPU only): the threaded oracle logits are
the single-call ones bit for bit, and the table-driven dequantisation equals
the oracle's element-wise decoding."""
import numpy as np

import oracle
import synth
from tests import _parity


def test_threaded_oracle_logits_equal_one_call():
    w = synth.workload("tiny", T=5, H=256, k=2, V=1000, S=4, seed=2)
    inp = synth.stage1_inputs(w)
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"])
    qw, sw = synth.lm_head_weights(w)
    toks = [0, 3, 4]
    one = oracle.lm_head_logits(ref["codes"], ref["scales"], qw, sw, tokens=toks)
    many = _parity.oracle_logits(ref["codes"], ref["scales"], qw, sw, toks)
    assert np.array_equal(one.view(np.uint32), many.view(np.uint32))


def test_threaded_oracle_logits_nvfp4_equal_one_call():
    w = synth.workload("tiny", T=3, H=512, k=2, V=700, S=7, seed=4)
    inp = synth.stage1_inputs(w)
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"])
    act = oracle.nvfp4_quant(ref["hidden"])
    qw, sw, gw = synth.lm_head_weights_nvfp4(w)
    args = (act["codes"], act["block_scales"], act["global_scales"], qw, sw, gw)
    one = oracle.lm_head_logits_nvfp4(*args, tokens=[0, 1, 2])
    many = _parity.oracle_logits_nvfp4(*args, [0, 1, 2])
    assert np.array_equal(one.view(np.uint32), many.view(np.uint32))


def test_table_dequant_equals_elementwise_decode():
    codes = np.random.default_rng(0).integers(0, 256, (3, 256), dtype=np.uint8)
    codes[0, :] = np.arange(256)
    scales = np.array([[0.5, 2.0], [1.0, 3.0], [0.25, 0.125]], np.float32)
    got = _parity.dequant_rows(codes, scales)
    want = oracle.e4m3_to_f32(codes.ravel()).reshape(codes.shape).astype(np.float64) * \
        np.repeat(scales.astype(np.float64), 128, axis=1)
    assert np.array_equal(np.nan_to_num(got, nan=7.0), np.nan_to_num(want, nan=7.0))
