"""Seeded random shapes (token counts, widths, input counts, vocab sizes and
shard counts within the ABI's limits) for both stages in both formats, each
checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import (bf16_host, check_stage1, check_stage1_fp4, check_stage2,
                           check_stage2_fp4, to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def _shape(seed, fp4):
    r = np.random.default_rng(seed)
    T = int(r.choice([1, 2, 3, 7, 16, 31, 33, 64, 65, 100, 128, 129, 200]))
    H = int(r.choice([256, 512, 768, 1024, 2048, 3072]))
    if not fp4 and r.random() < 0.3:
        H = int(r.choice([128, 384, 640, 896]))          # FP8 takes any multiple of 128
    k = int(r.integers(1, 17))
    S = int(r.choice([1, 2, 3, 4, 5, 8, 16]))
    V = S * int(r.integers(max(1, 128 // S), max(2, 6000 // S)))
    return T, H, k, V, S


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_fp8(nfq, seed):
    T, H, k, V, S = _shape(seed, False)
    w = synth.workload("tiny", T=T, H=H, k=k, V=V, S=S, seed=1000 + seed)
    inp = synth.stage1_inputs(w)
    h, c, s = nfq.mtp_reduce_norm_quant([to_dev_bf16(p) for p in inp["partials"]],
                                        to_dev_bf16(inp["residual"]), to_dev_bf16(inp["norm_w"]),
                                        w.eps)
    qw, sw = synth.lm_head_weights(w)
    t, mx, si, sv = nfq.lm_head_fp8_argmax(c, s, nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw),
                                           S, want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"], w.eps)
    check_stage1(bf16_host(h), c.cpu().numpy(), s.cpu().numpy(), ref)
    sample = list(range(T))
    check_stage2(t.cpu().numpy(), c.cpu().numpy(), s.cpu().numpy(), qw, sw, S, sample,
                 mx.cpu().numpy(), si.cpu().numpy(), sv.cpu().numpy())


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_nvfp4(nfq, seed):
    T, H, k, V, S = _shape(100 + seed, True)
    w = synth.workload("tiny", T=T, H=H, k=k, V=V, S=S, seed=2000 + seed)
    inp = synth.stage1_inputs(w)
    h, c, b, g = nfq.mtp_reduce_norm_quant_nvfp4([to_dev_bf16(p) for p in inp["partials"]],
                                                 to_dev_bf16(inp["residual"]),
                                                 to_dev_bf16(inp["norm_w"]), w.eps)
    qw, sw, gw = synth.lm_head_weights_nvfp4(w)
    wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
    t, mx, si, sv = nfq.lm_head_nvfp4_argmax(c, b, g, wp, S, want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"], w.eps)
    act = {"codes": c.cpu().numpy(), "block_scales": b.cpu().numpy(),
           "global_scales": g.cpu().numpy()}
    check_stage1_fp4(bf16_host(h), act["codes"], act["block_scales"], act["global_scales"],
                     ref["hidden"])
    sample = list(range(T))
    check_stage2_fp4(t.cpu().numpy(), act["codes"], act["block_scales"], act["global_scales"],
                     qw, sw, gw, S, sample, mx.cpu().numpy(), si.cpu().numpy(),
                     sv.cpu().numpy())
