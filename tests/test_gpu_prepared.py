"""Prepared calls (arguments checked once, issued many times) give the same
bytes as the ordinary calls, for both activation formats."""
import numpy as np
import pytest
import torch

import synth
from tests._parity import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def _inputs(w):
    inp = synth.stage1_inputs(w)
    return ([to_dev_bf16(p) for p in inp["partials"]], to_dev_bf16(inp["residual"]),
            to_dev_bf16(inp["norm_w"]))


def test_prepared_fp8_matches_plain_calls(nfq):
    w = synth.workload("tiny", T=24, H=1024, V=4096, S=4, seed=3)
    parts, res, nw = _inputs(w)
    qw, sw = synth.lm_head_weights(w)
    wp, swd = nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw)
    h0, c0, s0 = nfq.mtp_reduce_norm_quant(parts, res, nw, w.eps)
    t0 = nfq.lm_head_fp8_argmax(c0, s0, wp, swd, w.S)
    h1, c1, s1 = torch.empty_like(h0), torch.empty_like(c0), torch.empty_like(s0)
    ws = nfq.lm_head_workspace(w.T, w.S, "cuda")
    t1 = torch.empty_like(t0)
    st1 = nfq.prepare_reduce_norm_quant(parts, res, nw, w.eps, h1, c1, s1)
    st2 = nfq.prepare_lm_head_fp8_argmax(c1, s1, wp, swd, w.S, ws, t1)
    for _ in range(3):
        st1()
        st2()
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert torch.equal(h0.view(torch.int16), h1.view(torch.int16))
    assert torch.equal(c0, c1) and torch.equal(s0, s1) and torch.equal(t0, t1)


def test_prepared_nvfp4_matches_plain_calls(nfq):
    w = synth.workload("tiny", T=40, H=1024, V=8192, S=8, seed=4)
    parts, res, nw = _inputs(w)
    qw, sw, gw = synth.lm_head_weights_nvfp4(w)
    wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
    h0, c0, b0, g0 = nfq.mtp_reduce_norm_quant_nvfp4(parts, res, nw, w.eps)
    t0 = nfq.lm_head_nvfp4_argmax(c0, b0, g0, wp, w.S)
    h1, c1, b1, g1 = (torch.empty_like(x) for x in (h0, c0, b0, g0))
    ws = nfq.lm_head_workspace(w.T, w.S, "cuda")
    t1 = torch.empty_like(t0)
    st1 = nfq.prepare_reduce_norm_quant_nvfp4(parts, res, nw, w.eps, h1, c1, b1, g1)
    st2 = nfq.prepare_lm_head_nvfp4_argmax(c1, b1, g1, wp, w.S, ws, t1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):                # an explicit non-default stream
        for _ in range(3):
            st1()
            st2()
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    for a, b in ((h0.view(torch.int16), h1.view(torch.int16)), (c0, c1), (b0, b1), (g0, g1),
                 (t0, t1)):
        assert torch.equal(a, b)
    assert np.all(t1.cpu().numpy() < w.V)


def test_tokens_written_straight_to_pinned_host_memory(nfq):
    """tokens_out in pinned host memory (addressed by the device directly):
    the same tokens as a device buffer, for both LM heads."""
    w = synth.workload("tiny", T=33, H=1024, V=8192, S=4, seed=6)
    parts, res, nw = _inputs(w)
    h, c, s = nfq.mtp_reduce_norm_quant(parts, res, nw, w.eps)
    qw, sw = synth.lm_head_weights(w)
    wp, swd = nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw)
    ws = nfq.lm_head_workspace(w.T, w.S, "cuda")
    dev_tok = nfq.lm_head_fp8_argmax(c, s, wp, swd, w.S, workspace=ws)
    host_tok = torch.full((w.T,), -1, dtype=torch.int32).pin_memory()
    nfq.prepare_lm_head_fp8_argmax(c, s, wp, swd, w.S, ws, host_tok)()
    torch.cuda.synchronize()
    assert torch.equal(host_tok, dev_tok.cpu())
    h4, c4, b4, g4 = nfq.mtp_reduce_norm_quant_nvfp4(parts, res, nw, w.eps)
    q4, s4, gw = synth.lm_head_weights_nvfp4(w)
    wp4 = nfq.pack_lm_head_weights_nvfp4(to_dev(q4), to_dev(s4), gw)
    dev4 = nfq.lm_head_nvfp4_argmax(c4, b4, g4, wp4, w.S, workspace=ws)
    host4 = torch.full((w.T,), -1, dtype=torch.int32).pin_memory()
    nfq.prepare_lm_head_nvfp4_argmax(c4, b4, g4, wp4, w.S, ws, host4)()
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert torch.equal(host4, dev4.cpu())
