"""The fused step (stage 1 inside the LM-head launch) gives the same bytes as
the two launches, and the oracle's answers; where it does not apply it falls
back to the two launches."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import bf16_host, check_stage1, check_stage2, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def _case(nfq, w):
    inp = synth.stage1_inputs(w)
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    res, nw = to_dev_bf16(inp["residual"]), to_dev_bf16(inp["norm_w"])
    qw, sw = synth.lm_head_weights(w)
    wp, swd = nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw)
    return inp, parts, res, nw, qw, sw, wp, swd


@pytest.mark.parametrize("T,H,k,V,S", [(4, 1024, 2, 8192, 2), (64, 6144, 8, 151552, 8),
                                       (1, 7168, 8, 129280, 8), (17, 2048, 16, 20000, 5),
                                       (33, 4096, 1, 9000, 9), (64, 512, 3, 8192, 64),
                                       # not fused: falls back to the two launches
                                       (65, 1024, 2, 8192, 2), (5, 1152, 2, 8192, 4),
                                       (3, 16384, 2, 8192, 2), (8, 1024, 2, 640, 5)])
def test_fused_step_equals_two_launches(nfq, T, H, k, V, S):
    w = synth.workload("tiny", T=T, H=H, k=k, V=V, S=S, seed=T + H + k + V)
    inp, parts, res, nw, qw, sw, wp, swd = _case(nfq, w)
    h0, c0, s0 = nfq.mtp_reduce_norm_quant(parts, res, nw, w.eps)
    t0, m0, i0, v0 = nfq.lm_head_fp8_argmax(c0, s0, wp, swd, S, want_max=True, want_shards=True)
    ws = nfq.lm_head_workspace(T, S, "cuda")
    for _ in range(3):                       # the workspace (and its row counter) returns to zero
        out = nfq.mtp_step_fp8(parts, res, nw, wp, swd, S, w.eps, workspace=ws, want_max=True,
                               want_shards=True)
        torch.cuda.synchronize()
        assert nfq.device_error() == 0
        assert torch.count_nonzero(ws).item() == 0
        h1, c1, s1, t1, m1, i1, v1 = out
        assert torch.equal(h0.view(torch.int16), h1.view(torch.int16))
        for a, b in ((c0, c1), (s0, s1), (t0, t1), (m0, m1), (i0, i1), (v0, v1)):
            assert torch.equal(a, b)


def test_fused_step_against_the_oracle(nfq):
    w = synth.workload("tiny", T=24, H=2048, k=4, V=16384, S=4, seed=77)
    inp, parts, res, nw, qw, sw, wp, swd = _case(nfq, w)
    h, c, s, t, mx, si, sv = nfq.mtp_step_fp8(parts, res, nw, wp, swd, w.S, w.eps,
                                              want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"], w.eps)
    check_stage1(bf16_host(h), c.cpu().numpy(), s.cpu().numpy(), ref)
    # the LM head's part on the GPU's own activation
    check_stage2(t.cpu().numpy(), c.cpu().numpy(), s.cpu().numpy(), qw, sw, w.S,
                 list(range(w.T)), mx.cpu().numpy(), si.cpu().numpy(), sv.cpu().numpy())


def test_prepared_fused_step_in_a_graph(nfq):
    w = synth.workload("tiny", T=64, H=6144, k=8, V=32768, S=8, seed=5)
    inp, parts, res, nw, qw, sw, wp, swd = _case(nfq, w)
    h0, c0, s0, t0 = nfq.mtp_step_fp8(parts, res, nw, wp, swd, w.S, w.eps)
    hid, cod, sca = torch.empty_like(h0), torch.empty_like(c0), torch.empty_like(s0)
    tok = torch.empty_like(t0)
    ws = nfq.lm_head_workspace(w.T, w.S, "cuda")
    call = nfq.prepare_mtp_step_fp8(parts, res, nw, w.eps, hid, cod, sca, wp, swd, w.S, ws, tok)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
        call()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert nfq.device_error() == 0
        assert torch.count_nonzero(ws).item() == 0
        assert torch.equal(h0.view(torch.int16), hid.view(torch.int16))
        assert torch.equal(c0, cod) and torch.equal(s0, sca) and torch.equal(t0, tok)
