"""Both stages captured in a CUDA graph (prepared calls on the capturing
stream) and replayed give the same bytes as eager calls; the argmax workspace
returns to zero after every replay."""
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


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_graph_replay_matches_eager(nfq, fmt):
    w = synth.workload("tiny", T=48, H=1024, V=8192, S=8, seed=21)
    inp = synth.stage1_inputs(w)
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    res, nw = to_dev_bf16(inp["residual"]), to_dev_bf16(inp["norm_w"])
    T, H = w.T, w.H
    hidden = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    tok = torch.empty(T, dtype=torch.int32, device="cuda")
    ws = nfq.lm_head_workspace(T, w.S, "cuda")
    if fmt == "fp8":
        qw, sw = synth.lm_head_weights(w)
        wp, swd = nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw)
        codes = torch.empty((T, H), dtype=torch.uint8, device="cuda")
        scales = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")
        s1 = nfq.prepare_reduce_norm_quant(parts, res, nw, w.eps, hidden, codes, scales)
        s2 = nfq.prepare_lm_head_fp8_argmax(codes, scales, wp, swd, w.S, ws, tok)
        outs = (hidden, codes, scales, tok)
    else:
        qw, sw, gw = synth.lm_head_weights_nvfp4(w)
        wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
        codes = torch.empty((T, H // 2), dtype=torch.uint8, device="cuda")
        bs = torch.empty((T, H // 16), dtype=torch.uint8, device="cuda")
        gs = torch.empty(T, dtype=torch.float32, device="cuda")
        s1 = nfq.prepare_reduce_norm_quant_nvfp4(parts, res, nw, w.eps, hidden, codes, bs, gs)
        s2 = nfq.prepare_lm_head_nvfp4_argmax(codes, bs, gs, wp, w.S, ws, tok)
        outs = (hidden, codes, bs, gs, tok)
    s1()
    s2()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s1()
        s2()
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert nfq.device_error() == 0
        assert torch.count_nonzero(ws).item() == 0
        for a, b in zip(eager, outs):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
