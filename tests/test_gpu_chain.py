"""Chained MTP draft positions (the BF16 hidden of one position is the residual
of the next) through nfq_mtp_draft_chain, against the CPU oracle: every link
with the GPU's own previous hidden, and the whole chain end to end."""
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
    return m


def _hidden_within_one_ulp(gpu, ref):
    o = lambda b: np.where(b.astype(np.int32) & 0x8000, -(b.astype(np.int32) & 0x7FFF),
                           b.astype(np.int32) & 0x7FFF)
    assert np.abs(o(gpu) - o(ref)).max(initial=0) <= 1


@pytest.mark.parametrize("name,P,packed", [("tiny", 3, False), ("tiny", 5, True),
                                           ("decode_c64", 5, True)])
def test_chain_matches_oracle(nfq, name, P, packed):
    w = synth.workload(name)
    base = synth.stage1_inputs(w)
    pos = [synth.stage1_inputs(synth.workload(name, seed=p + 1))["partials"] for p in range(P)]
    qw, sw = synth.lm_head_weights(w)
    wd = to_dev(qw)
    if packed:
        wd = nfq.pack_lm_head_weights(wd)
    hidden = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    codes = torch.empty((w.T, w.H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((w.T, w.H // 128), dtype=torch.float32, device="cuda")
    toks, _ = nfq.mtp_draft_chain([[to_dev_bf16(x) for x in part] for part in pos],
                                  to_dev_bf16(base["residual"]), to_dev_bf16(base["norm_w"]),
                                  wd, to_dev(sw), w.S, w.eps, hidden_bufs=hidden,
                                  codes=codes, scales=scales)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    toks = toks.cpu().numpy()
    gh = [bf16_host(h) for h in hidden]
    sample = list(range(w.T))                 # every token of every link
    # every link: the oracle's stage 1 on the GPU's previous hidden
    for p in range(P):
        res = base["residual"] if p == 0 else gh[p - 1]
        ref = oracle.reduce_norm_quant(pos[p], res, base["norm_w"], w.eps)
        _hidden_within_one_ulp(gh[p], ref["hidden"])
        if p == P - 1:       # the packed activation buffer holds the last position
            check_stage1(gh[p], codes.cpu().numpy(), scales.cpu().numpy(), ref)
        check_stage2(toks[p], ref["codes"], ref["scales"], qw, sw, w.S, sample)
    # the whole chain in the oracle alone
    res = base["residual"]
    for p in range(P):
        ref = oracle.reduce_norm_quant(pos[p], res, base["norm_w"], w.eps)
        _hidden_within_one_ulp(gh[p], ref["hidden"]) if p == 0 else None
        if w.T <= 8:
            L = oracle.lm_head_logits(ref["codes"], ref["scales"], qw, sw)
            r = oracle.argmax(L, w.S)
            clear = (r["gap"] >= 1e-3) | (r["gap"] == 0)
            assert np.array_equal(toks[p][clear], r["tokens"][clear])
        res = ref["hidden"]


def test_chain_with_two_alternating_hidden_buffers(nfq):
    w = synth.workload("tiny", T=3, H=256, V=512, S=2)
    base = synth.stage1_inputs(w)
    pos = [synth.stage1_inputs(synth.workload("tiny", T=3, H=256, seed=p + 7))["partials"]
           for p in range(4)]
    qw, sw = synth.lm_head_weights(w)
    parts = [[to_dev_bf16(x) for x in part] for part in pos]
    res0, nw, wd, swd = to_dev_bf16(base["residual"]), to_dev_bf16(base["norm_w"]), to_dev(qw), to_dev(sw)
    t2, h2 = nfq.mtp_draft_chain(parts, res0, nw, wd, swd, w.S)      # two buffers
    hidden = [torch.empty_like(res0) for _ in range(4)]
    t4, h4 = nfq.mtp_draft_chain(parts, res0, nw, wd, swd, w.S, hidden_bufs=hidden)
    torch.cuda.synchronize()
    assert torch.equal(t2, t4)
    assert torch.equal(h2[3].view(torch.int16), h4[3].view(torch.int16))


@pytest.mark.parametrize("name,P", [("tiny", 3), ("decode_c64", 5)])
def test_nvfp4_chain_matches_oracle(nfq, name, P):
    """The NVFP4 chain: every link against the oracle fed the GPU's previous
    hidden (hidden within 1 ulp; the oracle's NVFP4 quantiser on the GPU's
    hidden is the activation the LM head saw, whose tokens the oracle checks)."""
    from tests._parity import check_stage2_fp4
    w = synth.workload(name)
    base = synth.stage1_inputs(w)
    pos = [synth.stage1_inputs(synth.workload(name, seed=p + 1))["partials"] for p in range(P)]
    qw, sw, gw = synth.lm_head_weights_nvfp4(w)
    wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
    hidden = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    toks, _ = nfq.mtp_draft_chain_nvfp4([[to_dev_bf16(x) for x in part] for part in pos],
                                        to_dev_bf16(base["residual"]), to_dev_bf16(base["norm_w"]),
                                        wp, w.S, w.eps, hidden_bufs=hidden)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    toks = toks.cpu().numpy()
    gh = [bf16_host(h) for h in hidden]
    sample = list(range(w.T))
    for p in range(P):
        res = base["residual"] if p == 0 else gh[p - 1]
        ref = oracle.reduce_norm_quant(pos[p], res, base["norm_w"], w.eps)
        _hidden_within_one_ulp(gh[p], ref["hidden"])
        act = oracle.nvfp4_quant(gh[p])
        check_stage2_fp4(toks[p], act["codes"], act["block_scales"], act["global_scales"], qw, sw,
                         gw, w.S, sample)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_chain_on_cta_pairs(nfq, fmt):
    """200 tokens a position: every LM head of a three-position chain runs on
    CTA pairs (cta_group::2), launched programmatically after the stage 1 that
    writes its activation while its weight stages are already requested.  Every
    token of every link against the oracle fed the GPU's previous hidden."""
    from tests._parity import check_stage2_fp4
    P = 3
    w = synth.workload("tiny", T=200, H=1024, k=2, V=32768, S=8, seed=41)
    base = synth.stage1_inputs(w)
    pos = [synth.stage1_inputs(synth.workload("tiny", T=200, H=1024, k=2, seed=p + 42))["partials"]
           for p in range(P)]
    parts = [[to_dev_bf16(x) for x in part] for part in pos]
    hidden = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    if fmt == "fp8":
        qw, sw = synth.lm_head_weights(w)
        toks, _ = nfq.mtp_draft_chain(parts, to_dev_bf16(base["residual"]),
                                      to_dev_bf16(base["norm_w"]),
                                      nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw), w.S, w.eps,
                                      hidden_bufs=hidden)
    else:
        qw, sw, gw = synth.lm_head_weights_nvfp4(w)
        wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
        toks, _ = nfq.mtp_draft_chain_nvfp4(parts, to_dev_bf16(base["residual"]),
                                            to_dev_bf16(base["norm_w"]), wp, w.S, w.eps,
                                            hidden_bufs=hidden)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    toks = toks.cpu().numpy()
    gh = [bf16_host(h) for h in hidden]
    sample = list(range(w.T))
    for p in range(P):
        res = base["residual"] if p == 0 else gh[p - 1]
        ref = oracle.reduce_norm_quant(pos[p], res, base["norm_w"], w.eps)
        _hidden_within_one_ulp(gh[p], ref["hidden"])
        if fmt == "fp8":
            check_stage2(toks[p], ref["codes"], ref["scales"], qw, sw, w.S, sample)
        else:
            act = oracle.nvfp4_quant(gh[p])
            check_stage2_fp4(toks[p], act["codes"], act["block_scales"], act["global_scales"], qw,
                             sw, gw, w.S, sample)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("T", [64, 200])
def test_chain_under_one_cuda_graph(nfq, fmt, T):
    """Five chained draft positions captured in one CUDA graph: every replay
    gives the bytes of the eager chain (tokens, every position's hidden, the
    activation), the argmax workspace returns to zero, and every link matches
    the oracle fed the previous link's hidden.  200 tokens run the LM heads on
    CTA pairs."""
    from tests._parity import check_stage2_fp4
    P = 5
    w = synth.workload("decode_c64", T=T, V=32768, S=8)
    base = synth.stage1_inputs(w)
    pos = [synth.stage1_inputs(synth.workload("decode_c64", T=T, seed=p + 1))["partials"]
           for p in range(P)]
    parts = [[to_dev_bf16(x) for x in part] for part in pos]
    res0, nw = to_dev_bf16(base["residual"]), to_dev_bf16(base["norm_w"])
    H = w.H
    hidden = [torch.empty((T, H), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    toks = torch.empty((P, T), dtype=torch.int32, device="cuda")
    ws = nfq.lm_head_workspace(T, w.S, "cuda")
    if fmt == "fp8":
        qw, sw = synth.lm_head_weights(w)
        wp, swd = nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw)
        codes = torch.empty((T, H), dtype=torch.uint8, device="cuda")
        scales = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")
        act = (codes, scales)
        run = lambda: nfq.mtp_draft_chain(parts, res0, nw, wp, swd, w.S, w.eps, hidden_bufs=hidden,
                                          codes=codes, scales=scales, tokens_out=toks, workspace=ws)
    else:
        qw, sw, gw = synth.lm_head_weights_nvfp4(w)
        wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
        codes = torch.empty((T, H // 2), dtype=torch.uint8, device="cuda")
        bs = torch.empty((T, H // 16), dtype=torch.uint8, device="cuda")
        gs = torch.empty(T, dtype=torch.float32, device="cuda")
        act = (codes, bs, gs)
        run = lambda: nfq.mtp_draft_chain_nvfp4(parts, res0, nw, wp, w.S, w.eps, hidden_bufs=hidden,
                                                codes=codes, block_scales=bs, row_scales=gs,
                                                tokens_out=toks, workspace=ws)
    outs = [toks, *hidden, *act]
    run()
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    eager = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert nfq.device_error() == 0
        assert torch.count_nonzero(ws).item() == 0
        for a, b in zip(eager, outs):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    tk = toks.cpu().numpy()
    gh = [bf16_host(h) for h in hidden]
    for p in range(P):
        res = base["residual"] if p == 0 else gh[p - 1]
        ref = oracle.reduce_norm_quant(pos[p], res, base["norm_w"], w.eps)
        _hidden_within_one_ulp(gh[p], ref["hidden"])
        if fmt == "fp8":
            check_stage2(tk[p], ref["codes"], ref["scales"], qw, sw, w.S, list(range(T)))
        else:
            a = oracle.nvfp4_quant(gh[p])
            check_stage2_fp4(tk[p], a["codes"], a["block_scales"], a["global_scales"], qw, sw, gw,
                             w.S, list(range(T)))
