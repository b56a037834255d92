"""The hand-derived end-to-end cases (tests/golden/e2e_two_tokens.txt and
tests/golden/nvfp4_e2e_two_tokens.txt) on the GPU through the C ABI: stage 1,
then the LM head with its sharded argmax, in the FP8 and the NVFP4 forms.
Every value of the cases is an exact dyadic number, so the GPU must reproduce
the hand-derived hidden, codes, scales, tokens, maxima and per-shard results
bit for bit, whatever its summation order."""
import numpy as np
import pytest
import torch

from tests._parity import bf16_host, to_dev, to_dev_bf16
from tests.test_oracle_pins import (check_nvfp4_e2e_stage1, e2e_golden_inputs,
                                    nvfp4_e2e_golden_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def _check_stage1(g, hidden, codes, scales):
    for t in range(2):
        h0, h1e, h1o = (int(v, 16) for v in g[f"hidden_t{t}"])
        assert np.all(hidden[t, :128] == h0)
        assert np.all(hidden[t, 128::2] == h1e) and np.all(hidden[t, 129::2] == h1o)
        c0, c1e, c1o = (int(v, 16) for v in g[f"codes_t{t}"])
        assert np.all(codes[t, :128] == c0)
        assert np.all(codes[t, 128::2] == c1e) and np.all(codes[t, 129::2] == c1o)
        assert scales[t].view(np.uint32).tolist() == [int(v, 16) for v in g["scales"]]


def _check_stage2(g, tok, mx, sidx, sval):
    assert tok.tolist() == [int(v) for v in g["tokens"]]
    assert mx.tolist() == [float(g["logits_t0"][0]), float(g["logits_t1"][3])]
    for t in range(2):
        assert sidx[:, t].tolist() == [int(v) for v in g[f"shard_idx_t{t}"]]
        assert sval[:, t].tolist() == [float(v) for v in g[f"shard_val_t{t}"]]


@pytest.mark.parametrize("layout", ["rowmajor", "packed"])
def test_e2e_golden_two_calls(nfq, layout):
    g, p, r, w, qw, sw = e2e_golden_inputs()
    h, c, s = nfq.mtp_reduce_norm_quant([to_dev_bf16(x) for x in p], to_dev_bf16(r),
                                        to_dev_bf16(w))
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    _check_stage1(g, bf16_host(h), c.cpu().numpy(), s.cpu().numpy())
    wd = to_dev(qw)
    if layout == "packed":
        wd = nfq.pack_lm_head_weights(wd)
    out = nfq.lm_head_fp8_argmax(c, s, wd, to_dev(sw), 2, want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    _check_stage2(g, *[x.cpu().numpy() for x in out])


def test_e2e_golden_step_call(nfq):
    """The one-call step API gives the same hand-derived results (at H = 256 it
    runs as its two launches; the one-launch form needs H % 512 == 0)."""
    g, p, r, w, qw, sw = e2e_golden_inputs()
    wp = nfq.pack_lm_head_weights(to_dev(qw))
    out = nfq.mtp_step_fp8([to_dev_bf16(x) for x in p], to_dev_bf16(r), to_dev_bf16(w), wp,
                           to_dev(sw), 2, want_max=True, want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    hidden, codes, scales, tok, mx, sidx, sval = out
    _check_stage1(g, bf16_host(hidden), codes.cpu().numpy(), scales.cpu().numpy())
    _check_stage2(g, *[x.cpu().numpy() for x in (tok, mx, sidx, sval)])


def test_nvfp4_e2e_golden(nfq):
    g, p, r, w, qw, sw, gw = nvfp4_e2e_golden_inputs()
    h, c, bs, gs = nfq.mtp_reduce_norm_quant_nvfp4([to_dev_bf16(x) for x in p], to_dev_bf16(r),
                                                   to_dev_bf16(w))
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    check_nvfp4_e2e_stage1(g, bf16_host(h), c.cpu().numpy(), bs.cpu().numpy(), gs.cpu().numpy())
    wp = nfq.pack_lm_head_weights_nvfp4(to_dev(qw), to_dev(sw), gw)
    tok, mx, sidx, sval = nfq.lm_head_nvfp4_argmax(c, bs, gs, wp, 2, want_max=True,
                                                   want_shards=True)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert tok.cpu().numpy().tolist() == [int(v) for v in g["tokens"]]
    assert mx.cpu().numpy().tolist() == [float(g["logits_t0"][0]), float(g["logits_t1"][2])]
    for t in range(2):
        assert sidx[:, t].cpu().numpy().tolist() == [int(v) for v in g[f"shard_idx_t{t}"]]
        assert sval[:, t].cpu().numpy().tolist() == [float(v) for v in g[f"shard_val_t{t}"]]


def test_unfused_e2e_golden(nfq):
    """The unfused arm's five kernels on the hand-derived case: BF16 all-reduce
    output, hidden, activation, BF16 logits and tokens as worked by hand."""
    g, p, r, w, qw, sw = e2e_golden_inputs()
    s = nfq.unfused_allreduce_bf16([to_dev_bf16(x) for x in p])
    h = nfq.unfused_add_rmsnorm(s, to_dev_bf16(r), to_dev_bf16(w))
    c, sc = nfq.unfused_quant_fp8(h)
    logits = nfq.unfused_lm_head_logits(c, sc, nfq.pack_lm_head_weights(to_dev(qw)), to_dev(sw))
    tok = nfq.unfused_argmax_bf16(logits)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    s_host = bf16_host(s)
    s0, s1 = (int(v, 16) for v in g["unfused_sum"])
    assert np.all(s_host[0] == s0) and np.all(s_host[1] == s1)
    _check_stage1(g, bf16_host(h), c.cpu().numpy(), sc.cpu().numpy())
    lb = bf16_host(logits)
    for t in range(2):
        assert lb[t].tolist() == [int(v, 16) for v in g[f"unfused_logits_t{t}"]]
    assert tok.cpu().numpy().tolist() == [int(v) for v in g["tokens"]]
