"""GPU parity of the fused reduce + residual + RMSNorm + packed-FP8 stage
against the CPU oracle, through the C ABI (via the Python binding)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import bf16_host, check_stage1, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def run_gpu(nfq, inp, eps=1e-6):
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    res = to_dev_bf16(inp["residual"])
    w = to_dev_bf16(inp["norm_w"])
    hidden, codes, scales = nfq.mtp_reduce_norm_quant(parts, res, w, eps)
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    return bf16_host(hidden), codes.cpu().numpy(), scales.cpu().numpy()


def run_oracle(inp, eps=1e-6):
    return oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"], eps)


@pytest.mark.parametrize("name", ["tiny", "decode_c1", "decode_c64", "tie_stress"])
def test_stage1_full_workloads(nfq, name):
    w = synth.workload(name)
    inp = synth.stage1_inputs(w)
    h, c, s = run_gpu(nfq, inp)
    info = check_stage1(h, c, s, run_oracle(inp))
    print(name, info)


def test_stage1_prefill_full_size_sampled_rows(nfq):
    """T = 8192, H = 7168, k = 8 in the launch configuration the benchmark uses;
    the oracle checks a spread of rows (first, last, and rows in between)."""
    w = synth.workload("prefill")
    inp = synth.stage1_inputs(w)
    h, c, s = run_gpu(nfq, inp)
    rows = sorted(set([0, 1, 151, 152, 4095, 8190, 8191] +
                      list(np.random.default_rng(0).integers(0, w.T, 25))))
    sub = synth.stage1_inputs(w, rows=rows)
    assert np.array_equal(sub["partials"][:, 0], inp["partials"][:, rows[0]])
    check_stage1(h[rows], c[rows], s[rows], run_oracle(sub))


@pytest.mark.parametrize("T,H,k", [(1, 128, 1), (3, 128, 1), (5, 896, 3), (17, 1024, 16),
                                   (150, 2048, 2), (153, 384, 5), (2, 16384, 4),
                                   (1, 32768, 2)])
def test_stage1_edge_shapes(nfq, T, H, k):
    w = synth.workload("tiny", T=T, H=H, k=k, seed=T * 7 + H + k)
    inp = synth.stage1_inputs(w)
    h, c, s = run_gpu(nfq, inp)
    check_stage1(h, c, s, run_oracle(inp))


def test_stage1_degenerate_rows(nfq):
    """Zero rows (scale 0, codes 0), a constant row, huge and tiny magnitudes,
    negative zero inputs and cancelling partials."""
    T, H, k = 6, 512, 3
    p = np.zeros((k, T, H), np.float32)
    r = np.zeros((T, H), np.float32)
    p[:, 1] = 0.25                     # constant row
    p[0, 2] = 3.0e4
    p[1, 2] = -3.0e4                   # cancelling partials, residual decides
    r[2] = np.linspace(-1, 1, H)
    p[0, 3, :128] = 1e-30              # tiny group next to normal ones
    p[0, 3, 128:] = 1.0
    p[:, 4] = -0.0                     # all negative zero
    p[0, 5] = np.random.default_rng(1).normal(0, 1, H) * 200.0
    bits = lambda a: synth.to_bf16_bits(a)
    inp = {"partials": np.stack([bits(p[i]) for i in range(k)]),
           "residual": bits(r), "norm_w": bits(np.linspace(-2, 2, H).astype(np.float32))}
    h, c, s = run_gpu(nfq, inp)
    ref = run_oracle(inp)
    check_stage1(h, c, s, ref)
    assert np.all(s[0] == 0) and np.all(c[0] & 0x7F == 0)
    assert np.all(s[4] == 0)


@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.1])
def test_stage1_eps_values(nfq, eps):
    w = synth.workload("tiny", T=9, H=256, k=2, seed=11)
    inp = synth.stage1_inputs(w)
    h, c, s = run_gpu(nfq, inp, eps)
    check_stage1(h, c, s, run_oracle(inp, eps))


def test_stage1_is_deterministic_and_reuses_outputs(nfq):
    w = synth.workload("decode_c64", T=40)
    inp = synth.stage1_inputs(w)
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    res, nw = to_dev_bf16(inp["residual"]), to_dev_bf16(inp["norm_w"])
    a = nfq.mtp_reduce_norm_quant(parts, res, nw)
    b = nfq.mtp_reduce_norm_quant(parts, res, nw)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.uint8) if y.dtype == torch.bfloat16 else y)


@pytest.mark.parametrize("cuts", [(0, 1, 40), (0, 17, 23, 40), (0, 39, 40)])
def test_stage1_row_ranges_compose(nfq, cuts):
    """A sequence-parallel rank owns a contiguous range of token rows: calling
    the stage on each range (pointer offsets into the same buffers) gives the
    same bytes as one call over all rows, because every row is independent."""
    w = synth.workload("decode_c64", T=cuts[-1], seed=5)
    inp = synth.stage1_inputs(w)
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    res, nw = to_dev_bf16(inp["residual"]), to_dev_bf16(inp["norm_w"])
    whole = nfq.mtp_reduce_norm_quant(parts, res, nw)
    hid = torch.empty_like(whole[0])
    cod = torch.empty_like(whole[1])
    sca = torch.empty_like(whole[2])
    for a, b in zip(cuts[:-1], cuts[1:]):
        nfq.mtp_reduce_norm_quant([p[a:b] for p in parts], res[a:b], nw,
                                  hidden_out=hid[a:b], codes_out=cod[a:b], scales_out=sca[a:b])
    torch.cuda.synchronize()
    assert nfq.device_error() == 0
    assert torch.equal(hid.view(torch.int16), whole[0].view(torch.int16))
    assert torch.equal(cod, whole[1]) and torch.equal(sca, whole[2])
    check_stage1(bf16_host(hid), cod.cpu().numpy(), sca.cpu().numpy(), run_oracle(inp))
