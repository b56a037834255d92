"""GPU parity of the unfused reference arm (BF16 all-reduce output, add +
RMSNorm, group quantisation, BF16 logits, full-vocab argmax) against the
oracle's unfused path, kernel by kernel."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import U, abs_dot, bf16_host, check_stage1, oracle_logits, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nfq():
    import norm_fp8_quant_gb300 as m
    from norm_fp8_quant_gb300 import build
    build.build()
    m.load()
    assert torch.cuda.is_available()
    return m


def _ordered(b):
    b = b.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode_c64", None), ("decode_c1", None),
                                    ("tiny", 37)])
def test_unfused_stage1_kernels(nfq, name, T):
    w = synth.workload(name) if T is None else synth.workload(name, T=T, H=2048, k=5, seed=9)
    inp = synth.stage1_inputs(w)
    parts = [to_dev_bf16(p) for p in inp["partials"]]
    s = nfq.unfused_allreduce_bf16(parts)
    torch.cuda.synchronize()
    s_ref = oracle.unfused_reduce_bf16(inp["partials"])
    assert np.array_equal(bf16_host(s), s_ref)                  # same order, one rounding
    hid = nfq.unfused_add_rmsnorm(s, to_dev_bf16(inp["residual"]), to_dev_bf16(inp["norm_w"]),
                                  w.eps)
    torch.cuda.synchronize()
    h_ref = oracle.unfused_add_rmsnorm(s_ref, inp["residual"], inp["norm_w"], w.eps)
    assert np.abs(_ordered(bf16_host(hid)) - _ordered(h_ref)).max() <= 1
    # the quantiser on the same hidden: bit for bit
    codes, scales = nfq.unfused_quant_fp8(to_dev_bf16(h_ref))
    torch.cuda.synchronize()
    q = oracle.quant_fp8_rows(h_ref)
    assert np.array_equal(scales.cpu().numpy(), q["scales"])
    zero = lambda c: np.where((c & 0x7F) == 0, 0, c)
    assert np.array_equal(zero(codes.cpu().numpy()), zero(q["codes"]))
    # and on the GPU's own hidden, with the fused stage's acceptance rule
    c2, s2 = nfq.unfused_quant_fp8(hid)
    torch.cuda.synchronize()
    check_stage1(bf16_host(hid), c2.cpu().numpy(), s2.cpu().numpy(),
                 {"hidden": h_ref, **q})
    assert nfq.device_error() == 0


@pytest.mark.parametrize("T,H,V", [(4, 1024, 4096), (64, 6144, 151552), (1, 7168, 129280),
                                   (100, 512, 3000), (129, 256, 1000)])
def test_unfused_logits_and_argmax(nfq, T, H, V):
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=1, seed=T + H)
    ref = oracle.reduce_norm_quant(*[synth.stage1_inputs(w)[x] for x in ("partials", "residual", "norm_w")])
    qw, sw = synth.lm_head_weights(w)
    wp = nfq.pack_lm_head_weights(to_dev(qw))
    logits = nfq.unfused_lm_head_logits(to_dev(ref["codes"]), to_dev(ref["scales"]), wp, to_dev(sw))
    torch.cuda.synchronize()
    Lg = bf16_host(logits)
    sample = list(range(T))                   # every token's whole logits row
    L32 = oracle_logits(ref["codes"], ref["scales"], qw, sw, sample)
    Lb = oracle.f32_to_bf16(L32.ravel()).reshape(L32.shape)
    # BF16 of fp32 logits that agree within the summation bound: equal almost
    # everywhere; elsewhere within the fp32 bound plus one BF16 rounding (near
    # zero the bound is absolute, so the BF16 patterns may be far apart)
    d = np.abs(_ordered(Lg[sample]) - _ordered(Lb))
    assert (d > 0).mean() < 0.01
    gamma = (H + 2) * U / (1 - (H + 2) * U)
    bad = np.argwhere(d > 1)[:200]
    for i, v in bad:
        t = sample[i]
        tol = 2 * gamma * abs_dot(ref["codes"][t], ref["scales"][t], qw, sw, [int(v)])[0]
        g = float(oracle.bf16_to_f32(np.array([Lg[t, v]], np.uint16))[0])
        assert abs(g - float(L32[i, v])) <= tol + 2.0 ** -8 * abs(float(L32[i, v])) + 1e-30
    # the argmax kernel on these logits: exactly the oracle's rule
    tok = nfq.unfused_argmax_bf16(logits)
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), oracle.argmax_bf16(Lg))
    assert nfq.device_error() == 0


def test_unfused_argmax_ties_and_signed_zero(nfq):
    L = np.zeros((3, 5000), np.float32)
    L[0, [7, 4000]] = 2.0                   # tie: lowest index
    L[1, :] = -0.0
    L[1, 4999] = 0.0                        # all zeros: index 0
    L[2] = np.linspace(-1, 1, 5000, dtype=np.float32)
    L[2, 4998] = L[2, 4999]
    bits = (L.view(np.uint32) >> 16).astype(np.uint16)
    tok = nfq.unfused_argmax_bf16(to_dev_bf16(bits)).cpu().numpy()
    assert tok.tolist() == [7, 0, int(oracle.argmax_bf16(bits)[2])]
