"""The allocation-free LM-head entry point, called through the C ABI.

Some callers cannot allocate device memory (a host engine that hands out only
fixed buffers, or a decode loop that must not touch the allocator because it
can synchronise the device); nfq_lm_head_fp8_argmax_noalloc serves them from a
scratch array the library owns.  This file is collected last so that a run
stopping at its first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests._parity import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import norm_fp8_quant_gb300 as nfq
    from norm_fp8_quant_gb300 import build
    build.build()
    lib = nfq.load()
    f = lib.nfq_lm_head_fp8_argmax_noalloc
    f.argtypes = [ctypes.POINTER(nfq.QuantAct)] + [ctypes.c_void_p] * 2 + [ctypes.c_int] * 2 + \
        [ctypes.c_void_p] * 5
    f.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("T,H,V,S", [(20, 512, 2048, 4), (64, 1024, 4096, 8)])
def test_noalloc_matches_workspace_entry_point(lib, T, H, V, S):
    import norm_fp8_quant_gb300 as nfq
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=T + V)
    inp = synth.stage1_inputs(w)
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"])
    qw, sw = synth.lm_head_weights(w)
    codes, scales, wd, swd = to_dev(ref["codes"]), to_dev(ref["scales"]), to_dev(qw), to_dev(sw)
    q = nfq.QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, 128)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def outputs():
        return (torch.full((T,), -7, dtype=torch.int32, device="cuda"),
                torch.zeros(T, dtype=torch.float32, device="cuda"),
                torch.full((S, T), -7, dtype=torch.int32, device="cuda"),
                torch.zeros((S, T), dtype=torch.float32, device="cuda"))

    # the existing entry point with a caller workspace
    ws = nfq.lm_head_workspace(T, S, "cuda")
    base = outputs()
    st = lib.nfq_lm_head_fp8_argmax(ctypes.byref(q), wd.data_ptr(), swd.data_ptr(), V, S,
                                    *[t.data_ptr() for t in base], ws.data_ptr(), ws.numel(),
                                    stream)
    assert st == 0
    # two allocation-free calls in a row
    for _ in range(2):
        got = outputs()
        st = lib.nfq_lm_head_fp8_argmax_noalloc(ctypes.byref(q), wd.data_ptr(), swd.data_ptr(),
                                                V, S, *[t.data_ptr() for t in got], stream)
        assert st == 0
        torch.cuda.synchronize()
        assert lib.nfq_device_error(1) == 0
        for a, b in zip(base, got):
            assert torch.equal(a, b)
    # and the tokens are the oracle's wherever the top-2 gap is clear
    L = oracle.lm_head_logits(ref["codes"], ref["scales"], qw, sw)
    r = oracle.argmax(L, S)
    clear = (r["gap"] >= 1e-3) | (r["gap"] == 0)
    assert np.array_equal(base[0].cpu().numpy()[clear], r["tokens"][clear])


def test_noalloc_rejects_too_many_shards(lib):
    import norm_fp8_quant_gb300 as nfq
    q = nfq.QuantAct(1 << 20, 1 << 20, 4, 256, 128)
    st = lib.nfq_lm_head_fp8_argmax_noalloc(ctypes.byref(q), 1 << 20, 1 << 20, 65 * 64, 65,
                                            1 << 20, None, None, None, None)
    assert st == nfq.NFQ_ERR_SHAPE
