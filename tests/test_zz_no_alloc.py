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


@pytest.mark.parametrize("T,H,V,S", [(20, 512, 2048, 4), (64, 1024, 4096, 8),
                                     # the largest shard count: the whole array in use
                                     (20, 256, 8192, 64),
                                     # more than 256 tokens: two launches share the array
                                     (300, 256, 2048, 4)])
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


def test_noalloc_rejects_bad_arguments_before_touching_the_array(lib):
    """More than 64 shards, a misaligned output or a NULL weight are refused
    with an error code and nothing is queued.  Real (small) device buffers are
    passed, so even a check that came too late could not read unmapped memory;
    a correct call made just before on the same stream keeps its results."""
    import norm_fp8_quant_gb300 as nfq
    T, H, V, S = 4, 256, 1024, 4
    w = synth.workload("tiny", T=T, H=H, k=2, V=V, S=S, seed=3)
    inp = synth.stage1_inputs(w)
    ref = oracle.reduce_norm_quant(inp["partials"], inp["residual"], inp["norm_w"])
    qw, sw = synth.lm_head_weights(w)
    codes, scales, wd, swd = to_dev(ref["codes"]), to_dev(ref["scales"]), to_dev(qw), to_dev(sw)
    q = nfq.QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, 128)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    tok = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    spare = torch.zeros(64, dtype=torch.int32, device="cuda")
    assert lib.nfq_lm_head_fp8_argmax_noalloc(ctypes.byref(q), wd.data_ptr(), swd.data_ptr(), V,
                                              S, tok.data_ptr(), None, None, None, stream) == 0
    call = lambda V_, S_, w_, t_: lib.nfq_lm_head_fp8_argmax_noalloc(
        ctypes.byref(q), w_, swd.data_ptr(), V_, S_, t_, None, None, None, stream)
    assert call(65 * 16, 65, wd.data_ptr(), spare.data_ptr()) == nfq.NFQ_ERR_SHAPE
    assert call(V, S, wd.data_ptr(), spare.data_ptr() + 2) == nfq.NFQ_ERR_ALIGN
    assert call(V, S, None, spare.data_ptr()) == nfq.NFQ_ERR_NULL
    torch.cuda.synchronize()
    assert lib.nfq_device_error(1) == 0
    assert torch.count_nonzero(spare).item() == 0
    L = oracle.lm_head_logits(ref["codes"], ref["scales"], qw, sw)
    r = oracle.argmax(L, S)
    clear = (r["gap"] >= 1e-3) | (r["gap"] == 0)
    assert np.array_equal(tok.cpu().numpy()[clear], r["tokens"][clear])
