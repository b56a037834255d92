"""The C-ABI library on the host: it loads, exports every declared symbol and
rejects bad arguments before touching a device (no GPU needed)."""
import ctypes
import os
import re

import pytest

import norm_fp8_quant_gb300 as nfq
from norm_fp8_quant_gb300 import build as nfq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nfq_build.build()
    return nfq.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "nfq.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(nfq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert len(syms) >= 7
    for s in syms:
        assert hasattr(lib, s), s
    assert lib.nfq_abi_version() >> 16 == 1
    for st in range(-7, 1):
        assert nfq.status_str(st) != "unknown status"


FAKE = 1 << 20          # aligned fake device addresses: never dereferenced
MIS = FAKE + 8


def _stage1(lib, partials, k=2, residual=FAKE, norm_w=FAKE, eps=1e-6, T=4, H=1024,
            hidden=FAKE, codes=FAKE, scales=FAKE, tokens=None, hidden_q=None, group=128):
    arr = (ctypes.c_void_p * max(len(partials), 1))(*partials) if partials is not None else None
    q = nfq.QuantAct(codes, scales, T if tokens is None else tokens,
                     H if hidden_q is None else hidden_q, group)
    return lib.nfq_mtp_reduce_norm_quant(arr, k, residual, norm_w, eps, T, H, hidden,
                                         ctypes.byref(q), None)


def test_stage1_argument_validation(lib):
    ok = [FAKE, FAKE]
    assert _stage1(lib, None) == nfq.NFQ_ERR_NULL
    assert _stage1(lib, [FAKE, 0]) == nfq.NFQ_ERR_NULL
    assert _stage1(lib, ok, residual=0) == nfq.NFQ_ERR_NULL
    assert _stage1(lib, ok, codes=0) == nfq.NFQ_ERR_NULL
    assert _stage1(lib, ok, k=0) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, [FAKE] * 17, k=17) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, H=1000) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, H=0) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, T=-1, tokens=-1) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, eps=-1.0) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, eps=float("nan")) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, group=64) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, tokens=5) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, ok, hidden_q=2048) == nfq.NFQ_ERR_SHAPE
    assert _stage1(lib, [FAKE, MIS]) == nfq.NFQ_ERR_ALIGN
    assert _stage1(lib, ok, hidden=MIS) == nfq.NFQ_ERR_ALIGN
    assert _stage1(lib, ok, scales=MIS) == nfq.NFQ_ERR_ALIGN
    # an empty batch is a no-op that needs no device
    assert _stage1(lib, ok, T=0, tokens=0) == nfq.NFQ_OK


def _stage2(lib, T=4, H=1024, group=128, codes=FAKE, scales=FAKE, w=FAKE, ws_=FAKE, V=4096,
            S=2, tokens=FAKE, ws=FAKE, ws_bytes=None, mx=None):
    q = nfq.QuantAct(codes, scales, T, H, group)
    if ws_bytes is None:
        ws_bytes = lib.nfq_lm_head_workspace_bytes(T, S)
    return lib.nfq_lm_head_fp8_argmax(ctypes.byref(q), w, ws_, V, S, tokens, mx, None, None,
                                      ws, ws_bytes, None)


def test_stage2_argument_validation(lib):
    assert lib.nfq_lm_head_workspace_bytes(4, 0) == 0
    assert lib.nfq_lm_head_workspace_bytes(4, 8) >= 8 * 8
    assert _stage2(lib, codes=0) == nfq.NFQ_ERR_NULL
    assert _stage2(lib, w=0) == nfq.NFQ_ERR_NULL
    assert _stage2(lib, tokens=0) == nfq.NFQ_ERR_NULL
    assert _stage2(lib, V=4095) == nfq.NFQ_ERR_SHAPE        # V % S != 0
    assert _stage2(lib, S=0) == nfq.NFQ_ERR_SHAPE
    assert _stage2(lib, S=65, V=65 * 64) == nfq.NFQ_ERR_SHAPE
    assert _stage2(lib, H=1000) == nfq.NFQ_ERR_SHAPE
    assert _stage2(lib, H=32768) == nfq.NFQ_ERR_SHAPE
    assert _stage2(lib, group=32) == nfq.NFQ_ERR_SHAPE
    assert _stage2(lib, ws=0) == nfq.NFQ_ERR_WORKSPACE
    assert _stage2(lib, ws_bytes=8) == nfq.NFQ_ERR_WORKSPACE
    assert _stage2(lib, w=MIS) == nfq.NFQ_ERR_ALIGN
    assert _stage2(lib, mx=FAKE + 2) == nfq.NFQ_ERR_ALIGN
    assert _stage2(lib, tokens=FAKE + 2) == nfq.NFQ_ERR_ALIGN
    assert _stage2(lib, mx=FAKE + 4, tokens=FAKE + 12, T=0) == nfq.NFQ_OK
    assert _stage2(lib, T=0) == nfq.NFQ_OK
    assert lib.nfq_lm_head_workspace_init(None, 16, None) == nfq.NFQ_ERR_NULL


def test_stage1_plans_cover_the_workload_shapes(lib):
    for (T, H, k) in [(4, 1024, 2), (1, 7168, 8), (64, 6144, 8), (8192, 7168, 8),
                      (256, 6144, 4), (3, 128, 1), (7, 896, 3), (2, 32768, 16)]:
        p = nfq.stage1_plan(T, H, k, 152)
        assert p["vpt"] >= 1 and (H // 128) % (p["cluster"] * p["vpt"]) == 0
        assert p["active_threads"] * p["vpt"] * 8 * p["cluster"] == H
        assert p["threads"] <= 1024 and p["smem"] <= 227 * 1024


def _split_valid(G, r, u):
    return G % r == 0 and (G // r) % u == 0 and -(-(16 * (G // r) // u) // 32) * 32 <= 512


def test_stage1_split_plans(lib):
    """The small-batch kernel: whole groups per CTA, whole 16-lane groups per
    vector slot, at most 512 threads.  Batches above 96 rows copy the inputs
    into shared memory when k > 8, with the smallest R whose (k+1) input
    slices fit in 112 KB (two CTAs an SM); the rest load into registers, with R and the
    vectors per thread by batch size (T <= 24: T*R >= 64, one vector; T <= 96:
    T*R >= 256, one vector); batches above 512 rows go to the persistent
    kernel (R = 0)."""
    for (T, H, k) in [(1, 7168, 8), (4, 1024, 2), (16, 6144, 8), (64, 6144, 8), (64, 7168, 8),
                      (128, 6144, 8), (256, 6144, 4), (256, 6144, 8), (300, 7168, 8),
                      (3, 128, 1), (2, 16384, 4), (1, 32768, 2), (17, 896, 3), (512, 2048, 16),
                      (200, 16384, 16)]:
        p = nfq.stage1_split_plan(T, H, k, num_sms=152)
        G = H // 128
        R, v = p["ctas_per_row"], p["vpt"]
        assert R >= 1 and _split_valid(G, R, v), (T, H)
        assert p["active_threads"] == 16 * (G // R) // v and p["threads"] <= 512
        want = None
        if T > 96 and k > 8:
            for r in range(1, 9):
                if G % r or (k + 1) * (H // r) * 2 > 112 * 1024:
                    continue
                u = next((u for u in (2, 1, 4) if _split_valid(G, r, u)), None)
                if u is not None:
                    want = (r, u, 1)
                    break
        if want is None:
            target, order = ((64, (1, 2, 4)) if T <= 24 else (256, (1, 2, 4)) if T <= 96 else
                             (1, (2, 1, 4)) if T <= 160 else (1, (4, 2, 1)))
            for r in range(1, 9):
                u = next((u for u in order if _split_valid(G, r, u)), None)
                if u is None:
                    continue
                want = (r, u, 0)
                if T * r >= target:
                    break
        assert (R, v, p["tma"]) == want, (T, H, k, R, v, p["tma"], want)
    assert nfq.stage1_split_plan(64, 6144, 8)["ctas_per_row"] == 4
    assert nfq.stage1_split_plan(256, 6144, 8)["tma"] == 0
    assert nfq.stage1_split_plan(256, 6144, 16)["tma"] == 1
    assert nfq.stage1_split_plan(513, 6144, 8)["ctas_per_row"] == 0
    assert nfq.stage1_split_plan(8192, 7168, 8)["ctas_per_row"] == 0
    nfq.stage1_split(0)
    try:
        assert nfq.stage1_split_plan(64, 6144, 8)["ctas_per_row"] == 0
    finally:
        nfq.stage1_split()
    nfq.stage1_split(-1, 4, 2, 0)
    try:
        p = nfq.stage1_split_plan(64, 6144, 8)
        assert (p["ctas_per_row"], p["vpt"], p["threads"], p["tma"]) == (4, 2, 96, 0)
        p = nfq.stage1_split_plan(256, 6144, 8)
        assert (p["ctas_per_row"], p["tma"]) == (4, 0)
    finally:
        nfq.stage1_split()
    nfq.stage1_split(-1, 0, 0, 1)
    try:
        p = nfq.stage1_split_plan(16, 6144, 8)
        assert (p["ctas_per_row"], p["vpt"], p["tma"]) == (1, 2, 1)
    finally:
        nfq.stage1_split()


def test_chain_argument_validation(lib):
    import ctypes as C
    q = nfq.QuantAct(FAKE, FAKE, 4, 1024, 128)
    parts = (C.c_void_p * 4)(FAKE, FAKE, FAKE, FAKE)
    same = (C.c_void_p * 2)(FAKE + 4096, FAKE + 4096)
    diff = (C.c_void_p * 2)(FAKE + 4096, FAKE + 8192)
    ws = lib.nfq_lm_head_workspace_bytes(4, 2)
    call = lambda P, h, res=FAKE, k=2: lib.nfq_mtp_draft_chain(
        P, parts, k, res, FAKE, 1e-6, 4, 1024, h, C.byref(q), FAKE, 0, FAKE, 4096, 2, FAKE, FAKE,
        ws, None)
    assert call(0, diff) == nfq.NFQ_ERR_SHAPE
    assert call(65, diff) == nfq.NFQ_ERR_SHAPE
    assert call(2, same) == nfq.NFQ_ERR_SHAPE            # consecutive positions share a buffer
    assert call(2, diff, res=FAKE + 4096) == nfq.NFQ_ERR_SHAPE   # hidden aliases the residual
    assert call(2, diff, k=0) == nfq.NFQ_ERR_SHAPE
    assert lib.nfq_mtp_draft_chain(2, None, 2, FAKE, FAKE, 1e-6, 4, 1024, diff, C.byref(q), FAKE,
                                   0, FAKE, 4096, 2, FAKE, FAKE, ws, None) == nfq.NFQ_ERR_NULL


def _stage1_fp4(lib, partials=(FAKE, FAKE), k=2, T=4, H=1024, codes=FAKE, bs=FAKE, gs=FAKE,
                tokens=None, block=16, hidden=FAKE):
    arr = (ctypes.c_void_p * len(partials))(*partials)
    q = nfq.Fp4Act(codes, bs, gs, T if tokens is None else tokens, H, block)
    return lib.nfq_mtp_reduce_norm_quant_nvfp4(arr, k, FAKE, FAKE, 1e-6, T, H, hidden,
                                               ctypes.byref(q), None)


def test_stage1_nvfp4_argument_validation(lib):
    assert _stage1_fp4(lib, codes=0) == nfq.NFQ_ERR_NULL
    assert _stage1_fp4(lib, bs=0) == nfq.NFQ_ERR_NULL
    assert _stage1_fp4(lib, gs=0) == nfq.NFQ_ERR_NULL
    assert _stage1_fp4(lib, H=1152) == nfq.NFQ_ERR_SHAPE          # not a multiple of 256
    assert _stage1_fp4(lib, H=32768) == nfq.NFQ_ERR_SHAPE         # a row must fit one CTA
    assert _stage1_fp4(lib, block=32) == nfq.NFQ_ERR_SHAPE
    assert _stage1_fp4(lib, tokens=5) == nfq.NFQ_ERR_SHAPE
    assert _stage1_fp4(lib, bs=MIS) == nfq.NFQ_ERR_ALIGN
    assert _stage1_fp4(lib, T=0, tokens=0) == nfq.NFQ_OK
    assert _stage1_fp4(lib, T=0, tokens=0, H=16384) == nfq.NFQ_OK


def _stage2_fp4(lib, T=4, H=1024, block=16, codes=FAKE, bs=FAKE, gs=FAKE, w=FAKE, V=4096, S=2,
                tokens=FAKE, ws=FAKE, ws_bytes=None):
    q = nfq.Fp4Act(codes, bs, gs, T, H, block)
    if ws_bytes is None:
        ws_bytes = lib.nfq_lm_head_workspace_bytes(T, S)
    return lib.nfq_lm_head_nvfp4_argmax(ctypes.byref(q), w, 0.5, V, S, tokens, None, None, None,
                                        ws, ws_bytes, None)


def test_stage2_nvfp4_argument_validation(lib):
    assert lib.nfq_lm_head_nvfp4_packed_bytes(4096, 1152) == 0
    assert lib.nfq_lm_head_nvfp4_packed_bytes(129280, 7168) == 1010 * 28 * 18432
    assert _stage2_fp4(lib, codes=0) == nfq.NFQ_ERR_NULL
    assert _stage2_fp4(lib, gs=0) == nfq.NFQ_ERR_NULL
    assert _stage2_fp4(lib, w=0) == nfq.NFQ_ERR_NULL
    assert _stage2_fp4(lib, H=1152) == nfq.NFQ_ERR_SHAPE
    assert _stage2_fp4(lib, block=32) == nfq.NFQ_ERR_SHAPE
    assert _stage2_fp4(lib, V=4095) == nfq.NFQ_ERR_SHAPE
    assert _stage2_fp4(lib, ws=0) == nfq.NFQ_ERR_WORKSPACE
    assert _stage2_fp4(lib, ws_bytes=8) == nfq.NFQ_ERR_WORKSPACE
    assert _stage2_fp4(lib, bs=MIS) == nfq.NFQ_ERR_ALIGN
    assert _stage2_fp4(lib, tokens=FAKE + 2) == nfq.NFQ_ERR_ALIGN
    assert _stage2_fp4(lib, T=0) == nfq.NFQ_OK
    pk = lambda codes=FAKE, bs=FAKE, V=4096, H=1024, n=None: lib.nfq_lm_head_nvfp4_pack_weights(
        codes, bs, V, H, FAKE, lib.nfq_lm_head_nvfp4_packed_bytes(V, H) if n is None else n, None)
    assert pk(codes=0) == nfq.NFQ_ERR_NULL
    assert pk(H=1000) == nfq.NFQ_ERR_SHAPE
    assert pk(n=16) == nfq.NFQ_ERR_WORKSPACE
    assert pk(bs=MIS) == nfq.NFQ_ERR_ALIGN


def test_probe_argument_validation(lib):
    """The measurement kernels reject their out-of-range arguments before any
    device call (so these run without a GPU)."""
    shape = nfq.NFQ_ERR_SHAPE
    assert lib.nfq_probe_handshake(0, 3, 1, 4, 16, None) == shape     # 3 buffers
    assert lib.nfq_probe_handshake(1, 8, 1, 4, 16, None) == shape     # pairs: 2 or 4 buffers
    assert lib.nfq_probe_handshake(0, 2, 4, 4, 16, None) == shape     # mode 4
    assert lib.nfq_probe_handshake(0, 2, 3, 4, 16, None) == shape     # mode 3: 4 buffers only
    assert lib.nfq_probe_handshake(0, 2, 1, 0, 16, None) == shape     # no CTAs
    assert lib.nfq_probe_handshake(0, 2, 1, 4, 0, None) == shape      # no K blocks
    assert lib.nfq_probe_fp8_mma(1, 4, 16, 0, None) == shape          # readers: one CTA only
    assert lib.nfq_probe_fp8_mma(0, 4, 16, 5, None) == shape
    assert lib.nfq_probe_nvfp4_mma(1, 0, 16, None) == shape
    assert lib.nfq_probe_nvfp4_mma(0, 4, 0, None) == shape
    assert lib.nfq_probe_handoff(4, 16, None) == shape
    assert lib.nfq_probe_fp8_mma_shape(96, 256, 4, 16, None) == shape
    assert lib.nfq_probe_fp8_mma_shape(128, 264, 4, 16, None) == shape
    assert lib.nfq_probe_fp8_mma_shape(64, 12, 4, 16, None) == shape
    assert lib.nfq_probe_handoff(1, 0, None) == shape
    assert lib.nfq_probe_tmem_ld(0, 0, 8, None) == shape
    assert lib.nfq_check_fp8_quotient(None, None, None) == nfq.NFQ_ERR_NULL
    assert lib.nfq_check_fp4_quotient(None, None, None) == nfq.NFQ_ERR_NULL
    assert lib.nfq_check_fp4_quotient(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4),
                                      None) == nfq.NFQ_ERR_ALIGN
    assert lib.nfq_check_fp8_quotient(ctypes.c_void_p(FAKE + 4), ctypes.c_void_p(FAKE),
                                      None) == nfq.NFQ_ERR_ALIGN
