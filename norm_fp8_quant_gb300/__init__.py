"""GB300 (sm_103a) MTP draft-layer tail: Python binding of the C-ABI library.

Thin argument marshalling over libnfq.so (include/nfq.h); every step of the
path runs in the library's CUDA kernels.  PyTorch only provides device memory
and the current stream.  There is no fallback: if the library is missing or
the device is not a compute-capability 10.3 GPU, calls raise.

  mtp_reduce_norm_quant(partials, residual, norm_w, eps=1e-6)
      -> (hidden bf16 [T][H], codes uint8 [T][H], scales fp32 [T][H/128])
  lm_head_fp8_argmax(codes, scales, w, w_scales, S, workspace=None)
      -> draft tokens int32 [T] (optionally max logit and per-shard results)
  mtp_reduce_norm_quant_nvfp4 / pack_lm_head_weights_nvfp4 / lm_head_nvfp4_argmax
      the same two stages with the NVFP4 activation and weight
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnfq.so")

NFQ_OK = 0
NFQ_ERR_NULL = -1
NFQ_ERR_SHAPE = -2
NFQ_ERR_ALIGN = -3
NFQ_ERR_WORKSPACE = -4
NFQ_ERR_CUDA = -5
NFQ_ERR_TIMEOUT = -6
NFQ_ERR_DEVICE = -7

GROUP = 128


class NfqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})")


class QuantAct(ctypes.Structure):
    """nfq_quant_act: packed FP8 activation descriptor (host struct)."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tokens", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("group", ctypes.c_int32)]


class Fp4Act(ctypes.Structure):
    """nfq_fp4_act: NVFP4 activation descriptor (host struct)."""
    _fields_ = [("codes", ctypes.c_void_p), ("block_scales", ctypes.c_void_p),
                ("row_scales", ctypes.c_void_p), ("tokens", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("block", ctypes.c_int32)]


FP4_BLOCK = 16

_lib = None
_P = ctypes.c_void_p


def load(path: str = LIB_PATH):
    """Load libnfq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with norm_fp8_quant_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.nfq_status_str.argtypes = [ctypes.c_int]
    lib.nfq_status_str.restype = ctypes.c_char_p
    lib.nfq_abi_version.argtypes = []
    lib.nfq_abi_version.restype = ctypes.c_int
    lib.nfq_mtp_reduce_norm_quant.argtypes = [_P, ctypes.c_int, _P, _P, ctypes.c_float,
                                              ctypes.c_int, ctypes.c_int, _P,
                                              ctypes.POINTER(QuantAct), _P]
    lib.nfq_mtp_reduce_norm_quant.restype = ctypes.c_int
    lib.nfq_lm_head_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.nfq_lm_head_workspace_bytes.restype = ctypes.c_size_t
    lib.nfq_lm_head_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
    lib.nfq_lm_head_workspace_init.restype = ctypes.c_int
    lib.nfq_lm_head_fp8_argmax.argtypes = [ctypes.POINTER(QuantAct), _P, _P, ctypes.c_int,
                                           ctypes.c_int, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.nfq_lm_head_fp8_argmax.restype = ctypes.c_int
    lib.nfq_lm_head_packed_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.nfq_lm_head_packed_bytes.restype = ctypes.c_size_t
    lib.nfq_lm_head_pack_weights.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, ctypes.c_size_t, _P]
    lib.nfq_lm_head_pack_weights.restype = ctypes.c_int
    lib.nfq_lm_head_fp8_argmax_packed.argtypes = lib.nfq_lm_head_fp8_argmax.argtypes
    lib.nfq_lm_head_fp8_argmax_packed.restype = ctypes.c_int
    lib.nfq_mtp_draft_chain.argtypes = [ctypes.c_int, _P, ctypes.c_int, _P, _P, ctypes.c_float,
                                        ctypes.c_int, ctypes.c_int, _P, ctypes.POINTER(QuantAct),
                                        _P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, _P, _P,
                                        ctypes.c_size_t, _P]
    lib.nfq_mtp_draft_chain.restype = ctypes.c_int
    lib.nfq_device_error.argtypes = [ctypes.c_int]
    lib.nfq_device_error.restype = ctypes.c_int
    lib.nfq_stage1_plan.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    lib.nfq_stage1_plan.restype = ctypes.c_int
    lib.nfq_stage1_tune.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.nfq_stage1_tune.restype = None
    lib.nfq_lm_head_small_batch.argtypes = [ctypes.c_int]
    lib.nfq_lm_head_small_batch.restype = None
    lib.nfq_lm_head_pair.argtypes = [ctypes.c_int]
    lib.nfq_lm_head_pair.restype = None
    lib.nfq_probe_fp8_mma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    lib.nfq_probe_fp8_mma.restype = ctypes.c_int
    lib.nfq_probe_nvfp4_mma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    lib.nfq_probe_nvfp4_mma.restype = ctypes.c_int
    lib.nfq_probe_handoff.argtypes = [ctypes.c_int, ctypes.c_int, _P]
    lib.nfq_probe_handoff.restype = ctypes.c_int
    lib.nfq_probe_fp8_mma_shape.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             _P]
    lib.nfq_probe_fp8_mma_shape.restype = ctypes.c_int
    lib.nfq_probe_tmem_ld.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    lib.nfq_probe_tmem_ld.restype = ctypes.c_int
    lib.nfq_probe_handshake.argtypes = [ctypes.c_int] * 5 + [_P]
    lib.nfq_probe_handshake.restype = ctypes.c_int
    lib.nfq_check_fp8_quotient.argtypes = [_P, _P, _P]
    lib.nfq_check_fp8_quotient.restype = ctypes.c_int
    lib.nfq_check_fp4_quotient.argtypes = [_P, _P, _P]
    lib.nfq_check_fp4_quotient.restype = ctypes.c_int
    lib.nfq_probe_wait_timeout.argtypes = [_P]
    lib.nfq_probe_wait_timeout.restype = ctypes.c_int
    lib.nfq_probe_stage1_reads.argtypes = [_P, ctypes.c_int, _P, ctypes.c_int, ctypes.c_int, _P]
    lib.nfq_probe_stage1_reads.restype = ctypes.c_int
    lib.nfq_mtp_reduce_norm_quant_nvfp4.argtypes = [_P, ctypes.c_int, _P, _P, ctypes.c_float,
                                                    ctypes.c_int, ctypes.c_int, _P,
                                                    ctypes.POINTER(Fp4Act), _P]
    lib.nfq_mtp_reduce_norm_quant_nvfp4.restype = ctypes.c_int
    lib.nfq_lm_head_nvfp4_packed_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.nfq_lm_head_nvfp4_packed_bytes.restype = ctypes.c_size_t
    lib.nfq_lm_head_nvfp4_pack_weights.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, _P,
                                                   ctypes.c_size_t, _P]
    lib.nfq_lm_head_nvfp4_pack_weights.restype = ctypes.c_int
    lib.nfq_lm_head_nvfp4_argmax.argtypes = [ctypes.POINTER(Fp4Act), _P, ctypes.c_float,
                                             ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P,
                                             ctypes.c_size_t, _P]
    lib.nfq_lm_head_nvfp4_argmax.restype = ctypes.c_int
    lib.nfq_lm_head_nvfp4_tune.argtypes = [ctypes.c_int]
    lib.nfq_lm_head_nvfp4_tune.restype = None
    lib.nfq_stage1_grid.argtypes = [ctypes.c_int]
    lib.nfq_stage1_grid.restype = None
    lib.nfq_stage1_split.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.nfq_stage1_split.restype = None
    lib.nfq_stage1_split_plan.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          _P]
    lib.nfq_stage1_split_plan.restype = ctypes.c_int
    lib.nfq_mtp_draft_chain_nvfp4.argtypes = [ctypes.c_int, _P, ctypes.c_int, _P, _P,
                                              ctypes.c_float, ctypes.c_int, ctypes.c_int, _P,
                                              ctypes.POINTER(Fp4Act), _P, ctypes.c_float,
                                              ctypes.c_int, ctypes.c_int, _P, _P,
                                              ctypes.c_size_t, _P]
    lib.nfq_mtp_draft_chain_nvfp4.restype = ctypes.c_int
    lib.nfq_mtp_step_fp8.argtypes = [_P, ctypes.c_int, _P, _P, ctypes.c_float, ctypes.c_int,
                                     ctypes.c_int, _P, ctypes.POINTER(QuantAct), _P, _P,
                                     ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P,
                                     ctypes.c_size_t, _P]
    lib.nfq_mtp_step_fp8.restype = ctypes.c_int
    lib.nfq_unfused_allreduce_bf16.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P]
    lib.nfq_unfused_add_rmsnorm.argtypes = [_P, _P, _P, ctypes.c_float, ctypes.c_int,
                                            ctypes.c_int, _P, _P]
    lib.nfq_unfused_quant_fp8.argtypes = [_P, ctypes.c_int, ctypes.c_int,
                                          ctypes.POINTER(QuantAct), _P]
    lib.nfq_unfused_lm_head_logits.argtypes = [ctypes.POINTER(QuantAct), _P, _P, ctypes.c_int,
                                               _P, _P]
    lib.nfq_unfused_argmax_bf16.argtypes = [_P, ctypes.c_int, ctypes.c_int, _P, _P]
    for fn in (lib.nfq_unfused_allreduce_bf16, lib.nfq_unfused_add_rmsnorm,
               lib.nfq_unfused_quant_fp8, lib.nfq_unfused_lm_head_logits,
               lib.nfq_unfused_argmax_bf16):
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().nfq_status_str(status).decode()


def _check(status: int, what: str):
    if status != NFQ_OK:
        raise NfqError(status, what)


def _stream_ptr(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _raw_stream(dev_index: int, stream=None) -> int:
    """cudaStream_t (as an int) of `stream`, or of the current stream of the device."""
    import torch
    if stream is not None:
        return stream.cuda_stream
    return torch._C._cuda_getCurrentRawStream(dev_index)


def _on_device(dev_index: int, fn, *args):
    """Call fn with dev_index as the current CUDA device (switching only if needed)."""
    import torch
    if torch._C._cuda_getDevice() == dev_index:
        return fn(*args)
    with torch.cuda.device(dev_index):
        return fn(*args)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _need_tokens_out(t):
    """Token outputs may be device memory or pinned host memory, which the
    device addresses directly under unified addressing (the LM head then writes
    the tokens straight to the host)."""
    import torch
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError("tokens_out must be a contiguous int32 tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("tokens_out must be device memory or pinned host memory")


# ----------------------------------------------------------------- stage 1 --

def mtp_reduce_norm_quant(partials, residual, norm_w, eps: float = 1e-6,
                          hidden_out=None, codes_out=None, scales_out=None, stream=None):
    """Sum k BF16 partials and the residual in fp32, RMSNorm, and emit the BF16
    hidden plus the packed FP8 activation (e4m3 codes, fp32 scale per 128)."""
    import torch
    k = len(partials)
    T, H = residual.shape
    _need_cuda(residual, norm_w, *partials)
    for p in partials:
        if p.dtype != torch.bfloat16 or p.shape != (T, H):
            raise ValueError("partials must be bf16 [T][H]")
    if residual.dtype != torch.bfloat16 or norm_w.dtype != torch.bfloat16:
        raise ValueError("residual and norm_w must be bf16")
    dev = residual.device
    hidden = hidden_out if hidden_out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    codes = codes_out if codes_out is not None else torch.empty((T, H), dtype=torch.uint8, device=dev)
    scales = scales_out if scales_out is not None else torch.empty((T, H // GROUP), dtype=torch.float32, device=dev)
    arr = (ctypes.c_void_p * max(k, 1))(*[p.data_ptr() for p in partials])
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    st = _on_device(dev.index, load().nfq_mtp_reduce_norm_quant, arr, k, residual.data_ptr(),
                    norm_w.data_ptr(), float(eps), T, H, hidden.data_ptr(), ctypes.byref(q),
                    _raw_stream(dev.index, stream))
    _check(st, "nfq_mtp_reduce_norm_quant")
    return hidden, codes, scales


# ----------------------------------------------------------------- stage 2 --

def lm_head_workspace_bytes(T: int, S: int) -> int:
    return int(load().nfq_lm_head_workspace_bytes(T, S))


def lm_head_workspace(T: int, S: int, device, stream=None):
    """A zero-filled workspace for nfq_lm_head_fp8_argmax (kept zero by every call)."""
    import torch
    n = lm_head_workspace_bytes(T, S)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    with torch.cuda.device(ws.device):
        _check(load().nfq_lm_head_workspace_init(_ptr(ws), n, _stream_ptr(stream)),
               "nfq_lm_head_workspace_init")
    return ws


def pack_lm_head_weights(w, stream=None):
    """Pack a row-major [V][H] e4m3 LM-head weight into the streaming layout
    (tile-contiguous, pre-swizzled 16 KB blocks); returns a PackedWeight."""
    import torch
    _need_cuda(w)
    V, H = w.shape
    n = int(load().nfq_lm_head_packed_bytes(V, H))
    if n == 0:
        raise ValueError("invalid LM-head weight shape")
    out = torch.empty(n, dtype=torch.uint8, device=w.device)
    with torch.cuda.device(w.device):
        _check(load().nfq_lm_head_pack_weights(_ptr(w), V, H, _ptr(out), n, _stream_ptr(stream)),
               "nfq_lm_head_pack_weights")
    return PackedWeight(out, V, H)


class PackedWeight:
    """LM-head weight in the packed streaming layout (see nfq_lm_head_pack_weights)."""

    def __init__(self, data, V: int, H: int):
        self.data, self.V, self.H = data, V, H
        self.device = data.device
        self.dtype = data.dtype

    @property
    def shape(self):
        return (self.V, self.H)

    @property
    def is_cuda(self):
        return self.data.is_cuda

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self.data.data_ptr()


def lm_head_fp8_argmax(codes, scales, w, w_scales, S: int, workspace=None,
                       tokens_out=None, want_max: bool = False, want_shards: bool = False,
                       stream=None):
    """Greedy draft token per row of the packed FP8 activation against the
    block-scaled FP8 LM head, via a vocab-sharded argmax (ties -> lowest id).
    `w` is the row-major e4m3 [V][H] weight or a PackedWeight.

    Returns tokens, or (tokens, max_logit, shard_idx, shard_val) with the
    optional ones None unless requested."""
    import torch
    T, H = codes.shape
    V = w.shape[0]
    packed = isinstance(w, PackedWeight)
    _need_cuda(codes, scales, w, w_scales)
    if codes.dtype != torch.uint8 or w.dtype != torch.uint8:
        raise ValueError("codes and w must be uint8 e4m3 patterns")
    if scales.dtype != torch.float32 or w_scales.dtype != torch.float32:
        raise ValueError("scales must be float32")
    dev = codes.device
    ws = workspace if workspace is not None else lm_head_workspace(T, S, dev, stream)
    tokens = tokens_out if tokens_out is not None else torch.empty(T, dtype=torch.int32, device=dev)
    mx = torch.empty(T, dtype=torch.float32, device=dev) if want_max else None
    sidx = torch.empty((S, T), dtype=torch.int32, device=dev) if want_shards else None
    sval = torch.empty((S, T), dtype=torch.float32, device=dev) if want_shards else None
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    opt = lambda t: None if t is None else t.data_ptr()
    fn = load().nfq_lm_head_fp8_argmax_packed if packed else load().nfq_lm_head_fp8_argmax
    st = _on_device(dev.index, fn, ctypes.byref(q), w.data_ptr(), w_scales.data_ptr(), V, S,
                    tokens.data_ptr(), opt(mx), opt(sidx), opt(sval), ws.data_ptr(), ws.numel(),
                    _raw_stream(dev.index, stream))
    _check(st, "nfq_lm_head_fp8_argmax")
    if want_max or want_shards:
        return tokens, mx, sidx, sval
    return tokens


def mtp_draft_chain(partials, residual0, norm_w, w, w_scales, S: int, eps: float = 1e-6,
                    hidden_bufs=None, codes=None, scales=None, tokens_out=None,
                    workspace=None, stream=None):
    """Chained MTP draft positions: partials is a list (one per position) of
    lists of k BF16 [T][H] tensors; the hidden of each position is the residual
    of the next.  Returns (tokens int32 [P][T], hidden of every position)."""
    import torch
    P = len(partials)
    k = len(partials[0])
    T, H = residual0.shape
    for ps in partials:
        if len(ps) != k:
            raise ValueError("every position needs k partials")
        _need_cuda(*ps)
    _need_cuda(residual0, norm_w, w_scales)
    dev = residual0.device
    if hidden_bufs is None:
        hidden_bufs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(min(P, 2))]
    hidden_of = [hidden_bufs[p % len(hidden_bufs)] for p in range(P)]
    codes = codes if codes is not None else torch.empty((T, H), dtype=torch.uint8, device=dev)
    scales = scales if scales is not None else torch.empty((T, H // GROUP), dtype=torch.float32, device=dev)
    tokens = tokens_out if tokens_out is not None else torch.empty((P, T), dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else lm_head_workspace(T, S, dev, stream)
    parr = (ctypes.c_void_p * (P * k))(*[t.data_ptr() for ps in partials for t in ps])
    harr = (ctypes.c_void_p * P)(*[h.data_ptr() for h in hidden_of])
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    packed = isinstance(w, PackedWeight)
    with torch.cuda.device(dev):
        st = load().nfq_mtp_draft_chain(P, parr, k, _ptr(residual0), _ptr(norm_w), float(eps), T, H,
                                        harr, ctypes.byref(q), _ptr(w), 1 if packed else 0,
                                        _ptr(w_scales), w.shape[0], S, _ptr(tokens), _ptr(ws),
                                        ws.numel(), _stream_ptr(stream))
    _check(st, "nfq_mtp_draft_chain")
    return tokens, hidden_of


def device_error(clear: bool = True) -> int:
    """Synchronise the current device and return its error-word status
    (NFQ_OK, or NFQ_ERR_TIMEOUT when a kernel gave up a bounded wait)."""
    return int(load().nfq_device_error(1 if clear else 0))


def stage1_plan(T: int, H: int, k: int, num_sms: int = 152):
    out = (ctypes.c_int * 7)()
    _check(load().nfq_stage1_plan(T, H, k, num_sms, out), "nfq_stage1_plan")
    return dict(zip(["cluster", "vpt", "active_threads", "threads", "slots", "smem",
                     "per_slot"], list(out)))


def stage1_tune(cluster: int = 0, vpt: int = 0, slots: int = 0, per_slot: int = 0):
    """Override the stage-1 launch plan (0 = automatic); for tuning sweeps."""
    load().nfq_stage1_tune(cluster, vpt, slots, per_slot)


def lm_head_small_batch(enabled: bool = True):
    """Choose the FP8 LM-head kernel family: the token-major kernel (default;
    up to 256 tokens per launch) or the weight-major kernel."""
    load().nfq_lm_head_small_batch(1 if enabled else 0)


def probe_fp8_mma(pair: bool, ctas: int, iters: int, stages: int = 1, stream=None):
    """Launch the FP8 MMA-rate measurement kernel (not part of the path):
    `ctas` CTAs (or CTA pairs) each issuing `iters` K blocks of four MMAs, K
    block i on operand set i % stages.  Returns the flops the launch performs."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_fp8_mma, 1 if pair else 0, ctas, iters, stages,
                      _raw_stream(dev, stream)), "nfq_probe_fp8_mma")
    M = 256 if pair else 128
    return 2.0 * M * 256 * 128 * iters * ctas


def probe_nvfp4_mma(pair: bool, ctas: int, iters: int, stream=None):
    """Launch the block-scaled NVFP4 MMA-rate measurement kernel (not part of
    the path): `ctas` CTAs (or CTA pairs) each issuing `iters` K steps of four
    MMAs of K = 64.  Returns the flops the launch performs."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_nvfp4_mma, 1 if pair else 0, ctas, iters,
                      _raw_stream(dev, stream)), "nfq_probe_nvfp4_mma")
    M = 256 if pair else 128
    return 2.0 * M * 256 * 256 * iters * ctas


def probe_fp8_mma_shape(m: int, n: int, ctas: int, iters: int, stream=None):
    """Launch the FP8 MMA-rate kernel (not part of the path) with MMAs of
    M = m x N = n x K = 32 on single CTAs.  Returns the flops the launch
    performs."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_fp8_mma_shape, m, n, ctas, iters,
                      _raw_stream(dev, stream)), "nfq_probe_fp8_mma_shape")
    return 2.0 * m * n * 128 * iters * ctas


def probe_handoff(mode: int, iters: int, stream=None):
    """Launch the barrier hand-off latency kernel (not part of the path):
    `iters` round trips; mode 0 within a CTA, 1..3 between the CTAs of a
    cluster (remote arrival at CTA scope, with cluster-scope release, by
    st.async).  Returns the number of one-way hand-offs."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_handoff, mode, iters, _raw_stream(dev, stream)),
           "nfq_probe_handoff")
    return 2 * iters


def probe_tmem_ld(batched: bool, ctas: int, iters: int, stream=None):
    """Launch the TMEM read-rate measurement kernel (not part of the path).
    Returns the bytes the launch reads from TMEM."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_tmem_ld, 1 if batched else 0, ctas, iters,
                      _raw_stream(dev, stream)), "nfq_probe_tmem_ld")
    return 128.0 * 256 * 4 * iters * ctas


def probe_handshake(pair: bool, buffers: int, mode: int, ctas: int, iters: int, stream=None):
    """Launch the accumulator hand-off measurement kernel (not part of the path):
    `ctas` CTAs (or CTA pairs) run `iters` K blocks through `buffers` TMEM
    buffers; mode 0 / 1: 16 epilogue warps release each buffer without / after
    reading it; mode 2: each group of MMAs waited for before the next.
    Returns the number of K blocks each CTA (pair) runs."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_handshake, 1 if pair else 0, buffers, mode, ctas,
                      iters, _raw_stream(dev, stream)), "nfq_probe_handshake")
    return iters


def check_fp8_quotient(stream=None):
    """Run the exhaustive check of stage 1's division-free FP8 scales,
    reciprocals and codes against IEEE arithmetic (a verification kernel, not
    part of the path).  Returns ([scale, reciprocal, code mismatches], first
    mismatch as (amax bits << 16) | hidden bits, or None)."""
    import torch
    dev = torch.cuda.current_device()
    count = torch.zeros(3, dtype=torch.int64, device=dev)
    first = torch.full((1,), -1, dtype=torch.int32, device=dev)
    _check(_on_device(dev, load().nfq_check_fp8_quotient, count.data_ptr(), first.data_ptr(),
                      _raw_stream(dev, stream)), "nfq_check_fp8_quotient")
    torch.cuda.synchronize(dev)
    f = int(first.item()) & 0xFFFFFFFF
    return [int(c) for c in count.tolist()], (None if f == 0xFFFFFFFF else f)


def probe_wait_timeout(stream=None):
    """Launch a kernel whose bounded wait runs out (about 2 s): afterwards
    device_error() reports NFQ_ERR_TIMEOUT.  A failure-detection check, not
    part of the path."""
    import torch
    dev = torch.cuda.current_device()
    _check(_on_device(dev, load().nfq_probe_wait_timeout, _raw_stream(dev, stream)),
           "nfq_probe_wait_timeout")


def check_fp4_quotient(stream=None):
    """Run the exhaustive check of the NVFP4 stage 1's division-free block-scale
    and e2m1 codes against IEEE arithmetic (a verification kernel, not part of
    the path).  Returns ([reciprocal of d, block-scale code, reciprocal of eff,
    e2m1 code mismatches], first mismatch as (scale code << 32) | (row max bits
    << 16) | value bits, or None)."""
    import torch
    dev = torch.cuda.current_device()
    count = torch.zeros(4, dtype=torch.int64, device=dev)
    first = torch.full((1,), -1, dtype=torch.int64, device=dev)
    _check(_on_device(dev, load().nfq_check_fp4_quotient, count.data_ptr(), first.data_ptr(),
                      _raw_stream(dev, stream)), "nfq_check_fp4_quotient")
    torch.cuda.synchronize(dev)
    f = int(first.item()) & 0xFFFFFFFFFFFFFFFF
    return [int(c) for c in count.tolist()], (None if f == 0xFFFFFFFFFFFFFFFF else f)


def prepare_probe_stage1_reads(partials, residual) -> "PreparedCall":
    """The small-batch stage-1 kernel's loads alone (a measurement kernel, not
    part of the path), as a PreparedCall."""
    import torch
    T, H = residual.shape
    _need_cuda(residual, *partials)
    if residual.dtype != torch.bfloat16 or any(p.dtype != torch.bfloat16 or p.shape != (T, H)
                                               for p in partials):
        raise ValueError("partials and residual must be bf16 [T][H]")
    arr = (ctypes.c_void_p * len(partials))(*[p.data_ptr() for p in partials])
    args = (arr, len(partials), residual.data_ptr(), T, H)
    return PreparedCall(load().nfq_probe_stage1_reads, args, residual.device.index,
                        "nfq_probe_stage1_reads", (partials, residual, arr))


def lm_head_pair(enabled: bool = True):
    """129..256 tokens: CTA pairs with cta_group::2 MMAs (default) or two
    independent 128-token groups."""
    load().nfq_lm_head_pair(1 if enabled else 0)


# ------------------------------------------------------------ NVFP4 form --

def mtp_reduce_norm_quant_nvfp4(partials, residual, norm_w, eps: float = 1e-6,
                                hidden_out=None, codes_out=None, block_scales_out=None,
                                row_scales_out=None, stream=None):
    """Stage 1 with the NVFP4 activation: returns (hidden bf16 [T][H], codes
    uint8 [T][H/2] (e2m1 pairs), block scales uint8 [T][H/16] (e4m3), row
    scales fp32 [T])."""
    import torch
    k = len(partials)
    T, H = residual.shape
    _need_cuda(residual, norm_w, *partials)
    for p in partials:
        if p.dtype != torch.bfloat16 or p.shape != (T, H):
            raise ValueError("partials must be bf16 [T][H]")
    if residual.dtype != torch.bfloat16 or norm_w.dtype != torch.bfloat16:
        raise ValueError("residual and norm_w must be bf16")
    dev = residual.device
    hidden = hidden_out if hidden_out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    codes = codes_out if codes_out is not None else torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    bs = (block_scales_out if block_scales_out is not None
          else torch.empty((T, H // FP4_BLOCK), dtype=torch.uint8, device=dev))
    gs = row_scales_out if row_scales_out is not None else torch.empty(T, dtype=torch.float32, device=dev)
    arr = (ctypes.c_void_p * max(k, 1))(*[p.data_ptr() for p in partials])
    q = Fp4Act(codes.data_ptr(), bs.data_ptr(), gs.data_ptr(), T, H, FP4_BLOCK)
    st = _on_device(dev.index, load().nfq_mtp_reduce_norm_quant_nvfp4, arr, k,
                    residual.data_ptr(), norm_w.data_ptr(), float(eps), T, H, hidden.data_ptr(),
                    ctypes.byref(q), _raw_stream(dev.index, stream))
    _check(st, "nfq_mtp_reduce_norm_quant_nvfp4")
    return hidden, codes, bs, gs


class PackedFp4Weight:
    """NVFP4 LM-head weight in the packed streaming layout, with its tensor scale."""

    def __init__(self, data, V: int, H: int, scale: float):
        self.data, self.V, self.H, self.scale = data, V, H, float(scale)
        self.device = data.device

    @property
    def shape(self):
        return (self.V, self.H)


def pack_lm_head_weights_nvfp4(codes, block_scales, scale: float, stream=None):
    """Pack row-major NVFP4 weight codes [V][H/2] and block scales [V][H/16]
    (with the tensor scale) into the streaming layout."""
    import torch
    _need_cuda(codes, block_scales)
    V, H2 = codes.shape
    H = 2 * H2
    if codes.dtype != torch.uint8 or block_scales.dtype != torch.uint8 or \
            tuple(block_scales.shape) != (V, H // FP4_BLOCK):
        raise ValueError("codes uint8 [V][H/2] and block scales uint8 [V][H/16] expected")
    n = int(load().nfq_lm_head_nvfp4_packed_bytes(V, H))
    if n == 0:
        raise ValueError("invalid NVFP4 LM-head weight shape")
    out = torch.empty(n, dtype=torch.uint8, device=codes.device)
    with torch.cuda.device(codes.device):
        _check(load().nfq_lm_head_nvfp4_pack_weights(_ptr(codes), _ptr(block_scales), V, H,
                                                     _ptr(out), n, _stream_ptr(stream)),
               "nfq_lm_head_nvfp4_pack_weights")
    return PackedFp4Weight(out, V, H, scale)


def lm_head_nvfp4_argmax(codes, block_scales, row_scales, w: PackedFp4Weight, S: int,
                         workspace=None, tokens_out=None, want_max: bool = False,
                         want_shards: bool = False, stream=None):
    """Greedy draft token per row of the NVFP4 activation against the packed
    NVFP4 LM head (vocab-sharded argmax, ties -> lowest id)."""
    import torch
    T, H2 = codes.shape
    H = 2 * H2
    _need_cuda(codes, block_scales, row_scales)
    if not isinstance(w, PackedFp4Weight):
        raise ValueError("w must be a PackedFp4Weight")
    if codes.dtype != torch.uint8 or block_scales.dtype != torch.uint8 or \
            row_scales.dtype != torch.float32:
        raise ValueError("codes/block scales uint8 and row scales float32 expected")
    dev = codes.device
    ws = workspace if workspace is not None else lm_head_workspace(T, S, dev, stream)
    tokens = tokens_out if tokens_out is not None else torch.empty(T, dtype=torch.int32, device=dev)
    mx = torch.empty(T, dtype=torch.float32, device=dev) if want_max else None
    sidx = torch.empty((S, T), dtype=torch.int32, device=dev) if want_shards else None
    sval = torch.empty((S, T), dtype=torch.float32, device=dev) if want_shards else None
    q = Fp4Act(codes.data_ptr(), block_scales.data_ptr(), row_scales.data_ptr(), T, H, FP4_BLOCK)
    opt = lambda t: None if t is None else t.data_ptr()
    st = _on_device(dev.index, load().nfq_lm_head_nvfp4_argmax, ctypes.byref(q), w.data.data_ptr(),
                    float(w.scale), w.V, S, tokens.data_ptr(), opt(mx), opt(sidx), opt(sval),
                    ws.data_ptr(), ws.numel(), _raw_stream(dev.index, stream))
    _check(st, "nfq_lm_head_nvfp4_argmax")
    if want_max or want_shards:
        return tokens, mx, sidx, sval
    return tokens


def lm_head_nvfp4_tune(stages: int = 0):
    """Pipeline stages of the NVFP4 LM head (0 = as many as fit); for sweeps."""
    load().nfq_lm_head_nvfp4_tune(stages)


# --------------------------------------------------------- prepared calls --

class PreparedCall:
    """One library call with its arguments checked and marshalled once.

    Calling it issues the C entry point on the given (or the current) stream of
    the tensors' device; the tensors it was prepared with must stay alive and
    unmoved (the object keeps references to them).  Each call costs a few
    microseconds of host time instead of the full argument checks, which
    matters in a decode loop that issues a step every ~100 us."""

    def __init__(self, fn, args, dev_index: int, what: str, keep):
        self._fn, self._args, self._dev, self._what, self._keep = fn, args, dev_index, what, keep

    def __call__(self, stream=None):
        st = _on_device(self._dev, self._fn, *self._args, _raw_stream(self._dev, stream))
        if st != NFQ_OK:
            raise NfqError(st, self._what)


def _check_stage1_args(partials, residual, norm_w):
    import torch
    T, H = residual.shape
    _need_cuda(residual, norm_w, *partials)
    for p in partials:
        if p.dtype != torch.bfloat16 or p.shape != (T, H):
            raise ValueError("partials must be bf16 [T][H]")
    if residual.dtype != torch.bfloat16 or norm_w.dtype != torch.bfloat16:
        raise ValueError("residual and norm_w must be bf16")
    return T, H


def prepare_reduce_norm_quant(partials, residual, norm_w, eps, hidden_out, codes_out,
                              scales_out) -> PreparedCall:
    """mtp_reduce_norm_quant with fixed buffers, as a PreparedCall."""
    T, H = _check_stage1_args(partials, residual, norm_w)
    _need_cuda(hidden_out, codes_out, scales_out)
    arr = (ctypes.c_void_p * len(partials))(*[p.data_ptr() for p in partials])
    q = QuantAct(codes_out.data_ptr(), scales_out.data_ptr(), T, H, GROUP)
    args = (arr, len(partials), residual.data_ptr(), norm_w.data_ptr(), float(eps), T, H,
            hidden_out.data_ptr(), ctypes.byref(q))
    return PreparedCall(load().nfq_mtp_reduce_norm_quant, args, residual.device.index,
                        "nfq_mtp_reduce_norm_quant",
                        (partials, residual, norm_w, hidden_out, codes_out, scales_out, arr, q))


def prepare_reduce_norm_quant_nvfp4(partials, residual, norm_w, eps, hidden_out, codes_out,
                                    block_scales_out, row_scales_out) -> PreparedCall:
    """mtp_reduce_norm_quant_nvfp4 with fixed buffers, as a PreparedCall."""
    T, H = _check_stage1_args(partials, residual, norm_w)
    _need_cuda(hidden_out, codes_out, block_scales_out, row_scales_out)
    arr = (ctypes.c_void_p * len(partials))(*[p.data_ptr() for p in partials])
    q = Fp4Act(codes_out.data_ptr(), block_scales_out.data_ptr(), row_scales_out.data_ptr(), T, H,
               FP4_BLOCK)
    args = (arr, len(partials), residual.data_ptr(), norm_w.data_ptr(), float(eps), T, H,
            hidden_out.data_ptr(), ctypes.byref(q))
    return PreparedCall(load().nfq_mtp_reduce_norm_quant_nvfp4, args, residual.device.index,
                        "nfq_mtp_reduce_norm_quant_nvfp4",
                        (partials, residual, norm_w, hidden_out, codes_out, block_scales_out,
                         row_scales_out, arr, q))


def prepare_lm_head_fp8_argmax(codes, scales, w, w_scales, S: int, workspace,
                               tokens_out) -> PreparedCall:
    """lm_head_fp8_argmax (tokens only) with fixed buffers, as a PreparedCall."""
    import torch
    T, H = codes.shape
    _need_cuda(codes, scales, w, w_scales, workspace)
    _need_tokens_out(tokens_out)
    if codes.dtype != torch.uint8 or w.dtype != torch.uint8 or scales.dtype != torch.float32 \
            or w_scales.dtype != torch.float32:
        raise ValueError("uint8 codes / weight and float32 scales expected")
    packed = isinstance(w, PackedWeight)
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    fn = load().nfq_lm_head_fp8_argmax_packed if packed else load().nfq_lm_head_fp8_argmax
    args = (ctypes.byref(q), w.data_ptr(), w_scales.data_ptr(), w.shape[0], S,
            tokens_out.data_ptr(), None, None, None, workspace.data_ptr(), workspace.numel())
    return PreparedCall(fn, args, codes.device.index, "nfq_lm_head_fp8_argmax",
                        (codes, scales, w, w_scales, workspace, tokens_out, q))


def prepare_lm_head_nvfp4_argmax(codes, block_scales, row_scales, w: PackedFp4Weight, S: int,
                                 workspace, tokens_out) -> PreparedCall:
    """lm_head_nvfp4_argmax (tokens only) with fixed buffers, as a PreparedCall."""
    import torch
    T, H2 = codes.shape
    _need_cuda(codes, block_scales, row_scales, workspace)
    _need_tokens_out(tokens_out)
    if not isinstance(w, PackedFp4Weight):
        raise ValueError("w must be a PackedFp4Weight")
    if codes.dtype != torch.uint8 or block_scales.dtype != torch.uint8 or \
            row_scales.dtype != torch.float32:
        raise ValueError("codes/block scales uint8 and row scales float32 expected")
    q = Fp4Act(codes.data_ptr(), block_scales.data_ptr(), row_scales.data_ptr(), T, 2 * H2,
               FP4_BLOCK)
    args = (ctypes.byref(q), w.data.data_ptr(), float(w.scale), w.V, S, tokens_out.data_ptr(),
            None, None, None, workspace.data_ptr(), workspace.numel())
    return PreparedCall(load().nfq_lm_head_nvfp4_argmax, args, codes.device.index,
                        "nfq_lm_head_nvfp4_argmax",
                        (codes, block_scales, row_scales, w, workspace, tokens_out, q))


def stage1_grid(max_ctas: int = 0):
    """Cap the stage-1 grid (each CTA then takes several rows); 0 = automatic."""
    load().nfq_stage1_grid(max_ctas)


def stage1_split(max_tokens: int = -1, ctas_per_row: int = 0, vpt: int = 0, tma: int = -1):
    """Small-batch stage-1 kernel: batches of at most max_tokens rows (-1 the
    default limit, 0 none), ctas_per_row CTAs per row and vpt vectors per
    thread (0 = automatic), inputs through registers (tma 0) or shared memory
    (tma 1; -1 automatic); for tuning sweeps and tests."""
    load().nfq_stage1_split(max_tokens, ctas_per_row, vpt, tma)


def stage1_split_plan(T: int, H: int, k: int = 8, num_sms: int = 152):
    out = (ctypes.c_int * 5)()
    _check(load().nfq_stage1_split_plan(T, H, k, num_sms, out), "nfq_stage1_split_plan")
    return dict(zip(["ctas_per_row", "vpt", "active_threads", "threads", "tma"], list(out)))


# ---------------------------------------------------- unfused reference arm --

def unfused_allreduce_bf16(partials, out=None, stream=None):
    """bf16(sum of the k BF16 partials): the separate all-reduce of the unfused path."""
    import torch
    T, H = partials[0].shape
    _need_cuda(*partials)
    dev = partials[0].device
    out = out if out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    arr = (ctypes.c_void_p * len(partials))(*[p.data_ptr() for p in partials])
    st = _on_device(dev.index, load().nfq_unfused_allreduce_bf16, arr, len(partials), T, H,
                    out.data_ptr(), _raw_stream(dev.index, stream))
    _check(st, "nfq_unfused_allreduce_bf16")
    return out


def unfused_add_rmsnorm(x, residual, norm_w, eps: float = 1e-6, hidden_out=None, stream=None):
    import torch
    T, H = x.shape
    _need_cuda(x, residual, norm_w)
    dev = x.device
    hidden = hidden_out if hidden_out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    st = _on_device(dev.index, load().nfq_unfused_add_rmsnorm, x.data_ptr(), residual.data_ptr(),
                    norm_w.data_ptr(), float(eps), T, H, hidden.data_ptr(),
                    _raw_stream(dev.index, stream))
    _check(st, "nfq_unfused_add_rmsnorm")
    return hidden


def unfused_quant_fp8(hidden, codes_out=None, scales_out=None, stream=None):
    import torch
    T, H = hidden.shape
    _need_cuda(hidden)
    dev = hidden.device
    codes = codes_out if codes_out is not None else torch.empty((T, H), dtype=torch.uint8, device=dev)
    scales = scales_out if scales_out is not None else torch.empty((T, H // GROUP), dtype=torch.float32, device=dev)
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    st = _on_device(dev.index, load().nfq_unfused_quant_fp8, hidden.data_ptr(), T, H,
                    ctypes.byref(q), _raw_stream(dev.index, stream))
    _check(st, "nfq_unfused_quant_fp8")
    return codes, scales


def unfused_lm_head_logits(codes, scales, w: PackedWeight, w_scales, logits_out=None,
                           stream=None):
    """BF16 logits [T][V] of the packed FP8 LM head."""
    import torch
    T, H = codes.shape
    _need_cuda(codes, scales, w_scales)
    if not isinstance(w, PackedWeight):
        raise ValueError("w must be a PackedWeight")
    dev = codes.device
    out = logits_out if logits_out is not None else torch.empty((T, w.V), dtype=torch.bfloat16, device=dev)
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    st = _on_device(dev.index, load().nfq_unfused_lm_head_logits, ctypes.byref(q), w.data_ptr(),
                    w_scales.data_ptr(), w.V, out.data_ptr(), _raw_stream(dev.index, stream))
    _check(st, "nfq_unfused_lm_head_logits")
    return out


def unfused_argmax_bf16(logits, tokens_out=None, stream=None):
    import torch
    T, V = logits.shape
    _need_cuda(logits)
    dev = logits.device
    tok = tokens_out if tokens_out is not None else torch.empty(T, dtype=torch.int32, device=dev)
    st = _on_device(dev.index, load().nfq_unfused_argmax_bf16, logits.data_ptr(), T, V,
                    tok.data_ptr(), _raw_stream(dev.index, stream))
    _check(st, "nfq_unfused_argmax_bf16")
    return tok


# ------------------------------------------------ sequence-parallel rows --

def sp_row_range(T: int, rank: int, world: int):
    """The contiguous token rows [r0, r1) that rank `rank` of `world`
    sequence-parallel ranks owns: after the reduce-scatter of the partials a
    rank holds the summed rows of its range and runs stage 1 on them alone
    (rows are independent).  Ranges differ in size by at most one row."""
    if world < 1 or not 0 <= rank < world or T < 0:
        raise ValueError("need 0 <= rank < world and T >= 0")
    return rank * T // world, (rank + 1) * T // world


def mtp_draft_chain_nvfp4(partials, residual0, norm_w, w: PackedFp4Weight, S: int,
                          eps: float = 1e-6, hidden_bufs=None, codes=None, block_scales=None,
                          row_scales=None, tokens_out=None, workspace=None, stream=None):
    """mtp_draft_chain with the NVFP4 forms of both stages.  Returns (tokens
    int32 [P][T], hidden of every position)."""
    import torch
    P = len(partials)
    k = len(partials[0])
    T, H = residual0.shape
    for ps in partials:
        if len(ps) != k:
            raise ValueError("every position needs k partials")
        _need_cuda(*ps)
    _need_cuda(residual0, norm_w)
    if not isinstance(w, PackedFp4Weight):
        raise ValueError("w must be a PackedFp4Weight")
    dev = residual0.device
    if hidden_bufs is None:
        hidden_bufs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(min(P, 2))]
    hidden_of = [hidden_bufs[p % len(hidden_bufs)] for p in range(P)]
    codes = codes if codes is not None else torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    bs = (block_scales if block_scales is not None
          else torch.empty((T, H // FP4_BLOCK), dtype=torch.uint8, device=dev))
    gs = row_scales if row_scales is not None else torch.empty(T, dtype=torch.float32, device=dev)
    tokens = tokens_out if tokens_out is not None else torch.empty((P, T), dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else lm_head_workspace(T, S, dev, stream)
    parr = (ctypes.c_void_p * (P * k))(*[t.data_ptr() for ps in partials for t in ps])
    harr = (ctypes.c_void_p * P)(*[h.data_ptr() for h in hidden_of])
    q = Fp4Act(codes.data_ptr(), bs.data_ptr(), gs.data_ptr(), T, H, FP4_BLOCK)
    st = _on_device(dev.index, load().nfq_mtp_draft_chain_nvfp4, P, parr, k, residual0.data_ptr(),
                    norm_w.data_ptr(), float(eps), T, H, harr, ctypes.byref(q), w.data.data_ptr(),
                    float(w.scale), w.V, S, tokens.data_ptr(), ws.data_ptr(), ws.numel(),
                    _raw_stream(dev.index, stream))
    _check(st, "nfq_mtp_draft_chain_nvfp4")
    return tokens, hidden_of


# ------------------------------------------------------------- fused step --

def _step_args(partials, residual, norm_w, eps, hidden, codes, scales, w, w_scales, S, ws,
               tokens, mx, sidx, sval):
    T, H = residual.shape
    arr = (ctypes.c_void_p * len(partials))(*[p.data_ptr() for p in partials])
    q = QuantAct(codes.data_ptr(), scales.data_ptr(), T, H, GROUP)
    opt = lambda t: None if t is None else t.data_ptr()
    args = (arr, len(partials), residual.data_ptr(), norm_w.data_ptr(), float(eps), T, H,
            hidden.data_ptr(), ctypes.byref(q), w.data_ptr(), w_scales.data_ptr(), w.V, S,
            tokens.data_ptr(), opt(mx), opt(sidx), opt(sval), ws.data_ptr(), ws.numel())
    return args, (arr, q)


def mtp_step_fp8(partials, residual, norm_w, w: PackedWeight, w_scales, S: int,
                 eps: float = 1e-6, hidden_out=None, codes_out=None, scales_out=None,
                 tokens_out=None, workspace=None, want_max: bool = False,
                 want_shards: bool = False, stream=None):
    """One whole draft step (stage 1 + the FP8 LM head, one launch where it
    applies).  Returns (hidden, codes, scales, tokens) or, with want_max /
    want_shards, (hidden, codes, scales, tokens, max_logit, shard_idx, shard_val)."""
    import torch
    T, H = _check_stage1_args(partials, residual, norm_w)
    if not isinstance(w, PackedWeight):
        raise ValueError("w must be a PackedWeight")
    _need_cuda(w_scales)
    dev = residual.device
    hidden = hidden_out if hidden_out is not None else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    codes = codes_out if codes_out is not None else torch.empty((T, H), dtype=torch.uint8, device=dev)
    scales = scales_out if scales_out is not None else torch.empty((T, H // GROUP), dtype=torch.float32, device=dev)
    tokens = tokens_out if tokens_out is not None else torch.empty(T, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else lm_head_workspace(T, S, dev, stream)
    mx = torch.empty(T, dtype=torch.float32, device=dev) if want_max else None
    sidx = torch.empty((S, T), dtype=torch.int32, device=dev) if want_shards else None
    sval = torch.empty((S, T), dtype=torch.float32, device=dev) if want_shards else None
    args, keep = _step_args(partials, residual, norm_w, eps, hidden, codes, scales, w, w_scales,
                            S, ws, tokens, mx, sidx, sval)
    st = _on_device(dev.index, load().nfq_mtp_step_fp8, *args, _raw_stream(dev.index, stream))
    _check(st, "nfq_mtp_step_fp8")
    if want_max or want_shards:
        return hidden, codes, scales, tokens, mx, sidx, sval
    return hidden, codes, scales, tokens


def prepare_mtp_step_fp8(partials, residual, norm_w, eps, hidden_out, codes_out, scales_out,
                         w: PackedWeight, w_scales, S: int, workspace, tokens_out) -> PreparedCall:
    """mtp_step_fp8 (tokens only) with fixed buffers, as a PreparedCall."""
    T, H = _check_stage1_args(partials, residual, norm_w)
    _need_cuda(hidden_out, codes_out, scales_out, w_scales, workspace)
    _need_tokens_out(tokens_out)
    if not isinstance(w, PackedWeight):
        raise ValueError("w must be a PackedWeight")
    args, keep = _step_args(partials, residual, norm_w, eps, hidden_out, codes_out, scales_out,
                            w, w_scales, S, workspace, tokens_out, None, None, None)
    return PreparedCall(load().nfq_mtp_step_fp8, args, residual.device.index, "nfq_mtp_step_fp8",
                        (partials, residual, norm_w, hidden_out, codes_out, scales_out, w,
                         w_scales, workspace, tokens_out, keep))
