// C ABI of the MTP draft-layer tail: argument validation, device properties,
// the device error word and dispatch to the stage kernels.  See include/nfq.h
// for the contract of every entry point.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/nfq.h"
#include "nfq_internal.h"

namespace nfq {

// bit 0: a stage-1 wait expired, bit 1: a stage-2 wait expired
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready;
  bool supported;
  int num_sms;
  unsigned *err;   // device address of g_device_error
};

DeviceInfo g_dev[kMaxDevices];

// Per-device facts, looked up once per device (the first call on a device does
// this set-up; it issues no device work).
int device_info(DeviceInfo **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NFQ_ERR_CUDA;
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NFQ_ERR_CUDA;
    void *err = nullptr;
    if (cudaGetSymbolAddress(&err, g_device_error) != cudaSuccess) return NFQ_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.err = static_cast<unsigned *>(err);
    d.ready = true;
  }
  if (!d.supported) return NFQ_ERR_DEVICE;
  *out = &d;
  return NFQ_OK;
}

// The LM heads request their first weight stages before they wait for the
// kernel that precedes them on the stream.  A pack call therefore ends with an
// ordering point (an event recorded and waited on the same stream), after which
// a following kernel starts only once the packed weight is complete.
int stream_ordering_point(cudaStream_t stream) {
  static cudaEvent_t ev[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NFQ_ERR_CUDA;
  if (!ev[dev] && cudaEventCreateWithFlags(&ev[dev], cudaEventDisableTiming) != cudaSuccess)
    return NFQ_ERR_CUDA;
  if (cudaEventRecord(ev[dev], stream) != cudaSuccess ||
      cudaStreamWaitEvent(stream, ev[dev], 0) != cudaSuccess)
    return NFQ_ERR_CUDA;
  return NFQ_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int map_cuda(cudaError_t e) { return e == cudaSuccess ? NFQ_OK : NFQ_ERR_CUDA; }

}  // namespace

}  // namespace nfq

using namespace nfq;

extern "C" {

const char *nfq_status_str(int status) {
  switch (status) {
    case NFQ_OK: return "ok";
    case NFQ_ERR_NULL: return "a required pointer is NULL";
    case NFQ_ERR_SHAPE: return "a size is out of range or inconsistent";
    case NFQ_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case NFQ_ERR_WORKSPACE: return "the workspace is missing or too small";
    case NFQ_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case NFQ_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case NFQ_ERR_DEVICE: return "the current device is not a compute capability 10.3 GPU";
    default: return "unknown status";
  }
}

int nfq_abi_version(void) { return (1 << 16) | 0; }

int nfq_mtp_reduce_norm_quant(const void *const *partials, int k, const void *residual,
                              const void *norm_w, float eps, int T, int H, void *hidden_out,
                              const nfq_quant_act *q_out, void *stream) {
  if (!partials || !residual || !norm_w || !hidden_out || !q_out) return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials) return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i)
    if (!partials[i]) return NFQ_ERR_NULL;
  if (!q_out->codes || !q_out->scales) return NFQ_ERR_NULL;
  if (T < 0 || H < 128 || H > 32768 || H % 128 != 0) return NFQ_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps > 1.0f) return NFQ_ERR_SHAPE;
  if (q_out->group != 128 || q_out->tokens != T || q_out->hidden != H) return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i)
    if (!aligned16(partials[i])) return NFQ_ERR_ALIGN;
  if (!aligned16(residual) || !aligned16(norm_w) || !aligned16(hidden_out) ||
      !aligned16(q_out->codes) || !aligned16(q_out->scales))
    return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  Stage1Params p;
  std::memset(&p, 0, sizeof(p));
  for (int i = 0; i < k; ++i) p.partials[i] = partials[i];
  p.residual = residual;
  p.norm_w = norm_w;
  p.hidden = hidden_out;
  p.codes = q_out->codes;
  p.scales = q_out->scales;
  p.err = d->err;
  p.eps = eps;
  p.k = k;
  p.T = T;
  p.H = H;
  const cudaError_t e = launch_stage1(p, d->num_sms, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
  return map_cuda(e);
}

int nfq_mtp_reduce_norm_quant_nvfp4(const void *const *partials, int k, const void *residual,
                                    const void *norm_w, float eps, int T, int H,
                                    void *hidden_out, const nfq_fp4_act *q_out, void *stream) {
  if (!partials || !residual || !norm_w || !hidden_out || !q_out) return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials) return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i)
    if (!partials[i]) return NFQ_ERR_NULL;
  if (!q_out->codes || !q_out->block_scales || !q_out->row_scales) return NFQ_ERR_NULL;
  if (T < 0 || H < 256 || H > 16384 || H % 256 != 0) return NFQ_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps > 1.0f) return NFQ_ERR_SHAPE;
  if (q_out->block != 16 || q_out->tokens != T || q_out->hidden != H) return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i)
    if (!aligned16(partials[i])) return NFQ_ERR_ALIGN;
  if (!aligned16(residual) || !aligned16(norm_w) || !aligned16(hidden_out) ||
      !aligned16(q_out->codes) || !aligned16(q_out->block_scales) ||
      !aligned16(q_out->row_scales))
    return NFQ_ERR_ALIGN;
  if (!stage1_fp4_supported(H)) return NFQ_ERR_SHAPE;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  Stage1Params p;
  std::memset(&p, 0, sizeof(p));
  for (int i = 0; i < k; ++i) p.partials[i] = partials[i];
  p.residual = residual;
  p.norm_w = norm_w;
  p.hidden = hidden_out;
  p.codes = q_out->codes;
  p.bscales = q_out->block_scales;
  p.gscales = q_out->row_scales;
  p.fp4 = 1;
  p.err = d->err;
  p.eps = eps;
  p.k = k;
  p.T = T;
  p.H = H;
  const cudaError_t e = launch_stage1(p, d->num_sms, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
  return map_cuda(e);
}

size_t nfq_lm_head_workspace_bytes(int T, int S) {
  (void)T;
  if (S < 1 || S > kMaxShards) return 0;
  return stage2_workspace_bytes(S);
}

int nfq_lm_head_workspace_init(void *workspace, size_t ws_bytes, void *stream) {
  if (!workspace) return NFQ_ERR_NULL;
  if (!aligned16(workspace)) return NFQ_ERR_ALIGN;
  return map_cuda(cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace nfq {

// The MMA-rate probe with `stages` sets of operand tiles, and with 16 warps
// reading TMEM meanwhile (probe.cu).
cudaError_t launch_probe_fp8_mma_stages(int pair, int ctas, int iters, int stages,
                                        unsigned *err, cudaStream_t stream);
cudaError_t launch_probe_mma_with_readers(int ctas, int iters, unsigned *err,
                                          cudaStream_t stream);
cudaError_t launch_probe_nvfp4_mma(int pair, int ctas, int iters, unsigned *err,
                                   cudaStream_t stream);
cudaError_t launch_probe_handoff(int mode, int iters, unsigned *err, cudaStream_t stream);
cudaError_t launch_probe_fp8_mma_shape(int m, int n, int ctas, int iters, unsigned *err,
                                       cudaStream_t stream);
// The LM head's accumulator hand-off without data (probe.cu).
cudaError_t launch_probe_handshake(int pair, int buffers, int mode, int ctas, int iters,
                                   unsigned *err, cudaStream_t stream);
// Stage 1's division-free quotient against IEEE division (probe.cu).
cudaError_t launch_check_fp8_quotient(unsigned long long *count, unsigned *first,
                                      cudaStream_t stream);
cudaError_t launch_check_fp4_quotient(unsigned long long *count, unsigned long long *first,
                                      cudaStream_t stream);
// A bounded wait on a barrier nothing arrives on (probe.cu).
cudaError_t launch_probe_wait_timeout(unsigned *err, cudaStream_t stream);
// The form of the NVFP4 LM head for 129..256 tokens (lm_head_fp4.cu).
void stage2_fp4_set_pair(int enabled);

// Every argument of an FP8 LM-head call except the workspace: NULL pointers,
// shapes and alignment.  Queues nothing.
int lm_head_check_args(const nfq_quant_act *a, const uint8_t *w, const float *w_scales, int V,
                       int S, const int32_t *tokens_out, const float *max_logit_out,
                       const int32_t *shard_idx_out, const float *shard_val_out) {
  if (!a || !w || !w_scales || !tokens_out) return NFQ_ERR_NULL;
  if (!a->codes || !a->scales) return NFQ_ERR_NULL;
  const int T = a->tokens, H = a->hidden;
  if (a->group != 128 || H < 128 || H > 16384 || H % 128 != 0 || T < 0) return NFQ_ERR_SHAPE;
  if (V < 1 || S < 1 || S > kMaxShards || V % S != 0) return NFQ_ERR_SHAPE;
  // the per-token outputs are written with 4-byte stores
  if (!aligned16(a->codes) || !aligned16(a->scales) || !aligned16(w) || !aligned16(w_scales) ||
      !aligned4(tokens_out) || (max_logit_out && !aligned4(max_logit_out)) ||
      (shard_idx_out && !aligned4(shard_idx_out)) ||
      (shard_val_out && !aligned4(shard_val_out)))
    return NFQ_ERR_ALIGN;
  return NFQ_OK;
}

// NFQ_OK when the current device runs this library's kernels (looked up once
// per device).
int current_device_supported() {
  DeviceInfo *d = nullptr;
  return device_info(&d);
}

}  // namespace nfq

namespace {

int lm_head_common(const nfq_quant_act *a, const uint8_t *w, bool packed, const float *w_scales,
                   int V, int S, int32_t *tokens_out, float *max_logit_out,
                   int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                   size_t ws_bytes, void *stream) {
  const int chk = lm_head_check_args(a, w, w_scales, V, S, tokens_out, max_logit_out,
                                     shard_idx_out, shard_val_out);
  if (chk != NFQ_OK) return chk;
  if (!workspace) return NFQ_ERR_WORKSPACE;
  if (ws_bytes < stage2_workspace_bytes(S)) return NFQ_ERR_WORKSPACE;
  if (!aligned16(workspace)) return NFQ_ERR_ALIGN;
  const int T = a->tokens, H = a->hidden;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  const int G = H / 128;
  Stage2Params p;
  std::memset(&p, 0, sizeof(p));
  p.w_scales = w_scales;
  p.w_packed = packed ? w : nullptr;
  p.shard_idx_out = shard_idx_out;
  p.shard_val_out = shard_val_out;
  p.keys = static_cast<unsigned long long *>(workspace);
  p.counter = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(workspace) +
                                           stage2_workspace_bytes(S) - 16u);
  p.err = d->err;
  p.T_total = T;
  p.H = H;
  p.G = G;
  p.V = V;
  p.S = S;
  p.shard_width = V / S;
  p.n_vtiles = (V + 127) / 128;
  const int chunk = stage2_token_chunk();
  for (int t0 = 0; t0 < T; t0 += chunk) {
    const int Tc = (T - t0) < chunk ? (T - t0) : chunk;
    p.tok0 = t0;
    p.T = Tc;
    p.act_codes = a->codes + (size_t)t0 * H;
    p.act_scales = a->scales + (size_t)t0 * G;
    p.tokens_out = tokens_out + t0;
    p.max_logit_out = max_logit_out ? max_logit_out + t0 : nullptr;
    const cudaError_t e =
        launch_stage2(p, p.act_codes, w, d->num_sms, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
    if (e != cudaSuccess) return NFQ_ERR_CUDA;
  }
  return NFQ_OK;
}

}  // namespace

extern "C" {

int nfq_lm_head_fp8_argmax(const nfq_quant_act *a, const uint8_t *w, const float *w_scales,
                           int V, int S, int32_t *tokens_out, float *max_logit_out,
                           int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                           size_t ws_bytes, void *stream) {
  return lm_head_common(a, w, false, w_scales, V, S, tokens_out, max_logit_out, shard_idx_out,
                        shard_val_out, workspace, ws_bytes, stream);
}

size_t nfq_lm_head_packed_bytes(int V, int H) {
  if (V < 1 || H < 128 || H % 128 != 0) return 0;
  return packed_weight_bytes(V, H);
}

int nfq_lm_head_pack_weights(const uint8_t *w, int V, int H, uint8_t *w_packed,
                             size_t packed_bytes, void *stream) {
  if (!w || !w_packed) return NFQ_ERR_NULL;
  if (V < 1 || H < 128 || H > 16384 || H % 128 != 0) return NFQ_ERR_SHAPE;
  if (packed_bytes < packed_weight_bytes(V, H)) return NFQ_ERR_WORKSPACE;
  if (!aligned16(w) || !aligned16(w_packed)) return NFQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  const int r = map_cuda(launch_pack_weights(w, V, H, w_packed, static_cast<cudaStream_t>(stream)));
  return r != NFQ_OK ? r : stream_ordering_point(static_cast<cudaStream_t>(stream));
}

int nfq_lm_head_fp8_argmax_packed(const nfq_quant_act *a, const uint8_t *w_packed,
                                  const float *w_scales, int V, int S, int32_t *tokens_out,
                                  float *max_logit_out, int32_t *shard_idx_out,
                                  float *shard_val_out, void *workspace, size_t ws_bytes,
                                  void *stream) {
  return lm_head_common(a, w_packed, true, w_scales, V, S, tokens_out, max_logit_out,
                        shard_idx_out, shard_val_out, workspace, ws_bytes, stream);
}

int nfq_unfused_allreduce_bf16(const void *const *partials, int k, int T, int H, void *out,
                               void *stream) {
  if (!partials || !out) return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials || T < 0 || H < 8 || H % 8 != 0) return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i) {
    if (!partials[i]) return NFQ_ERR_NULL;
    if (!aligned16(partials[i])) return NFQ_ERR_ALIGN;
  }
  if (!aligned16(out)) return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  UnfusedReduceParams p;
  std::memset(&p, 0, sizeof(p));
  for (int i = 0; i < k; ++i) p.partials[i] = partials[i];
  p.k = k;
  p.n_vec = (size_t)T * (size_t)H / 8u;
  p.out = out;
  return map_cuda(launch_unfused_reduce(p, d->num_sms, static_cast<cudaStream_t>(stream)));
}

int nfq_unfused_add_rmsnorm(const void *x, const void *residual, const void *norm_w, float eps,
                            int T, int H, void *hidden_out, void *stream) {
  if (!x || !residual || !norm_w || !hidden_out) return NFQ_ERR_NULL;
  if (T < 0 || H < 128 || H > 16384 || H % 128 != 0) return NFQ_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps > 1.0f) return NFQ_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(norm_w) || !aligned16(hidden_out))
    return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_unfused_add_rmsnorm(x, residual, norm_w, eps, T, H, hidden_out,
                                             static_cast<cudaStream_t>(stream)));
}

int nfq_unfused_quant_fp8(const void *hidden, int T, int H, const nfq_quant_act *q_out,
                          void *stream) {
  if (!hidden || !q_out || !q_out->codes || !q_out->scales) return NFQ_ERR_NULL;
  if (T < 0 || H < 128 || H > 32768 || H % 128 != 0) return NFQ_ERR_SHAPE;
  if (q_out->group != 128 || q_out->tokens != T || q_out->hidden != H) return NFQ_ERR_SHAPE;
  if (!aligned16(hidden) || !aligned16(q_out->codes) || !aligned16(q_out->scales))
    return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_unfused_quant(hidden, T, H, q_out->codes, q_out->scales,
                                       static_cast<cudaStream_t>(stream)));
}

int nfq_unfused_lm_head_logits(const nfq_quant_act *a, const uint8_t *w_packed,
                               const float *w_scales, int V, void *logits_out, void *stream) {
  if (!a || !w_packed || !w_scales || !logits_out || !a->codes || !a->scales)
    return NFQ_ERR_NULL;
  const int T = a->tokens, H = a->hidden;
  if (a->group != 128 || H < 128 || H > 16384 || H % 128 != 0 || T < 0 || V < 1)
    return NFQ_ERR_SHAPE;
  if (!aligned16(a->codes) || !aligned16(a->scales) || !aligned16(w_packed) ||
      !aligned16(w_scales) || !aligned16(logits_out))
    return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  Stage2Params p;
  std::memset(&p, 0, sizeof(p));
  p.w_scales = w_scales;
  p.w_packed = w_packed;
  p.err = d->err;
  p.H = H;
  p.G = H / 128;
  p.V = V;
  p.S = 1;
  p.shard_width = V;
  p.n_vtiles = (V + 127) / 128;
  for (int t0 = 0; t0 < T; t0 += 128) {
    const int Tc = (T - t0) < 128 ? (T - t0) : 128;
    p.T = Tc;
    p.T_total = T;
    p.tok0 = t0;
    p.act_codes = a->codes + (size_t)t0 * H;
    p.act_scales = a->scales + (size_t)t0 * (H / 128);
    p.logits_out = static_cast<uint16_t *>(logits_out) + (size_t)t0 * (size_t)V;
    const cudaError_t e = launch_lm_head_logits(p, d->num_sms, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
    if (e != cudaSuccess) return NFQ_ERR_CUDA;
  }
  return NFQ_OK;
}

int nfq_unfused_argmax_bf16(const void *logits, int T, int V, int32_t *tokens_out,
                            void *stream) {
  if (!logits || !tokens_out) return NFQ_ERR_NULL;
  if (T < 0 || V < 1) return NFQ_ERR_SHAPE;
  if (!aligned16(logits) || !aligned4(tokens_out)) return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_unfused_argmax(logits, T, V, tokens_out,
                                        static_cast<cudaStream_t>(stream)));
}

size_t nfq_lm_head_nvfp4_packed_bytes(int V, int H) {
  if (V < 1 || H < 256 || H > 16384 || H % 256 != 0) return 0;
  return fp4_packed_weight_bytes(V, H);
}

int nfq_lm_head_nvfp4_pack_weights(const uint8_t *codes, const uint8_t *block_scales, int V,
                                   int H, void *w_packed, size_t packed_bytes, void *stream) {
  if (!codes || !block_scales || !w_packed) return NFQ_ERR_NULL;
  if (V < 1 || H < 256 || H > 16384 || H % 256 != 0) return NFQ_ERR_SHAPE;
  if (packed_bytes < fp4_packed_weight_bytes(V, H)) return NFQ_ERR_WORKSPACE;
  if (!aligned16(codes) || !aligned16(block_scales) || !aligned16(w_packed)) return NFQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  const int r = map_cuda(launch_pack_fp4_weights(codes, block_scales, V, H,
                                                 static_cast<uint8_t *>(w_packed),
                                                 static_cast<cudaStream_t>(stream)));
  return r != NFQ_OK ? r : stream_ordering_point(static_cast<cudaStream_t>(stream));
}

int nfq_lm_head_nvfp4_argmax(const nfq_fp4_act *a, const void *w_packed, float w_scale, int V,
                             int S, int32_t *tokens_out, float *max_logit_out,
                             int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                             size_t ws_bytes, void *stream) {
  if (!a || !w_packed || !tokens_out) return NFQ_ERR_NULL;
  if (!a->codes || !a->block_scales || !a->row_scales) return NFQ_ERR_NULL;
  const int T = a->tokens, H = a->hidden;
  if (a->block != 16 || H < 256 || H > 16384 || H % 256 != 0 || T < 0) return NFQ_ERR_SHAPE;
  if (V < 1 || S < 1 || S > kMaxShards || V % S != 0) return NFQ_ERR_SHAPE;
  if (!workspace) return NFQ_ERR_WORKSPACE;
  if (ws_bytes < stage2_workspace_bytes(S)) return NFQ_ERR_WORKSPACE;
  if (!aligned16(a->codes) || !aligned16(a->block_scales) || !aligned16(a->row_scales) ||
      !aligned16(w_packed) || !aligned4(tokens_out) || !aligned16(workspace) ||
      (max_logit_out && !aligned4(max_logit_out)) ||
      (shard_idx_out && !aligned4(shard_idx_out)) ||
      (shard_val_out && !aligned4(shard_val_out)))
    return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  Stage2Params p;
  std::memset(&p, 0, sizeof(p));
  p.w_packed = static_cast<const uint8_t *>(w_packed);
  p.w_scale = w_scale;
  p.shard_idx_out = shard_idx_out;
  p.shard_val_out = shard_val_out;
  p.keys = static_cast<unsigned long long *>(workspace);
  p.counter = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(workspace) +
                                           stage2_workspace_bytes(S) - 16u);
  p.err = d->err;
  p.T_total = T;
  p.H = H;
  p.G = H / 256;
  p.V = V;
  p.S = S;
  p.shard_width = V / S;
  p.n_vtiles = (V + 127) / 128;
  for (int t0 = 0; t0 < T; t0 += kFp4LaunchMaxT) {
    const int Tc = (T - t0) < kFp4LaunchMaxT ? (T - t0) : kFp4LaunchMaxT;
    p.tok0 = t0;
    p.T = Tc;
    p.act_codes = a->codes + (size_t)t0 * (size_t)(H / 2);
    p.act_bscales = a->block_scales + (size_t)t0 * (size_t)(H / 16);
    p.act_gscales = a->row_scales + t0;
    p.tokens_out = tokens_out + t0;
    p.max_logit_out = max_logit_out ? max_logit_out + t0 : nullptr;
    const cudaError_t e = launch_stage2_fp4(p, d->num_sms, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
    if (e != cudaSuccess) return NFQ_ERR_CUDA;
  }
  return NFQ_OK;
}

int nfq_mtp_draft_chain(int positions, const void *const *partials, int k,
                        const void *residual0, const void *norm_w, float eps, int T, int H,
                        void *const *hidden_out, const nfq_quant_act *q, const uint8_t *w,
                        int w_is_packed, const float *w_scales, int V, int S,
                        int32_t *tokens_out, void *workspace, size_t ws_bytes, void *stream) {
  if (positions < 1 || positions > 64) return NFQ_ERR_SHAPE;
  if (!partials || !hidden_out || !q || !tokens_out) return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials) return NFQ_ERR_SHAPE;
  for (int p = 0; p < positions; ++p) {
    if (!hidden_out[p]) return NFQ_ERR_NULL;
    // the residual of position p is the hidden of position p-1: distinct buffers
    if (p > 0 && hidden_out[p] == hidden_out[p - 1]) return NFQ_ERR_SHAPE;
    if (hidden_out[p] == residual0) return NFQ_ERR_SHAPE;
  }
  for (int p = 0; p < positions; ++p) {
    const void *residual = p == 0 ? residual0 : hidden_out[p - 1];
    int st = nfq_mtp_reduce_norm_quant(partials + (size_t)p * k, k, residual, norm_w, eps, T, H,
                                       hidden_out[p], q, stream);
    if (st != NFQ_OK) return st;
    int32_t *tok = tokens_out + (size_t)p * (size_t)T;
    st = w_is_packed ? nfq_lm_head_fp8_argmax_packed(q, w, w_scales, V, S, tok, nullptr, nullptr,
                                                     nullptr, workspace, ws_bytes, stream)
                     : nfq_lm_head_fp8_argmax(q, w, w_scales, V, S, tok, nullptr, nullptr,
                                              nullptr, workspace, ws_bytes, stream);
    if (st != NFQ_OK) return st;
  }
  return NFQ_OK;
}

int nfq_mtp_step_fp8(const void *const *partials, int k, const void *residual,
                     const void *norm_w, float eps, int T, int H, void *hidden_out,
                     const nfq_quant_act *q, const uint8_t *w_packed, const float *w_scales,
                     int V, int S, int32_t *tokens_out, float *max_logit_out,
                     int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                     size_t ws_bytes, void *stream) {
  if (!partials || !residual || !norm_w || !hidden_out || !q || !w_packed || !w_scales ||
      !tokens_out || !q->codes || !q->scales)
    return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials) return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i) {
    if (!partials[i]) return NFQ_ERR_NULL;
    if (!aligned16(partials[i])) return NFQ_ERR_ALIGN;
  }
  if (T < 0 || H < 128 || H > 16384 || H % 128 != 0) return NFQ_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps > 1.0f) return NFQ_ERR_SHAPE;
  if (q->group != 128 || q->tokens != T || q->hidden != H) return NFQ_ERR_SHAPE;
  if (V < 1 || S < 1 || S > kMaxShards || V % S != 0) return NFQ_ERR_SHAPE;
  if (!workspace || ws_bytes < stage2_workspace_bytes(S)) return NFQ_ERR_WORKSPACE;
  if (!aligned16(residual) || !aligned16(norm_w) || !aligned16(hidden_out) ||
      !aligned16(q->codes) || !aligned16(q->scales) || !aligned16(w_packed) ||
      !aligned16(w_scales) || !aligned16(workspace) || !aligned4(tokens_out) ||
      (max_logit_out && !aligned4(max_logit_out)) ||
      (shard_idx_out && !aligned4(shard_idx_out)) ||
      (shard_val_out && !aligned4(shard_val_out)))
    return NFQ_ERR_ALIGN;
  if (T == 0) return NFQ_OK;
  DeviceInfo *d = nullptr;
  int st = device_info(&d);
  if (st != NFQ_OK) return st;
  if (!fused_step_supported(T, H, k, V, d->num_sms)) {
    // the same results as two launches
    st = nfq_mtp_reduce_norm_quant(partials, k, residual, norm_w, eps, T, H, hidden_out, q,
                                   stream);
    if (st != NFQ_OK) return st;
    return nfq_lm_head_fp8_argmax_packed(q, w_packed, w_scales, V, S, tokens_out,
                                         max_logit_out, shard_idx_out, shard_val_out,
                                         workspace, ws_bytes, stream);
  }
  Stage2Params p;
  std::memset(&p, 0, sizeof(p));
  p.act_codes = q->codes;
  p.act_scales = q->scales;
  p.w_scales = w_scales;
  p.w_packed = w_packed;
  p.tokens_out = tokens_out;
  p.max_logit_out = max_logit_out;
  p.shard_idx_out = shard_idx_out;
  p.shard_val_out = shard_val_out;
  p.keys = static_cast<unsigned long long *>(workspace);
  p.counter = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(workspace) +
                                           stage2_workspace_bytes(S) - 16u);
  p.err = d->err;
  p.T = T;
  p.T_total = T;
  p.tok0 = 0;
  p.H = H;
  p.G = H / 128;
  p.V = V;
  p.S = S;
  p.shard_width = V / S;
  p.n_vtiles = (V + 127) / 128;
  for (int i = 0; i < k; ++i) p.s1.partials[i] = partials[i];
  p.s1.residual = residual;
  p.s1.norm_w = norm_w;
  p.s1.hidden = hidden_out;
  p.s1.codes = q->codes;
  p.s1.scales = q->scales;
  p.s1.ready = p.counter + 1;
  p.s1.eps = eps;
  p.s1.k = k;
  p.s1.na = H / 16;
  const cudaError_t e = launch_fused_step(p, d->num_sms, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
  return map_cuda(e);
}

int nfq_mtp_draft_chain_nvfp4(int positions, const void *const *partials, int k,
                              const void *residual0, const void *norm_w, float eps, int T, int H,
                              void *const *hidden_out, const nfq_fp4_act *q,
                              const void *w_packed, float w_scale, int V, int S,
                              int32_t *tokens_out, void *workspace, size_t ws_bytes,
                              void *stream) {
  if (positions < 1 || positions > 64) return NFQ_ERR_SHAPE;
  if (!partials || !hidden_out || !q || !tokens_out) return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials) return NFQ_ERR_SHAPE;
  for (int p = 0; p < positions; ++p) {
    if (!hidden_out[p]) return NFQ_ERR_NULL;
    if (p > 0 && hidden_out[p] == hidden_out[p - 1]) return NFQ_ERR_SHAPE;
    if (hidden_out[p] == residual0) return NFQ_ERR_SHAPE;
  }
  for (int p = 0; p < positions; ++p) {
    const void *residual = p == 0 ? residual0 : hidden_out[p - 1];
    int st = nfq_mtp_reduce_norm_quant_nvfp4(partials + (size_t)p * k, k, residual, norm_w, eps,
                                             T, H, hidden_out[p], q, stream);
    if (st != NFQ_OK) return st;
    st = nfq_lm_head_nvfp4_argmax(q, w_packed, w_scale, V, S, tokens_out + (size_t)p * (size_t)T,
                                  nullptr, nullptr, nullptr, workspace, ws_bytes, stream);
    if (st != NFQ_OK) return st;
  }
  return NFQ_OK;
}

int nfq_device_error(int clear) {
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return NFQ_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return NFQ_ERR_CUDA;
  if (v && clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess)
      return NFQ_ERR_CUDA;
  }
  return v ? NFQ_ERR_TIMEOUT : NFQ_OK;
}

// Launch-plan query and override for the stage-1 kernel (tuning sweeps; 0 = automatic).
void nfq_lm_head_nvfp4_tune(int stages) { stage2_fp4_set_stages(stages); }

void nfq_stage1_grid(int max_ctas) { stage1_set_grid(max_ctas); }

void nfq_stage1_split(int max_tokens, int ctas_per_row, int vpt, int tma) {
  stage1_set_split(max_tokens, ctas_per_row, vpt, tma);
}

int nfq_stage1_split_plan(int T, int H, int k, int num_sms, int *out5) {
  if (!out5) return NFQ_ERR_NULL;
  if (H < 128 || H % 128 || T < 1 || k < 1 || k > kMaxPartials || num_sms < 1)
    return NFQ_ERR_SHAPE;
  return stage1_split_plan(T, H, k, num_sms, out5);
}

int nfq_stage1_plan(int T, int H, int k, int num_sms, int *out7) {
  if (!out7) return NFQ_ERR_NULL;
  if (H < 128 || H % 128 || T < 1 || k < 1 || num_sms < 1) return NFQ_ERR_SHAPE;
  return stage1_plan(T, H, k, num_sms, out7);
}

void nfq_stage1_tune(int cluster, int vpt, int slots, int per_slot) {
  stage1_set_tuning(cluster, vpt, slots, per_slot);
}

// Selects the LM-head kernel family for T <= 64: 1 (default) the token-major
// small-batch kernel, 0 the weight-major kernel used for larger batches.
void nfq_lm_head_small_batch(int enabled) { stage2_set_small(enabled); }

int nfq_probe_fp8_mma(int pair, int ctas, int iters, int stages, void *stream) {
  if (ctas < 1 || ctas > 4096 || iters < 1 || iters > (1 << 20) || stages < 0 || stages > 4 ||
      (pair && stages == 0))
    return NFQ_ERR_SHAPE;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  if (stages == 0)   // one CTA per SM, with 16 warps reading TMEM during the MMAs
    return map_cuda(launch_probe_mma_with_readers(ctas, iters, d->err,
                                                  static_cast<cudaStream_t>(stream)));
  return map_cuda(launch_probe_fp8_mma_stages(pair ? 1 : 0, ctas, iters, stages, d->err,
                                              static_cast<cudaStream_t>(stream)));
}

int nfq_probe_nvfp4_mma(int pair, int ctas, int iters, void *stream) {
  if (ctas < 1 || ctas > 4096 || iters < 1 || iters > (1 << 20)) return NFQ_ERR_SHAPE;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_probe_nvfp4_mma(pair ? 1 : 0, ctas, iters, d->err,
                                         static_cast<cudaStream_t>(stream)));
}

int nfq_probe_fp8_mma_shape(int m, int n, int ctas, int iters, void *stream) {
  if (!((m == 64 && n % 8 == 0) || (m == 128 && n % 16 == 0)) || n < 16 || n > 256 || ctas < 1 ||
      ctas > 4096 || iters < 1 || iters > (1 << 20))
    return NFQ_ERR_SHAPE;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_probe_fp8_mma_shape(m, n, ctas, iters, d->err,
                                             static_cast<cudaStream_t>(stream)));
}

int nfq_probe_handoff(int mode, int iters, void *stream) {
  if (mode < 0 || mode > 3 || iters < 1 || iters > (1 << 20)) return NFQ_ERR_SHAPE;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_probe_handoff(mode, iters, d->err, static_cast<cudaStream_t>(stream)));
}

int nfq_probe_stage1_reads(const void *const *partials, int k, const void *residual, int T,
                           int H, void *stream) {
  if (!partials || !residual) return NFQ_ERR_NULL;
  if (k < 1 || k > kMaxPartials || T < 1 || H < 128 || H > 32768 || H % 128 != 0)
    return NFQ_ERR_SHAPE;
  for (int i = 0; i < k; ++i) {
    if (!partials[i]) return NFQ_ERR_NULL;
    if (!aligned16(partials[i])) return NFQ_ERR_ALIGN;
  }
  if (!aligned16(residual)) return NFQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  Stage1Params p;
  std::memset(&p, 0, sizeof(p));
  for (int i = 0; i < k; ++i) p.partials[i] = partials[i];
  p.residual = residual;
  p.k = k;
  p.T = T;
  p.H = H;
  const cudaError_t e = launch_stage1_reads(p, d->num_sms, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidConfiguration) return NFQ_ERR_SHAPE;
  return map_cuda(e);
}

int nfq_probe_handshake(int pair, int buffers, int mode, int ctas, int iters, void *stream) {
  if (ctas < 1 || ctas > 4096 || iters < 1 || iters > (1 << 20) || mode < 0 || mode > 3)
    return NFQ_ERR_SHAPE;
  if (!(buffers == 2 || buffers == 4 || (!pair && buffers == 8))) return NFQ_ERR_SHAPE;
  if (mode == 3 && buffers != 4) return NFQ_ERR_SHAPE;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_probe_handshake(pair ? 1 : 0, buffers, mode, ctas, iters, d->err,
                                         static_cast<cudaStream_t>(stream)));
}

int nfq_check_fp8_quotient(unsigned long long *mismatches, unsigned *first_bad, void *stream) {
  if (!mismatches || !first_bad) return NFQ_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(mismatches) & 7u) || (reinterpret_cast<uintptr_t>(first_bad) & 3u))
    return NFQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(
      launch_check_fp8_quotient(mismatches, first_bad, static_cast<cudaStream_t>(stream)));
}

int nfq_check_fp4_quotient(unsigned long long *mismatches, unsigned long long *first_bad,
                           void *stream) {
  if (!mismatches || !first_bad) return NFQ_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(mismatches) & 7u) || (reinterpret_cast<uintptr_t>(first_bad) & 7u))
    return NFQ_ERR_ALIGN;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(
      launch_check_fp4_quotient(mismatches, first_bad, static_cast<cudaStream_t>(stream)));
}

int nfq_probe_wait_timeout(void *stream) {
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(launch_probe_wait_timeout(d->err, static_cast<cudaStream_t>(stream)));
}

int nfq_probe_tmem_ld(int batched, int ctas, int iters, void *stream) {
  if (ctas < 1 || ctas > 4096 || iters < 1 || iters > (1 << 20)) return NFQ_ERR_SHAPE;
  DeviceInfo *d = nullptr;
  const int st = device_info(&d);
  if (st != NFQ_OK) return st;
  return map_cuda(
      launch_probe_tmem_ld(batched ? 1 : 0, ctas, iters, static_cast<cudaStream_t>(stream)));
}

// Selects the form of the FP8 and NVFP4 LM heads for 129..256 tokens: 1
// (default) CTA pairs issuing cta_group::2 MMAs, 0 two independent 128-token
// groups over one weight stream.
void nfq_lm_head_pair(int enabled) {
  stage2_set_pair(enabled);
  stage2_fp4_set_pair(enabled);
}

}  // extern "C"
