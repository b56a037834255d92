// nfq_lm_head_fp8_argmax_noalloc: the LM head + argmax without a caller
// workspace.  Its scratch (the per-shard argmax keys and the CTA counter) is a
// fixed array in this library's device memory, so the call allocates nothing.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "../../include/nfq.h"
#include "nfq_internal.h"

namespace nfq {
// Defined with the other entry points (abi.cu).
int lm_head_check_args(const nfq_quant_act *a, const uint8_t *w, const float *w_scales, int V,
                       int S, const int32_t *tokens_out, const float *max_logit_out,
                       const int32_t *shard_idx_out, const float *shard_val_out);
int current_device_supported();
}  // namespace nfq

namespace {

// Largest workspace any valid call needs: 64 shards x 256 keys x 8 bytes plus
// the 16-byte counter block (128 KiB + 16 B).  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 64u * 256u * 8u + 16u;
static_assert(kNoAllocScratchBytes == nfq::stage2_workspace_bytes_for(nfq::kMaxShards),
              "the array must hold the workspace of the largest shard count a call accepts");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
// Device address of the array, per device.  Two host threads making their
// first call on one device at the same time may both look it up; they store
// the same value, and the atomic makes that race well defined.
std::atomic<void *> g_scratch_ptr[kMaxDevices];

// Once per device, with that device current: look up where the array lives.
// In host code the array's name is only a host-side stand-in, so its device
// address has to come from the runtime.
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NFQ_ERR_CUDA;
  void *ptr = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return NFQ_ERR_CUDA;
    g_scratch_ptr[dev].store(ptr, std::memory_order_relaxed);
  }
  *out = ptr;
  return NFQ_OK;
}

}  // namespace

extern "C" int nfq_lm_head_fp8_argmax_noalloc(const nfq_quant_act *a, const uint8_t *w,
                                              const float *w_scales, int V, int S,
                                              int32_t *tokens_out, float *max_logit_out,
                                              int32_t *shard_idx_out, float *shard_val_out,
                                              void *stream) {
  // every argument is checked before the shared array is touched, so a
  // rejected call cannot disturb another call in flight
  const int chk = nfq::lm_head_check_args(a, w, w_scales, V, S, tokens_out, max_logit_out,
                                          shard_idx_out, shard_val_out);
  if (chk != NFQ_OK) return chk;
  if (a->tokens == 0) return NFQ_OK;
  const int dv = nfq::current_device_supported();
  if (dv != NFQ_OK) return dv;
  const size_t need = nfq_lm_head_workspace_bytes(a->tokens, S);   // S <= 64: fits the array
  void *scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != NFQ_OK) return st;
  // the keys and the counter must start at zero; the array keeps whatever the
  // previous call left, so clear the part this call uses (a memset, no allocation)
  const int z = nfq_lm_head_workspace_init(scratch, need, stream);
  if (z != NFQ_OK) return z;
  return nfq_lm_head_fp8_argmax(a, w, w_scales, V, S, tokens_out, max_logit_out, shard_idx_out,
                                shard_val_out, scratch, need, stream);
}
