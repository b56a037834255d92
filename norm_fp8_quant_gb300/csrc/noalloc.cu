// nfq_lm_head_fp8_argmax_noalloc: the LM head + argmax without a caller
// workspace.  Its scratch (the per-shard argmax keys and the CTA counter) is a
// fixed array in this library's device memory, so the call allocates nothing.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/nfq.h"

namespace {

// Largest workspace any valid call needs: 64 shards x 256 keys x 8 bytes plus
// the 16-byte counter block (128 KiB + 16 B).  Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 64u * 256u * 8u + 16u;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];   // device address of the array, per device

// Once per device, with that device current: look up where the array lives.
// In host code the array's name is only a host-side stand-in, so its device
// address has to come from the runtime.
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NFQ_ERR_CUDA;
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return NFQ_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return NFQ_OK;
}

}  // namespace

extern "C" int nfq_lm_head_fp8_argmax_noalloc(const nfq_quant_act *a, const uint8_t *w,
                                              const float *w_scales, int V, int S,
                                              int32_t *tokens_out, float *max_logit_out,
                                              int32_t *shard_idx_out, float *shard_val_out,
                                              void *stream) {
  if (!a) return NFQ_ERR_NULL;
  const size_t need = nfq_lm_head_workspace_bytes(a->tokens, S);
  if (need == 0) return NFQ_ERR_SHAPE;
  if (need > kNoAllocScratchBytes) return NFQ_ERR_WORKSPACE;
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
