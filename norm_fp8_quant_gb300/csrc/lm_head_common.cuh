// Pieces shared by the LM-head kernels (FP8 and NVFP4): the packed argmax key,
// the last-CTA finalisation, the block schedule and the host-side launch and
// tensor-map helpers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "nfq_internal.h"

namespace nfq {

namespace {

constexpr int kErrBitStage2 = 2;
constexpr int kKeyStride = kArgmaxKeysPerShard;   // keys per shard in the workspace
constexpr uint32_t kWTileBytes = 128 * 128;

// Ordered 64-bit key: larger value first, then lower index; -0 counts as +0.
__device__ __forceinline__ unsigned long long pack_key(float v, uint32_t idx) {
  uint32_t u = (v == 0.0f) ? 0u : __float_as_uint(v);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

__device__ __forceinline__ float key_value(unsigned long long key) {
  const uint32_t ord = (uint32_t)(key >> 32);
  const uint32_t u = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(u);
}

__device__ __forceinline__ int32_t key_index(unsigned long long key) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

// After every CTA has merged its keys: the last CTA to finish turns the keys
// into outputs and returns the workspace to zero.  All threads call this.
__device__ __forceinline__ void finish_launch(const Stage2Params &p, int *last_flag) {
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.counter, 1u);
    *last_flag = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*last_flag) {
    __threadfence();
    for (int n = (int)threadIdx.x; n < p.T; n += (int)blockDim.x) {
      unsigned long long best = 0ull;
      for (int s = 0; s < p.S; ++s) {
        const unsigned long long k = atomicExch(&p.keys[(size_t)s * kKeyStride + n], 0ull);
        if (p.shard_idx_out) p.shard_idx_out[(size_t)s * p.T_total + p.tok0 + n] = key_index(k);
        if (p.shard_val_out) p.shard_val_out[(size_t)s * p.T_total + p.tok0 + n] = key_value(k);
        if (k > best) best = k;
      }
      p.tokens_out[n] = key_index(best);
      if (p.max_logit_out) p.max_logit_out[n] = key_value(best);
    }
    if (threadIdx.x == 0) {
      *p.counter = 0u;
      if (p.s1.ready) *p.s1.ready = 0u;     // the fused step's row counter
    }
  }
}

// Tile ti of a CTA's block range [b_begin, b_end): pairs of 128-row blocks.
// An odd range starts with its single block, so that the one tile whose MMAs
// carry half the weight bytes runs while every CTA is still sharing HBM, not
// at the end where it would set the finishing time.
__device__ __forceinline__ void small_tile(int b_begin, int b_end, int ti, int &blk0, int &nb) {
  const bool odd = ((b_end - b_begin) & 1) != 0;
  if (odd && ti == 0) {
    blk0 = b_begin;
    nb = 1;
  } else {
    blk0 = b_begin + 2 * ti - (odd ? 1 : 0);
    nb = 2;
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Launch with programmatic stream serialization: the kernel's set-up may
// overlap the previous kernel on the stream; it waits (griddepcontrol) before
// touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// 2-D uint8 map over [rows][cols] (cols contiguous), box 128 x box_rows, 128B swizzle.
inline bool encode_u8_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 map over [rows][cols] with an unswizzled box of box_cols x box_rows.
inline bool encode_u8_map_plain(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                                uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

}  // namespace nfq
