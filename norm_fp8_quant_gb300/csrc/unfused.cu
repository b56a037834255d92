// The unfused reference arm: the MTP draft tail as separate kernels, the way
// it runs without the two fusions.
//
// "[Spec Decode][Perf] Fuse the MTP trailing all-reduce; local-argmax draft
// tokens", intro and Accuracy: without the fusion the trailing all-reduce is a
// separate BF16 collective ahead of the final RMSNorm, and the greedy draft
// tokens come from the argmax over the gathered full-vocab logits (64 x 151k
// x 2 bytes per draft step at c=64, Benchmarks).  On one GPU the collective is
// the sum of the k partials, rounded to BF16:
//   unfused_reduce      s = bf16(p_0 + ... + p_{k-1})        (fp32 sum, one rounding)
//   unfused_add_rmsnorm hidden = bf16((s + residual) * rsqrt(mean(.^2) + eps) * w)
//   unfused_quant       per 128 group: scale = amax / 448, codes = e4m3(hidden / scale)
//   (LM head writing BF16 logits: lm_head.cu, kLogits form)
//   unfused_argmax      token = lowest index of the maximum BF16 logit
// Each is a plain HBM-streaming kernel; together they measure what the fused
// path saves in bytes, launches and latency.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "nfq_internal.h"

namespace nfq {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// s = bf16(sum of k partials), one 16-byte vector per thread and step.
__global__ void __launch_bounds__(256) unfused_reduce_kernel(const UnfusedReduceParams p) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n_vec;
       i += (size_t)gridDim.x * blockDim.x) {
    float acc[8];
    bf16x8_to_f32(reinterpret_cast<const uint4 *>(p.partials[0])[i], acc);
    for (int j = 1; j < p.k; ++j) {
      float f[8];
      bf16x8_to_f32(reinterpret_cast<const uint4 *>(p.partials[j])[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
    }
    reinterpret_cast<uint4 *>(p.out)[i] =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

constexpr int kNormThreads = 256;
constexpr int kNormMaxVec = 8;     // vectors per thread: H <= 256 * 8 * 8 = 16384

// One CTA per row: v = x + residual (fp32), RMSNorm, BF16 hidden.
__global__ void __launch_bounds__(kNormThreads) unfused_add_rmsnorm_kernel(
    const uint4 *__restrict__ x, const uint4 *__restrict__ residual,
    const uint4 *__restrict__ norm_w, float eps, int H, uint4 *__restrict__ hidden) {
  __shared__ float red[kNormThreads / 32];
  const int nv = H / 8;
  const size_t row = (size_t)blockIdx.x * (size_t)nv;
  float v[kNormMaxVec][8];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int j = (int)threadIdx.x + i * kNormThreads;
    if (j < nv) {
      float a[8], b[8];
      bf16x8_to_f32(x[row + j], a);
      bf16x8_to_f32(residual[row + j], b);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[i][e] = __fadd_rn(a[e], b[e]);
        ss = fmaf(v[i][e], v[i][e], ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float rr = __frsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), eps));
#pragma unroll
  for (int i = 0; i < kNormMaxVec; ++i) {
    const int j = (int)threadIdx.x + i * kNormThreads;
    if (j < nv) {
      float w[8];
      bf16x8_to_f32(norm_w[j], w);
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2)
        o[e / 2] = pack_bf16x2(__fmul_rn(__fmul_rn(v[i][e], rr), w[e]),
                               __fmul_rn(__fmul_rn(v[i][e + 1], rr), w[e + 1]));
      hidden[row + j] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Group quantisation: 16 lanes per 128-channel group, one 16-byte vector each.
__global__ void __launch_bounds__(256) unfused_quant_kernel(const uint4 *__restrict__ hidden,
                                                            size_t n_groups,
                                                            uint2 *__restrict__ codes,
                                                            float *__restrict__ scales) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t grp = t / 16;
  const bool ok = grp < n_groups;
  float y[8];
  if (ok) {
    bf16x8_to_f32(hidden[t], y);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.0f;
  }
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[e]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = __fdiv_rn(amax, 448.0f);
  uint32_t q[2] = {0u, 0u};
  if (scale != 0.0f) {
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      uint16_t pr;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
          : "=h"(pr)
          : "f"(__fdiv_rn(y[e + 1], scale)), "f"(__fdiv_rn(y[e], scale)));
      q[e / 4] |= (uint32_t)pr << ((e % 4) * 8);
    }
  }
  if (ok) {
    codes[t] = make_uint2(q[0], q[1]);
    if ((t & 15) == 0) scales[grp] = scale;
  }
}

constexpr int kArgmaxThreads = 1024;

__device__ __forceinline__ void take(float x, int v, float &best, int &bi) {
  if (bi == 0x7FFFFFFF || x > best) {          // ascending within a thread: first wins
    best = x;
    bi = v;
  }
}

// One CTA per token row: the lowest index of the maximum BF16 logit (-0 == +0).
// Rows whose length is a multiple of 8 are read 16 bytes at a time, four loads
// in flight per thread.
__global__ void __launch_bounds__(kArgmaxThreads) unfused_argmax_kernel(
    const uint16_t *__restrict__ logits, int V, int32_t *__restrict__ tokens) {
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  const uint16_t *row = logits + (size_t)blockIdx.x * (size_t)V;
  float best = -INFINITY;
  int bi = 0x7FFFFFFF;
  if ((V & 7) == 0) {
    const uint4 *rv = reinterpret_cast<const uint4 *>(row);
    const int nv = V / 8;
    for (int c0 = (int)threadIdx.x; c0 < nv; c0 += 4 * kArgmaxThreads) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * kArgmaxThreads;
        q[u] = c < nv ? __ldg(rv + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * kArgmaxThreads;
        if (c < nv) {
          float f[8];
          bf16x8_to_f32(q[u], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) take(f[e], 8 * c + e, best, bi);
        }
      }
    }
  } else {
    for (int v = (int)threadIdx.x; v < V; v += kArgmaxThreads)
      take(__uint_as_float((uint32_t)row[v] << 16), v, best, bi);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = best;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = sv[0];
    int i = si[0];
    for (int w = 1; w < kArgmaxThreads / 32; ++w)
      if (sv[w] > b || (sv[w] == b && si[w] < i)) {
        b = sv[w];
        i = si[w];
      }
    tokens[blockIdx.x] = i;
  }
}

}  // namespace

cudaError_t launch_unfused_reduce(const UnfusedReduceParams &p, int num_sms,
                                  cudaStream_t stream) {
  if (p.k < 1 || p.k > kMaxPartials || p.n_vec == 0) return cudaErrorInvalidConfiguration;
  size_t blocks = (p.n_vec + 255) / 256;
  const size_t cap = (size_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  unfused_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_unfused_add_rmsnorm(const void *x, const void *residual, const void *norm_w,
                                       float eps, int T, int H, void *hidden,
                                       cudaStream_t stream) {
  if (T < 1 || H % 8 != 0 || H / 8 > kNormThreads * kNormMaxVec)
    return cudaErrorInvalidConfiguration;
  unfused_add_rmsnorm_kernel<<<(unsigned)T, kNormThreads, 0, stream>>>(
      static_cast<const uint4 *>(x), static_cast<const uint4 *>(residual),
      static_cast<const uint4 *>(norm_w), eps, H, static_cast<uint4 *>(hidden));
  return cudaGetLastError();
}

cudaError_t launch_unfused_quant(const void *hidden, int T, int H, uint8_t *codes,
                                 float *scales, cudaStream_t stream) {
  const size_t n_groups = (size_t)T * (size_t)(H / 128);
  if (n_groups == 0 || H % 128 != 0) return cudaErrorInvalidConfiguration;
  const size_t threads = n_groups * 16;
  unfused_quant_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(
      static_cast<const uint4 *>(hidden), n_groups, reinterpret_cast<uint2 *>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_unfused_argmax(const void *logits, int T, int V, int32_t *tokens,
                                  cudaStream_t stream) {
  if (T < 1 || V < 1) return cudaErrorInvalidConfiguration;
  unfused_argmax_kernel<<<(unsigned)T, kArgmaxThreads, 0, stream>>>(
      static_cast<const uint16_t *>(logits), V, tokens);
  return cudaGetLastError();
}

}  // namespace nfq
