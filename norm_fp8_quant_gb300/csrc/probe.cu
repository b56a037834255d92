// Measurement kernels (not on the hot path): the rate at which tcgen05 FP8
// and block-scaled NVFP4 MMAs run when nothing else competes for the SM (the
// tensor rooflines that the LM heads' tensor-pipe figures are read against),
// the latency of the barrier hand-offs (within a CTA and between the CTAs of
// a pair), the rate at
// which TMEM accumulators can be read into registers, the time of the
// LM head's accumulator hand-off between the MMA thread and the epilogue
// warps through two (or more) TMEM buffers, with no data to stream;
// exhaustive checks of stage 1's division-free FP8 and NVFP4 quotients; and a
// bounded wait that is made to run out.
//
// fp8_mma_rate_kernel<kPair>: every CTA (kPair: every CTA pair, cta_group::2)
// zeroes `stages` pairs of A and B tiles in shared memory, allocates one
// 256-column TMEM accumulator and has one thread issue `iters` K blocks of
// four back-to-back tcgen05.mma kind::f8f6f4 (K = 32 bytes each), K block i
// reading the tiles of stage i % stages, with the shapes the LM head uses:
// M = 128 tokens x N = 256 weight rows per CTA, or M = 256 x N = 256 per pair
// (each CTA holding 128 A rows and 128 B rows).  A commit at the end arrives
// on an mbarrier, waited for with the usual time limit.
#include <cuda_runtime.h>

#include <cstdint>

#include "nfq_internal.h"
#include "ptx.cuh"
#include "stage1_math.cuh"

namespace nfq {

namespace {

constexpr int kProbeErrBit = 4;

template <bool kPair>
__global__ void __launch_bounds__(128, 1)
    fp8_mma_rate_kernel(int iters, int stages, int m, int n, unsigned *err) {
  // A: 128 rows x 128 bytes; B: 256 rows (one CTA) or 128 rows (each CTA of a pair)
  constexpr uint32_t kA = 128 * 128, kB = (kPair ? 128 : 256) * 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = (int)(threadIdx.x / 32), lane = (int)(threadIdx.x % 32);
  const bool issuer = !kPair || cluster_ctarank() == 0;

  uint4 *z = reinterpret_cast<uint4 *>(smem);
  for (uint32_t i = threadIdx.x; i < (uint32_t)stages * (kA + kB) / 16; i += blockDim.x)
    z[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(&tmem_base), 256);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&tmem_base), 256);
      tmem_relinquish();
    }
  }
  // the zeroed tiles are read by the tensor cores (async proxy)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();

  if (warp == 0) {
    if (issuer && lane == 0) {
      // m x n per CTA (pairs: 256 x 256); the tiles hold the largest shape
      const uint32_t idesc = idesc_e4m3_f32(kPair ? 256u : (uint32_t)m, kPair ? 256u : (uint32_t)n);
      int st = 0;
      for (int it = 0; it < iters; ++it) {
        const uint32_t a = smem_u32(smem + (size_t)st * (kA + kB)), b = a + kA;
        st = (st + 1 == stages) ? 0 : st + 1;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if constexpr (kPair)
            mma_f8_pair(tmem_base, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32),
                        idesc, (it | kk) ? 1u : 0u);
          else
            mma_f8(tmem_base, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32),
                   idesc, (it | kk) ? 1u : 0u);
        }
      }
      if constexpr (kPair)
        mma_commit_pair(smem_u32(&done), (uint16_t)3);
      else
        mma_commit(smem_u32(&done));
    }
    __syncwarp();
    // every CTA waits for the last MMAs (a pair's commit arrives on both CTAs)
    if (lane == 0 &&
        !mbar_wait(smem_u32(&done), 0u, (volatile int *)&abort_flag, err, kProbeErrBit)) {
      // gave up: the MMAs still in flight are waited for, again with a limit
      mbar_wait_drain(smem_u32(&done), 0u);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, 256);
    else
      tmem_dealloc(tmem_base, 256);
  }
}

// tmem_ld_rate_kernel: the rate at which 16 warps of one CTA per SM read a
// 128-lane x 512-column TMEM allocation into registers with the LM head
// epilogue's access pattern: warp w reads lane quadrant w % 4, columns
// 64 (w / 4) .. +63 of one of two 256-column accumulators (alternating), as
// four 32x32b.x16 loads, waiting for each (kBatched: for all four at once).
__device__ unsigned g_tmem_probe_sink;   // bumped only by an (unexpected) checksum match

template <bool kBatched>
__global__ void __launch_bounds__(512, 1) tmem_ld_rate_kernel(int iters) {
  __shared__ uint32_t tmem_base;
  const int warp = (int)(threadIdx.x / 32);
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t t0 = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(64 * (warp >> 2));
  uint32_t x = 0;
  for (int it = 0; it < iters; ++it) {
    const uint32_t ta = t0 + (uint32_t)(it & 1) * 256u;
    if constexpr (kBatched) {
      uint32_t r0[16], r1[16], r2[16], r3[16];
      tmem_ld16(ta, r0);
      tmem_ld16(ta + 16, r1);
      tmem_ld16(ta + 32, r2);
      tmem_ld16(ta + 48, r3);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) x ^= r0[j] ^ r1[j] ^ r2[j] ^ r3[j];
    } else {
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t r[16];
        tmem_ld16(ta + (uint32_t)c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) x ^= r[j];
      }
    }
  }
  if (x == 0x9E3779B9u) atomicAdd(&g_tmem_probe_sink, 1u);   // keeps the loads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem_base, 512);
}

// mma_with_readers_kernel: fp8_mma_rate_kernel's issue loop (one CTA, one
// operand set, accumulator in TMEM columns 0..255) while 16 other warps read
// TMEM columns 256..511 with the LM head epilogue's pattern, as long as the
// MMAs run: the MMA rate the LM head's promotion leaves.  The readers stop
// when the issuing thread's last MMA has completed (a flag in shared memory),
// or after a fixed number of passes.
__global__ void __launch_bounds__(17 * 32, 1) mma_with_readers_kernel(int iters, unsigned *err) {
  constexpr uint32_t kA = 128 * 128, kB = 256 * 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ volatile int finished;
  const int warp = (int)(threadIdx.x / 32), lane = (int)(threadIdx.x % 32);
  uint4 *z = reinterpret_cast<uint4 *>(smem);
  for (uint32_t i = threadIdx.x; i < (kA + kB) / 16; i += blockDim.x)
    z[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    abort_flag = 0;
    finished = 0;
    fence_mbarrier_init();
  }
  if (warp == 16) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 16) {
    if (lane == 0) {
      const uint32_t a = smem_u32(smem), b = smem_u32(smem + kA);
      const uint32_t idesc = idesc_e4m3_f32(128, 256);
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f8(tmem_base, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32),
                 idesc, (it | kk) ? 1u : 0u);
      }
      mma_commit(smem_u32(&done));
      if (!mbar_wait(smem_u32(&done), 0u, (volatile int *)&abort_flag, err, kProbeErrBit))
        mbar_wait_drain(smem_u32(&done), 0u);
      finished = 1;
    }
    __syncwarp();
  } else {
    const uint32_t ta = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + 256u +
                        (uint32_t)(64 * (warp >> 2));
    uint32_t x = 0;
    for (int pass = 0; pass < (1 << 22); ++pass) {
      if (__shfl_sync(0xffffffffu, finished, 0)) break;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t r[16];
        tmem_ld16(ta + (uint32_t)c, r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) x ^= r[j];
      }
    }
    if (x == 0x9E3779B9u) atomicAdd(&g_tmem_probe_sink, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 16) tmem_dealloc(tmem_base, 512);
}

// handshake_kernel<kPair, NB>: the LM head's accumulator hand-off without
// any data to stream.  One thread (of the even CTA) issues, per K block, NB / 2
// groups of four MMAs (M = 128 per CTA, 256 per pair, x N = 512 / NB x K = 32,
// from one zeroed operand set), each group into its own N-column TMEM buffer
// (NB buffers fill the 512 columns), and commits each group to that buffer's
// full barrier.  16 epilogue warps per CTA wait for each buffer, read their
// N / 4 columns of it 16 at a time with a wait after each (mode 1; mode 0:
// no reads) and arrive on its empty barrier (CTA pairs: 16 local and 16
// remote arrivals on the even CTA's barrier), which the issuing thread waits
// for before it reuses the buffer.  mode 2: no epilogue; the issuing thread
// waits for each group to complete before it issues the next (the MMAs'
// issue-to-completion latency).  mode 3 (NB = 4): each 128-column buffer has
// its own half of the epilogue: warps 4h + 2j + q' with column group
// g = warp / 4, half h = g / 2, read 64 columns of the buffers of group h only
// (8 warps per buffer, 16 on CTA pairs), so the two halves of a K block are
// handed off independently.
template <bool kPair, int NB>
__global__ void __launch_bounds__(17 * 32, 1) handshake_kernel(int iters, int mode, unsigned *err) {
  constexpr int N = 512 / NB, GROUPS = NB / 2, C = N / 4;
  static_assert(!kPair || NB == 2 || NB == 4, "CTA pairs: two or four buffers");
  constexpr uint32_t kA = 128 * 128, kB = (kPair ? 128 : 256) * 128;
  constexpr int kRowsPerGroup = kPair ? N / 2 : N;   // B rows per CTA per group
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  __shared__ uint64_t full[NB], empty[NB], fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = (int)(threadIdx.x / 32), lane = (int)(threadIdx.x % 32);
  const bool even = !kPair || cluster_ctarank() == 0;

  uint4 *z = reinterpret_cast<uint4 *>(smem);
  for (uint32_t i = threadIdx.x; i < (kA + kB) / 16; i += blockDim.x)
    z[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    const uint32_t readers = mode == 3 ? 8u : 16u;
    for (int b = 0; b < NB; ++b) {
      mbar_init(smem_u32(&full[b]), 1);
      mbar_init(smem_u32(&empty[b]), kPair ? 2u * readers : readers);
    }
    mbar_init(smem_u32(&fin), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 16) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(&tmem_base), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&tmem_base), 512);
      tmem_relinquish();
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  volatile int *ab = &abort_flag;
  const int total = iters * GROUPS;

  if (warp == 16) {
    if (lane == 0 && even) {
      const uint64_t a_desc = sw128_kmajor_desc(smem_u32(smem));
      const uint64_t b_desc = sw128_kmajor_desc(smem_u32(smem + kA));
      const uint32_t idesc = idesc_e4m3_f32(kPair ? 256 : 128, (uint32_t)N);
      for (int i = 0; i < total; ++i) {
        const int buf = i % NB, use = i / NB, grp = i % GROUPS;
        if (mode != 2) {
          if (!mbar_wait(smem_u32(&empty[buf]), (uint32_t)(use & 1) ^ 1u, ab, err, kProbeErrBit))
            break;
          tc_fence_after();
        }
        // group grp multiplies this CTA's B rows grp * kRowsPerGroup .. (128 bytes each)
        const uint64_t bd = b_desc + (uint64_t)((grp * kRowsPerGroup * 128) >> 4);
        const uint32_t d = tmem_base + (uint32_t)(buf * N);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if constexpr (kPair)
            mma_f8_pair(d, a_desc + 2u * kk, bd + 2u * kk, idesc, kk ? 1u : 0u);
          else
            mma_f8(d, a_desc + 2u * kk, bd + 2u * kk, idesc, kk ? 1u : 0u);
        }
        if (mode == 2) {
          if constexpr (kPair)
            mma_commit_pair(smem_u32(&full[buf]), (uint16_t)1);
          else
            mma_commit(smem_u32(&full[buf]));
          if (!mbar_wait(smem_u32(&full[buf]), (uint32_t)(use & 1), ab, err, kProbeErrBit)) break;
        } else {
          if constexpr (kPair)
            mma_commit_pair(smem_u32(&full[buf]), (uint16_t)3);
          else
            mma_commit(smem_u32(&full[buf]));
        }
      }
      // every MMA issued has completed before the TMEM is given back
      if constexpr (kPair)
        mma_commit_pair(smem_u32(&fin), (uint16_t)1);
      else
        mma_commit(smem_u32(&fin));
      mbar_wait_drain(smem_u32(&fin), 0u);
    }
    __syncwarp();
  } else if (mode != 2) {
    // mode 3: this warp's half (group) and its 64 columns of that half's buffers
    const int g = warp >> 2;
    const int cols = mode == 3 ? 64 : C;
    const uint32_t t0 = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) +
                        (uint32_t)(mode == 3 ? 64 * (g & 1) : C * g);
    uint32_t x = 0;
    for (int i = 0; i < total; ++i) {
      const int buf = i % NB, use = i / NB;
      if (mode == 3 && (i % GROUPS) != (g >> 1)) continue;
      const bool got = mbar_wait(smem_u32(&full[buf]), (uint32_t)(use & 1), ab, err, kProbeErrBit);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      if (mode == 1 || mode == 3) {
        for (int c = 0; c < cols; c += 16) {
          uint32_t r[16];
          tmem_ld16(t0 + (uint32_t)(buf * N + c), r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) x ^= r[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (even)
          mbar_arrive(smem_u32(&empty[buf]));
        else
          mbar_arrive_remote_cta(smem_u32(&empty[buf]), 0u);
      }
    }
    if (x == 0x9E3779B9u) atomicAdd(&g_tmem_probe_sink, 1u);   // keeps the loads
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  if (warp == 16) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, 512);
    else
      tmem_dealloc(tmem_base, 512);
  }
}

// quotient_check_kernel: block a takes the bf16 pattern a (0 .. +inf) as the
// group maximum amax and checks stage 1's division-free steps against IEEE
// arithmetic: the scale fp8_scale(amax) against RN(amax / 448) bit for bit;
// where quot_rn stands for the division (quot_rn_ok), recip_rn(scale)
// against the IEEE reciprocal bit for bit, and for every bf16 pattern y with
// |y| <= amax, and every NaN, the e4m3 code of quot_rn(y, scale, recip_rn)
// against that of IEEE y / scale.  Differences are counted in count[0]
// (scales), count[1] (reciprocals) and count[2] (codes); the first one seen
// is kept as (a << 16) | y (y = 0 for a scale or reciprocal).
__global__ void __launch_bounds__(256) quotient_check_kernel(unsigned long long *count,
                                                             unsigned *first) {
  const uint32_t a = blockIdx.x;
  const float amax = __uint_as_float(a << 16);
  const float s = fp8_scale(amax);
  const float s_ieee = __fdiv_rn(amax, 448.0f);
  if (threadIdx.x == 0 && __float_as_uint(s) != __float_as_uint(s_ieee)) {
    atomicAdd(&count[0], 1ull);
    atomicCAS(first, 0xFFFFFFFFu, a << 16);
  }
  if (!quot_rn_ok(s_ieee)) return;
  const float r = recip_rn(s);
  if (threadIdx.x == 0 && __float_as_uint(r) != __float_as_uint(__frcp_rn(s_ieee))) {
    atomicAdd(&count[1], 1ull);
    atomicCAS(first, 0xFFFFFFFFu, a << 16);
  }
  for (uint32_t yb = threadIdx.x; yb < 65536u; yb += blockDim.x) {
    const float y = __uint_as_float(yb << 16);
    if (!isnan(y) && !(fabsf(y) <= amax)) continue;
    if (e4m3x2(quot_rn(y, s, r), 0.0f) != e4m3x2(__fdiv_rn(y, s_ieee), 0.0f)) {
      atomicAdd(&count[2], 1ull);
      atomicCAS(first, 0xFFFFFFFFu, (a << 16) | yb);
    }
  }
}

// quotient_check_fp4_kernel: block (a, c) takes the bf16 pattern a (0 .. +inf)
// as the row maximum, g = RN(amax_row / 2688), d = RN(6 g), and the e4m3 code
// c (0 .. 0x7E) as a block scale, eff = RN(value(c) g); it checks stage 1's
// division-free NVFP4 steps against IEEE arithmetic: (c = 0 only) recip_rn(d)
// against the IEEE reciprocal, counted in count[0], and for every bf16 block
// maximum ab <= amax_row the block-scale code e4m3(RN(ab / d)), count[1];
// recip_rn(eff) against the IEEE reciprocal, count[2]; for every bf16 y with
// |y| <= amax_row, and every NaN, the e2m1 code of RN(y / eff), count[3].
// The first difference seen is kept as (c << 32) | (a << 16) | y.
__global__ void __launch_bounds__(256) quotient_check_fp4_kernel(unsigned long long *count,
                                                                 unsigned long long *first) {
  const uint32_t a = blockIdx.x, c = blockIdx.y;
  const float amax_row = __uint_as_float(a << 16);
  const float g = __fdiv_rn(amax_row, 2688.0f);
  if (g == 0.0f) return;
  const float d = __fmul_rn(6.0f, g);
  const unsigned long long tag = ((unsigned long long)c << 32) | ((unsigned long long)a << 16);
  if (c == 0 && quot_rn_ok(d)) {
    const float rd = recip_rn(d);
    if (threadIdx.x == 0 && __float_as_uint(rd) != __float_as_uint(__frcp_rn(d))) {
      atomicAdd(&count[0], 1ull);
      atomicCAS(first, ~0ull, tag);
    }
    for (uint32_t ab_bits = threadIdx.x; ab_bits <= 0x7F80u; ab_bits += blockDim.x) {
      const float ab = __uint_as_float(ab_bits << 16);
      if (!(ab <= amax_row)) continue;
      if ((e4m3x2(quot_rn(ab, d, rd), 0.0f) & 0xFFu) != (e4m3x2(__fdiv_rn(ab, d), 0.0f) & 0xFFu)) {
        atomicAdd(&count[1], 1ull);
        atomicCAS(first, ~0ull, tag | ab_bits);
      }
    }
  }
  const float eff = __fmul_rn(e4m3_value(c), g);
  if (!quot_rn_ok(eff)) return;
  const float re = recip_rn(eff);
  if (threadIdx.x == 0 && __float_as_uint(re) != __float_as_uint(__frcp_rn(eff))) {
    atomicAdd(&count[2], 1ull);
    atomicCAS(first, ~0ull, tag);
  }
  for (uint32_t yb = threadIdx.x; yb < 65536u; yb += blockDim.x) {
    const float y = __uint_as_float(yb << 16);
    if (!isnan(y) && !(fabsf(y) <= amax_row)) continue;
    if (e2m1x2(quot_rn(y, eff, re), 0.0f) != e2m1x2(__fdiv_rn(y, eff), 0.0f)) {
      atomicAdd(&count[3], 1ull);
      atomicCAS(first, ~0ull, tag | yb);
    }
  }
}

// wait_timeout_kernel: one thread waits, with the bounded wait every kernel
// of the path uses, on an mbarrier that nothing arrives on.  The wait gives
// up after its time limit, sets the device error word's probe bit and the
// kernel returns: the failure a stuck peer would cause, made on purpose
// without faulting or hanging anything.
__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned *err) {
  __shared__ uint64_t never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&never), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0)
    (void)mbar_wait(smem_u32(&never), 0u, (volatile int *)&abort_flag, err, kProbeErrBit);
  __syncwarp();
}

}  // namespace

cudaError_t launch_probe_mma_with_readers(int ctas, int iters, unsigned *err,
                                          cudaStream_t stream) {
  const size_t smem = 120u * 1024u;
  cudaError_t e = cudaFuncSetAttribute(mma_with_readers_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  mma_with_readers_kernel<<<(unsigned)ctas, 17 * 32, smem, stream>>>(iters, err);
  return cudaGetLastError();
}

cudaError_t launch_probe_tmem_ld(int batched, int ctas, int iters, cudaStream_t stream) {
  // the whole TMEM (512 columns) and most of shared memory: one CTA per SM
  const size_t smem = 120u * 1024u;
  auto kern = batched ? tmem_ld_rate_kernel<true> : tmem_ld_rate_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)ctas, 512, smem, stream>>>(iters);
  return cudaGetLastError();
}

// nvfp4_mma_rate_kernel<kPair>: as fp8_mma_rate_kernel with the LM head's
// block-scaled NVFP4 MMA (tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X,
// K = 64 e2m1 elements each, four per 256-element K step) on one operand set:
// M = 128 x N = 256 per CTA or M = 256 x N = 256 per pair.  The block scales
// (e4m3 1.0) sit in TMEM columns 256..303 in the LM head's layout.
__device__ __forceinline__ void probe_mma_fp4_pair(uint32_t d, uint64_t a, uint64_t b,
                                                   uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                                   uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

template <bool kPair>
__global__ void __launch_bounds__(128, 1) nvfp4_mma_rate_kernel(int iters, unsigned *err) {
  constexpr uint32_t kA = 128 * 128, kB = (kPair ? 128 : 256) * 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = (int)(threadIdx.x / 32), lane = (int)(threadIdx.x % 32);
  const bool issuer = !kPair || cluster_ctarank() == 0;

  uint4 *z = reinterpret_cast<uint4 *>(smem);
  for (uint32_t i = threadIdx.x; i < (kA + kB) / 16; i += blockDim.x)
    z[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(&tmem_base), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&tmem_base), 512);
      tmem_relinquish();
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  {
    // every warp its own lane quadrant: 48 scale columns of e4m3 1.0
    uint32_t one[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) one[j] = 0x38383838u;
    const uint32_t col = tmem_base + ((uint32_t)(32 * warp) << 16) + 256u;
    tmem_st32(col, one);
    tmem_st16(col + 32u, *reinterpret_cast<const uint32_t(*)[16]>(one));
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();

  if (warp == 0) {
    if (issuer && lane == 0) {
      const uint32_t idesc = idesc_nvfp4(kPair ? 256 : 128, 256);
      const uint64_t ad = sw128_kmajor_desc(smem_u32(smem)), bd = sw128_kmajor_desc(smem_u32(smem + kA));
      const uint32_t sf = tmem_base + 256u;
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if constexpr (kPair)
            probe_mma_fp4_pair(tmem_base, ad + 2u * kk, bd + 2u * kk, idesc, sf + 4u * kk,
                               sf + 16u + 8u * kk, (it | kk) ? 1u : 0u);
          else
            mma_fp4_block16(tmem_base, ad + 2u * kk, bd + 2u * kk, idesc, sf + 4u * kk,
                            sf + 16u + 8u * kk, (it | kk) ? 1u : 0u);
        }
      }
      if constexpr (kPair)
        mma_commit_pair(smem_u32(&done), (uint16_t)3);
      else
        mma_commit(smem_u32(&done));
    }
    __syncwarp();
    if (lane == 0 &&
        !mbar_wait(smem_u32(&done), 0u, (volatile int *)&abort_flag, err, kProbeErrBit))
      mbar_wait_drain(smem_u32(&done), 0u);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, 512);
    else
      tmem_dealloc(tmem_base, 512);
  }
}

// handoff_kernel<MODE>: the latency of the barrier hand-offs the LM heads'
// pipelines are built from, as a ping-pong of `iters` round trips between two
// threads, each waiting (bounded) on its own mbarrier for the other's signal:
//   0: two warps of one CTA, local arrivals;
//   1: the two CTAs of a cluster, remote arrivals at CTA scope (the form the
//      CTA-pair kernels use);
//   2: the same with release at cluster scope;
//   3: the same by st.async of one word, counted (complete_tx) on the peer's
//      barrier.
template <int MODE>
__global__ void __launch_bounds__(64, 1) handoff_kernel(int iters, unsigned *err) {
  constexpr bool kPair = MODE != 0;
  __shared__ uint64_t bar[2];   // MODE 0: one per thread; pairs: bar[0] in each CTA
  __shared__ int abort_flag;
  __shared__ float box;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int warp = (int)(threadIdx.x / 32), lane = (int)(threadIdx.x % 32);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar[0]), 1);
    mbar_init(smem_u32(&bar[1]), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();
  const bool ping = lane == 0 && (kPair ? (rank == 0 && warp == 0) : warp == 0);
  const bool pong = lane == 0 && (kPair ? (rank == 1 && warp == 0) : warp == 1);
  if (ping || pong) {
    // own barrier to wait on, and where the signal goes
    const uint32_t mine = smem_u32(&bar[kPair ? 0 : (ping ? 0 : 1)]);
    const uint32_t theirs = smem_u32(&bar[kPair ? 0 : (ping ? 1 : 0)]);
    const uint32_t peer = rank ^ 1u;
    for (int i = 0; i < iters; ++i) {
      const bool first = ping;   // ping signals, then waits; pong waits, then signals
      for (int step = 0; step < 2; ++step) {
        if ((step == 0) == first) {
          if constexpr (MODE == 0) mbar_arrive(theirs);
          else if constexpr (MODE == 1) mbar_arrive_remote_cta(theirs, peer);
          else if constexpr (MODE == 2) mbar_arrive_remote(theirs, peer);
          else st_async_remote_f32(smem_u32(&box), theirs, peer, 1.0f);
        } else {
          if constexpr (MODE == 3) mbar_arrive_expect_tx(mine, 4u);
          if (!mbar_wait(mine, (uint32_t)(i & 1), (volatile int *)&abort_flag, err, kProbeErrBit)) {
            i = iters;
            break;
          }
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();   // no CTA leaves while its peer may signal it
}

// `stages` sets of tiles (1..4): each K block reads fresh operands from shared
// memory, as the LM head's pipeline does, instead of the same tiles again.
cudaError_t launch_probe_fp8_mma_stages(int pair, int ctas, int iters, int stages,
                                        unsigned *err, cudaStream_t stream) {
  if (stages < 1 || stages > 4) return cudaErrorInvalidValue;
  // the tiles need at most 4 x 48 KB; at least 120 KB keeps one CTA per SM
  const size_t tiles = 1024 + (size_t)stages * (128 * 128 + (pair ? 128 : 256) * 128);
  const size_t smem = tiles > 120u * 1024u ? tiles : 120u * 1024u;
  auto kern = pair ? fp8_mma_rate_kernel<true> : fp8_mma_rate_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pair ? 2 * ctas : ctas));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, iters, stages, 128, 256, err);
}

// One operand set, one CTA per SM, MMAs of M = m x N = n (cta_group::1):
// m 64 or 128, n a multiple of 8 (m = 64) or 16 (m = 128) in 16..256.
cudaError_t launch_probe_fp8_mma_shape(int m, int n, int ctas, int iters, unsigned *err,
                                       cudaStream_t stream) {
  if (!((m == 64 && n % 8 == 0) || (m == 128 && n % 16 == 0)) || n < 16 || n > 256)
    return cudaErrorInvalidValue;
  const size_t smem = 120u * 1024u;
  auto kern = fp8_mma_rate_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)ctas, 128, smem, stream>>>(iters, 1, m, n, err);
  return cudaGetLastError();
}

cudaError_t launch_probe_fp8_mma(int pair, int ctas, int iters, unsigned *err,
                                 cudaStream_t stream) {
  return launch_probe_fp8_mma_stages(pair, ctas, iters, 1, err, stream);
}

cudaError_t launch_probe_handoff(int mode, int iters, unsigned *err, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(mode == 0 ? 1u : 2u);
  cfg.blockDim = dim3(64);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = mode == 0 ? 1 : 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (mode) {
    case 0: return cudaLaunchKernelEx(&cfg, handoff_kernel<0>, iters, err);
    case 1: return cudaLaunchKernelEx(&cfg, handoff_kernel<1>, iters, err);
    case 2: return cudaLaunchKernelEx(&cfg, handoff_kernel<2>, iters, err);
    case 3: return cudaLaunchKernelEx(&cfg, handoff_kernel<3>, iters, err);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_probe_nvfp4_mma(int pair, int ctas, int iters, unsigned *err,
                                   cudaStream_t stream) {
  const size_t smem = 120u * 1024u;   // the tiles need 48 KB; 120 KB keeps one CTA per SM
  auto kern = pair ? nvfp4_mma_rate_kernel<true> : nvfp4_mma_rate_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pair ? 2 * ctas : ctas));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, iters, err);
}

// The accumulator hand-off probe: `ctas` CTAs (pair: `ctas` CTA pairs) with
// `buffers` TMEM buffers (2, 4 or 8; pairs: 2), `iters` K blocks each.
cudaError_t launch_probe_handshake(int pair, int buffers, int mode, int ctas, int iters,
                                   unsigned *err, cudaStream_t stream) {
  void (*kern)(int, int, unsigned *) = nullptr;
  if (pair && buffers == 2) kern = handshake_kernel<true, 2>;
  else if (pair && buffers == 4) kern = handshake_kernel<true, 4>;
  else if (!pair && buffers == 2) kern = handshake_kernel<false, 2>;
  else if (!pair && buffers == 4) kern = handshake_kernel<false, 4>;
  else if (!pair && buffers == 8) kern = handshake_kernel<false, 8>;
  if (!kern || mode < 0 || mode > 3 || (mode == 3 && buffers != 4)) return cudaErrorInvalidValue;
  // 48 KB of tiles; 120 KB keeps one CTA per SM
  const size_t smem = 120u * 1024u;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pair ? 2 * ctas : ctas));
  cfg.blockDim = dim3(17 * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, iters, mode, err);
}

// Every bf16 group maximum from 0 to +inf (0x0000 .. 0x7F80), one block each;
// count holds three counters.
cudaError_t launch_check_fp8_quotient(unsigned long long *count, unsigned *first,
                                      cudaStream_t stream) {
  quotient_check_kernel<<<0x7F81u, 256, 0, stream>>>(count, first);
  return cudaGetLastError();
}

// Every bf16 row maximum from 0 to +inf times every finite e4m3 block scale;
// count holds four counters.
cudaError_t launch_check_fp4_quotient(unsigned long long *count, unsigned long long *first,
                                      cudaStream_t stream) {
  quotient_check_fp4_kernel<<<dim3(0x7F81u, 0x7Fu), 256, 0, stream>>>(count, first);
  return cudaGetLastError();
}

cudaError_t launch_probe_wait_timeout(unsigned *err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace nfq
