// Stage 2: shared LM head on the prequantised FP8 activation with a fused,
// vocab-sharded greedy argmax.  Logits never leave the chip.
//
// "[Quant][MTP] Reuse packed FP8 logits inputs", Dependencies: the LM-head GEMM
// consumes the packed activation as already quantised.  "[Spec Decode][Perf]
// Fuse the MTP trailing all-reduce; local-argmax draft tokens", intro: greedy
// draft tokens come from a vocab-parallel local argmax instead of gathering the
// full-vocab logits; Accuracy: ties at shard boundaries are decided by the
// local-argmax rule (here: the lowest global vocab index).
//
// Formulation (swap-AB): the weight is the MMA's M operand (128 vocab rows =
// one 128x128 scale block row) and the tokens are N.  Per 128-wide K block:
//   P[v][n] = sum_{k in block} qw[v][k] * qa[n][k]     tcgen05.mma kind::f8f6f4,
//                                                      fp32 accumulator in TMEM
//   acc[v][n] += P[v][n] * (sw[v/128][kb] * sa[n][kb]) fp32, in registers
// The scales are arbitrary fp32 values (amax / 448), which the hardware block
// scaling (power-of-two scale factors) cannot express, hence the per-block
// promotion out of TMEM.
//
// Warp roles (one CTA per SM, persistent over contiguous vocab tiles):
//   warps 0 .. 4*EPI-1   epilogue: TMEM -> registers, promotion, argmax
//   warp  4*EPI          TMA producer: weight tile 128x128 + activation tile
//                        Nx128 per K block into a ring of swizzled stages
//   warp  4*EPI+1        TMEM allocator and MMA issuer (one thread)
// TMEM holds NBUF accumulators of N columns so the MMA of the next K block
// overlaps the promotion of the previous one.  After the last K block of a
// tile each warp reduces its 32 rows per token to (max, lowest row) per shard
// and merges it into a packed 64-bit key with atomicMax; the last CTA to
// finish turns the keys into tokens and resets the workspace.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "nfq_internal.h"
#include "ptx.cuh"

namespace nfq {

namespace {

constexpr int kErrBitStage2 = 2;
constexpr int kMaxStages = 16;
constexpr int kKeyStride = 256;   // keys per shard in the workspace
constexpr uint32_t kWTileBytes = 128 * 128;

struct Stage2Smem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[4];
  uint64_t tempty[4];
  uint32_t tmem_base;
  int abort;
  int last;
};

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

template <int NCOL, int EPI>
__global__ void __launch_bounds__(128 * EPI + 64, 1)
    lm_head_argmax_kernel(const __grid_constant__ CUtensorMap tmap_w,
                          const __grid_constant__ CUtensorMap tmap_a, const Stage2Params p,
                          int nstage) {
  constexpr int N = NCOL * EPI;                  // MMA N (token columns)
  constexpr int NBUF = (512 / N) < 4 ? (512 / N) : 4;
  constexpr int TM_COLS_RAW = NBUF * N;
  constexpr uint32_t TM_COLS = TM_COLS_RAW <= 32 ? 32 : TM_COLS_RAW <= 64 ? 64
                               : TM_COLS_RAW <= 128 ? 128 : TM_COLS_RAW <= 256 ? 256 : 512;
  constexpr uint32_t kATileBytes = N * 128;
  constexpr uint32_t kIdesc = idesc_e4m3_f32(128, N);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  uint8_t *w_tiles = smem;
  uint8_t *a_tiles = w_tiles + (size_t)nstage * kWTileBytes;
  float *sa_s = reinterpret_cast<float *>(a_tiles + (size_t)nstage * kATileBytes);  // [G][N]
  Stage2Smem *sh = reinterpret_cast<Stage2Smem *>(sa_s + (size_t)p.G * N);
  volatile int *abort_flag = &sh->abort;

  const int warp = (int)(threadIdx.x / 32);
  const int lane = (int)(threadIdx.x % 32);
  const int G = p.G;

  // contiguous tile range of this CTA
  const int t_begin = (int)(((long)blockIdx.x * p.n_vtiles) / gridDim.x);
  const int t_end = (int)(((long)(blockIdx.x + 1) * p.n_vtiles) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(smem_u32(&sh->tfull[b]), 1);
      mbar_init(smem_u32(&sh->tempty[b]), 4 * EPI);
    }
    sh->abort = 0;
    sh->last = 0;
    fence_mbarrier_init();
  }
  if (warp == 4 * EPI) {
    if (lane == 0) {
      prefetch_tmap(&tmap_w);
      prefetch_tmap(&tmap_a);
    }
  }
  if (warp == 4 * EPI + 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), TM_COLS);
    tmem_relinquish();
  }
  // activation scales of this token chunk, transposed to [kb][n]; zero beyond T
  for (int i = (int)threadIdx.x; i < G * N; i += (int)blockDim.x) {
    const int kb = i / N, n = i % N;
    sa_s[i] = (n < p.T) ? p.act_scales[(size_t)n * G + kb] : 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  if (warp == 4 * EPI) {
    // -------------------------------------------------------------- producer --
    // The whole warp walks the schedule; lane 0 waits and issues.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    uint32_t it = 0;
    bool ok = true;
    for (int vt = t_begin; vt < t_end && ok; ++vt) {
      for (int kb = 0; kb < G; ++kb, ++it) {
        const uint32_t s = it % (uint32_t)nstage;
        const uint32_t ph = (it / (uint32_t)nstage) & 1u;
        int got = 1;
        if (lane == 0)
          got = mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, abort_flag, p.err, kErrBitStage2);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&sh->full[s]);
          mbar_arrive_expect_tx(fb, kWTileBytes + kATileBytes);
          tma_load_2d(smem_u32(w_tiles + (size_t)s * kWTileBytes), &tmap_w, kb * 128, vt * 128,
                      fb, pol_w);
          tma_load_2d(smem_u32(a_tiles + (size_t)s * kATileBytes), &tmap_a, kb * 128, 0, fb,
                      pol_a);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      const uint32_t issued = it;
      const uint32_t first = issued > (uint32_t)nstage ? issued - (uint32_t)nstage : 0u;
      for (uint32_t j = first; j < issued; ++j)
        mbar_wait_drain(smem_u32(&sh->full[j % (uint32_t)nstage]), (j / (uint32_t)nstage) & 1u);
    }
    __syncwarp();
  } else if (warp == 4 * EPI + 1) {
    // ------------------------------------------------------------------- MMA --
    // The whole warp walks the schedule; lane 0 waits, issues the MMAs and
    // commits them to the stage's empty barrier and the accumulator's full one.
    uint32_t it = 0, kbi = 0;
    bool ok = true;
    for (int vt = t_begin; vt < t_end && ok; ++vt) {
      for (int kb = 0; kb < G; ++kb, ++it, ++kbi) {
        const uint32_t s = it % (uint32_t)nstage;
        const uint32_t ph = (it / (uint32_t)nstage) & 1u;
        const uint32_t b = kbi % NBUF;
        const uint32_t bph = (kbi / NBUF) & 1u;
        int got = 1;
        if (lane == 0)
          got = mbar_wait(smem_u32(&sh->tempty[b]), bph ^ 1u, abort_flag, p.err, kErrBitStage2) &&
                mbar_wait(smem_u32(&sh->full[s]), ph, abort_flag, p.err, kErrBitStage2);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_addr = smem_u32(w_tiles + (size_t)s * kWTileBytes);
          const uint32_t b_addr = smem_u32(a_tiles + (size_t)s * kATileBytes);
          const uint32_t d_tmem = tmem_base + b * N;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(d_tmem, sw128_kmajor_desc(a_addr + kk * 32),
                   sw128_kmajor_desc(b_addr + kk * 32), kIdesc, kk > 0 ? 1u : 0u);
          mma_commit(smem_u32(&sh->empty[s]));
          mma_commit(smem_u32(&sh->tfull[b]));
        }
        __syncwarp();
      }
    }
    // every MMA issued has finished before TMEM is released
    if (lane == 0 && kbi > 0) {
      const uint32_t last = kbi - 1;
      mbar_wait_drain(smem_u32(&sh->tfull[last % NBUF]), (last / NBUF) & 1u);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    const int quad = warp & 3;          // TMEM lanes 32*quad .. 32*quad+31
    const int grp = warp >> 2;          // column group: columns grp*NCOL ..
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(grp * NCOL);
    uint32_t kbi = 0;
    bool ok = true;

    // wait for accumulator kbi and start reading this warp's NCOL columns of it
    auto issue = [&](uint32_t (&r)[NCOL], uint32_t kb_i) -> bool {
      const uint32_t b = kb_i % NBUF;
      const bool got = mbar_wait(smem_u32(&sh->tfull[b]), (kb_i / NBUF) & 1u, abort_flag, p.err,
                                 kErrBitStage2);
      if (!__all_sync(0xffffffffu, got)) return false;
      tc_fence_after();
      if constexpr (NCOL == 16) {
        tmem_ld16(lane_base + b * N, r);
      } else {
#pragma unroll
        for (int c = 0; c < NCOL; c += 32)
          tmem_ld32(lane_base + b * N + c, *reinterpret_cast<uint32_t(*)[32]>(&r[c]));
      }
      return true;
    };
    // finish the reads and hand the accumulator back to the MMA warp
    auto release = [&](uint32_t (&r)[NCOL], uint32_t kb_i) {
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < NCOL; ++j) asm volatile("" : "+r"(r[j]));   // uses stay after the wait
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[kb_i % NBUF]));
    };

    for (int vt = t_begin; vt < t_end && ok; ++vt) {
      const float *swrow = p.w_scales + (size_t)vt * G;
      float acc[NCOL];
#pragma unroll
      for (int j = 0; j < NCOL; ++j) acc[j] = 0.0f;
      // acc += P * (sw * sa) for K block kb
      auto promote = [&](const uint32_t (&r)[NCOL], int kb, float swv) {
        const float *sak = sa_s + (size_t)kb * N + grp * NCOL;
#pragma unroll
        for (int j = 0; j < NCOL; j += 4) {
          const float4 sa4 = *reinterpret_cast<const float4 *>(sak + j);
          acc[j + 0] = fmaf(__uint_as_float(r[j + 0]), swv * sa4.x, acc[j + 0]);
          acc[j + 1] = fmaf(__uint_as_float(r[j + 1]), swv * sa4.y, acc[j + 1]);
          acc[j + 2] = fmaf(__uint_as_float(r[j + 2]), swv * sa4.z, acc[j + 2]);
          acc[j + 3] = fmaf(__uint_as_float(r[j + 3]), swv * sa4.w, acc[j + 3]);
        }
      };

      if constexpr (NCOL <= 32) {
        // two register sets: block kb+1 is read from TMEM while kb is promoted
        uint32_t ra[NCOL], rb[NCOL];
        if (!issue(ra, kbi)) { ok = false; break; }
        release(ra, kbi);
        float sw_cur = __ldg(swrow);
        for (int kb = 0; kb < G; kb += 2) {
          const uint32_t k1 = kbi + (uint32_t)kb + 1u, k2 = k1 + 1u;
          const bool more1 = kb + 1 < G;
          float sw_nxt = more1 ? __ldg(swrow + kb + 1) : 0.0f;
          if (more1 && !issue(rb, k1)) { ok = false; break; }
          promote(ra, kb, sw_cur);
          if (!more1) break;
          release(rb, k1);
          const bool more2 = kb + 2 < G;
          sw_cur = more2 ? __ldg(swrow + kb + 2) : 0.0f;
          if (more2 && !issue(ra, k2)) { ok = false; break; }
          promote(rb, kb + 1, sw_nxt);
          if (more2) release(ra, k2);
        }
        kbi += (uint32_t)G;
      } else {
        // wide column groups: 32 columns at a time to bound register use
        for (int kb = 0; kb < G; ++kb, ++kbi) {
          const float swv = __ldg(swrow + kb);
          const uint32_t b = kbi % NBUF;
          const bool got = mbar_wait(smem_u32(&sh->tfull[b]), (kbi / NBUF) & 1u, abort_flag,
                                     p.err, kErrBitStage2);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          tc_fence_after();
          const float *sak = sa_s + (size_t)kb * N + grp * NCOL;
#pragma unroll
          for (int c = 0; c < NCOL; c += 32) {
            uint32_t r[32];
            tmem_ld32(lane_base + b * N + c, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(r[j]));
            if (c + 32 >= NCOL) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 sa4 = *reinterpret_cast<const float4 *>(sak + c + j);
              acc[c + j + 0] = fmaf(__uint_as_float(r[j + 0]), swv * sa4.x, acc[c + j + 0]);
              acc[c + j + 1] = fmaf(__uint_as_float(r[j + 1]), swv * sa4.y, acc[c + j + 1]);
              acc[c + j + 2] = fmaf(__uint_as_float(r[j + 2]), swv * sa4.z, acc[c + j + 2]);
              acc[c + j + 3] = fmaf(__uint_as_float(r[j + 3]), swv * sa4.w, acc[c + j + 3]);
            }
          }
        }
      }
      if (!ok) break;

      // per-warp argmax over its 32 rows, per shard present in the warp
      const int row0 = vt * 128 + quad * 32;
      const int v = row0 + lane;
      const bool valid = v < p.V;
      const int my_shard = valid ? v / p.shard_width : -1;
      const int last_row = min(row0 + 31, p.V - 1);
      if (row0 < p.V) {
        const int s_lo = row0 / p.shard_width;
        const int s_hi = last_row / p.shard_width;
        for (int s = s_lo; s <= s_hi; ++s) {
          const bool mine = (my_shard == s);
#pragma unroll
          for (int j = 0; j < NCOL; ++j) {
            const float val = mine ? acc[j] : -INFINITY;
            float mx = val;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const unsigned ball = __ballot_sync(0xffffffffu, mine && val == mx);
            const int n = grp * NCOL + j;
            if (lane == (j & 31) && n < p.T && ball != 0u) {
              const uint32_t idx = (uint32_t)(row0 + __ffs((int)ball) - 1);
              atomicMax(&p.keys[(size_t)s * kKeyStride + n], pack_key(mx, idx));
            }
          }
        }
      }
    }
    __threadfence();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4 * EPI + 1) tmem_dealloc(tmem_base, TM_COLS);

  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.counter, 1u);
    sh->last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (sh->last) {
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
    if (threadIdx.x == 0) *p.counter = 0u;
  }
}

// ------------------------------------------------------------------- host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

// 2-D uint8 map over [rows][cols] (cols contiguous), box 128 x box_rows, 128B swizzle.
bool encode_u8_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
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

template <int NCOL, int EPI>
cudaError_t launch_cfg(const Stage2Params &p, const void *act_codes, const void *w, int num_sms,
                       cudaStream_t stream) {
  constexpr int N = NCOL * EPI;
  CUtensorMap tw, ta;
  if (!encode_u8_map(&tw, w, (uint64_t)p.V, (uint64_t)p.H, 128)) return cudaErrorInvalidValue;
  if (!encode_u8_map(&ta, act_codes, (uint64_t)p.T, (uint64_t)p.H, (uint32_t)N))
    return cudaErrorInvalidValue;
  const size_t fixed = 1024 /*align pad*/ + (size_t)p.G * N * 4 + sizeof(Stage2Smem) + 64;
  const size_t per_stage = kWTileBytes + (size_t)N * 128;
  const size_t budget = 227u * 1024u;
  int nstage = (int)((budget - fixed) / per_stage);
  if (nstage > 12) nstage = 12;
  if (nstage < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)nstage * per_stage;
  auto kern = lm_head_argmax_kernel<NCOL, EPI>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = num_sms < p.n_vtiles ? num_sms : p.n_vtiles;
  kern<<<grid, 128 * EPI + 64, smem, stream>>>(tw, ta, p, nstage);
  return cudaGetLastError();
}

}  // namespace

size_t stage2_workspace_bytes(int S) {
  return (size_t)S * kKeyStride * sizeof(unsigned long long) + 16u;
}

cudaError_t launch_stage2(const Stage2Params &p, const void *act_codes, const void *w,
                          int num_sms, cudaStream_t stream) {
  if (p.T <= 16) return launch_cfg<16, 1>(p, act_codes, w, num_sms, stream);
  if (p.T <= 32) return launch_cfg<16, 2>(p, act_codes, w, num_sms, stream);
  if (p.T <= 64) return launch_cfg<32, 2>(p, act_codes, w, num_sms, stream);
  if (p.T <= 128) return launch_cfg<32, 4>(p, act_codes, w, num_sms, stream);
  return launch_cfg<128, 2>(p, act_codes, w, num_sms, stream);
}

}  // namespace nfq
