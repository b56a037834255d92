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
// Per 128-wide K block kb, with the products summed by the tensor cores:
//   P[v][n] = sum_{k in block} qw[v][k] * qa[n][k]     tcgen05.mma kind::f8f6f4,
//                                                      fp32 accumulator in TMEM
//   acc[v][n] += P[v][n] * (sw[v/128][kb] * sa[n][kb]) fp32, in registers
// The scales are arbitrary fp32 values (amax / 448), which the hardware block
// scaling (power-of-two scale factors) cannot express, hence the per-block
// promotion out of TMEM.
//
// Two kernel families:
//  - lm_head_small_kernel (the default, up to 256 tokens a launch): the tokens
//    are the MMA's M operand (64 or 128) and 256 weight rows (two scale blocks)
//    are N, so each MMA consumes twice the weight bytes; 129..256 tokens run
//    as two token groups over one weight stream.  Described before the kernel.
//  - lm_head_argmax_kernel (weight-major, below; selected with
//    nfq_lm_head_small_batch(0)): the weight is M (128 vocab rows = one scale
//    block row) and up to 256 tokens are N.
//
// Warp roles of the weight-major kernel (one CTA per SM, persistent over
// contiguous vocab tiles):
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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "lm_head_common.cuh"
#include "nfq_internal.h"
#include "ptx.cuh"
#include "stage1_math.cuh"

namespace nfq {

namespace {

constexpr int kMaxStages = 16;
#ifndef NFQ_TMEM_BUFS
#define NFQ_TMEM_BUFS 16
#endif
constexpr int kMaxTmemBufs = NFQ_TMEM_BUFS;   // accumulators in flight (TMEM holds 512 columns)

struct Stage2Smem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[16];
  uint64_t tempty[16];
  uint32_t tmem_base;
  int abort;
  int last;
};


template <int NCOL, int EPI, bool kPacked>
__global__ void __launch_bounds__(128 * EPI + 64, 1)
    lm_head_argmax_kernel(const __grid_constant__ CUtensorMap tmap_w,
                          const __grid_constant__ CUtensorMap tmap_a, const Stage2Params p,
                          int nstage) {
  constexpr int N = NCOL * EPI;                  // MMA N (token columns)
  constexpr int NBUF = (512 / N) < kMaxTmemBufs ? (512 / N) : kMaxTmemBufs;
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
      if constexpr (!kPacked) prefetch_tmap(&tmap_w);
      prefetch_tmap(&tmap_a);
    }
  }
  if (warp == 4 * EPI + 1) {
    tmem_alloc(smem_u32(&sh->tmem_base), TM_COLS);
    tmem_relinquish();
  }
  // everything below reads memory the previous kernel on the stream may write
  grid_dependency_wait();
  grid_launch_dependents();
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
          if constexpr (kPacked) {
            // one contiguous, already swizzled 16 KB block per (tile, K block)
            bulk_g2s(smem_u32(w_tiles + (size_t)s * kWTileBytes),
                     p.w_packed + ((size_t)vt * G + kb) * kWTileBytes, kWTileBytes, fb, pol_w);
          } else {
            tma_load_2d(smem_u32(w_tiles + (size_t)s * kWTileBytes), &tmap_w, kb * 128, vt * 128,
                        fb, pol_w);
          }
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

    // acc[j] += P[j] * (sw * sa[kb][grp*NCOL + j]) for one K block
    auto promote = [&](float (&acc)[NCOL], const uint32_t (&r)[NCOL], int kb, float swv) {
      const float *sak = sa_s + (size_t)kb * N + grp * NCOL;
#pragma unroll
      for (int j = 0; j < NCOL; j += 4) {
        const float4 sa4 = *reinterpret_cast<const float4 *>(sak + j);
        promote4(&acc[j], &r[j], swv, sa4);
      }
    };
    // per-warp argmax over its 32 rows for every token column, merged per shard
    auto argmax_tile = [&](const float (&acc)[NCOL], int vt) {
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
    };

    // double-buffered TMEM reads when two register sets fit next to the accumulators
    constexpr bool kPipe = NCOL <= 32 && (3 * NCOL + 40) * (128 * EPI + 64) <= 65536;
    static_assert(kPipe || NCOL % 16 == 0, "unpipelined epilogue reads 16 or 32 columns at a time");
    if constexpr (kPipe) {
      // One flat pipeline over every (tile, K block) of this CTA: the TMEM read
      // of step q+1 is in flight while step q is promoted (and, at a tile's
      // last K block, while the tile's argmax runs).  The weight-scale row of
      // a tile sits in lane registers (lane l holds sw[32 i + l]) and is
      // broadcast with shuffles.
      const int n_steps = (t_end - t_begin) * G;
      auto load_sw = [&](int vt, float (&r)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = 32 * i + lane;
          r[i] = (vt < t_end && kk < G) ? __ldg(p.w_scales + (size_t)vt * G + kk) : 0.0f;
        }
      };
      auto sw_of = [&](const float (&r)[4], int kb) {
        const float src = kb < 32 ? r[0] : kb < 64 ? r[1] : kb < 96 ? r[2] : r[3];
        return __shfl_sync(0xffffffffu, src, kb & 31);
      };
      float acc[NCOL];
      float swc[4], swn[4];
      uint32_t ra[NCOL], rb[NCOL];
      int vt = t_begin, kb = 0;
      load_sw(vt, swc);
      load_sw(vt + 1, swn);
      if (n_steps > 0) {
        if (!issue(ra, 0)) ok = false;
        if (ok) release(ra, 0);
      }
      // one step: promote `cur` (step q), with step q+1 already issued into `nxt`
      auto step = [&](uint32_t (&cur)[NCOL], uint32_t (&nxt)[NCOL], int q) -> bool {
        const bool more = q + 1 < n_steps;
        if (more && !issue(nxt, (uint32_t)(q + 1))) return false;
        if (kb == 0) {
#pragma unroll
          for (int j = 0; j < NCOL; ++j) acc[j] = 0.0f;
        }
        promote(acc, cur, kb, sw_of(swc, kb));
        if (kb == G - 1) {
          argmax_tile(acc, vt);
          ++vt;
          kb = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) swc[i] = swn[i];
          load_sw(vt + 1, swn);
        } else {
          ++kb;
        }
        if (more) release(nxt, (uint32_t)(q + 1));
        return true;
      };
      for (int q = 0; q < n_steps && ok; q += 2) {
        if (!step(ra, rb, q)) { ok = false; break; }
        if (q + 1 < n_steps && !step(rb, ra, q + 1)) { ok = false; break; }
      }
    } else {
      for (int vt = t_begin; vt < t_end && ok; ++vt) {
        const float *swrow = p.w_scales + (size_t)vt * G;
        float acc[NCOL];
#pragma unroll
        for (int j = 0; j < NCOL; ++j) acc[j] = 0.0f;
        // wide column groups: 32 columns at a time to bound register use
        for (int kb = 0; kb < G; ++kb, ++kbi) {
          const float swv = __ldg(swrow + kb);
          const uint32_t b = kbi % NBUF;
          const bool got = mbar_wait(smem_u32(&sh->tfull[b]), (kbi / NBUF) & 1u, abort_flag,
                                     p.err, kErrBitStage2);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          tc_fence_after();
          const float *sak = sa_s + (size_t)kb * N + grp * NCOL;
          // 16 columns at a time when the accumulators leave little room
          constexpr int CHK = (16 * NCOL * EPI >= 4096) ? 16 : 32;
#pragma unroll
          for (int c = 0; c < NCOL; c += CHK) {
            uint32_t r[CHK];
            if constexpr (CHK == 16) {
              tmem_ld16(lane_base + b * N + c, r);
            } else {
              tmem_ld32(lane_base + b * N + c, r);
            }
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < CHK; ++j) asm volatile("" : "+r"(r[j]));
            if (c + CHK >= NCOL) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
            }
#pragma unroll
            for (int j = 0; j < CHK; j += 4) {
              const float4 sa4 = *reinterpret_cast<const float4 *>(sak + c + j);
              promote4(&acc[c + j], &r[j], swv, sa4);
            }
          }
        }
        if (!ok) break;
        argmax_tile(acc, vt);
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

// ------------------------------------------------------- small token batch --
//
// T <= 64 form.  One tcgen05.mma K=32 step costs the same for any M in {64,
// 128} and N up to 256, so the weight is made the N operand: a tile is 256
// vocab rows (two 128-row scale blocks), the tokens are the M = 64 operand.
// Each MMA then consumes 8 KB of weight instead of 4 KB.  The M = 64
// accumulator puts token r in TMEM lane 32*(r/16) + r%16; a 16x64b load gives
// every thread one token and 32 of a warp's 64 columns, so the promotion is one
// multiply per K block (activation scale x weight scale) and 32 FMAs.
//
// Warps: 0..15 epilogue (lane quadrant w%4 = tokens 16*(w%4)..+15, column
// group w/4 = tile columns 64*(w/4)..+63), 16 producer, 17 TMEM + MMA.
// A CTA streams a contiguous range of 128-row blocks, two per tile (the first
// tile of an odd range holds one).  Two 256-column accumulators in TMEM.
// Batches of 129..256 tokens run in one launch as two token groups: CTAs 2i
// and 2i+1 stream the same block range for tokens 0..127 and 128.., so every
// weight block is fetched from HBM once and served to the second CTA by L2.

constexpr int kSmallMaxT = 128;                 // tokens per token group of the token-major form
constexpr int kFusedMaxGroups = 64;             // the fused step's rows: H <= 8192
constexpr int kSmallEpiWarps = 16;
template <int MT>
__host__ __device__ constexpr uint32_t small_stage_bytes() { return 2 * kWTileBytes + MT * 128; }

struct SmallSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int abort;
  int last;
};



// The fused step's stage 1, run by the 16 epilogue warps (512 threads) of a
// CTA.  CTA r < T computes token row r exactly as the stand-alone stage-1
// kernel does (same per-thread vectors, same order of every fp32 operation),
// reading its inputs straight from global memory, and publishes the row with
// a release increment of s1.ready.  Every CTA then waits (bounded) until all T
// rows are published.  Returns false when the wait gave up.
__device__ bool fused_stage1(const Stage2Params &p, float *red, int *flag,
                             volatile int *abort_flag) {
  const FusedStage1 &s = p.s1;
  const int tc = (int)threadIdx.x;
  const int lane = tc & 31, warp = tc >> 5;
  const int r = (int)blockIdx.x;
  if (r < p.T) {                                          // CTA-uniform
    const int NA = s.na;
    const bool active = tc < NA;
    const size_t rowv = (size_t)r * (size_t)(p.H / 8);     // first 16-byte vector of the row
    float x[2][8];
    // inputs p_0 .. p_{k-1}, then the residual, in batches of up to 9 loads a vector
    for (int i0 = 0; i0 <= s.k; i0 += 9) {
      uint4 in[9][2];
#pragma unroll
      for (int c = 0; c < 9; ++c) {
        const int i = i0 + c;
        if (active && i <= s.k) {
          const uint4 *src = static_cast<const uint4 *>(i < s.k ? s.partials[i] : s.residual) + rowv;
          in[c][0] = __ldg(src + tc);
          in[c][1] = __ldg(src + NA + tc);
        } else {
          in[c][0] = in[c][1] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int c = 0; c < 9; ++c) {
        const int i = i0 + c;
        if (i > s.k) break;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          if (i == 0) unpack_bf16x8(in[c][v], x[v]);
          else add_bf16x8(x[v], in[c][v]);
        }
      }
    }
    // sum of squares in the canonical order of stage1_math.cuh: group sums
    // (one per 128 channels) in shared memory, then the row total
    float gsv[2];
#pragma unroll
    for (int v = 0; v < 2; ++v) gsv[v] = group_sum16(vec_sumsq(x[v]));   // all lanes (shuffles)
    if (active && (tc & 15) == 0) {
#pragma unroll
      for (int v = 0; v < 2; ++v) red[(v * NA + tc) / 16] = gsv[v];
    }
    named_bar_sync(1, kSmallEpiWarps * 32);
    const float tot = row_total(red, p.H / 128);
    const float ms = __fdiv_rn(tot, (float)p.H);
    const float rr = __frsqrt_rn(__fadd_rn(ms, s.eps));
    const uint4 *wsrc = static_cast<const uint4 *>(s.norm_w);
    uint4 *hid = static_cast<uint4 *>(s.hidden) + rowv;
    uint2 *cod = reinterpret_cast<uint2 *>(s.codes) + rowv;
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      const int j = v * NA + tc;
      const uint4 wpk = active ? __ldg(wsrc + j) : make_uint4(0u, 0u, 0u, 0u);
      uint4 hv;
      uint2 cv;
      float scale;
      fp8_vector_epilogue(x[v], wpk, rr, hv, cv, scale);     // all lanes (group shuffles)
      if (active) {
        hid[j] = hv;
        cod[j] = cv;
        if ((tc & 15) == 0) s.scales[(size_t)r * (size_t)(p.H / 128) + (size_t)(j / 16)] = scale;
      }
    }
    __threadfence();
    named_bar_sync(1, kSmallEpiWarps * 32);
    if (tc == 0) red_release_gpu_add(s.ready, 1u);
  }
  // every row of the batch is published before any CTA reads the activation
  if (tc == 0) {
    int ok = 1;
    if (ld_acquire_gpu(s.ready) < (unsigned)p.T) {
      const unsigned long long t0 = globaltimer();
      while (ld_acquire_gpu(s.ready) < (unsigned)p.T) {
        if (*abort_flag || globaltimer() - t0 > kWaitLimitNs) {
          atomicOr(p.err, (unsigned)kErrBitStage2);
          *abort_flag = 1;
          ok = 0;
          break;
        }
      }
    }
    fence_proxy_async_global();
    *flag = ok;
  }
  named_bar_sync(1, kSmallEpiWarps * 32);
  return *flag != 0;
}

template <int MT, bool kPacked, bool kLogits = false, bool kFused = false>
__global__ void __launch_bounds__(kSmallEpiWarps * 32 + 64, 1)
    lm_head_small_kernel(const __grid_constant__ CUtensorMap tmap_w,
                         const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_a2, const Stage2Params p,
                         int nstage) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const int G = p.G;
  constexpr uint32_t kStage = small_stage_bytes<MT>();
  float *sa_s = reinterpret_cast<float *>(smem + (size_t)nstage * kStage);  // [G][MT]
  SmallSmem *sh = reinterpret_cast<SmallSmem *>(sa_s + (size_t)G * MT);
  volatile int *abort_flag = &sh->abort;

  const int warp = (int)(threadIdx.x / 32);
  const int lane = (int)(threadIdx.x % 32);
  constexpr int kProducer = kSmallEpiWarps, kMma = kSmallEpiWarps + 1;

  // token group: tokens t_base .. t_base + Tc - 1 of the launch
  const int n_grp = p.n_groups;
  const int grp = (int)blockIdx.x % n_grp;
  const int cta = (int)blockIdx.x / n_grp, n_cta = (int)gridDim.x / n_grp;
  const int t_base = grp * MT;
  const int Tc = min(p.T - t_base, MT);
  const CUtensorMap *tmap_act = grp ? &tmap_a2 : &tmap_a;
  // contiguous range of 128-row blocks, processed two per tile
  const int b_begin = (int)(((long)cta * p.n_vtiles) / n_cta);
  const int b_end = (int)(((long)(cta + 1) * p.n_vtiles) / n_cta);
  const int n_tiles = (b_end - b_begin + 1) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh->tfull[b]), 1);
      mbar_init(smem_u32(&sh->tempty[b]), kSmallEpiWarps);
    }
    sh->abort = 0;
    sh->last = 0;
    fence_mbarrier_init();
  }
  if (warp == kProducer && lane == 0) {
    if constexpr (!kPacked) prefetch_tmap(&tmap_w);
    prefetch_tmap(tmap_act);
  }
  if (warp == kMma) {
    tmem_alloc(smem_u32(&sh->tmem_base), 512);
    tmem_relinquish();
  }
  __syncthreads();   // the barriers exist
  // The weight is a constant of the model, never written by the kernel this
  // one may overlap: the weight part of the first stages is requested before
  // the wait for the previous kernel (whose output is the activation).
  const int total_steps = n_tiles * G;
  const int npre = total_steps < nstage ? total_steps : nstage;
  if (warp == kProducer && lane == 0) {
    const uint64_t pol_w = n_grp > 1 ? policy_evict_normal() : policy_evict_first();
    for (int it = 0; it < npre; ++it) {
      int blk0, nb;
      small_tile(b_begin, b_end, it / G, blk0, nb);
      const int kb = it % G;
      uint8_t *st = smem + (size_t)it * kStage;
      const uint32_t fb = smem_u32(&sh->full[it]);
      mbar_expect_tx(fb, (uint32_t)nb * kWTileBytes);
      for (int h = 0; h < nb; ++h) {
        if constexpr (kPacked) {
          bulk_g2s(smem_u32(st + h * kWTileBytes),
                   p.w_packed + ((size_t)(blk0 + h) * G + kb) * kWTileBytes, kWTileBytes, fb,
                   pol_w);
        } else {
          tma_load_2d(smem_u32(st + h * kWTileBytes), &tmap_w, kb * 128, (blk0 + h) * 128, fb,
                      pol_w);
        }
      }
    }
  }
  // everything below reads memory the previous kernel on the stream may write
  grid_dependency_wait();
  grid_launch_dependents();
  if constexpr (kFused) {
    // stage 1 of the step, then the activation scales, by the epilogue warps
    __shared__ float s1_red[kFusedMaxGroups];
    __shared__ int s1_flag;
    if (warp < kSmallEpiWarps && fused_stage1(p, s1_red, &s1_flag, abort_flag)) {
      for (int i = (int)threadIdx.x; i < G * MT; i += kSmallEpiWarps * 32) {
        const int kb = i / MT, n = i % MT;
        sa_s[i] = (n < Tc) ? p.act_scales[(size_t)(t_base + n) * G + kb] : 0.0f;
      }
    }
  } else {
    for (int i = (int)threadIdx.x; i < G * MT; i += (int)blockDim.x) {
      const int kb = i / MT, n = i % MT;
      sa_s[i] = (n < Tc) ? p.act_scales[(size_t)(t_base + n) * G + kb] : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  if (warp == kProducer) {
    // -------------------------------------------------------------- producer --
    const uint64_t pol_w = n_grp > 1 ? policy_evict_normal() : policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    // the fused step's activation was written by other CTAs' generic stores
    if constexpr (kFused) fence_proxy_async_global();
    // One thread waits for free stages and issues the copies.
    if (lane == 0) {
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = !(kFused && *abort_flag);
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        for (int kb = 0; kb < G; ++kb, ++it) {
          const bool pre = (int)it < npre;           // weight part already requested
          if (!pre &&
              !mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          {
            uint8_t *st = smem + (size_t)s * kStage;
            const uint32_t fb = smem_u32(&sh->full[s]);
            mbar_arrive_expect_tx(fb,
                                  (pre ? 0u : (uint32_t)nb * kWTileBytes) + (uint32_t)Tc * 128u);
            for (int h = 0; h < nb && !pre; ++h) {
              if constexpr (kPacked) {
                bulk_g2s(smem_u32(st + h * kWTileBytes),
                         p.w_packed + ((size_t)(blk0 + h) * G + kb) * kWTileBytes, kWTileBytes, fb,
                         pol_w);
              } else {
                tma_load_2d(smem_u32(st + h * kWTileBytes), &tmap_w, kb * 128, (blk0 + h) * 128,
                            fb, pol_w);
              }
            }
            tma_load_2d(smem_u32(st + 2 * kWTileBytes), tmap_act, kb * 128, 0, fb, pol_a);
          }
          if (++s == (uint32_t)nstage) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // stages whose weight was requested but which the loop never reached:
      // arrive, so their phase completes once those bytes have landed
      for (uint32_t j = it; j < (uint32_t)npre; ++j) mbar_arrive(smem_u32(&sh->full[j]));
      const uint32_t issued = it > (uint32_t)npre ? it : (uint32_t)npre;
      const uint32_t first = issued > (uint32_t)nstage ? issued - (uint32_t)nstage : 0u;
      for (uint32_t j = first; j < issued; ++j)
        mbar_wait_drain(smem_u32(&sh->full[j % (uint32_t)nstage]), (j / (uint32_t)nstage) & 1u);
    }
    __syncwarp();
  } else if (warp == kMma) {
    // ------------------------------------------------------------------- MMA --
    // One thread issues; the descriptors of stage s are the stage-0 ones
    // advanced by s stages, K step kk adds 32 bytes (2 in the address field).
    if (lane == 0) {
      const uint64_t w_desc0 = sw128_kmajor_desc(smem_u32(smem));
      const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(smem + 2 * kWTileBytes));
      constexpr uint64_t kStageDesc = kStage >> 4;
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        const uint32_t idesc = idesc_e4m3_f32(MT, (uint32_t)(nb * 128));
        for (int kb = 0; kb < G; ++kb, ++it) {
          const uint32_t b = it & 1u;
          const uint64_t ad = a_desc0 + kStageDesc * s, wd = w_desc0 + kStageDesc * s;
          const uint32_t d_tmem = tmem_base + b * 256u;
          if (!mbar_wait(smem_u32(&sh->tempty[b]), ((it >> 1) & 1u) ^ 1u, abort_flag, p.err,
                         kErrBitStage2) ||
              !mbar_wait(smem_u32(&sh->full[s]), ph, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(d_tmem, ad + 2u * kk, wd + 2u * kk, idesc, kk > 0 ? 1u : 0u);
          mma_commit(smem_u32(&sh->empty[s]));
          mma_commit(smem_u32(&sh->tfull[b]));
          if (++s == (uint32_t)nstage) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (it > 0) {
        const uint32_t last = it - 1;
        mbar_wait_drain(smem_u32(&sh->tfull[last & 1u]), (last >> 1) & 1u);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    // MT = 64: the accumulator puts token r in TMEM lane 32*(r/16) + r%16; a
    //   16x64b load gives thread t token 16q + t/4 + 8*(t&1) and columns
    //   64g + 2j + ((t>>1)&1), j < 32 (two lanes share a token).
    // MT = 128: token r is TMEM lane r; 32x32b loads give thread t token
    //   32q + t and columns 64g + j, j < 64, read 16 at a time.
    constexpr int CPT = MT == 64 ? 32 : 64;        // columns per thread
    const int q = warp & 3;                        // TMEM lane quadrant
    const int g = warp >> 2;                       // tile columns 64g .. 64g+63
    const int tok = MT == 64 ? 16 * q + (lane >> 2) + 8 * (lane & 1) : 32 * q + lane;
    const int colpar = (lane >> 1) & 1;
    const bool quad_active = (MT == 64 ? 16 : 32) * q < Tc;
    const uint32_t taddr0 = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * g);
    auto col_of = [&](int j) { return MT == 64 ? 2 * j + colpar : j; };
    uint32_t it = 0;
    bool ok = true;
    for (int ti = 0; ti < n_tiles && ok; ++ti) {
      int blk0, nb;
      small_tile(b_begin, b_end, ti, blk0, nb);
      const bool active = quad_active && (g < 2 * nb);
      const int blk = blk0 + (g >> 1);             // the 128-row scale block of this group
      // this tile's weight-scale row, spread over the lanes (lane l: sw[32i + l])
      float swr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kk = 32 * i + lane;
        swr[i] = (active && kk < G) ? __ldg(p.w_scales + (size_t)blk * G + kk) : 0.0f;
      }
      float acc[CPT];
#pragma unroll
      for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < G; ++kb, ++it) {
        const uint32_t b = it & 1u;
        // this K block's scale does not depend on the accumulator: taken while the MMAs run
        const float src = kb < 32 ? swr[0] : kb < 64 ? swr[1] : kb < 96 ? swr[2] : swr[3];
        const float swv = __shfl_sync(0xffffffffu, src, kb & 31);
        const float sc = active ? sa_s[kb * MT + tok] * swv : 0.0f;
        const bool got = mbar_wait(smem_u32(&sh->tfull[b]), (it >> 1) & 1u, abort_flag, p.err,
                                   kErrBitStage2);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (MT == 64) {
          uint32_t r[32];
          if (active) {
            tmem_ld_16x64b_x32(taddr0 + b * 256u, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(r[j]));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
          if (active) {
#pragma unroll
            for (int j = 0; j < 32; j += 2)
              fma2(acc[j], acc[j + 1], __uint_as_float(r[j]), __uint_as_float(r[j + 1]), sc, sc);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            uint32_t r[16];
            if (active) {
              tmem_ld16(taddr0 + b * 256u + (uint32_t)c, r);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 16; ++j) asm volatile("" : "+r"(r[j]));
            }
            if (c == 48) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
            }
            if (active) {
#pragma unroll
              for (int j = 0; j < 16; j += 2)
                fma2(acc[c + j], acc[c + j + 1], __uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                     sc, sc);
            }
          }
        }
      }
      if (!ok) break;
      if (!active) continue;

      if constexpr (kLogits) {
        // unfused reference arm: the promoted logits go to memory as BF16,
        // two adjacent columns per 4-byte store when the row allows it
        const int row0 = blk0 * 128 + 64 * g;
        uint16_t *dst = p.logits_out + (size_t)(t_base + (tok < Tc ? tok : 0)) * (size_t)p.V;
        const bool pairs = (p.V & 1) == 0;
        if constexpr (MT == 64) {
          // this lane holds columns 2j + colpar, its partner (lane ^ 2) the others
#pragma unroll
          for (int j = 0; j < CPT; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, acc[j], 2);
            const int v0 = row0 + 2 * j;
            if (tok < Tc && (j & 1) == colpar) {
              const float lo = colpar ? other : acc[j], hi = colpar ? acc[j] : other;
              if (pairs && v0 + 1 < p.V) {
                *reinterpret_cast<uint32_t *>(dst + v0) =
                    (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                    ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
              } else {
                if (v0 < p.V) dst[v0] = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
                if (v0 + 1 < p.V) dst[v0 + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
              }
            }
          }
        } else if (tok < Tc) {
#pragma unroll
          for (int j = 0; j < CPT; j += 2) {
            const int v0 = row0 + j;
            if (pairs && v0 + 1 < p.V) {
              *reinterpret_cast<uint32_t *>(dst + v0) =
                  (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[j])) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[j + 1])) << 16);
            } else {
              if (v0 < p.V) dst[v0] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j]));
              if (v0 + 1 < p.V) dst[v0 + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j + 1]));
            }
          }
        }
        continue;
      }

      // argmax over this thread's columns (ascending rows), then merge
      const int row0 = blk0 * 128 + 64 * g;          // first row of the group
      const int last_row = min(row0 + 63, p.V - 1);
      const bool tok_ok = tok < Tc;
      const int key = t_base + tok;                  // the token's index in the launch
      if (row0 / p.shard_width == last_row / p.shard_width) {
        // the whole group is one shard: thread max, then (MT = 64) the partner lane
        float best = -INFINITY;
        int bi = -1;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int v = row0 + col_of(j);
          if (v < p.V && (bi < 0 || acc[j] > best)) {
            best = acc[j];
            bi = v;
          }
        }
        if constexpr (MT == 64) {
          const float ob = __shfl_xor_sync(0xffffffffu, best, 2);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, 2);
          if (oi >= 0 && (bi < 0 || ob > best || (ob == best && oi < bi))) {
            best = ob;
            bi = oi;
          }
        }
        if ((MT == 128 || (lane & 2) == 0) && tok_ok && bi >= 0)
          atomicMax(&p.keys[(size_t)(row0 / p.shard_width) * kKeyStride + key],
                    pack_key(best, (uint32_t)bi));
      } else {
        // shard boundaries inside the group: flush at every shard change
        float best = -INFINITY;
        int bi = -1, cur = -1;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          const int v = row0 + col_of(j);
          if (v >= p.V) break;
          const int sv = v / p.shard_width;
          if (sv != cur) {
            if (bi >= 0 && tok_ok)
              atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
            cur = sv;
            bi = -1;
          }
          if (bi < 0 || acc[j] > best) {
            best = acc[j];
            bi = v;
          }
        }
        if (bi >= 0 && tok_ok)
          atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
      }
    }
    __threadfence();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMma) tmem_dealloc(tmem_base, 512);
  if constexpr (!kLogits) finish_launch(p, &sh->last);
}

// ------------------------------------------------ CTA pairs, 129..256 tokens --
//
// Batches of 129..256 tokens run on CTA pairs (clusters of two) with
// cta_group::2 MMAs of M = 256 tokens: the even CTA holds tokens 0..127 and
// the odd one tokens 128.. as the A operand, and each holds HALF of the tile's
// weight rows as the B operand (block blk0 + rank of a two-block tile, or rows
// 64*rank.. of a one-block tile).  The even CTA's single MMA thread issues the
// MMAs; each CTA's TMEM receives its 128 tokens x the tile's 256 columns.
// Against two independent 128-token CTAs streaming the same weight, a stage
// moves 32 KB per CTA through shared memory instead of 48 KB (and the MMAs
// read 32 KB instead of 48 KB), which is what bounds that form.
//
// Hand-offs between the two CTAs:
//  - both CTAs' tensor copies of a stage complete on the EVEN CTA's full
//    barrier (cta_group::2 copies may signal the peer's barrier); the even
//    producer's arrive.expect_tx carries the stage's bytes of both CTAs;
//  - the MMA commits arrive, multicast, on both CTAs' empty (stage reusable)
//    and tfull (accumulator ready) barriers;
//  - both CTAs' epilogue warps arrive on the even CTA's tempty barriers.
// A cluster barrier after the set-up (barriers initialised, TMEM allocated)
// and one before the teardown (every MMA, copy and remote arrival done) bound
// every cross-CTA access.  The barriers carry no generic-memory data between
// the CTAs (copies and MMAs complete through the async proxy, TMEM reads and
// writes are ordered by the tcgen05 fences), so every wait is the CTA-scope
// one.

constexpr uint32_t kPairATile = 128 * 128;         // 128 tokens x 128 K bytes
constexpr uint32_t kPairStage = 2 * kPairATile;    // A tile + half of the tile's weight rows

struct PairSmem {
  uint64_t full[kMaxStages];   // even CTA: both CTAs' bytes of a stage have landed
  uint64_t empty[kMaxStages];  // each CTA: its part of the stage may be refilled
  uint64_t tfull[2];           // each CTA: accumulator b is ready
  uint64_t tempty[2];          // even CTA: both CTAs' epilogues are done with accumulator b
  uint32_t tmem_base;
  int abort;
  int last;
};

template <bool kPacked>
__global__ void __launch_bounds__(kSmallEpiWarps * 32 + 64, 1)
    lm_head_pair_kernel(const __grid_constant__ CUtensorMap tmap_w128,
                        const __grid_constant__ CUtensorMap tmap_w64,
                        const __grid_constant__ CUtensorMap tmap_a0,
                        const __grid_constant__ CUtensorMap tmap_a1, const Stage2Params p,
                        int nstage) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  const int G = p.G;
  float *sa_s = reinterpret_cast<float *>(smem + (size_t)nstage * kPairStage);  // [G][128]
  PairSmem *sh = reinterpret_cast<PairSmem *>(sa_s + (size_t)G * 128);
  volatile int *abort_flag = &sh->abort;

  const int warp = (int)(threadIdx.x / 32);
  const int lane = (int)(threadIdx.x % 32);
  constexpr int kProducer = kSmallEpiWarps, kMma = kSmallEpiWarps + 1;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int pair = (int)cluster_id_x(), n_pair = (int)nclusters_x();
  const int t_base = (int)rank * 128;
  const int Tc = min(p.T - t_base, 128);                    // this CTA's tokens (>= 1)
  const int Tc_pair = p.T;                                   // both CTAs' tokens
  const CUtensorMap *tmap_act = rank ? &tmap_a1 : &tmap_a0;
  const int b_begin = (int)(((long)pair * p.n_vtiles) / n_pair);
  const int b_end = (int)(((long)(pair + 1) * p.n_vtiles) / n_pair);
  const int n_tiles = (b_end - b_begin + 1) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sh->tfull[b]), 1);
      mbar_init(smem_u32(&sh->tempty[b]), 2 * kSmallEpiWarps);
    }
    sh->abort = 0;
    sh->last = 0;
    fence_mbarrier_init();
  }
  if (warp == kProducer && lane == 0) {
    if constexpr (!kPacked) {
      prefetch_tmap(&tmap_w128);
      prefetch_tmap(&tmap_w64);
    }
    prefetch_tmap(tmap_act);
  }
  if (warp == kMma) {
    tmem_alloc_pair(smem_u32(&sh->tmem_base), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers exist and the TMEM columns are allocated
  tc_fence_after();
  // everything below reads memory the previous kernel on the stream may write
  grid_dependency_wait();
  grid_launch_dependents();
  for (int i = (int)threadIdx.x; i < G * 128; i += (int)blockDim.x) {
    const int kb = i / 128, n = i % 128;
    sa_s[i] = (n < Tc) ? p.act_scales[(size_t)(t_base + n) * G + kb] : 0.0f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  // the even CTA's full barriers, as seen from this CTA
  const uint32_t full0 = mapa_shared(smem_u32(&sh->full[0]), 0u);

  if (warp == kProducer) {
    // -------------------------------------------------------------- producer --
    // One thread waits for free stages and issues both CTAs' copies.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        for (int kb = 0; kb < G; ++kb, ++it) {
          if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          uint8_t *st = smem + (size_t)s * kPairStage;
          const uint32_t fb = full0 + 8u * s;
          if (even)   // the stage's bytes of both CTAs: two activation tiles, the weight rows
            mbar_arrive_expect_tx(smem_u32(&sh->full[s]),
                                  (uint32_t)Tc_pair * 128u + (uint32_t)nb * kWTileBytes);
          tma_load_2d_pair(smem_u32(st), tmap_act, kb * 128, 0, fb, pol_a);
          if (nb == 2) {
            if constexpr (kPacked)
              tma_load_2d_pair(smem_u32(st + kPairATile), &tmap_w128, 0,
                               ((blk0 + (int)rank) * G + kb) * 128, fb, pol_w);
            else
              tma_load_2d_pair(smem_u32(st + kPairATile), &tmap_w128, kb * 128,
                               (blk0 + (int)rank) * 128, fb, pol_w);
          } else {
            if constexpr (kPacked)
              tma_load_2d_pair(smem_u32(st + kPairATile), &tmap_w64, 0,
                               (blk0 * G + kb) * 128 + 64 * (int)rank, fb, pol_w);
            else
              tma_load_2d_pair(smem_u32(st + kPairATile), &tmap_w64, kb * 128,
                               blk0 * 128 + 64 * (int)rank, fb, pol_w);
          }
          if (++s == (uint32_t)nstage) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (even) {
        // the even CTA counts both CTAs' copies: wait until every stage issued has landed
        const uint32_t first = it > (uint32_t)nstage ? it - (uint32_t)nstage : 0u;
        for (uint32_t q = first; q < it; ++q)
          mbar_wait_drain(smem_u32(&sh->full[q % (uint32_t)nstage]), (q / (uint32_t)nstage) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == kMma) {
    // ------------------------------------------------------------------- MMA --
    // One thread of the even CTA issues for the pair.  The descriptors of
    // stage s are the stage-0 ones advanced by s stages; K step kk adds 32 bytes
    // (2 in the descriptor's address field).
    if (lane == 0 && even) {
      const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(smem));
      const uint64_t w_desc0 = sw128_kmajor_desc(smem_u32(smem + kPairATile));
      constexpr uint64_t kStageDesc = kPairStage >> 4;
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        const uint32_t idesc = idesc_e4m3_f32(256, (uint32_t)(nb * 128));
        for (int kb = 0; kb < G; ++kb, ++it) {
          const uint32_t b = it & 1u;
          const uint64_t ad = a_desc0 + kStageDesc * s, wd = w_desc0 + kStageDesc * s;
          const uint32_t d_tmem = tmem_base + b * 256u;
          if (!mbar_wait(smem_u32(&sh->tempty[b]), ((it >> 1) & 1u) ^ 1u, abort_flag, p.err,
                         kErrBitStage2) ||
              !mbar_wait(smem_u32(&sh->full[s]), ph, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_pair(d_tmem, ad + 2u * kk, wd + 2u * kk, idesc, kk > 0 ? 1u : 0u);
          mma_commit_pair(smem_u32(&sh->empty[s]), (uint16_t)3);
          mma_commit_pair(smem_u32(&sh->tfull[b]), (uint16_t)3);
          if (++s == (uint32_t)nstage) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (it > 0) {
        const uint32_t last = it - 1;
        mbar_wait_drain(smem_u32(&sh->tfull[last & 1u]), (last >> 1) & 1u);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    // Token r of this CTA is TMEM lane r; thread t of warp w holds token
    // 32 (w%4) + t and the tile columns 64 (w/4) .. +63, read 16 at a time.
    const int q = warp & 3;
    const int g = warp >> 2;
    const int tok = 32 * q + lane;
    const bool quad_active = 32 * q < Tc;
    const uint32_t taddr0 = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * g);
    uint32_t it = 0;
    bool ok = true;
    for (int ti = 0; ti < n_tiles && ok; ++ti) {
      int blk0, nb;
      small_tile(b_begin, b_end, ti, blk0, nb);
      const bool active = quad_active && (g < 2 * nb);
      const int blk = blk0 + (g >> 1);
      float swr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kk = 32 * i + lane;
        swr[i] = (active && kk < G) ? __ldg(p.w_scales + (size_t)blk * G + kk) : 0.0f;
      }
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
      for (int kb = 0; kb < G; ++kb, ++it) {
        const uint32_t b = it & 1u;
        // this K block's scale does not depend on the accumulator: taken while the MMAs run
        const float src = kb < 32 ? swr[0] : kb < 64 ? swr[1] : kb < 96 ? swr[2] : swr[3];
        const float swv = __shfl_sync(0xffffffffu, src, kb & 31);
        const float sc = active ? sa_s[kb * 128 + tok] * swv : 0.0f;
        const bool got = mbar_wait(smem_u32(&sh->tfull[b]), (it >> 1) & 1u, abort_flag,
                                         p.err, kErrBitStage2);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          uint32_t r[16];
          if (active) {
            tmem_ld16(taddr0 + b * 256u + (uint32_t)c, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) asm volatile("" : "+r"(r[j]));
          }
          if (c == 48) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // the even CTA's tempty: an execution dependency only
              if (even) mbar_arrive(smem_u32(&sh->tempty[b]));
              else mbar_arrive_remote_cta(smem_u32(&sh->tempty[b]), 0u);
            }
          }
          if (active) {
#pragma unroll
            for (int j = 0; j < 16; j += 2)
              fma2(acc[c + j], acc[c + j + 1], __uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                   sc, sc);
          }
        }
      }
      if (!ok) break;
      if (!active) continue;

      // argmax over this thread's 64 columns (ascending rows), merged per shard
      const int row0 = blk0 * 128 + 64 * g;
      const bool tok_ok = tok < Tc;
      const int key = t_base + tok;
      const int shard0 = row0 / p.shard_width;
      if (row0 + 63 < p.V && (row0 + 63) / p.shard_width == shard0) {
        // all 64 rows valid and in one shard: first maximum in ascending row order
        float best = acc[0];
        int bj = 0;
#pragma unroll
        for (int j = 1; j < 64; ++j)
          if (acc[j] > best) {
            best = acc[j];
            bj = j;
          }
        if (tok_ok)
          atomicMax(&p.keys[(size_t)shard0 * kKeyStride + key],
                    pack_key(best, (uint32_t)(row0 + bj)));
      } else {
        float best = -INFINITY;
        int bi = -1, cur = -1;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int v = row0 + j;
          if (v >= p.V) break;
          const int sv = v / p.shard_width;
          if (sv != cur) {
            if (bi >= 0 && tok_ok)
              atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
            cur = sv;
            bi = -1;
          }
          if (bi < 0 || acc[j] > best) {
            best = acc[j];
            bi = v;
          }
        }
        if (bi >= 0 && tok_ok)
          atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
      }
    }
    __threadfence();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  // After an expired wait the odd CTA cannot see its copies complete (they
  // count on the even CTA's barriers, which may never have been armed for
  // them): it gives copies in flight 50 us to land before leaving.
  if (!even && threadIdx.x == 0 && *abort_flag) {
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 50000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // every MMA, copy and remote arrival of the pair is done
  tc_fence_after();
  if (warp == kMma) tmem_dealloc_pair(tmem_base, 512);
  finish_launch(p, &sh->last);
}

// ------------------------------------------------------------------- host --




template <int NCOL, int EPI, bool kPacked>
cudaError_t launch_cfg(const Stage2Params &p, const void *act_codes, const void *w, int num_sms,
                       cudaStream_t stream) {
  constexpr int N = NCOL * EPI;
  CUtensorMap tw, ta;
  std::memset(&tw, 0, sizeof(tw));
  if (!kPacked && !encode_u8_map(&tw, w, (uint64_t)p.V, (uint64_t)p.H, 128))
    return cudaErrorInvalidValue;
  if (!encode_u8_map(&ta, act_codes, (uint64_t)p.T, (uint64_t)p.H, (uint32_t)N))
    return cudaErrorInvalidValue;
  const size_t fixed = 1024 /*align pad*/ + (size_t)p.G * N * 4 + sizeof(Stage2Smem) + 64;
  const size_t per_stage = kWTileBytes + (size_t)N * 128;
  const size_t budget = 227u * 1024u;
  int nstage = (int)((budget - fixed) / per_stage);
  if (nstage > 12) nstage = 12;
  if (nstage < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)nstage * per_stage;
  auto kern = lm_head_argmax_kernel<NCOL, EPI, kPacked>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = num_sms < p.n_vtiles ? num_sms : p.n_vtiles;
  return launch_pdl(kern, grid, 128 * EPI + 64, smem, stream, tw, ta, p, nstage);
}

bool g_small_enabled = true;

template <bool kPacked>
cudaError_t launch_by_tokens(const Stage2Params &p, const void *act_codes, const void *w,
                             int num_sms, cudaStream_t stream) {
  if (p.T <= 16) return launch_cfg<16, 1, kPacked>(p, act_codes, w, num_sms, stream);
  if (p.T <= 32) return launch_cfg<16, 2, kPacked>(p, act_codes, w, num_sms, stream);
  if (p.T <= 64) return launch_cfg<16, 4, kPacked>(p, act_codes, w, num_sms, stream);
  if (p.T <= 128) return launch_cfg<32, 4, kPacked>(p, act_codes, w, num_sms, stream);
  return launch_cfg<64, 4, kPacked>(p, act_codes, w, num_sms, stream);
}

// Re-lays the row-major [V][H] e4m3 weight into [ceil(V/128)][H/128] blocks of
// 128 rows x 128 bytes, each row's 16-byte chunks permuted by the 128-byte
// swizzle (chunk c of row r stored at chunk c ^ (r mod 8)); rows past V are 0.
__global__ void __launch_bounds__(256) pack_weights_kernel(const uint8_t *__restrict__ w, int V,
                                                           int H, uint8_t *__restrict__ out) {
  const int G = H / 128;
  const size_t block = blockIdx.x;           // vt * G + kb
  const int vt = (int)(block / (size_t)G), kb = (int)(block % (size_t)G);
  uint4 *dst = reinterpret_cast<uint4 *>(out + block * kWTileBytes);
  for (int i = (int)threadIdx.x; i < 1024; i += (int)blockDim.x) {
    const int r = i >> 3, c = i & 7;
    const int row = vt * 128 + r;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < V)
      v = *reinterpret_cast<const uint4 *>(w + (size_t)row * H + (size_t)kb * 128 + c * 16);
    dst[r * 8 + (c ^ (r & 7))] = v;
  }
}

}  // namespace

size_t stage2_workspace_bytes(int S) { return stage2_workspace_bytes_for(S); }

template <int MT, bool kPacked, bool kLogits = false, bool kFused = false>
cudaError_t launch_small(const Stage2Params &p_in, const void *act_codes, const void *w,
                         int num_sms, cudaStream_t stream) {
  // two token groups (the second CTA of each pair reads the weight from L2)
  // for 129..256 tokens in the plain argmax form
  const int n_grp = (MT == 128 && !kLogits && !kFused && p_in.T > MT) ? 2 : 1;
  if (p_in.T < 1 || p_in.T > n_grp * MT || num_sms < n_grp) return cudaErrorInvalidConfiguration;
  Stage2Params p = p_in;
  p.n_groups = n_grp;
  CUtensorMap tw, ta[2];
  std::memset(&tw, 0, sizeof(tw));
  if (!kPacked && !encode_u8_map(&tw, w, (uint64_t)p.V, (uint64_t)p.H, 128))
    return cudaErrorInvalidValue;
  // per group a box of exactly its token count: rows Tc..MT-1 of the tile keep
  // stale bytes, which only reach accumulator rows of tokens that do not exist
  // (never read)
  for (int g = 0; g < n_grp; ++g) {
    const int Tg = (p.T - g * MT) < MT ? (p.T - g * MT) : MT;
    if (!encode_u8_map(&ta[g], static_cast<const uint8_t *>(act_codes) + (size_t)g * MT * p.H,
                       (uint64_t)Tg, (uint64_t)p.H, (uint32_t)Tg))
      return cudaErrorInvalidValue;
  }
  if (n_grp == 1) ta[1] = ta[0];
  constexpr uint32_t kStage = small_stage_bytes<MT>();
  const size_t fixed = 1024 /*align pad*/ + (size_t)p.G * MT * 4 + sizeof(SmallSmem) + 64;
  const size_t budget = 227u * 1024u;
  int nstage = (int)((budget - fixed) / kStage);
  if (nstage > 8) nstage = 8;
  if (nstage < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)nstage * kStage;
  auto kern = lm_head_small_kernel<MT, kPacked, kLogits, kFused>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int per_grp = (num_sms / n_grp) < p.n_vtiles ? (num_sms / n_grp) : p.n_vtiles;
  return launch_pdl(kern, per_grp * n_grp, kSmallEpiWarps * 32 + 64, smem, stream, tw, ta[0],
                    ta[1], p, nstage);
}

bool g_pair_enabled = true;

// 129..256 tokens on CTA pairs (cta_group::2).  Weight tiles come through 2-D
// tensor maps with boxes of 128 and 64 rows: over the row-major [V][H] weight
// (128-byte swizzle), or over the packed layout seen as [blocks x 128][128]
// bytes (already swizzled, copied as is).
template <bool kPacked>
cudaError_t launch_pair(const Stage2Params &p_in, const void *act_codes, const void *w,
                        int num_sms, cudaStream_t stream) {
  if (p_in.T <= kSmallMaxT || p_in.T > 2 * kSmallMaxT || num_sms < 2)
    return cudaErrorInvalidConfiguration;
  Stage2Params p = p_in;
  p.n_groups = 2;
  CUtensorMap tw128, tw64, ta[2];
  if constexpr (kPacked) {
    const uint64_t rows = (uint64_t)p.n_vtiles * (uint64_t)p.G * 128u;
    if (!encode_u8_map_plain(&tw128, w, rows, 128, 128, 128) ||
        !encode_u8_map_plain(&tw64, w, rows, 128, 128, 64))
      return cudaErrorInvalidValue;
  } else {
    if (!encode_u8_map(&tw128, w, (uint64_t)p.V, (uint64_t)p.H, 128) ||
        !encode_u8_map(&tw64, w, (uint64_t)p.V, (uint64_t)p.H, 64))
      return cudaErrorInvalidValue;
  }
  for (int g = 0; g < 2; ++g) {
    const int Tg = (p.T - g * 128) < 128 ? (p.T - g * 128) : 128;
    if (!encode_u8_map(&ta[g], static_cast<const uint8_t *>(act_codes) + (size_t)g * 128 * p.H,
                       (uint64_t)Tg, (uint64_t)p.H, (uint32_t)Tg))
      return cudaErrorInvalidValue;
  }
  const size_t fixed = 1024 /*align pad*/ + (size_t)p.G * 128 * 4 + sizeof(PairSmem) + 64;
  const size_t budget = 227u * 1024u;
  int nstage = (int)((budget - fixed) / kPairStage);
  if (nstage > kMaxStages) nstage = kMaxStages;
  if (nstage < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)nstage * kPairStage;
  auto kern = lm_head_pair_kernel<kPacked>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int pairs = (num_sms / 2) < p.n_vtiles ? (num_sms / 2) : p.n_vtiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3((unsigned)(kSmallEpiWarps * 32 + 64));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tw128, tw64, ta[0], ta[1], p, nstage);
}

cudaError_t launch_stage2(const Stage2Params &p, const void *act_codes, const void *w,
                          int num_sms, cudaStream_t stream) {
  if (p.T > kSmallMaxT && p.T <= 2 * kSmallMaxT && g_small_enabled && g_pair_enabled)
    return p.w_packed ? launch_pair<true>(p, act_codes, w, num_sms, stream)
                      : launch_pair<false>(p, act_codes, w, num_sms, stream);
  if (p.T <= 2 * kSmallMaxT && g_small_enabled) {
    if (p.T <= 64)
      return p.w_packed ? launch_small<64, true>(p, act_codes, w, num_sms, stream)
                        : launch_small<64, false>(p, act_codes, w, num_sms, stream);
    return p.w_packed ? launch_small<128, true>(p, act_codes, w, num_sms, stream)
                      : launch_small<128, false>(p, act_codes, w, num_sms, stream);
  }
  if (p.w_packed) return launch_by_tokens<true>(p, act_codes, w, num_sms, stream);
  return launch_by_tokens<false>(p, act_codes, w, num_sms, stream);
}

void stage2_set_small(int enabled) { g_small_enabled = enabled != 0; }

void stage2_set_pair(int enabled) { g_pair_enabled = enabled != 0; }

// The fused step: batches of at most 64 tokens (one CTA per row among the
// grid), rows whose H/16 data-holding threads are whole warps within the 512
// epilogue threads, at most 16 inputs, packed weight.
bool fused_step_supported(int T, int H, int k, int V, int num_sms) {
  const int n_vtiles = (V + 127) / 128;
  const int grid = num_sms < n_vtiles ? num_sms : n_vtiles;
  return T >= 1 && T <= 64 && T <= grid && H % 512 == 0 && H / 16 <= kSmallEpiWarps * 32 &&
         k >= 1 && k <= kMaxPartials;
}

cudaError_t launch_fused_step(const Stage2Params &p, int num_sms, cudaStream_t stream) {
  if (!p.w_packed || !p.s1.ready || !fused_step_supported(p.T, p.H, p.s1.k, p.V, num_sms))
    return cudaErrorInvalidConfiguration;
  return launch_small<64, true, false, true>(p, p.act_codes, p.w_packed, num_sms, stream);
}

cudaError_t launch_lm_head_logits(const Stage2Params &p, int num_sms, cudaStream_t stream) {
  if (!p.w_packed || !p.logits_out || p.T < 1 || p.T > kSmallMaxT)
    return cudaErrorInvalidConfiguration;
  return p.T <= 64 ? launch_small<64, true, true>(p, p.act_codes, p.w_packed, num_sms, stream)
                   : launch_small<128, true, true>(p, p.act_codes, p.w_packed, num_sms, stream);
}

// Tokens per launch: up to 256 in either family (the token-major form runs
// 129..256 tokens as two token groups over one weight stream).
int stage2_token_chunk() { return 2 * kSmallMaxT; }

size_t packed_weight_bytes(int V, int H) {
  return (size_t)((V + 127) / 128) * (size_t)(H / 128) * kWTileBytes;
}

cudaError_t launch_pack_weights(const uint8_t *w, int V, int H, uint8_t *out,
                                cudaStream_t stream) {
  const size_t blocks = (size_t)((V + 127) / 128) * (size_t)(H / 128);
  if (blocks == 0 || blocks > 0x7FFFFFFFu) return cudaErrorInvalidValue;
  pack_weights_kernel<<<(unsigned)blocks, 256, 0, stream>>>(w, V, H, out);
  return cudaGetLastError();
}

}  // namespace nfq
