// Stage 2, NVFP4 form: the shared LM head on the NVFP4 activation and the
// packed NVFP4 weight, with the same fused vocab-sharded argmax as the FP8 form.
//
// "[Spec Decode][Perf] Fuse the MTP trailing all-reduce; local-argmax draft
// tokens", Benchmarks: the served checkpoint is NVFP4.  The FP4 format (e2m1
// values, an unsigned e4m3 scale per 16 elements, an fp32 scale per row) is
// the published NVFP4 one; the pages fix none of it.
//
// Unlike the FP8 form, whose fp32 128x128 block scales need a promotion out of
// TMEM after every K block, the NVFP4 block scales are what the tensor cores'
// block scaling consumes: tcgen05.mma kind::mxf4nvf4 with scale_vec::4X reads
// one e4m3 scale per 16 K elements of every row of both operands from TMEM and
// accumulates the scaled products over the whole hidden dimension.  The
// epilogue only applies the two fp32 row scales and takes the argmax.
//
// Token-major, as the FP8 small-batch form: a tile is 256 vocab rows (two
// 128-row blocks, the MMA's N), the tokens (up to 128, zero-padded; MT = 64
// rows loaded for batches of at most 64) are M.  129..256 tokens run in one
// launch as two token groups: CTAs 2i and 2i+1 stream the same block range for
// tokens 0..127 and 128.., the weight with the normal L2 policy so that the
// second request for every block is served from L2.  Without a per-K-block
// promotion the epilogue reads each tile once, so the second group costs the
// SM little more than the weight stream it shares.
// One K step is 128 code bytes = 256 elements = four MMAs of K = 64.
//
// Warps (704 threads):
//   0 .. 15   epilogue: warp w reads TMEM lane quadrant w%4 (tokens
//             32(w%4) .. +31), tile columns 64(w/4) .. +63, all 64 at once,
//             releases the accumulator, then reduces them
//   16 .. 19  scale writers: per K step, copy the stage's activation and
//             weight scales from shared memory into this step's TMEM scale
//             slot, each warp into its own lane quadrant (every quadrant holds
//             the same copy)
//   20        producer: 1-D bulk copies of the packed weight codes and scales,
//             2-D tensor copies of the activation codes and scales
//   21        TMEM allocator and MMA issuer
// TMEM (512 columns): the fp32 accumulator in columns 0..255, then one scale
// slot of 48 columns per pipeline stage (16 for the activation: column
// 4kk + c holds rows 32c + lane for MMA kk; 32 for the weight: column 8kk + c
// holds rows 32c + lane).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "lm_head_common.cuh"
#include "nfq_internal.h"
#include "ptx.cuh"

namespace nfq {

namespace {

constexpr int kF4EpiWarps = 16;
constexpr int kF4SfWarps = 4;
constexpr int kF4SfWarp0 = kF4EpiWarps;
constexpr int kF4Producer = kF4EpiWarps + kF4SfWarps;
constexpr int kF4Mma = kF4Producer + 1;
constexpr int kF4Threads = (kF4Mma + 1) * 32;
constexpr int kF4MaxStages = 5;
constexpr uint32_t kF4ScaleBlock = 2048;                 // 128 rows x 16 scale bytes
constexpr uint32_t kF4WBytes = 2 * kWTileBytes;          // 256 rows x 128 code bytes
constexpr uint32_t kF4SfbBytes = 2 * kF4ScaleBlock;      // 256 rows x 16 scale bytes
constexpr uint32_t kF4SfBase = 256;                      // first scale column in TMEM
constexpr uint32_t kF4SfCols = 48;                       // scale columns per stage
static_assert(kF4SfBase + kF4MaxStages * kF4SfCols <= 512, "scale slots fit in TMEM");

// Stage layout for MT token rows: [A codes MT x 128 B][W 256 x 128 B][W scales
// 4 KB][A scales MT x 16 B].  Only the T <= MT rows of the batch are copied in.
// The MMA always reads 128 A rows; rows T..127 hold whatever the buffer held
// before (with MT = 64, rows 64..127 are the first weight rows of the stage).
// They only produce accumulator rows of tokens that do not exist — a row of D
// depends on the same row of A and its scales alone — and are never read.
template <int MT>
struct Fp4Layout {
  static constexpr uint32_t kA = 0;
  static constexpr uint32_t kABytes = MT * 128;
  static constexpr uint32_t kW = kABytes;
  static constexpr uint32_t kSfb = kW + kF4WBytes;
  static constexpr uint32_t kSfa = kSfb + kF4SfbBytes;
  static constexpr uint32_t kStage = kSfa + MT * 16 + (MT == 64 ? 1024 - 64 * 16 : 0);
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
};

struct Fp4Smem {
  uint64_t full[kF4MaxStages];
  uint64_t empty[kF4MaxStages];
  uint64_t sfready[kF4MaxStages];
  uint64_t tfull;
  uint64_t tempty;
  uint32_t tmem_base;
  int abort;
  int last;
};

template <int MT>
__global__ void __launch_bounds__(kF4Threads, 1)
    lm_head_fp4_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_sa,
                       const __grid_constant__ CUtensorMap tmap_a2,
                       const __grid_constant__ CUtensorMap tmap_sa2, const Stage2Params p,
                       int nstage) {
  using L = Fp4Layout<MT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *smem = smem_raw + pad;
  float *gs_s = reinterpret_cast<float *>(smem + (size_t)nstage * L::kStage);   // [128]
  Fp4Smem *sh = reinterpret_cast<Fp4Smem *>(gs_s + kFp4MaxT);
  volatile int *abort_flag = &sh->abort;

  const int warp = (int)(threadIdx.x / 32);
  const int lane = (int)(threadIdx.x % 32);
  const int G = p.G;                                           // K steps of 256 elements
  const size_t scale_region = (size_t)p.n_vtiles * (size_t)G * kWTileBytes;

  // token group: tokens t_base .. t_base + Tc - 1 of the launch
  const int n_grp = p.n_groups;
  const int grp = (int)blockIdx.x % n_grp;
  const int cta = (int)blockIdx.x / n_grp, n_cta = (int)gridDim.x / n_grp;
  const int t_base = grp * kFp4MaxT;
  const int Tc = min(p.T - t_base, kFp4MaxT);
  const CUtensorMap *tm_a = grp ? &tmap_a2 : &tmap_a;
  const CUtensorMap *tm_sa = grp ? &tmap_sa2 : &tmap_sa;
  const int b_begin = (int)(((long)cta * p.n_vtiles) / n_cta);
  const int b_end = (int)(((long)(cta + 1) * p.n_vtiles) / n_cta);
  const int n_tiles = (b_end - b_begin + 1) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 1);
      mbar_init(smem_u32(&sh->empty[s]), 1);
      mbar_init(smem_u32(&sh->sfready[s]), kF4SfWarps);
    }
    mbar_init(smem_u32(&sh->tfull), 1);
    mbar_init(smem_u32(&sh->tempty), kF4EpiWarps);
    sh->abort = 0;
    sh->last = 0;
    fence_mbarrier_init();
  }
  if (warp == kF4Producer && lane == 0) {
    prefetch_tmap(tm_a);
    prefetch_tmap(tm_sa);
  }
  if (warp == kF4Mma) {
    tmem_alloc(smem_u32(&sh->tmem_base), 512);
    tmem_relinquish();
  }
  __syncthreads();   // the barriers exist
  // The weight is a constant of the model, never written by the kernel this
  // one may overlap: the weight part of the first stages is requested before
  // the wait for the previous kernel (whose output is the activation), so
  // the pipeline is full when the activation becomes readable.
  const int total_steps = n_tiles * G;
  const int npre = total_steps < nstage ? total_steps : nstage;
  if (warp == kF4Producer && lane == 0) {
    const uint64_t pol_w = n_grp > 1 ? policy_evict_normal() : policy_evict_first();
    for (int it = 0; it < npre; ++it) {
      int blk0, nb;
      small_tile(b_begin, b_end, it / G, blk0, nb);
      const int ks = it % G;
      uint8_t *st = smem + (size_t)it * L::kStage;
      const uint32_t fb = smem_u32(&sh->full[it]);
      mbar_expect_tx(fb, (uint32_t)nb * (kWTileBytes + kF4ScaleBlock));
      for (int h = 0; h < nb; ++h) {
        const size_t blk = (size_t)(blk0 + h) * (size_t)G + (size_t)ks;
        bulk_g2s(smem_u32(st + L::kW + h * kWTileBytes), p.w_packed + blk * kWTileBytes,
                 kWTileBytes, fb, pol_w);
        bulk_g2s(smem_u32(st + L::kSfb + h * kF4ScaleBlock),
                 p.w_packed + scale_region + blk * kF4ScaleBlock, kF4ScaleBlock, fb, pol_w);
      }
    }
  }
  // everything below reads memory the previous kernel on the stream may write
  grid_dependency_wait();
  grid_launch_dependents();
  for (int i = (int)threadIdx.x; i < kFp4MaxT; i += (int)blockDim.x)
    gs_s[i] = (i < Tc) ? __fmul_rn(p.act_gscales[t_base + i], p.w_scale) : 0.0f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  if (warp == kF4Producer) {
    // -------------------------------------------------------------- producer --
    // One thread waits for free stages and issues the copies.
    if (lane == 0) {
      const uint64_t pol_w = n_grp > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        for (int ks = 0; ks < G; ++ks, ++it) {
          const bool pre = (int)it < npre;           // weight part already requested
          if (!pre &&
              !mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          {
            uint8_t *st = smem + (size_t)s * L::kStage;
            const uint32_t fb = smem_u32(&sh->full[s]);
            // the activation boxes hold exactly the group's Tc token rows
            mbar_arrive_expect_tx(fb, (pre ? 0u : (uint32_t)nb * (kWTileBytes + kF4ScaleBlock)) +
                                          (uint32_t)Tc * (128u + 16u));
            for (int h = 0; h < nb && !pre; ++h) {
              const size_t blk = (size_t)(blk0 + h) * (size_t)G + (size_t)ks;
              bulk_g2s(smem_u32(st + L::kW + h * kWTileBytes), p.w_packed + blk * kWTileBytes,
                       kWTileBytes, fb, pol_w);
              bulk_g2s(smem_u32(st + L::kSfb + h * kF4ScaleBlock),
                       p.w_packed + scale_region + blk * kF4ScaleBlock, kF4ScaleBlock, fb, pol_w);
            }
            tma_load_2d(smem_u32(st + L::kA), tm_a, ks * 128, 0, fb, pol_a);
            tma_load_2d(smem_u32(st + L::kSfa), tm_sa, ks * 16, 0, fb, pol_a);
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
  } else if (warp == kF4Mma) {
    // ------------------------------------------------------------------- MMA --
    // One thread issues; the descriptors of stage s are the stage-0 ones
    // advanced by s stages, K step kk adds 32 bytes (2 in the address field).
    if (lane == 0) {
      const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(smem + L::kA));
      const uint64_t w_desc0 = sw128_kmajor_desc(smem_u32(smem + L::kW));
      constexpr uint64_t kStageDesc = L::kStage >> 4;
      uint32_t s = 0, ph = 0;
      int committed = 0;
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        const uint32_t idesc = idesc_nvfp4(128, (uint32_t)(nb * 128));
        if (!mbar_wait(smem_u32(&sh->tempty), (uint32_t)(ti & 1) ^ 1u, abort_flag, p.err,
                       kErrBitStage2))
          break;
        for (int ks = 0; ks < G; ++ks) {
          const uint64_t ad = a_desc0 + kStageDesc * s, wd = w_desc0 + kStageDesc * s;
          const uint32_t sfa = tmem_base + kF4SfBase + s * kF4SfCols;
          if (!mbar_wait(smem_u32(&sh->full[s]), ph, abort_flag, p.err, kErrBitStage2) ||
              !mbar_wait(smem_u32(&sh->sfready[s]), ph, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_fp4_block16(tmem_base, ad + 2u * kk, wd + 2u * kk, idesc, sfa + 4u * kk,
                            sfa + 16u + 8u * kk, (ks > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(&sh->empty[s]));
          if (ks == G - 1) mma_commit(smem_u32(&sh->tfull));
          if (++s == (uint32_t)nstage) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) committed = ti + 1;
      }
      if (committed > 0) mbar_wait_drain(smem_u32(&sh->tfull), (uint32_t)((committed - 1) & 1));
    }
    __syncwarp();
  } else if (warp >= kF4SfWarp0) {
    // --------------------------------------------------------- scale writers --
    const int q = warp & 3;                        // this warp's TMEM lane quadrant
    uint32_t s = 0, ph = 0;
    bool ok = true;
    for (int ti = 0; ti < n_tiles && ok; ++ti) {
      for (int ks = 0; ks < G; ++ks) {
        const bool got = mbar_wait(smem_u32(&sh->full[s]), ph, abort_flag, p.err, kErrBitStage2);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint8_t *sfb_s = smem + (size_t)s * L::kStage + L::kSfb;
        const uint8_t *sfa_s = smem + (size_t)s * L::kStage + L::kSfa;
        uint32_t ra[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // token row 32c + lane: its 16 scale bytes = words for MMAs 0..3
          // (rows past MT feed accumulator rows that are never read)
          const uint4 v = (32 * c + lane < Tc)
                              ? *reinterpret_cast<const uint4 *>(sfa_s + (32 * c + lane) * 16)
                              : make_uint4(0u, 0u, 0u, 0u);
          ra[0 + c] = v.x;
          ra[4 + c] = v.y;
          ra[8 + c] = v.z;
          ra[12 + c] = v.w;
        }
        uint32_t rb[32];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // packed scale block: words (kk, lane, c = 0..3) = rows 32c + lane
            const uint4 v = *reinterpret_cast<const uint4 *>(sfb_s + h * kF4ScaleBlock +
                                                             (kk * 32 + lane) * 16);
            rb[kk * 8 + h * 4 + 0] = v.x;
            rb[kk * 8 + h * 4 + 1] = v.y;
            rb[kk * 8 + h * 4 + 2] = v.z;
            rb[kk * 8 + h * 4 + 3] = v.w;
          }
        const uint32_t col =
            tmem_base + ((uint32_t)(32 * q) << 16) + kF4SfBase + s * kF4SfCols;
        tmem_st16(col, ra);
        tmem_st32(col + 16u, rb);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh->sfready[s]));
        if (++s == (uint32_t)nstage) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    // Token 32q + lane is TMEM lane 32q + lane; column n of the accumulator is
    // row n of the tile.  Each thread streams its 64 columns 16 at a time,
    // keeping the running (max, lowest row) of the current shard.
    const int q = warp & 3;
    const int g = warp >> 2;
    const int tok = 32 * q + lane;
    const bool quad_active = 32 * q < Tc && 32 * q < MT;
    const bool tok_ok = tok < Tc;
    const int key = t_base + tok;                   // the token's index in the launch
    const float sc = gs_s[tok];
    const uint32_t taddr0 = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * g);
    for (int ti = 0; ti < n_tiles; ++ti) {
      int blk0, nb;
      small_tile(b_begin, b_end, ti, blk0, nb);
      const bool got = mbar_wait(smem_u32(&sh->tfull), (uint32_t)(ti & 1), abort_flag, p.err,
                                 kErrBitStage2);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const bool active = quad_active && (g < 2 * nb);
      const int row0 = blk0 * 128 + 64 * g;
      int cur = active ? row0 / p.shard_width : 0;     // shard of the running maximum
      int next_bound = (cur + 1) * p.shard_width;      // first row of the next shard
      float best = -INFINITY;
      int bi = -1;
      uint32_t r0[32], r1[32];
      if (active) {
        tmem_ld32(taddr0, r0);
        tmem_ld32(taddr0 + 32u, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(r0[j]), "+r"(r1[j]));
      }
      // every TMEM read of this tile is complete: the MMA may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh->tempty));
#pragma unroll
      for (int c4 = 0; c4 < 2; ++c4) {
        const uint32_t(&r)[32] = c4 ? r1 : r0;
        if (active) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int v = row0 + 32 * c4 + j;
            if (v >= p.V) break;
            if (v >= next_bound) {
              if (bi >= 0 && tok_ok)
                atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
              cur = v / p.shard_width;
              next_bound = (cur + 1) * p.shard_width;
              bi = -1;
            }
            const float logit = __fmul_rn(__uint_as_float(r[j]), sc);
            if (bi < 0 || logit > best) {
              best = logit;
              bi = v;
            }
          }
        }
      }
      if (active && bi >= 0 && tok_ok)
        atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
    }
    __threadfence();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kF4Mma) tmem_dealloc(tmem_base, 512);
  finish_launch(p, &sh->last);
}

// ------------------------------------------------ CTA pairs, 129..256 tokens --
//
// 129..256 tokens on CTA pairs (clusters of two) with cta_group::2 block-scaled
// MMAs of M = 256 tokens: the even CTA holds tokens 0..127 and the odd one
// tokens 128.. as the A operand, and each holds HALF of the tile's weight
// codes as the B operand (block blk0 + rank of a two-block tile, rows
// 64*rank.. of a one-block tile).  The pair streams every weight block once,
// and a CTA moves 38 KB per K step through shared memory where a 128-token
// CTA holding the whole tile moves 54 KB: the per-SM ingest that bounds the
// two-group form.
//
// Both CTAs keep the single-CTA layout of the block scales in TMEM: the
// activation scales of the CTA's own 128 tokens (column 4kk + c: rows
// 32c + lane) and the weight scales of ALL the tile's rows (column 8kk + c),
// which is what the pair MMA reads from each CTA.  Each CTA therefore loads the
// scale blocks of the whole tile (4 KB per K step; the second request of each
// is served from L2).
//
// Two rings per CTA.  The weight ring holds this CTA's codes and the tile's
// scales (20 KB a K step, streamed from HBM).  The activation ring holds this
// CTA's tokens' codes and scales (18 KB a step, served from L2 for every
// tile).  Each weight slot owns one TMEM scale slot, so the weight ring is 5
// deep, as many slots as TMEM holds beside the accumulator; the activation
// ring is 4 deep (2 slots measured 25 % slower, 3 slots 4 %, more nothing).
// Both producers arrive on one full barrier per step, so the scale writers
// wait once per step: their loop, not the copies, is what bounded the step
// time while they waited on three barriers (the K loop ran at about 0.53 us a
// step with the copies switched off altogether).  The activation ring must
// not be deeper than the weight ring: the activation producer may run as many
// steps ahead as it has slots, and it must never arrive on a full barrier
// whose previous phase (nw steps back) is still pending.  A build that broke
// this rule (6 activation slots, 5 full barriers) let a CTA exit with copies
// still in flight and faulted the GPU; the launcher enforces it.
//
// Warps (736 threads):
//   0 .. 15   epilogue: warp w reads TMEM lane quadrant w%4 (tokens
//             32(w%4) .. +31 of this CTA), tile columns 64(w/4) .. +63
//   16 .. 19  scale writers: per K step, the step's activation and weight
//             scales from shared memory into its TMEM scale slot
//   20        weight producer (1-D bulk copies)
//   21        TMEM allocator and, in the even CTA, the MMA issuer
//   22        activation producer (2-D tensor copies)
//
// Hand-offs between the two CTAs:
//  - each CTA's copies complete on its own full barrier; its scale writers
//    wait there, store the step's scales into TMEM and arrive on the EVEN
//    CTA's sfready barrier, which therefore completes once both CTAs' bytes
//    have landed and both CTAs' scales are in TMEM: the MMA thread waits on it
//    alone;
//  - one MMA commit per step arrives, multicast, on both CTAs' empty barrier
//    of the step (which frees its weight, TMEM and activation slots), and one
//    per tile on both tfull barriers;
//  - both CTAs' epilogue warps arrive on the even CTA's tempty barrier.
// The remote arrivals carry execution dependencies only (the copies and the
// MMAs go through the async proxy, TMEM accesses are ordered by the tcgen05
// fences), so they and the waits use the CTA scope: a cluster-scope release
// and acquire per K step measured about 1 us each, a step's whole budget.
// A cluster barrier after the set-up (barriers initialised, TMEM allocated)
// and one before the teardown (every MMA, copy and remote arrival done) bound
// every cross-CTA access.  Each CTA drains its own copies.

constexpr int kP4WProducer = kF4Producer;
constexpr int kP4Mma = kF4Mma;
constexpr int kP4AProducer = kF4Mma + 1;
constexpr int kP4Threads = (kP4AProducer + 1) * 32;
constexpr int kP4MaxW = kF4MaxStages;                       // weight ring depth (at most)
constexpr int kP4NA = 4;                                    // activation ring depth
constexpr uint32_t kP4WStage = kWTileBytes + kF4SfbBytes;   // codes (or half), the tile's scales
constexpr uint32_t kP4WSfb = kWTileBytes;
constexpr uint32_t kP4AStage = 128 * 128 + 128 * 16;        // 128 tokens' codes, then scales
constexpr uint32_t kP4ASfa = 128 * 128;
static_assert(kP4WStage % 1024 == 0 && kP4AStage % 1024 == 0,
              "ring slots keep the 1024-byte swizzle alignment");
static_assert(kP4NA <= kP4MaxW, "the activation producer stays within the full-barrier ring");

struct Fp4PairSmem {
  uint64_t full[kP4MaxW];         // this CTA's weight and activation bytes of a step have landed
  uint64_t empty[kP4MaxW];        // the step's MMAs are done: its weight, TMEM and activation slots are free
  uint64_t sfready[kF4MaxStages]; // even CTA: both CTAs' bytes landed, scales in TMEM
  uint64_t tfull;
  uint64_t tempty;                // even CTA: both CTAs' epilogues are done with the tile
  uint32_t tmem_base;
  int abort;
  int last;
};

__device__ __forceinline__ void mma_fp4_block16_pair(uint32_t d_tmem, uint64_t a_desc,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     uint32_t sfa, uint32_t sfb,
                                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], "
      "[%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// The weight copies of K step ks of tile (blk0, nb) into weight slot st: this
// CTA's codes and the tile's scales.
__device__ __forceinline__ void issue_pair_weight(const Stage2Params &p, size_t scale_region,
                                                  uint8_t *st, uint32_t fb, int blk0, int nb,
                                                  int ks, uint32_t rank, uint64_t pol_w,
                                                  uint64_t pol_s) {
  const size_t G = (size_t)p.G;
  const uint8_t *codes =
      nb == 2 ? p.w_packed + ((size_t)(blk0 + (int)rank) * G + (size_t)ks) * kWTileBytes
              : p.w_packed + ((size_t)blk0 * G + (size_t)ks) * kWTileBytes +
                    (size_t)rank * (kWTileBytes / 2);
  bulk_g2s(smem_u32(st), codes, nb == 2 ? kWTileBytes : kWTileBytes / 2, fb, pol_w);
  for (int h = 0; h < nb; ++h)
    bulk_g2s(smem_u32(st + kP4WSfb + h * kF4ScaleBlock),
             p.w_packed + scale_region + ((size_t)(blk0 + h) * G + (size_t)ks) * kF4ScaleBlock,
             kF4ScaleBlock, fb, pol_s);
}

__device__ __forceinline__ uint32_t pair_weight_bytes(int nb) {
  return (nb == 2 ? kWTileBytes : kWTileBytes / 2) + (uint32_t)nb * kF4ScaleBlock;
}

// nw: weight ring depth = TMEM scale slots
__global__ void __launch_bounds__(kP4Threads, 1)
    lm_head_fp4_pair_kernel(const __grid_constant__ CUtensorMap tmap_a0,
                            const __grid_constant__ CUtensorMap tmap_sa0,
                            const __grid_constant__ CUtensorMap tmap_a1,
                            const __grid_constant__ CUtensorMap tmap_sa1, const Stage2Params p,
                            int nw) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t *aring = smem_raw + pad;                              // kP4NA activation slots
  uint8_t *wring = aring + (size_t)kP4NA * kP4AStage;           // nw weight slots
  float *gs_s = reinterpret_cast<float *>(wring + (size_t)nw * kP4WStage);   // [128]
  Fp4PairSmem *sh = reinterpret_cast<Fp4PairSmem *>(gs_s + kFp4MaxT);
  volatile int *abort_flag = &sh->abort;

  const int warp = (int)(threadIdx.x / 32);
  const int lane = (int)(threadIdx.x % 32);
  const int G = p.G;                                           // K steps of 256 elements
  const size_t scale_region = (size_t)p.n_vtiles * (size_t)G * kWTileBytes;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int pair = (int)cluster_id_x(), n_pair = (int)nclusters_x();
  const int t_base = (int)rank * kFp4MaxT;
  const int Tc = min(p.T - t_base, kFp4MaxT);                  // this CTA's tokens (>= 1)
  const CUtensorMap *tm_a = rank ? &tmap_a1 : &tmap_a0;
  const CUtensorMap *tm_sa = rank ? &tmap_sa1 : &tmap_sa0;
  const int b_begin = (int)(((long)pair * p.n_vtiles) / n_pair);
  const int b_end = (int)(((long)(pair + 1) * p.n_vtiles) / n_pair);
  const int n_tiles = (b_end - b_begin + 1) / 2;
  const uint32_t total = (uint32_t)(n_tiles * G);              // K steps of the pair

  if (threadIdx.x == 0) {
    for (int s = 0; s < nw; ++s) {
      mbar_init(smem_u32(&sh->full[s]), 2);      // the two producers
      mbar_init(smem_u32(&sh->empty[s]), 1);
    }
    for (int s = 0; s < nw; ++s) mbar_init(smem_u32(&sh->sfready[s]), 2 * kF4SfWarps);
    mbar_init(smem_u32(&sh->tfull), 1);
    mbar_init(smem_u32(&sh->tempty), 2 * kF4EpiWarps);
    sh->abort = 0;
    sh->last = 0;
    fence_mbarrier_init();
  }
  if (warp == kP4AProducer && lane == 0) {
    prefetch_tmap(tm_a);
    prefetch_tmap(tm_sa);
  }
  if (warp == kP4Mma) {
    tmem_alloc_pair(smem_u32(&sh->tmem_base), 512);
    tmem_relinquish_pair();
  }
  __syncthreads();   // this CTA's barriers exist
  // The weight does not depend on the previous kernel on the stream: the
  // first nw weight steps are requested before the wait for it.  They
  // complete on this CTA's own barriers only.
  const uint32_t npre = total < (uint32_t)nw ? total : (uint32_t)nw;
  if (warp == kP4WProducer) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_s = policy_evict_normal();
      int ti = 0, ks = 0, blk0 = 0, nb = 0;
      if (n_tiles > 0) small_tile(b_begin, b_end, 0, blk0, nb);
      for (uint32_t it = 0; it < npre; ++it) {
        const uint32_t fb = smem_u32(&sh->full[it]);
        mbar_arrive_expect_tx(fb, pair_weight_bytes(nb));
        issue_pair_weight(p, scale_region, wring + (size_t)it * kP4WStage, fb, blk0, nb, ks, rank,
                          pol_w, pol_s);
        if (++ks == G) {
          ks = 0;
          if (++ti < n_tiles) small_tile(b_begin, b_end, ti, blk0, nb);
        }
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist and the TMEM columns are allocated
  tc_fence_after();
  // everything below reads memory the previous kernel on the stream may write
  grid_dependency_wait();
  grid_launch_dependents();
  for (int i = (int)threadIdx.x; i < kFp4MaxT; i += (int)blockDim.x)
    gs_s[i] = (i < Tc) ? __fmul_rn(p.act_gscales[t_base + i], p.w_scale) : 0.0f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;

  if (warp == kP4WProducer) {
    // ------------------------------------------------------- weight producer --
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_s = policy_evict_normal();
      uint32_t s = npre % (uint32_t)nw, ph = (npre / (uint32_t)nw) & 1u;
      int ti = (int)npre / G, ks = (int)npre % G, blk0 = 0, nb = 0;
      if (ti < n_tiles) small_tile(b_begin, b_end, ti, blk0, nb);
      uint32_t it = npre;
      for (; it < total; ++it) {
        if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1u, abort_flag, p.err, kErrBitStage2))
          break;
        const uint32_t fb = smem_u32(&sh->full[s]);
        mbar_arrive_expect_tx(fb, pair_weight_bytes(nb));
        issue_pair_weight(p, scale_region, wring + (size_t)s * kP4WStage, fb, blk0, nb, ks, rank,
                          pol_w, pol_s);
        if (++s == (uint32_t)nw) {
          s = 0;
          ph ^= 1u;
        }
        if (++ks == G) {
          ks = 0;
          if (++ti < n_tiles) small_tile(b_begin, b_end, ti, blk0, nb);
        }
      }
      // the steps whose weight copies may still be in flight (their full
      // barrier also needs the activation producer's arrival: after an
      // expired wait that may never come, and the drain gives up in time)
      const uint32_t first = it > (uint32_t)nw ? it - (uint32_t)nw : 0u;
      bool drained = true;
      for (uint32_t j = first; j < it && drained; ++j)
        drained = mbar_wait(smem_u32(&sh->full[j % (uint32_t)nw]), (j / (uint32_t)nw) & 1u,
                            abort_flag, p.err, 0u);
      if (!drained) {   // after an expired wait: give copies in flight 50 us to land
        const unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 50000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == kP4AProducer) {
    // --------------------------------------------------- activation producer --
    // The activation boxes hold exactly this CTA's Tc token rows.  Slot s of
    // step it is free once the MMAs of step it - kP4NA are done: their commit
    // on empty[(it - kP4NA) % nw] (that barrier cannot have moved on by a
    // further phase, which needs this producer's arrival for a later step).
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      uint32_t s = 0, f = 0, e = 0, eph = 0, it = 0;   // activation slot; full barrier; empty barrier of step it - kP4NA
      int ks = 0;
      for (; it < total; ++it) {
        if (it >= (uint32_t)kP4NA) {
          if (!mbar_wait(smem_u32(&sh->empty[e]), eph, abort_flag, p.err, kErrBitStage2)) break;
          if (++e == (uint32_t)nw) {
            e = 0;
            eph ^= 1u;
          }
        }
        uint8_t *st = aring + (size_t)s * kP4AStage;
        const uint32_t fb = smem_u32(&sh->full[f]);
        mbar_arrive_expect_tx(fb, (uint32_t)Tc * (128u + 16u));
        tma_load_2d(smem_u32(st), tm_a, ks * 128, 0, fb, pol_a);
        tma_load_2d(smem_u32(st + kP4ASfa), tm_sa, ks * 16, 0, fb, pol_a);
        if (++s == (uint32_t)kP4NA) s = 0;
        if (++f == (uint32_t)nw) f = 0;
        if (++ks == G) ks = 0;
      }
    }
    __syncwarp();
  } else if (warp == kP4Mma) {
    // ------------------------------------------------------------------- MMA --
    // One thread of the even CTA issues for the pair, one commit per step: this
    // thread's per-step path (wait, fence, four MMAs, commits) is what bounds the
    // K loop.  The last commit on an empty barrier covers every MMA issued
    // before it: the thread waits for it before the teardown, also when it gave
    // up within a tile.
    if (lane == 0 && even) {
      const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(aring));
      const uint64_t w_desc0 = sw128_kmajor_desc(smem_u32(wring));
      constexpr uint64_t kADesc = kP4AStage >> 4, kWDesc = kP4WStage >> 4;
      uint32_t ws = 0, wph = 0, as = 0;
      uint32_t n_issued = 0, ws_last = 0, wph_last = 0;
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        int blk0, nb;
        small_tile(b_begin, b_end, ti, blk0, nb);
        const uint32_t idesc = idesc_nvfp4(256, (uint32_t)(nb * 128));
        if (!mbar_wait(smem_u32(&sh->tempty), (uint32_t)(ti & 1) ^ 1u, abort_flag, p.err,
                       kErrBitStage2))
          break;
        for (int ks = 0; ks < G; ++ks) {
          if (!mbar_wait(smem_u32(&sh->sfready[ws]), wph, abort_flag, p.err, kErrBitStage2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a_desc0 + kADesc * as, wd = w_desc0 + kWDesc * ws;
          const uint32_t sf = tmem_base + kF4SfBase + ws * kF4SfCols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_fp4_block16_pair(tmem_base, ad + 2u * kk, wd + 2u * kk, idesc, sf + 4u * kk,
                                 sf + 16u + 8u * kk, (ks > 0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(smem_u32(&sh->empty[ws]), (uint16_t)3);
          if (ks == G - 1) mma_commit_pair(smem_u32(&sh->tfull), (uint16_t)3);
          ++n_issued;
          ws_last = ws;
          wph_last = wph;
          if (++ws == (uint32_t)nw) {
            ws = 0;
            wph ^= 1u;
          }
          if (++as == (uint32_t)kP4NA) as = 0;
        }
      }
      if (n_issued > 0) mbar_wait_drain(smem_u32(&sh->empty[ws_last]), wph_last);
    }
    __syncwarp();
  } else if (warp >= kF4SfWarp0) {
    // --------------------------------------------------------- scale writers --
    // Step it takes TMEM slot it % nw (as many slots as weight slots): its full
    // barrier completes only after the weight producer waited for the MMAs of
    // step it - nw, the slot's previous user.  One wait per step: the loop of
    // these four warps is on the K loop's critical path.
    const int q = warp & 3;                        // this warp's TMEM lane quadrant
    uint32_t ws = 0, wph = 0, as = 0;
    for (uint32_t it = 0; it < total; ++it) {
      const bool got = mbar_wait(smem_u32(&sh->full[ws]), wph, abort_flag, p.err, kErrBitStage2);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const uint8_t *sfb_s = wring + (size_t)ws * kP4WStage + kP4WSfb;
      const uint8_t *sfa_s = aring + (size_t)as * kP4AStage + kP4ASfa;
      uint32_t ra[16];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // this CTA's token row 32c + lane (rows past Tc feed accumulator rows
        // that are never read)
        const uint4 v = (32 * c + lane < Tc)
                            ? *reinterpret_cast<const uint4 *>(sfa_s + (32 * c + lane) * 16)
                            : make_uint4(0u, 0u, 0u, 0u);
        ra[0 + c] = v.x;
        ra[4 + c] = v.y;
        ra[8 + c] = v.z;
        ra[12 + c] = v.w;
      }
      uint32_t rb[32];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // the tile's rows 128h + 32c + lane (for a one-block tile, h = 1
          // fills columns the MMA of N = 128 does not read)
          const uint4 v = *reinterpret_cast<const uint4 *>(sfb_s + h * kF4ScaleBlock +
                                                           (kk * 32 + lane) * 16);
          rb[kk * 8 + h * 4 + 0] = v.x;
          rb[kk * 8 + h * 4 + 1] = v.y;
          rb[kk * 8 + h * 4 + 2] = v.z;
          rb[kk * 8 + h * 4 + 3] = v.w;
        }
      const uint32_t col = tmem_base + ((uint32_t)(32 * q) << 16) + kF4SfBase + ws * kF4SfCols;
      tmem_st16(col, ra);
      tmem_st32(col + 16u, rb);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (even) mbar_arrive(smem_u32(&sh->sfready[ws]));
        else mbar_arrive_remote_cta(smem_u32(&sh->sfready[ws]), 0u);
      }
      if (++ws == (uint32_t)nw) {
        ws = 0;
        wph ^= 1u;
      }
      if (++as == (uint32_t)kP4NA) as = 0;
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    // Token 32q + lane of this CTA is TMEM lane 32q + lane; column n of the
    // accumulator is row n of the tile.  Each thread reads its 64 columns at
    // once, releases the accumulator and then takes their argmax per shard.
    const int q = warp & 3;
    const int g = warp >> 2;
    const int tok = 32 * q + lane;
    const bool quad_active = 32 * q < Tc;
    const bool tok_ok = tok < Tc;
    const int key = t_base + tok;                   // the token's index in the launch
    const float sc = gs_s[tok];
    const uint32_t taddr0 = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * g);
    for (int ti = 0; ti < n_tiles; ++ti) {
      int blk0, nb;
      small_tile(b_begin, b_end, ti, blk0, nb);
      const bool got = mbar_wait(smem_u32(&sh->tfull), (uint32_t)(ti & 1), abort_flag, p.err,
                                 kErrBitStage2);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const bool active = quad_active && (g < 2 * nb);
      uint32_t r0[32], r1[32];
      if (active) {
        tmem_ld32(taddr0, r0);
        tmem_ld32(taddr0 + 32u, r1);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(r0[j]), "+r"(r1[j]));
      }
      // every TMEM read of this tile is complete: the MMA may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {   // the even CTA's tempty: an execution dependency only
        if (even) mbar_arrive(smem_u32(&sh->tempty));
        else mbar_arrive_remote_cta(smem_u32(&sh->tempty), 0u);
      }
      if (!active) continue;
      const int row0 = blk0 * 128 + 64 * g;
      int cur = row0 / p.shard_width;                 // shard of the running maximum
      int next_bound = (cur + 1) * p.shard_width;     // first row of the next shard
      float best = -INFINITY;
      int bi = -1;
#pragma unroll
      for (int c4 = 0; c4 < 2; ++c4) {
        const uint32_t(&r)[32] = c4 ? r1 : r0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int v = row0 + 32 * c4 + j;
          if (v >= p.V) break;
          if (v >= next_bound) {
            if (bi >= 0 && tok_ok)
              atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
            cur = v / p.shard_width;
            next_bound = (cur + 1) * p.shard_width;
            bi = -1;
          }
          const float logit = __fmul_rn(__uint_as_float(r[j]), sc);
          if (bi < 0 || logit > best) {
            best = logit;
            bi = v;
          }
        }
      }
      if (bi >= 0 && tok_ok)
        atomicMax(&p.keys[(size_t)cur * kKeyStride + key], pack_key(best, (uint32_t)bi));
    }
    __threadfence();
    __syncwarp();
  }

  // ------------------------------------------------------------- teardown --
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // every MMA, copy and remote arrival of the pair is done
  tc_fence_after();
  if (warp == kF4Mma) tmem_dealloc_pair(tmem_base, 512);
  finish_launch(p, &sh->last);
}

// Scale blocks of the packed NVFP4 weight: block (vt, s) holds, at word
// (kk * 32 + i) * 4 + c, the four block scales 4kk .. 4kk+3 of K step s for
// row vt * 128 + 32c + i (zero past V).
__global__ void __launch_bounds__(256) pack_fp4_scales_kernel(const uint8_t *__restrict__ bs,
                                                              int V, int H,
                                                              uint8_t *__restrict__ out) {
  const int G = H / 256, B16 = H / 16;
  const size_t block = blockIdx.x;                // vt * G + s
  const int vt = (int)(block / (size_t)G), s = (int)(block % (size_t)G);
  uint32_t *dst = reinterpret_cast<uint32_t *>(out + block * kF4ScaleBlock);
  for (int w = (int)threadIdx.x; w < (int)(kF4ScaleBlock / 4); w += (int)blockDim.x) {
    const int kk = w >> 7, i = (w >> 2) & 31, c = w & 3;
    const int row = vt * 128 + 32 * c + i;
    uint32_t val = 0u;
    if (row < V)
      val = *reinterpret_cast<const uint32_t *>(bs + (size_t)row * B16 + (size_t)s * 16 + 4 * kk);
    dst[w] = val;
  }
}

}  // namespace

size_t fp4_packed_weight_bytes(int V, int H) {
  return (size_t)((V + 127) / 128) * (size_t)(H / 256) * (kWTileBytes + kF4ScaleBlock);
}

cudaError_t launch_pack_fp4_weights(const uint8_t *codes, const uint8_t *bscales, int V, int H,
                                    uint8_t *out, cudaStream_t stream) {
  const size_t blocks = (size_t)((V + 127) / 128) * (size_t)(H / 256);
  if (blocks == 0 || blocks > 0x7FFFFFFFu) return cudaErrorInvalidValue;
  // the code blocks have the FP8 layout of a [V][H/2] byte matrix
  cudaError_t e = launch_pack_weights(codes, V, H / 2, out, stream);
  if (e != cudaSuccess) return e;
  pack_fp4_scales_kernel<<<(unsigned)blocks, 256, 0, stream>>>(bscales, V, H,
                                                                out + blocks * kWTileBytes);
  return cudaGetLastError();
}

namespace {

int g_fp4_stages = 0;   // 0: as many as fit

template <int MT>
cudaError_t launch_fp4(const Stage2Params &p_in, int num_sms, cudaStream_t stream) {
  using L = Fp4Layout<MT>;
  Stage2Params p = p_in;
  const int n_grp = (MT == kFp4MaxT && p.T > kFp4MaxT) ? 2 : 1;
  if (p.T < 1 || p.T > n_grp * MT || num_sms < n_grp) return cudaErrorInvalidConfiguration;
  p.n_groups = n_grp;
  CUtensorMap ta[2], tsa[2];
  // per group, boxes of exactly its token rows: a box reaching past the
  // tensor's last row is filled with zeros by the copy engine, which measured
  // slow for tiny T
  for (int g = 0; g < n_grp; ++g) {
    const int Tg = (p.T - g * MT) < MT ? (p.T - g * MT) : MT;
    if (!encode_u8_map(&ta[g], p.act_codes + (size_t)g * MT * (size_t)(p.H / 2), (uint64_t)Tg,
                       (uint64_t)(p.H / 2), (uint32_t)Tg))
      return cudaErrorInvalidValue;
    if (!encode_u8_map_plain(&tsa[g], p.act_bscales + (size_t)g * MT * (size_t)(p.H / 16),
                             (uint64_t)Tg, (uint64_t)(p.H / 16), 16u, (uint32_t)Tg))
      return cudaErrorInvalidValue;
  }
  if (n_grp == 1) {
    ta[1] = ta[0];
    tsa[1] = tsa[0];
  }
  const size_t fixed = 1024 /*align pad*/ + kFp4MaxT * sizeof(float) + sizeof(Fp4Smem) + 64;
  const size_t budget = 227u * 1024u;
  int nstage = (int)((budget - fixed) / L::kStage);
  if (nstage > kF4MaxStages) nstage = kF4MaxStages;
  if (g_fp4_stages >= 2 && g_fp4_stages < nstage) nstage = g_fp4_stages;
  if (nstage < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)nstage * L::kStage;
  auto kern = lm_head_fp4_kernel<MT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int per_grp = (num_sms / n_grp) < p.n_vtiles ? (num_sms / n_grp) : p.n_vtiles;
  return launch_pdl(kern, per_grp * n_grp, kF4Threads, smem, stream, ta[0], tsa[0], ta[1],
                    tsa[1], p, nstage);
}

bool g_fp4_pair = true;  // 129..256 tokens on CTA pairs (false: two token groups)

cudaError_t launch_fp4_pair(const Stage2Params &p_in, int num_sms, cudaStream_t stream) {
  Stage2Params p = p_in;
  if (p.T <= kFp4MaxT || p.T > 2 * kFp4MaxT || num_sms < 2) return cudaErrorInvalidConfiguration;
  p.n_groups = 1;
  CUtensorMap ta[2], tsa[2];
  // per CTA of the pair, boxes of exactly its token rows
  for (int r = 0; r < 2; ++r) {
    const int Tr = (p.T - r * kFp4MaxT) < kFp4MaxT ? (p.T - r * kFp4MaxT) : kFp4MaxT;
    if (!encode_u8_map(&ta[r], p.act_codes + (size_t)r * kFp4MaxT * (size_t)(p.H / 2),
                       (uint64_t)Tr, (uint64_t)(p.H / 2), (uint32_t)Tr))
      return cudaErrorInvalidValue;
    if (!encode_u8_map_plain(&tsa[r], p.act_bscales + (size_t)r * kFp4MaxT * (size_t)(p.H / 16),
                             (uint64_t)Tr, (uint64_t)(p.H / 16), 16u, (uint32_t)Tr))
      return cudaErrorInvalidValue;
  }
  // the weight ring (and the TMEM scale slots) as deep as shared memory and
  // TMEM allow
  const size_t fixed = 1024 /*align pad*/ + (size_t)kP4NA * kP4AStage +
                       kFp4MaxT * sizeof(float) + sizeof(Fp4PairSmem) + 64;
  const size_t budget = 227u * 1024u;
  int nw = (int)((budget - fixed) / kP4WStage);
  if (nw > kP4MaxW) nw = kP4MaxW;
  if (g_fp4_stages >= kP4NA && g_fp4_stages < nw) nw = g_fp4_stages;
  if (nw < kP4NA) return cudaErrorInvalidConfiguration;   // see the activation ring's rule
  const size_t smem = fixed + (size_t)nw * kP4WStage;
  cudaError_t e = cudaFuncSetAttribute(lm_head_fp4_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int pairs = (num_sms / 2) < p.n_vtiles ? (num_sms / 2) : p.n_vtiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3((unsigned)kP4Threads);
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
  return cudaLaunchKernelEx(&cfg, lm_head_fp4_pair_kernel, ta[0], tsa[0], ta[1], tsa[1], p, nw);
}

}  // namespace

void stage2_fp4_set_stages(int n) { g_fp4_stages = n; }

void stage2_fp4_set_pair(int enabled) { g_fp4_pair = enabled != 0; }

cudaError_t launch_stage2_fp4(const Stage2Params &p, int num_sms, cudaStream_t stream) {
  if (p.T < 1 || p.T > kFp4LaunchMaxT) return cudaErrorInvalidConfiguration;
  if (p.T > kFp4MaxT && g_fp4_pair) return launch_fp4_pair(p, num_sms, stream);
  return p.T <= 64 ? launch_fp4<64>(p, num_sms, stream) : launch_fp4<128>(p, num_sms, stream);
}

}  // namespace nfq
