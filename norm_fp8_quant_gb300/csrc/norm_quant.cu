// Stage 1: fused k-way partial-sum reduction + residual + RMSNorm + packed FP8.
//
// "[Quant][MTP] Reuse packed FP8 logits inputs", Purpose: the MTP layer's final
// all-reduce and RMSNorm are fused with packed FP8 quantisation and the layer
// returns both the packed activation and the post-norm BF16 hidden state.
// "[Spec Decode][Perf] Fuse the MTP trailing all-reduce; local-argmax draft
// tokens", intro and Accuracy: the trailing all-reduce goes into the final
// RMSNorm and the fused kernel accumulates in fp32.
//
// Design (HBM-bound streaming kernel):
//  * A row of H channels is split over a cluster of C CTAs (C = 1 for long
//    inputs, up to 8 when there are too few rows to occupy every SM); each CTA
//    owns E = H / C consecutive channels (whole 128-channel groups).
//  * Warp 0 is the producer: one thread streams (row, input) chunks of E BF16
//    values — the k partials, then the residual — into a ring of shared-memory
//    slots with 1-D TMA bulk copies completing on per-slot mbarriers.
//  * The consumer warps own fixed 16-byte vectors of the slice: vector j of the
//    slice is held by thread j mod NA in register slot j / NA, so the 16
//    vectors of a 128-channel group sit in 16 consecutive lanes.  They add the
//    inputs in fp32 in input order (no intermediate rounding), square-sum
//    per warp with shuffles, combine warps in shared memory and, when C > 1,
//    exchange the CTA partial sums through distributed shared memory.
//  * Epilogue per vector: y = bf16((x * rsqrt(ms + eps)) * w); the group
//    maximum |y| is a 16-lane shuffle reduction; scale = amax / 448 (IEEE
//    division); codes = cvt.rn.satfinite.e4m3x2(y / scale).  Hidden (16 B),
//    codes (8 B) and scales go straight to global memory, coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "nfq_internal.h"
#include "ptx.cuh"
#include "stage1_math.cuh"

namespace nfq {

namespace {

constexpr int kErrBitStage1 = 1;
// register budget: one vector per thread with up to 992 consumers, two with up
// to 512 (17 warps leave 96 registers a thread), more with up to 256
__host__ __device__ constexpr int stage1_max_threads(int vpt) {
  return vpt == 1 ? 1024 : vpt == 2 ? 544 : 288;
}

constexpr int kMaxGroups = 256;   // 128-channel groups of the widest row (H = 32768)

struct RowSums {
  float gs[2][kMaxGroups];   // per group: sum of squares, double-buffered by row parity
  float amx[2][32];          // per consumer warp: row maximum |hidden| (NVFP4 form)
};

template <int VPT, bool kFp4>
__global__ void __launch_bounds__(stage1_max_threads(VPT), 1)
    reduce_norm_quant_kernel(const Stage1Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int E = p.E;
  const uint32_t in_bytes = (uint32_t)E * 2u;                  // one input's slice of a row
  const int m = p.per_slot;                                      // inputs per ring slot
  const uint32_t slot_bytes = in_bytes * (uint32_t)m;
  uint8_t *ring = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)p.nslot * slot_bytes);
  uint64_t *empty = full + p.nslot;
  uint64_t *ss_bar = empty + p.nslot;               // [2], the row's group sums (cluster-wide)
  uint64_t *amx_bar = ss_bar + 2;                   // [2], row maximum (NVFP4 form)
  RowSums *sums = reinterpret_cast<RowSums *>(amx_bar + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sums + 1);

  const int C = p.C;
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const int cid = (C > 1) ? (int)cluster_id_x() : (int)blockIdx.x;
  const int ncl = (C > 1) ? (int)nclusters_x() : (int)gridDim.x;
  const int col0 = (int)rank * E;
  const int n_cons_warps = (int)(blockDim.x / 32) - 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nslot; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), (uint32_t)n_cons_warps);
    }
    // one arrival per consumer warp (one CTA), or per 128-channel group of the
    // row from whichever CTA of the cluster holds it
    const uint32_t ss_count = C > 1 ? (uint32_t)(p.H / 128) : (uint32_t)n_cons_warps;
    mbar_init(smem_u32(&ss_bar[0]), ss_count);
    mbar_init(smem_u32(&ss_bar[1]), ss_count);
    mbar_init(smem_u32(&amx_bar[0]), (uint32_t)n_cons_warps);
    mbar_init(smem_u32(&amx_bar[1]), (uint32_t)n_cons_warps);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (C > 1) cluster_sync_all();   // peers' barriers exist before any remote arrive
  // The set-up above overlaps the previous kernel's tail; every global read
  // and write below waits for it (its outputs may be this kernel's inputs, and
  // it may still read the buffers this kernel writes).
  grid_dependency_wait();
  grid_launch_dependents();

  const int warp = (int)(threadIdx.x / 32);
  const int lane = (int)(threadIdx.x % 32);

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // The whole warp walks the schedule (so it stays converged for the
    // barriers at the end); lane 0 waits and issues, the others follow.
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    for (int r = cid; r < p.T && ok; r += ncl) {
      const size_t off = ((size_t)r * (size_t)p.H + (size_t)col0) * 2u;
      for (int i0 = 0; i0 <= p.k; i0 += m, ++it) {
        const int cnt = (p.k + 1 - i0) < m ? (p.k + 1 - i0) : m;
        const uint32_t s = it % (uint32_t)p.nslot;
        const uint32_t ph = (it / (uint32_t)p.nslot) & 1u;
        int got = 1;
        if (lane == 0)
          got = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, abort_flag, p.err, kErrBitStage1);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&full[s]), in_bytes * (uint32_t)cnt);
          for (int c = 0; c < cnt; ++c) {
            const int i = i0 + c;
            const uint8_t *src =
                static_cast<const uint8_t *>(i < p.k ? p.partials[i] : p.residual) + off;
            bulk_g2s(smem_u32(ring + (size_t)s * slot_bytes + (size_t)c * in_bytes), src,
                     in_bytes, smem_u32(&full[s]), pol);
          }
        }
        __syncwarp();
      }
    }
    // every copy issued lands before the CTA can leave
    if (lane == 0) {
      const uint32_t issued = it;
      const uint32_t first = issued > (uint32_t)p.nslot ? issued - (uint32_t)p.nslot : 0u;
      for (uint32_t j = first; j < issued; ++j)
        mbar_wait_drain(smem_u32(&full[j % (uint32_t)p.nslot]), (j / (uint32_t)p.nslot) & 1u);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers --
    // Every lane of a consumer warp executes every shuffle and wait; lanes
    // past n_active carry no data (whole 16-lane groups, as NA % 16 == 0).
    const int tc = (int)threadIdx.x - 32;
    const int cw = warp - 1;
    const int NA = p.n_active;
    const bool active = tc < NA;

    uint4 wpk[VPT];   // norm weight, packed BF16 pairs
    if (active) {
      const uint4 *wsrc = reinterpret_cast<const uint4 *>(
          static_cast<const uint8_t *>(p.norm_w) + (size_t)col0 * 2u);
#pragma unroll
      for (int v = 0; v < VPT; ++v) wpk[v] = __ldg(wsrc + v * NA + tc);
    } else {
#pragma unroll
      for (int v = 0; v < VPT; ++v) wpk[v] = make_uint4(0u, 0u, 0u, 0u);
    }

    uint32_t it = 0;
    int row_iter = 0;
    for (int r = cid; r < p.T; r += ncl, ++row_iter) {
      float x[VPT][8];
#pragma unroll
      for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int e = 0; e < 8; ++e) x[v][e] = 0.0f;
      bool ok = true;
      for (int i0 = 0; i0 <= p.k; i0 += m, ++it) {
        const int cnt = (p.k + 1 - i0) < m ? (p.k + 1 - i0) : m;
        const uint32_t s = it % (uint32_t)p.nslot;
        const uint32_t ph = (it / (uint32_t)p.nslot) & 1u;
        const bool got = mbar_wait(smem_u32(&full[s]), ph, abort_flag, p.err, kErrBitStage1);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (active) {
          for (int c = 0; c < cnt; ++c) {
            const uint4 *src = reinterpret_cast<const uint4 *>(ring + (size_t)s * slot_bytes +
                                                               (size_t)c * in_bytes);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
              const uint4 d = src[v * NA + tc];
              if (i0 + c == 0) {
                unpack_bf16x8(d, x[v]);
              } else {
                add_bf16x8(x[v], d);   // x += input, element-wise, fp32, in input order
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      }
      if (!ok) break;

      // sum of squares in the canonical order (stage1_math.cuh): each group's
      // leader lane sends the group sum to every CTA of the cluster, and the
      // row total is formed from all G group sums
      const int par = row_iter & 1;
      const uint32_t pph = (uint32_t)((row_iter >> 1) & 1);
      float gsv_[VPT];
#pragma unroll
      for (int v = 0; v < VPT; ++v) gsv_[v] = group_sum16(vec_sumsq(x[v]));   // all lanes
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const float gsv = gsv_[v];
        if (active && (tc & 15) == 0) {
          const int g = (col0 + (v * NA + tc) * 8) / 128;
          if (C > 1) {
            const uint32_t a = smem_u32(&sums->gs[par][g]);
            for (int q = 0; q < C; ++q) {
              st_remote_f32(a, (uint32_t)q, gsv);
              mbar_arrive_remote(smem_u32(&ss_bar[par]), (uint32_t)q);
            }
          } else {
            sums->gs[par][g] = gsv;
          }
        }
      }
      // one CTA: the warp's group sums are ordered before lane 0's release
      // arrival by the warp barrier
      __syncwarp();
      if (C == 1 && lane == 0) mbar_arrive(smem_u32(&ss_bar[par]));
      const bool got_ss =
          C > 1 ? mbar_wait<true>(smem_u32(&ss_bar[par]), pph, abort_flag, p.err, kErrBitStage1)
                : mbar_wait(smem_u32(&ss_bar[par]), pph, abort_flag, p.err, kErrBitStage1);
      if (!__all_sync(0xffffffffu, got_ss)) break;
      const float tot = row_total(sums->gs[par], p.H / 128);
      const float ms = __fdiv_rn(tot, (float)p.H);
      const float rr = __frsqrt_rn(__fadd_rn(ms, p.eps));

      const size_t rowbase = (size_t)r * (size_t)p.H + (size_t)col0;
      uint4 *hid = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.hidden) + rowbase * 2u);
      if constexpr (kFp4) {
        // NVFP4 form (one CTA holds the row): hidden, then the row maximum
        // over the CTA, then per 16-element block (two adjacent lanes) the
        // e4m3 block scale and the e2m1 codes.
        float yv[VPT][8];
        uint32_t hbv[VPT][4];
        float am = 0.0f;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          float wv[8];
          unpack_bf16x8(wpk[v], wv);
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const __nv_bfloat162 h2 =
                __floats2bfloat162_rn(__fmul_rn(__fmul_rn(x[v][e], rr), wv[e]),
                                      __fmul_rn(__fmul_rn(x[v][e + 1], rr), wv[e + 1]));
            const uint32_t hu = *reinterpret_cast<const uint32_t *>(&h2);
            hbv[v][e / 2] = hu;
            yv[v][e] = __uint_as_float(hu << 16);
            yv[v][e + 1] = __uint_as_float(hu & 0xFFFF0000u);
            am = fmaxf(am, fmaxf(fabsf(yv[v][e]), fabsf(yv[v][e + 1])));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) {
          sums->amx[par][cw] = am;
          mbar_arrive(smem_u32(&amx_bar[par]));
        }
        __syncwarp();
        const bool got_am = mbar_wait(smem_u32(&amx_bar[par]), pph, abort_flag, p.err,
                                      kErrBitStage1);
        if (!__all_sync(0xffffffffu, got_am)) break;
        float amax_row = 0.0f;
        for (int q = 0; q < n_cons_warps; ++q) amax_row = fmaxf(amax_row, sums->amx[par][q]);
        const float g = __fdiv_rn(amax_row, 2688.0f);     // 448 * 6
        const float d = __fmul_rn(6.0f, g);
        const bool d_fast = quot_rn_ok(d);
        const float rd = d_fast ? recip_rn(d) : 0.0f;
        uint32_t *cod4 = reinterpret_cast<uint32_t *>(p.codes + rowbase / 2u);
        uint8_t *bsc = p.bscales + (size_t)r * (size_t)(p.H / 16);
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
          float ab = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) ab = fmaxf(ab, fabsf(yv[v][e]));
          ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 1));   // the block's other half
          uint32_t sb;
          const uint32_t packed = fp4_vector_codes(yv[v], ab, g, d, rd, d_fast, sb);
          if (active) {
            const int j = v * NA + tc;
            hid[j] = make_uint4(hbv[v][0], hbv[v][1], hbv[v][2], hbv[v][3]);
            cod4[j] = packed;
            if ((tc & 1) == 0) bsc[j / 2] = (uint8_t)sb;
          }
        }
        if (active && tc == 0) p.gscales[r] = g;
        continue;
      }
      uint2 *cod = reinterpret_cast<uint2 *>(p.codes + rowbase);
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        uint4 hv;
        uint2 cv;
        float scale;
        fp8_vector_epilogue(x[v], wpk[v], rr, hv, cv, scale);   // all lanes (group shuffles)
        if (active) {
          const int j = v * NA + tc;
          hid[j] = hv;
          cod[j] = cv;
          if ((tc & 15) == 0)
            p.scales[(size_t)r * (size_t)(p.H / 128) + (size_t)((col0 + j * 8) / 128)] = scale;
        }
      }
    }
    __syncwarp();
  }

  __syncthreads();
  if (C > 1) cluster_sync_all();   // no CTA leaves while a peer may still write to it
}

// ------------------------------------------------------ small batches --
//
// One row per cluster of R CTAs (R = 1: one CTA per row, no cluster); CTA
// `rank` of the cluster holds E = H / R consecutive channels, E / 8 vectors,
// VPT per thread (vector j in thread j mod NA, slot j / NA: the 16 vectors of
// a group in 16 consecutive lanes).  A CTA handles exactly one row slice, so
// nothing is pipelined across rows: every thread issues all of its 16-byte
// loads at once (the k partials, the residual and the norm weight; up to NB
// inputs per batch), and with T * R CTAs spread over the SMs the whole batch
// is in flight together.  That is what a latency-bound small batch needs: at
// T = 64 one CTA per row would leave most SMs idle and each of the others
// streaming a whole row.
//
// The CTAs of a cluster exchange the row's group sums through distributed
// shared memory: each group's leader lane stores its sum into every CTA's
// gsum[] (after a cluster barrier whose arrive was issued at the start, so
// that every peer has begun), then one cluster barrier publishes them.  The
// NVFP4 form repeats that exchange for the row maximum of |hidden|.  No wait
// is data-dependent: every thread reaches every barrier.
//
// kTma (batches above 96 rows with more than 9 inputs): the slice's k + 1
// inputs are instead copied into shared memory by 1-D bulk copies, all
// requested at once under one mbarrier, and the threads add from there, so
// registers do not split the loads into several rounds.  Two CTAs of up to
// 112 KB of slices fit on an SM.
constexpr int kSplitMaxThreads = 512;

template <int VPT, bool kFp4, bool kTma>
__global__ void __launch_bounds__(kSplitMaxThreads)
    stage1_split_kernel(const Stage1Params p) {
  constexpr int NB = VPT == 1 ? 17 : VPT == 2 ? 9 : 4;   // inputs per batch of loads
  __shared__ float gsum[kMaxGroups];
  __shared__ float gmax[kMaxGroups];
  __shared__ uint64_t in_full;        // kTma: every input slice has landed
  __shared__ uint64_t xch[2];         // R > 1: the row's group sums / maxima have landed
  __shared__ int abort_word;
  extern __shared__ __align__(128) uint8_t in_slices[];   // kTma: [k + 1][E] BF16
  const int R = p.C;
  const uint32_t rank = R > 1 ? cluster_ctarank() : 0u;
  const int r = R > 1 ? (int)cluster_id_x() : (int)blockIdx.x;
  const int E = p.E, G = p.H / 128, NA = p.n_active;
  const int col0 = (int)rank * E;
  const int tc = (int)threadIdx.x;
  const bool active = tc < NA;
  if (kTma || R > 1) {
    if (tc == 0) {
      if (kTma) mbar_init(smem_u32(&in_full), 1);
      if (R > 1) {
        // the exchanges: each group's value arrives from the CTA that holds it
        // as 4 bytes counted on these barriers (st.async)
        mbar_init(smem_u32(&xch[0]), 1);
        mbar_init(smem_u32(&xch[1]), 1);
      }
      abort_word = 0;
      fence_mbarrier_init();
      if (R > 1) {
        mbar_arrive_expect_tx(smem_u32(&xch[0]), (uint32_t)G * 4u);
        if (kFp4) mbar_arrive_expect_tx(smem_u32(&xch[1]), (uint32_t)G * 4u);
      }
    }
    __syncthreads();
  }
  // this CTA has started and its exchange barriers exist (release: the peers
  // see them initialised once their wait returns)
  if (R > 1) cluster_arrive_release();
  // the previous kernel on the stream may write this one's inputs, or still
  // read the buffers this one writes
  grid_dependency_wait();
  grid_launch_dependents();

  const size_t rowv = ((size_t)r * (size_t)p.H + (size_t)col0) / 8u;   // first vector of the slice
  const uint64_t pol = policy_evict_first();
  if constexpr (kTma) {
    if (tc == 0) {
      const uint32_t in_bytes = (uint32_t)E * 2u;
      mbar_arrive_expect_tx(smem_u32(&in_full), in_bytes * (uint32_t)(p.k + 1));
      for (int i = 0; i <= p.k; ++i)
        bulk_g2s(smem_u32(in_slices + (size_t)i * in_bytes),
                 static_cast<const uint4 *>(i < p.k ? p.partials[i] : p.residual) + rowv,
                 in_bytes, smem_u32(&in_full), pol);
    }
  }
  uint4 wpk[VPT];
  const uint4 *wsrc = static_cast<const uint4 *>(p.norm_w) + col0 / 8;
#pragma unroll
  for (int v = 0; v < VPT; ++v)
    wpk[v] = active ? __ldg(wsrc + v * NA + tc) : make_uint4(0u, 0u, 0u, 0u);
  float x[VPT][8];
  if constexpr (kTma) {
    // every thread waits (bounded); after an expired wait the copies still in
    // flight are waited for, again with a limit, and the results are garbage
    // (the device error word says so) but every barrier below is still reached
    if (!mbar_wait(smem_u32(&in_full), 0u, &abort_word, p.err, kErrBitStage1))
      mbar_wait_drain(smem_u32(&in_full), 0u);
    const uint4 *sl = reinterpret_cast<const uint4 *>(in_slices);
    const int vecs = E / 8;
    for (int i = 0; i <= p.k; ++i) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const uint4 d = active ? sl[(size_t)i * vecs + v * NA + tc] : make_uint4(0u, 0u, 0u, 0u);
        if (i == 0) unpack_bf16x8(d, x[v]);
        else add_bf16x8(x[v], d);   // x += input, fp32, in input order
      }
    }
  }
  for (int i0 = 0; i0 <= p.k && !kTma; i0 += NB) {
    uint4 in[NB][VPT];
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const int i = i0 + c;
      const uint4 *src =
          static_cast<const uint4 *>(i < p.k ? p.partials[i < p.k ? i : 0] : p.residual) + rowv;
#pragma unroll
      for (int v = 0; v < VPT; ++v)
        in[c][v] = (active && i <= p.k) ? ld_stream16(src + v * NA + tc, pol)
                                         : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const int i = i0 + c;
      if (i > p.k) break;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (i == 0) unpack_bf16x8(in[c][v], x[v]);
        else add_bf16x8(x[v], in[c][v]);   // x += input, fp32, in input order
      }
    }
  }

  // the row's sum of squares in the canonical order (stage1_math.cuh)
  float lead[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) lead[v] = group_sum16(vec_sumsq(x[v]));   // all lanes
  if (R > 1) cluster_wait();   // every CTA of the cluster has started
  if (active && (tc & 15) == 0) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int g = (col0 + (v * NA + tc) * 8) / 128;
      if (R > 1) {
        for (int q = 0; q < R; ++q)
          st_async_remote_f32(smem_u32(&gsum[g]), smem_u32(&xch[0]), (uint32_t)q, lead[v]);
      } else {
        gsum[g] = lead[v];
      }
    }
  }
  if (R > 1) {
    // all G group sums are in this CTA's gsum once the barrier has counted
    // their bytes; after an expired wait the results are garbage (the device
    // error word says so) but every barrier below is still reached
    mbar_wait(smem_u32(&xch[0]), 0u, &abort_word, p.err, kErrBitStage1);
  } else {
    __syncthreads();
  }
  const float tot = row_total(gsum, G);
  const float ms = __fdiv_rn(tot, (float)p.H);
  const float rr = __frsqrt_rn(__fadd_rn(ms, p.eps));

  uint4 *hid = static_cast<uint4 *>(p.hidden) + rowv;
  if constexpr (kFp4) {
    // hidden, then the row maximum |hidden| over the cluster (group maxima
    // exchanged like the sums), then per 16-element block (two adjacent
    // lanes) the e4m3 block scale and the e2m1 codes
    float yv[VPT][8];
    uint32_t hbv[VPT][4];
    float gm[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      float wv[8];
      unpack_bf16x8(wpk[v], wv);
      float am = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat162 h2 =
            __floats2bfloat162_rn(__fmul_rn(__fmul_rn(x[v][e], rr), wv[e]),
                                  __fmul_rn(__fmul_rn(x[v][e + 1], rr), wv[e + 1]));
        const uint32_t hu = *reinterpret_cast<const uint32_t *>(&h2);
        hbv[v][e / 2] = hu;
        yv[v][e] = __uint_as_float(hu << 16);
        yv[v][e + 1] = __uint_as_float(hu & 0xFFFF0000u);
        am = fmaxf(am, fmaxf(fabsf(yv[v][e]), fabsf(yv[v][e + 1])));
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      gm[v] = am;
    }
    if (active && (tc & 15) == 0) {
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        const int g = (col0 + (v * NA + tc) * 8) / 128;
        if (R > 1) {
          for (int q = 0; q < R; ++q)
            st_async_remote_f32(smem_u32(&gmax[g]), smem_u32(&xch[1]), (uint32_t)q, gm[v]);
        } else {
          gmax[g] = gm[v];
        }
      }
    }
    if (R > 1) mbar_wait(smem_u32(&xch[1]), 0u, &abort_word, p.err, kErrBitStage1);
    else __syncthreads();
    const float amax_row = row_max(gmax, G);
    const float g = __fdiv_rn(amax_row, 2688.0f);     // 448 * 6
    const float d = __fmul_rn(6.0f, g);
    const bool d_fast = quot_rn_ok(d);
    const float rd = d_fast ? recip_rn(d) : 0.0f;
    uint32_t *cod4 = reinterpret_cast<uint32_t *>(p.codes) + rowv;
    uint8_t *bsc = p.bscales + ((size_t)r * (size_t)p.H + (size_t)col0) / 16u;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      float ab = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ab = fmaxf(ab, fabsf(yv[v][e]));
      ab = fmaxf(ab, __shfl_xor_sync(0xffffffffu, ab, 1));   // the block's other half
      uint32_t sb;
      const uint32_t packed = fp4_vector_codes(yv[v], ab, g, d, rd, d_fast, sb);
      if (active) {
        const int j = v * NA + tc;
        hid[j] = make_uint4(hbv[v][0], hbv[v][1], hbv[v][2], hbv[v][3]);
        cod4[j] = packed;
        if ((tc & 1) == 0) bsc[j / 2] = (uint8_t)sb;
      }
    }
    if (active && tc == 0 && rank == 0) p.gscales[r] = g;
  } else {
    uint2 *cod = reinterpret_cast<uint2 *>(p.codes) + rowv;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      uint4 hv;
      uint2 cv;
      float scale;
      fp8_vector_epilogue(x[v], wpk[v], rr, hv, cv, scale);   // all lanes (group shuffles)
      if (active) {
        const int j = v * NA + tc;
        hid[j] = hv;
        cod[j] = cv;
        if ((tc & 15) == 0)
          p.scales[(size_t)r * (size_t)G + (size_t)((col0 + j * 8) / 128)] = scale;
      }
    }
  }
}

// Measurement (not on the path): the loads of stage1_split_kernel alone, in
// the same grid, clusters and per-thread pattern, with no arithmetic beyond a
// checksum and no stores: the floor under the small-batch kernel's time.
__device__ unsigned g_stage1_probe_sink;

template <int VPT>
__global__ void __launch_bounds__(kSplitMaxThreads) stage1_reads_kernel(const Stage1Params p) {
  constexpr int NB = VPT == 1 ? 17 : VPT == 2 ? 9 : 4;
  const int R = p.C;
  const uint32_t rank = R > 1 ? cluster_ctarank() : 0u;
  const int r = R > 1 ? (int)cluster_id_x() : (int)blockIdx.x;
  const int NA = p.n_active;
  const int tc = (int)threadIdx.x;
  const bool active = tc < NA;
  grid_dependency_wait();
  grid_launch_dependents();
  const size_t rowv = ((size_t)r * (size_t)p.H + (size_t)rank * (size_t)p.E) / 8u;
  const uint64_t pol = policy_evict_first();
  // the same loads and fp32 accumulation as stage1_split_kernel
  float x[VPT][8];
  for (int i0 = 0; i0 <= p.k; i0 += NB) {
    uint4 in[NB][VPT];
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const int i = i0 + c;
      const uint4 *src =
          static_cast<const uint4 *>(i < p.k ? p.partials[i < p.k ? i : 0] : p.residual) + rowv;
#pragma unroll
      for (int v = 0; v < VPT; ++v)
        in[c][v] = (active && i <= p.k) ? ld_stream16(src + v * NA + tc, pol)
                                         : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      const int i = i0 + c;
      if (i > p.k) break;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        if (i == 0) unpack_bf16x8(in[c][v], x[v]);
        else add_bf16x8(x[v], in[c][v]);
      }
    }
  }
  float t = 0.0f;
#pragma unroll
  for (int v = 0; v < VPT; ++v)
#pragma unroll
    for (int e = 0; e < 8; ++e) t += x[v][e];
  if (t == 1.2345e-30f) atomicAdd(&g_stage1_probe_sink, 1u);   // keeps the loads
}

}  // namespace

// ------------------------------------------------------------------- host --

namespace {

struct Stage1Choice {
  int C, VPT, NA, threads, nslot, per_slot;
  size_t smem;
};

int g_tune_C = 0, g_tune_vpt = 0, g_tune_slots = 0, g_tune_per_slot = 0, g_tune_ctas = 0;

// ---- small batches: which rows go to stage1_split_kernel, and its shape --

constexpr int kSplitDefaultMaxT = 512;   // largest batch run by the small-batch kernel
int g_split_max_T = -1;                  // tuning: -1 automatic, 0 never, else the limit
int g_split_R = 0, g_split_vpt = 0;      // tuning: 0 automatic
int g_split_tma = -1;                    // tuning: -1 automatic, 0 register loads, 1 bulk copies
constexpr size_t kTmaSliceMax = 112u * 1024u;   // input slices of a CTA: two CTAs per SM

struct SplitChoice {
  int R, VPT, NA, threads, tma;
};

// R CTAs per row and VPT vectors per thread: whole groups per CTA, whole
// 16-lane groups per vector slot, at most kSplitMaxThreads threads.
bool split_shape(int G, int R, int vpt, SplitChoice &c) {
  if (R < 1 || R > 8 || G % R != 0) return false;
  const int gc = G / R;
  if (gc % vpt != 0) return false;
  const int na = 16 * gc / vpt;
  const int threads = (na + 31) / 32 * 32;
  if (threads > kSplitMaxThreads) return false;
  c = SplitChoice{R, vpt, na, threads, 0};
  return true;
}

// R = 0 when the batch goes to the persistent kernel.  The defaults follow a
// CUDA-graph sweep on GB300 (H = 6144 and 7168, k = 8):
//  - T <= 24: one vector per thread, the smallest R with T * R >= 64 (or the
//    largest R): at T = 1 eight CTAs per row take 2.8 us against 3.5 us for one;
//  - T <= 96: one vector per thread, the smallest R with T * R >= 256 (T = 64:
//    R = 4, 4.4 us; one CTA per row with two vectors per thread: 4.5 us);
//  - T <= 160: one CTA per row, two vectors per thread (T = 128: 5.6 us);
//  - T <= 512: one CTA per row, four vectors per thread, so that two CTAs fit
//    on an SM (T = 256: 9.2 us, the persistent kernel 10.5 us);
//  - above: the persistent kernel (T = 1024: 29.0 us against 30.0 us).
// A shape the width does not allow falls back to the next vectors-per-thread
// choice, then to the next R.
SplitChoice choose_split(int T, int H, int k, int num_sms) {
  (void)num_sms;
  SplitChoice none{0, 0, 0, 0, 0};
  const int max_T = g_split_max_T >= 0 ? g_split_max_T : kSplitDefaultMaxT;
  if (T < 1 || T > max_T) return none;
  const int G = H / 128;
  // Above 96 rows with more than 9 inputs (more than a register batch of two
  // vectors a thread): the inputs through shared memory (bulk copies), the
  // smallest R whose slices of the k + 1 inputs leave room for two CTAs an
  // SM.  With k <= 8 the register loads measured as fast or faster (T = 128:
  // 5.6 against 6.1 us; T = 256: 9.4 against 9.1 us; tie stress, k = 4: 7.5
  // against 7.8 us).
  const bool want_tma = g_split_tma >= 0 ? g_split_tma != 0 : (T > 96 && k > 8);
  if (want_tma) {
    const int order[3] = {2, 1, 4};
    for (int R = 1; R <= 8; ++R) {
      if (g_split_R > 0 && R != g_split_R) continue;
      if (G % R != 0 || (size_t)(k + 1) * (size_t)(H / R) * 2u > kTmaSliceMax) continue;
      for (int v : order) {
        if (g_split_vpt > 0 && v != g_split_vpt) continue;
        SplitChoice c = none;
        if (split_shape(G, R, v, c)) {
          c.tma = 1;
          return c;
        }
      }
    }
    if (g_split_tma > 0) return none;   // forced, but no shape fits: the persistent kernel
  }
  int target;   // CTAs the batch should reach
  int order[3];
  if (T <= 24) {
    target = 64; order[0] = 1; order[1] = 2; order[2] = 4;
  } else if (T <= 96) {
    target = 256; order[0] = 1; order[1] = 2; order[2] = 4;
  } else if (T <= 160) {
    target = 1; order[0] = 2; order[1] = 1; order[2] = 4;
  } else {
    target = 1; order[0] = 4; order[1] = 2; order[2] = 1;
  }
  SplitChoice best = none;
  for (int R = 1; R <= 8; ++R) {
    if (g_split_R > 0 && R != g_split_R) continue;
    SplitChoice c = none;
    for (int v : order) {
      if (g_split_vpt > 0 && v != g_split_vpt) continue;
      if (split_shape(G, R, v, c)) break;
      c = none;
    }
    if (!c.R) continue;
    best = c;
    if ((long)T * R >= target) break;
  }
  return best;
}

template <int VPT>
cudaError_t launch_split_vpt(const Stage1Params &p, const SplitChoice &c, cudaStream_t stream) {
  auto kern = c.tma ? (p.fp4 ? stage1_split_kernel<VPT, true, true>
                             : stage1_split_kernel<VPT, false, true>)
                    : (p.fp4 ? stage1_split_kernel<VPT, true, false>
                             : stage1_split_kernel<VPT, false, false>);
  const size_t smem = c.tma ? (size_t)(p.k + 1) * (size_t)p.E * 2u : 0u;
  if (c.tma) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.T * c.R));
  cfg.blockDim = dim3((unsigned)c.threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (c.R > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)c.R;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_split(Stage1Params p, const SplitChoice &c, cudaStream_t stream) {
  p.C = c.R;
  p.E = p.H / c.R;
  p.n_active = c.NA;
  switch (c.VPT) {
    case 1: return launch_split_vpt<1>(p, c, stream);
    case 2: return launch_split_vpt<2>(p, c, stream);
    case 4: return launch_split_vpt<4>(p, c, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

size_t stage1_smem_bytes(int nslot, int per_slot, int E) {
  return (size_t)nslot * (size_t)per_slot * (size_t)E * 2u + (size_t)nslot * 16u + 48u +
         sizeof(RowSums) + 16u;
}

// Vectors per consumer thread for a slice of Gc groups: two where possible (on
// GB300 two vectors a thread beat one and four for both one row per CTA and
// streaming many rows per CTA), whole warps first, within the register budget
// of each variant.
int pick_vpt(int Gc) {
  const int order[8] = {2, 1, 3, 4, 5, 6, 7, 8};   // two vectors per thread measured best
  for (int pass = 0; pass < 2; ++pass)
    for (int v : order) {
      if (Gc % v) continue;
      const int na = 16 * Gc / v;
      if (na + 32 > stage1_max_threads(v)) continue;
      if (pass == 0 && na % 32 != 0) continue;
      return v;
    }
  return 0;
}

Stage1Choice choose_stage1(int T, int H, int k, int num_sms, bool fp4 = false) {
  const int G = H / 128;
  Stage1Choice ch{};
  // one CTA per row slice; a row is split over a cluster only when no single
  // CTA can hold it (very wide H) or when tuning asks for it
  int C = 0, vpt = 0;
  const int opts[4] = {1, 2, 4, 8};
  for (int c : opts) {
    if (G % c) continue;
    if (fp4 && c != 1) continue;           // the NVFP4 row maximum is taken inside one CTA
    if (!fp4 && g_tune_C > 0 && c != g_tune_C) continue;
    int v = 0;
    if (g_tune_vpt > 0 && (G / c) % g_tune_vpt == 0 &&
        16 * (G / c) / g_tune_vpt + 32 <= stage1_max_threads(g_tune_vpt))
      v = g_tune_vpt;
    else
      v = pick_vpt(G / c);
    if (!v) continue;
    C = c;
    vpt = v;
    break;
  }
  if (!C) return ch;   // VPT == 0 signals an unsupported width
  ch.C = C;
  ch.VPT = vpt;
  ch.NA = 16 * (G / C) / vpt;
  ch.threads = 32 + ((ch.NA + 31) / 32) * 32;
  const int E = H / C;
  const size_t in_bytes = (size_t)E * 2u;
  // inputs per slot: a row's k + 1 inputs in as few slots as leave room for
  // two slots in the ring, split evenly (k = 8: two slots of 5 and 4 inputs
  // for H = 6144 and 7168; a CUDA-graph sweep at T = 2048 and 8192 found this
  // 3-5 % faster than three slots of 3, and far faster than smaller slots)
  const size_t budget = 200u * 1024u;
  int per_row = 1;
  while ((k + per_row) / per_row > 1 &&
         2u * in_bytes * (size_t)((k + per_row) / per_row) > budget)
    ++per_row;
  int m = (k + per_row) / per_row;   // ceil((k + 1) / per_row)
  if (g_tune_per_slot > 0) m = g_tune_per_slot < k + 1 ? g_tune_per_slot : k + 1;
  while (m > 1 && 2u * in_bytes * (size_t)m > budget) --m;   // room for two slots
  const int slots_per_row = (k + 1 + m - 1) / m;
  int nslot = (int)(budget / (in_bytes * (size_t)m));
  // slots one CTA fills when the grid covers every SM
  const long clusters = (long)num_sms / C;
  const long rows_each = (T + clusters - 1) / clusters;
  const long total_slots = rows_each * slots_per_row;
  if (nslot > total_slots) nslot = (int)total_slots;
  if (nslot > 64) nslot = 64;
  if (nslot < 2) nslot = 2;
  if (g_tune_slots > 0) nslot = g_tune_slots;
  ch.nslot = nslot;
  ch.per_slot = m;
  ch.smem = stage1_smem_bytes(nslot, m, E);
  return ch;
}

template <int VPT>
cudaError_t launch_vpt(const Stage1Params &p, const Stage1Choice &ch, int grid,
                       cudaStream_t stream) {
  auto kern = p.fp4 ? reduce_norm_quant_kernel<VPT, true> : reduce_norm_quant_kernel<VPT, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)ch.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)ch.threads);
  cfg.dynamicSmemBytes = ch.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ch.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

void stage1_set_grid(int max_ctas) { g_tune_ctas = max_ctas; }

void stage1_set_tuning(int cluster, int vpt, int slots, int per_slot) {
  g_tune_C = cluster;
  g_tune_vpt = vpt;
  g_tune_slots = slots;
  g_tune_per_slot = per_slot;
}

int stage1_plan(int T, int H, int k, int num_sms, int *out7) {
  Stage1Choice ch = choose_stage1(T, H, k, num_sms);
  out7[0] = ch.C;
  out7[1] = ch.VPT;
  out7[2] = ch.NA;
  out7[3] = ch.threads;
  out7[4] = ch.nslot;
  out7[5] = (int)ch.smem;
  out7[6] = ch.per_slot;
  return 0;
}

bool stage1_fp4_supported(int H) {
  return H % 256 == 0 && H >= 256 && H <= 16384 && choose_stage1(1, H, 1, 1, true).VPT != 0;
}

void stage1_set_split(int max_tokens, int ctas_per_row, int vpt, int tma) {
  g_split_max_T = max_tokens;
  g_split_R = ctas_per_row;
  g_split_vpt = vpt;
  g_split_tma = tma;
}

int stage1_split_plan(int T, int H, int k, int num_sms, int *out5) {
  const SplitChoice c = choose_split(T, H, k, num_sms);
  out5[0] = c.R;
  out5[1] = c.VPT;
  out5[2] = c.NA;
  out5[3] = c.threads;
  out5[4] = c.tma;
  return 0;
}

// The small-batch kernel's loads alone, in the grid launch_stage1 would use
// for the small-batch kernel at this size (forced for any T).
cudaError_t launch_stage1_reads(Stage1Params p, int num_sms, cudaStream_t stream) {
  const int saved = g_split_max_T, saved_tma = g_split_tma;
  g_split_max_T = 1 << 30;
  g_split_tma = 0;   // the register-load form: its loads are what the probe mirrors
  const SplitChoice c = choose_split(p.T, p.H, p.k, num_sms);
  g_split_max_T = saved;
  g_split_tma = saved_tma;
  if (c.R == 0) return cudaErrorInvalidConfiguration;
  p.C = c.R;
  p.E = p.H / c.R;
  p.n_active = c.NA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.T * c.R));
  cfg.blockDim = dim3((unsigned)c.threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (c.R > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)c.R;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (unsigned)n;
  switch (c.VPT) {
    case 1: return cudaLaunchKernelEx(&cfg, stage1_reads_kernel<1>, p);
    case 2: return cudaLaunchKernelEx(&cfg, stage1_reads_kernel<2>, p);
    case 4: return cudaLaunchKernelEx(&cfg, stage1_reads_kernel<4>, p);
    default: return cudaErrorInvalidConfiguration;
  }
}

cudaError_t launch_stage1(Stage1Params p, int num_sms, cudaStream_t stream) {
  const SplitChoice sc = choose_split(p.T, p.H, p.k, num_sms);
  if (sc.R > 0) return launch_split(p, sc, stream);
  Stage1Choice ch = choose_stage1(p.T, p.H, p.k, num_sms, p.fp4 != 0);
  if (ch.VPT == 0) return cudaErrorInvalidConfiguration;
  p.C = ch.C;
  p.E = p.H / ch.C;
  p.nslot = ch.nslot;
  p.per_slot = ch.per_slot;
  p.n_active = ch.NA;
  // persistent grid: at most one CTA per SM, whole clusters, no more rows than exist
  long clusters = num_sms / ch.C;
  if (g_tune_ctas > 0 && g_tune_ctas / ch.C >= 1 && g_tune_ctas / ch.C < clusters)
    clusters = g_tune_ctas / ch.C;
  if (clusters > p.T) clusters = p.T;
  if (clusters < 1) clusters = 1;
  const int grid = (int)(clusters * ch.C);
  switch (ch.VPT) {
    case 1: return launch_vpt<1>(p, ch, grid, stream);
    case 2: return launch_vpt<2>(p, ch, grid, stream);
    case 3: return launch_vpt<3>(p, ch, grid, stream);
    case 4: return launch_vpt<4>(p, ch, grid, stream);
    case 5: return launch_vpt<5>(p, ch, grid, stream);
    case 6: return launch_vpt<6>(p, ch, grid, stream);
    case 7: return launch_vpt<7>(p, ch, grid, stream);
    case 8: return launch_vpt<8>(p, ch, grid, stream);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace nfq
