// Internal interfaces between the C ABI layer (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace nfq {

constexpr int kMaxPartials = 16;
constexpr int kMaxShards = 64;          // vocabulary shards of one LM-head call
constexpr int kArgmaxKeysPerShard = 256; // argmax keys per shard: one per token of a launch

// Bytes of the LM head's scratch for S shards: S x 256 packed 64-bit argmax
// keys, then a 16-byte block holding the CTA-done counter (and the fused
// step's row counter).
__host__ __device__ constexpr size_t stage2_workspace_bytes_for(int S) {
  return (size_t)S * kArgmaxKeysPerShard * 8u + 16u;
}

// Stage 1 launch parameters (passed by value to the kernel).
struct Stage1Params {
  const void *partials[kMaxPartials];  // k BF16 [T][H]
  const void *residual;                // BF16 [T][H]
  const void *norm_w;                  // BF16 [H]
  void *hidden;                        // BF16 [T][H]
  uint8_t *codes;                      // e4m3 [T][H], or NVFP4 e2m1 pairs [T][H/2]
  float *scales;                       // fp32 [T][H/128] (FP8 form)
  uint8_t *bscales;                    // e4m3 [T][H/16] (NVFP4 form)
  float *gscales;                      // fp32 [T] (NVFP4 form)
  unsigned *err;                       // device error word
  float eps;
  int k, T, H;
  int C;          // CTAs per cluster (channel split of a row)
  int E;          // channels per CTA = H / C
  int nslot;      // shared-memory ring slots
  int per_slot;   // inputs (E BF16 values each) per ring slot
  int n_active;   // consumer threads holding data
  int fp4;        // 1: NVFP4 activation (codes, bscales, gscales), 0: FP8 (codes, scales)
};

cudaError_t launch_stage1(Stage1Params p, int num_sms, cudaStream_t stream);
void stage1_set_tuning(int cluster, int vpt, int slots, int per_slot);
void stage1_set_grid(int max_ctas);   // 0: one CTA (cluster) per SM at most
// Small batches: batches of at most max_tokens rows (-1: the default limit, 0:
// none) run one row per cluster of ctas_per_row CTAs (0: automatic) with vpt
// vectors per thread (0: automatic), the inputs loaded into registers (tma 0)
// or copied into shared memory (tma 1; -1: automatic).
void stage1_set_split(int max_tokens, int ctas_per_row, int vpt, int tma);
int stage1_split_plan(int T, int H, int k, int num_sms, int *out5);
// Measurement: the small-batch kernel's loads alone (its grid at this size).
cudaError_t launch_stage1_reads(Stage1Params p, int num_sms, cudaStream_t stream);
int stage1_plan(int T, int H, int k, int num_sms, int *out7);
bool stage1_fp4_supported(int H);

// Stage 1 folded into the LM-head launch (the fused step): the epilogue warps
// of CTA r < T compute row r and publish it through `ready`.
struct FusedStage1 {
  const void *partials[kMaxPartials];  // k BF16 [T][H]
  const void *residual;                // BF16 [T][H]
  const void *norm_w;                  // BF16 [H]
  void *hidden;                        // BF16 [T][H]
  uint8_t *codes;                      // the activation the LM head reads (act_codes)
  float *scales;                       // (act_scales)
  unsigned *ready;                     // workspace word: rows published (reset by the last CTA)
  float eps;
  int k;
  int na;                              // threads holding data: H / 16 (two vectors each)
};

// Stage 2 launch parameters.
struct Stage2Params {
  const uint8_t *act_codes;   // e4m3 [T][H]   (this launch's token chunk)
  const float *act_scales;    // fp32 [T][G]
  const float *w_scales;      // fp32 [ceil(V/128)][G]
  const uint8_t *w_packed;    // tile-contiguous weight blocks, or null for row-major [V][H]
  int32_t *tokens_out;        // [T]
  float *max_logit_out;       // [T] or null
  int32_t *shard_idx_out;     // [S][T_total] or null, column offset tok0
  float *shard_val_out;       // [S][T_total] or null
  unsigned long long *keys;   // workspace [S][NPAD] packed (value, index) maxima
  unsigned *counter;          // workspace: CTAs finished
  unsigned *err;              // device error word
  int T;                      // tokens in this launch (<= 256)
  int T_total;                // row stride of the per-shard outputs
  int tok0;                   // first token of this chunk
  int H, G, V, S;
  int shard_width;            // V / S
  int n_vtiles;               // ceil(V / 128)
  int n_groups;               // token-major form: token groups of 128 (1 or 2), set at launch
  uint16_t *logits_out;       // unfused arm: BF16 logits [T][V] instead of the argmax
  FusedStage1 s1;             // the fused step (s1.ready != null)
  // NVFP4 form: act_codes are e2m1 pairs [T][H/2], G = H / 256 (K steps)
  const uint8_t *act_bscales; // e4m3 [T][H/16]
  const float *act_gscales;   // fp32 [T]
  float w_scale;              // the weight's tensor scale
};

cudaError_t launch_stage2(const Stage2Params &p, const void *act_codes_base, const void *w,
                          int num_sms, cudaStream_t stream);

size_t stage2_workspace_bytes(int S);
void stage2_set_small(int enabled);   // 0: always use the wide-batch kernel (tests, tuning)
void stage2_set_pair(int enabled);    // 0: 129..256 tokens as two independent token groups
int stage2_token_chunk();             // tokens per LM-head launch
size_t packed_weight_bytes(int V, int H);
cudaError_t launch_pack_weights(const uint8_t *w, int V, int H, uint8_t *out, cudaStream_t stream);

// Unfused reference arm: the FP8 LM head writing BF16 logits (packed weight,
// T <= 128 per launch), and the separate kernels of the unfused path.
cudaError_t launch_lm_head_logits(const Stage2Params &p, int num_sms, cudaStream_t stream);
// The fused FP8 step (stage 1 inside the token-major LM head), when it applies.
bool fused_step_supported(int T, int H, int k, int V, int num_sms);
cudaError_t launch_fused_step(const Stage2Params &p, int num_sms, cudaStream_t stream);
struct UnfusedReduceParams {
  const void *partials[kMaxPartials];
  int k;
  size_t n_vec;                        // 16-byte vectors per tensor
  void *out;
};
cudaError_t launch_unfused_reduce(const UnfusedReduceParams &p, int num_sms, cudaStream_t stream);
cudaError_t launch_unfused_add_rmsnorm(const void *x, const void *residual, const void *norm_w,
                                       float eps, int T, int H, void *hidden,
                                       cudaStream_t stream);
cudaError_t launch_unfused_quant(const void *hidden, int T, int H, uint8_t *codes,
                                 float *scales, cudaStream_t stream);
cudaError_t launch_unfused_argmax(const void *logits, int T, int V, int32_t *tokens,
                                  cudaStream_t stream);

// NVFP4 LM head (token-major, block-scaled tensor cores): up to 128 tokens per
// token group, two groups (256 tokens) per launch
constexpr int kFp4MaxT = 128;
constexpr int kFp4LaunchMaxT = 2 * kFp4MaxT;
cudaError_t launch_stage2_fp4(const Stage2Params &p, int num_sms, cudaStream_t stream);
void stage2_fp4_set_stages(int n);   // 0: as many pipeline stages as fit
size_t fp4_packed_weight_bytes(int V, int H);
cudaError_t launch_pack_fp4_weights(const uint8_t *codes, const uint8_t *bscales, int V, int H,
                                    uint8_t *out, cudaStream_t stream);

// Measurement: `ctas` CTAs (pair: CTA pairs) each issue `iters` K blocks of
// four FP8 MMAs from shared memory (probe.cu).
cudaError_t launch_probe_fp8_mma(int pair, int ctas, int iters, unsigned *err, cudaStream_t stream);
// Measurement: `ctas` CTAs of 16 warps each read 64 TMEM columns x 32 lanes
// per warp, `iters` times (probe.cu).
cudaError_t launch_probe_tmem_ld(int batched, int ctas, int iters, cudaStream_t stream);

}  // namespace nfq
