/*
 * nfq.h — C ABI of the GB300 (sm_103a) MTP draft-layer tail.
 *
 * Two operations, each one asynchronous launch sequence on a caller stream:
 *
 *   nfq_mtp_reduce_norm_quant   k BF16 partial sums + residual -> RMSNorm ->
 *                               (BF16 hidden, packed FP8 activation)
 *   nfq_lm_head_fp8_argmax      packed FP8 activation x block-scaled FP8 LM
 *                               head -> greedy draft token per row, via a
 *                               vocab-sharded argmax; logits are never stored
 * and their NVFP4 variants (…_nvfp4), which carry the activation and the
 * weight in the NVFP4 format and use the tensor cores' block scaling.
 *
 * Sources (page title, section):
 *   [R] "[Quant][MTP] Reuse packed FP8 logits inputs" (vLLM pull request 51947),
 *       Purpose and Dependencies.
 *   [F] "[Spec Decode][Perf] Fuse the MTP trailing all-reduce; local-argmax
 *       draft tokens" (vLLM pull request 49793), intro bullets, Benchmarks and
 *       Accuracy.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers unless stated otherwise; the caller
 *    owns every buffer.  The library never allocates device memory, never frees
 *    and never synchronises (except nfq_device_error, which says so).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous on it; results are valid once the stream
 *    has reached the call.
 *  - Every argument is validated on the host before anything is launched; the
 *    first violation is returned and nothing runs.  Launch failures return
 *    NFQ_ERR_CUDA.  No C++ exception crosses this boundary.
 *  - Tensor values are not inspected: NaN or infinite inputs give unspecified
 *    (but memory-safe) results.
 *  - Row-major layouts throughout.  Every device pointer must be 16-byte aligned,
 *    except the LM head's int32 / fp32 per-token outputs (4-byte aligned).
 *  - Kernels are launched with programmatic stream serialisation: a launch may
 *    begin while the previous kernel on the stream is finishing, and waits for
 *    it before it touches that kernel's outputs.  The LM-head calls read the
 *    LM-head weight (FP8 codes, or NVFP4 codes and block scales) before that
 *    wait: the weight is a constant, which the kernel immediately preceding an
 *    LM-head call must not write.  The pack calls below end with an ordering
 *    point that makes their output safe to use right away; a weight written by
 *    another kernel needs an event or a synchronisation before the LM head.
 */
#ifndef NFQ_H_
#define NFQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NFQ_OK = 0,
  NFQ_ERR_NULL = -1,       /* a required pointer is NULL                       */
  NFQ_ERR_SHAPE = -2,      /* a size is out of range or inconsistent           */
  NFQ_ERR_ALIGN = -3,      /* a device pointer is not 16-byte aligned          */
  NFQ_ERR_WORKSPACE = -4,  /* the workspace is missing or too small            */
  NFQ_ERR_CUDA = -5,       /* a CUDA runtime call or launch failed             */
  NFQ_ERR_TIMEOUT = -6,    /* a kernel gave up a bounded wait (nfq_device_error) */
  NFQ_ERR_DEVICE = -7      /* the current device is not sm_103 / sm_100 class  */
} nfq_status;

/* Packed FP8 QuantizedActivation ([R] Purpose: the draft layer's first output,
 * consumed by the LM head without unpacking or requantising it).
 *   codes  : e4m3fn bytes [tokens][hidden]
 *   scales : fp32 [tokens][hidden / group]; element (t, h) represents
 *            decode(codes[t][h]) * scales[t][h / group]
 *   group  : must be 128 (one scale per 1x128 token group)            */
typedef struct {
  uint8_t *codes;
  float *scales;
  int32_t tokens;
  int32_t hidden;
  int32_t group;
} nfq_quant_act;

/* Human-readable name of a status code (static string, never NULL). */
const char *nfq_status_str(int status);

/* ABI version: (major << 16) | minor. */
int nfq_abi_version(void);

/*
 * Stage 1 — fused trailing all-reduce + residual + final RMSNorm + packed FP8.
 * [R] Purpose: the MTP layer's final all-reduce and RMSNorm are fused with
 * packed FP8 quantisation, and the layer returns two deliberately different
 * values: the packed activation for the logits projection and the post-norm
 * BF16 hidden state recycled into the next MTP position.  [F] intro: the
 * trailing all-reduce is fused into the final RMSNorm.  [F] Accuracy: the fused
 * kernel accumulates in fp32.
 *
 * On one GPU the tensor-parallel partial outputs are k BF16 tensors in HBM and
 * the all-reduce is their sum.  For every token t and channel h:
 *   x      = ((p_0 + p_1) + ... + p_{k-1}) + residual      fp32, this order
 *   hidden = bf16_rne( x * rsqrt(mean_h(x^2) + eps) * w )
 *   per 128-channel group g: scale = max_g |hidden| / 448  (fp32 division)
 *   code   = e4m3fn_rne_satfinite(hidden / scale), 0 when scale == 0
 *
 *   partials   HOST array of k device pointers, each BF16 [T][H]
 *   k          1..16
 *   residual   BF16 [T][H]
 *   norm_w     BF16 [H]
 *   eps        added to mean(x^2); must be >= 0 (the MTP layers use 1e-6)
 *   T, H       T >= 1 (T == 0 is a no-op returning NFQ_OK), H % 128 == 0,
 *              128 <= H <= 32768
 *   hidden_out BF16 [T][H]; must not overlap any input
 *   q_out      host struct; q_out->codes [T][H], q_out->scales [T][H/128];
 *              q_out->tokens == T, q_out->hidden == H, q_out->group == 128
 * Bounded waits inside the kernel that expire set the device error word read
 * by nfq_device_error.
 */
int nfq_mtp_reduce_norm_quant(const void *const *partials, int k, const void *residual,
                              const void *norm_w, float eps, int T, int H, void *hidden_out,
                              const nfq_quant_act *q_out, void *stream);

/*
 * Stage 2 — shared LM head on the prequantised activation, greedy draft token.
 * [R] Dependencies: the LM-head GEMM consumes prequantised activations (block
 * linear, prequantised-input contract).  [F] intro: greedy draft tokens come
 * from a vocab-parallel local argmax, skipping the full-vocab all-gather of the
 * logits; [F] Benchmarks: at 64 tokens that gather is 64 x 151k x 2 bytes per
 * draft step.  [F] Accuracy: local argmax changes how ties at shard boundaries
 * are broken; here every tie goes to the lowest global vocab index.
 *
 *   L[t][v] = sum_k decode(a.codes[t][k]) * a.scales[t][k/128]
 *                 * decode(w[v][k]) * w_scales[v/128][k/128]     (fp32 accumulate)
 * The V vocab rows form S equal shards [s*V/S, (s+1)*V/S).  Outputs:
 *   tokens_out    int32 [T]    argmax_v L[t][v], lowest index among equal maxima; may
 *                              also be pinned host memory that the device addresses
 *                              directly (unified addressing): the tokens are then
 *                              written straight to the host by the kernel's last CTA
 *   max_logit_out fp32 [T]     L at that index, or NULL
 *   shard_idx_out int32 [S][T] per-shard argmax (global index), or NULL
 *   shard_val_out fp32 [S][T]  per-shard maximum, or NULL
 * A -0 logit compares equal to +0 (the value reported is +0).  The full [T][V]
 * logits are never written to memory.
 *
 *   a          host struct describing the activation (group == 128, hidden % 128 == 0)
 *   w          e4m3fn [V][H], H = a->hidden
 *   w_scales   fp32 [ceil(V/128)][H/128]
 *   V, S       V >= 1, 1 <= S <= 64, V % S == 0
 *   workspace  device scratch of at least nfq_lm_head_workspace_bytes(T, S) bytes.
 *              It must be zero-filled before its first use (nfq_lm_head_workspace_init);
 *              every call returns it to all-zero, so one zeroing suffices for
 *              any number of calls that run one after another on a stream.
 *              Concurrent calls need separate workspaces.
 * T = a->tokens may be any size >= 1; rows are processed 256 at a time, and
 * each such chunk streams the weights from HBM once.
 */
size_t nfq_lm_head_workspace_bytes(int T, int S);

int nfq_lm_head_workspace_init(void *workspace, size_t ws_bytes, void *stream);

int nfq_lm_head_fp8_argmax(const nfq_quant_act *a, const uint8_t *w, const float *w_scales,
                           int V, int S, int32_t *tokens_out, float *max_logit_out,
                           int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                           size_t ws_bytes, void *stream);

/*
 * Packed LM-head weight: the same e4m3 bytes re-laid for streaming.  The
 * row-major [V][H] weight is cut into blocks of 128 vocab rows x 128 columns
 * (the 128x128 scale blocks); block (vt, kb) is stored contiguously at byte
 * offset (vt * H/128 + kb) * 16384, row r of the block at r * 128, and within
 * a row the 16-byte chunk c at chunk position c XOR (r mod 8) (the 128-byte
 * shared-memory swizzle the tensor cores read).  Rows past V are zero.  Each
 * K step of the LM head then fetches one contiguous 16 KB block.
 *
 * nfq_lm_head_packed_bytes: size of the packed weight, ceil(V/128) * H * 128
 *   bytes (0 for invalid sizes).
 * nfq_lm_head_pack_weights: one kernel on `stream` that writes w_packed from w
 *   (device pointers, 16-byte aligned, no overlap).  Done once per weight;
 *   errors as for the calls above (NFQ_ERR_WORKSPACE if packed_bytes is short).
 * nfq_lm_head_fp8_argmax_packed: nfq_lm_head_fp8_argmax with the weight given
 *   in the packed layout; identical results.
 */
size_t nfq_lm_head_packed_bytes(int V, int H);

int nfq_lm_head_pack_weights(const uint8_t *w, int V, int H, uint8_t *w_packed,
                             size_t packed_bytes, void *stream);

int nfq_lm_head_fp8_argmax_packed(const nfq_quant_act *a, const uint8_t *w_packed,
                                  const float *w_scales, int V, int S, int32_t *tokens_out,
                                  float *max_logit_out, int32_t *shard_idx_out,
                                  float *shard_val_out, void *workspace, size_t ws_bytes,
                                  void *stream);

/*
 * Reads the current device's error word that kernels set when a bounded wait
 * expires (bit 0: stage 1, bit 1: stage 2).  SYNCHRONISES the current device.
 * Returns NFQ_OK when clear, NFQ_ERR_TIMEOUT when set (and clears it when
 * `clear` != 0), NFQ_ERR_CUDA if the device cannot be read.
 */
int nfq_device_error(int clear);

/*
 * nfq_mtp_draft_chain — `positions` chained MTP draft steps on one stream.
 * [R] Purpose: the post-final-norm BF16 hidden state is recycled into the next
 * MTP position; [F] Benchmarks: the draft runs five positions per accepted
 * token (MTP=5).  Position p runs nfq_mtp_reduce_norm_quant on its k partials
 * with residual = residual0 (p = 0) or the hidden of position p-1, writing
 * hidden_out[p], then the LM head on the packed activation, writing
 * tokens_out[p][0..T).  (The transformer block that turns a draft token into
 * the next position's partials is not part of this library: the caller
 * supplies every position's partials.)
 *   positions   1..64
 *   partials    HOST array [positions][k] of device pointers, BF16 [T][H] each
 *   hidden_out  HOST array [positions] of device pointers, BF16 [T][H]; buffers of
 *               consecutive positions must differ (two alternating buffers do)
 *               and none may be residual0
 *   q           the packed activation buffer, reused by every position
 *   w, w_is_packed  LM-head weight, row-major (0) or packed (1)
 *   tokens_out  int32 [positions][T]
 *   workspace   as for nfq_lm_head_fp8_argmax (one suffices for the chain)
 * Errors are those of the two calls; the first failing position stops the chain.
 */
int nfq_mtp_draft_chain(int positions, const void *const *partials, int k,
                        const void *residual0, const void *norm_w, float eps, int T, int H,
                        void *const *hidden_out, const nfq_quant_act *q, const uint8_t *w,
                        int w_is_packed, const float *w_scales, int V, int S,
                        int32_t *tokens_out, void *workspace, size_t ws_bytes, void *stream);

/*
 * nfq_lm_head_fp8_argmax_noalloc — the same LM head and argmax, for callers
 * that cannot allocate device memory: code that runs where cudaMalloc is not
 * allowed or not wanted (inside a host engine that hands out only fixed
 * buffers, or a decode loop that must not hit the allocator, which may
 * synchronise the device).  The source pages have no counterpart to this call.
 *
 * Instead of a caller workspace it uses a scratch array of 131,088 bytes that
 * the library keeps in device memory for the life of the process on every GPU
 * that loads it.  That is the workspace of the largest shard count any LM-head
 * call accepts (64); S outside 1..64 returns NFQ_ERR_SHAPE, as it does for
 * nfq_lm_head_fp8_argmax.  It allocates nothing and frees nothing.  Arguments,
 * outputs and errors are those of nfq_lm_head_fp8_argmax minus the workspace.
 * - Every argument is checked before the array is touched: a rejected call
 *   queues nothing.
 * - The first call on a device looks up the array's device address for that
 *   device (the current one); make that first call before any stream capture.
 * - Each call clears the part of the array it uses with an asynchronous memset
 *   on `stream`, then launches the LM head on `stream`.
 * - All calls on a device share the one array: calls that overlap on the GPU
 *   (different streams, no ordering between them) race and give wrong results.
 *   Calls ordered on one stream are safe.
 */
int nfq_lm_head_fp8_argmax_noalloc(const nfq_quant_act *a, const uint8_t *w,
                                   const float *w_scales, int V, int S, int32_t *tokens_out,
                                   float *max_logit_out, int32_t *shard_idx_out,
                                   float *shard_val_out, void *stream);

/*
 * NVFP4 variant of both stages.  [F] Benchmarks serve an NVFP4 checkpoint
 * (GLM-5.2-NVFP4); the pages define no FP4 arithmetic, so the published NVFP4
 * format is used: OCP FP4 e2m1 values, one unsigned e4m3 scale per 16
 * consecutive hidden elements, and one fp32 scale per row (per token for the
 * activation, per tensor for the weight) so that a row's largest block scale is
 * 448.  Element (t, h) represents
 *   e2m1(codes[t][h/2] nibble h%2) * e4m3(block_scales[t][h/16]) * row_scales[t]
 * with element 2i in the low nibble of byte i.
 *   codes        uint8 [tokens][hidden/2]
 *   block_scales uint8 [tokens][hidden/16]   (unsigned e4m3 codes, < 0x80)
 *   row_scales   fp32  [tokens]
 *   block        must be 16
 */
typedef struct {
  uint8_t *codes;
  uint8_t *block_scales;
  float *row_scales;
  int32_t tokens;
  int32_t hidden;
  int32_t block;
} nfq_fp4_act;

/*
 * nfq_mtp_reduce_norm_quant_nvfp4 — stage 1 with the NVFP4 activation instead
 * of the packed FP8 one; the reduction, residual, RMSNorm and BF16 hidden are
 * those of nfq_mtp_reduce_norm_quant (same arguments and rules).  Per token:
 *   g    = max_h |hidden| / (448 * 6)                            fp32
 *   per block b of 16: sb = e4m3_rne_satfinite(max_b |hidden| / (6 * g)), 0 when g == 0
 *   eff  = e4m3(sb) * g;  code = e2m1_rne_satfinite(hidden / eff), 0 when eff == 0
 *   q_out  codes [T][H/2], block_scales [T][H/16], row_scales [T];
 *          q_out->tokens == T, q_out->hidden == H, q_out->block == 16
 *   H      H % 256 == 0 and 256 <= H <= 16384 (one CTA holds a row)
 */
int nfq_mtp_reduce_norm_quant_nvfp4(const void *const *partials, int k, const void *residual,
                                    const void *norm_w, float eps, int T, int H,
                                    void *hidden_out, const nfq_fp4_act *q_out, void *stream);

/*
 * NVFP4 LM-head weight in the streaming layout, built once from the row-major
 * codes [V][H/2] and block scales [V][H/16].  Rows are cut into blocks of 128
 * and the hidden dimension into steps of 256 elements (128 code bytes, 16 block
 * scales).  The packed buffer holds ceil(V/128) * (H/256) code blocks of 16 KB
 * (block (vt, s) at (vt * H/256 + s) * 16384; row r at r * 128, 16-byte chunk c
 * at chunk position c XOR (r mod 8)) followed by as many 2 KB scale blocks
 * (block (vt, s) at the same index * 2048 after the codes): word (kk, i, c) at
 * ((kk * 32 + i) * 4 + c) * 4 holds the scales of the four 16-element blocks
 * 4kk .. 4kk+3 of step s for row 32c + i, one byte each, lowest block first.
 * Rows past V are zero.
 * nfq_lm_head_nvfp4_packed_bytes: ceil(V/128) * (H/256) * 18432 (0 if invalid;
 *   H % 256 == 0).
 * nfq_lm_head_nvfp4_pack_weights: one kernel on `stream`; device pointers,
 *   16-byte aligned, no overlap; NFQ_ERR_WORKSPACE if packed_bytes is short.
 */
size_t nfq_lm_head_nvfp4_packed_bytes(int V, int H);

int nfq_lm_head_nvfp4_pack_weights(const uint8_t *codes, const uint8_t *block_scales, int V,
                                   int H, void *w_packed, size_t packed_bytes, void *stream);

/*
 * nfq_lm_head_nvfp4_argmax — the LM head and argmax of nfq_lm_head_fp8_argmax
 * on the NVFP4 activation and the packed NVFP4 weight (tensor scale w_scale):
 *   L[t][v] = (sum_b e4m3(a.block_scales[t][b]) * e4m3(w_block_scales[v][b])
 *                  * sum_{j<16} e2m1(a[t][16b+j]) * e2m1(w[v][16b+j]))
 *             * (a.row_scales[t] * w_scale)
 * The block-scaled products are summed by the tensor cores in fp32.  Outputs,
 * shards, ties, workspace and errors as for nfq_lm_head_fp8_argmax; V >= 1,
 * H % 256 == 0; rows are processed 128 tokens at a time.
 */
int nfq_lm_head_nvfp4_argmax(const nfq_fp4_act *a, const void *w_packed, float w_scale, int V,
                             int S, int32_t *tokens_out, float *max_logit_out,
                             int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                             size_t ws_bytes, void *stream);

/*
 * nfq_mtp_step_fp8 — one whole draft step: nfq_mtp_reduce_norm_quant followed by
 * nfq_lm_head_fp8_argmax_packed, with the same arguments, rules, outputs (the
 * hidden, the packed activation in q, the tokens and the optional maxima) and
 * the same results bit for bit.  Where it applies (1 <= T <= 64, H % 512 == 0,
 * H <= 8192, at least T CTAs in the LM head's grid) it is ONE launch: the
 * LM-head kernel's epilogue warps compute stage 1 for one token row per CTA
 * while its producer already streams the first weight stages, and the MMAs
 * start once every row is published through a counter in the workspace (the
 * counter returns to zero with the rest of the workspace).  Otherwise it is
 * the two launches.  Requires the packed weight (nfq_lm_head_pack_weights).
 */
int nfq_mtp_step_fp8(const void *const *partials, int k, const void *residual,
                     const void *norm_w, float eps, int T, int H, void *hidden_out,
                     const nfq_quant_act *q, const uint8_t *w_packed, const float *w_scales,
                     int V, int S, int32_t *tokens_out, float *max_logit_out,
                     int32_t *shard_idx_out, float *shard_val_out, void *workspace,
                     size_t ws_bytes, void *stream);

/*
 * nfq_mtp_draft_chain_nvfp4 — nfq_mtp_draft_chain with the NVFP4 forms of both
 * stages: q is the NVFP4 activation buffer reused by every position, w_packed
 * the packed NVFP4 weight with its tensor scale w_scale.  Rules and errors as
 * for nfq_mtp_draft_chain and the two NVFP4 calls.
 */
int nfq_mtp_draft_chain_nvfp4(int positions, const void *const *partials, int k,
                              const void *residual0, const void *norm_w, float eps, int T, int H,
                              void *const *hidden_out, const nfq_fp4_act *q,
                              const void *w_packed, float w_scale, int V, int S,
                              int32_t *tokens_out, void *workspace, size_t ws_bytes,
                              void *stream);

/*
 * The unfused reference arm: the same step as separate kernels, the way it runs
 * without the two fusions of [F] (intro, Accuracy): the trailing all-reduce as a
 * separate BF16 collective (here the BF16-rounded sum of the partials), then
 * add + RMSNorm, then the group quantisation, then an LM head that writes the
 * full BF16 logits, then a full-vocab argmax ([F] Benchmarks: the gathered
 * logits are 64 x 151k x 2 bytes per draft step at c=64).  For measuring what
 * the fused path saves; arguments follow the fused calls.
 *   nfq_unfused_allreduce_bf16  out = bf16(p_0 + ... + p_{k-1}), fp32 sum in order,
 *                               out BF16 [T][H]; H % 8 == 0
 *   nfq_unfused_add_rmsnorm     hidden = bf16((x + residual) * rsqrt(mean(.^2) + eps) * w)
 *                               for BF16 x, residual [T][H]; 128 <= H <= 16384
 *   nfq_unfused_quant_fp8       the packed FP8 quantisation of stage 1 applied to a
 *                               BF16 hidden [T][H]
 *   nfq_unfused_lm_head_logits  BF16 logits [T][V] (round to nearest even of the fp32
 *                               logit) from the activation and the packed FP8 weight
 *                               (nfq_lm_head_pack_weights) with its block scales
 *   nfq_unfused_argmax_bf16     tokens_out[t] = lowest index of the maximum of the BF16
 *                               logits row t (-0 == +0)
 */
int nfq_unfused_allreduce_bf16(const void *const *partials, int k, int T, int H, void *out,
                               void *stream);
int nfq_unfused_add_rmsnorm(const void *x, const void *residual, const void *norm_w, float eps,
                            int T, int H, void *hidden_out, void *stream);
int nfq_unfused_quant_fp8(const void *hidden, int T, int H, const nfq_quant_act *q_out,
                          void *stream);
int nfq_unfused_lm_head_logits(const nfq_quant_act *a, const uint8_t *w_packed,
                               const float *w_scales, int V, void *logits_out, void *stream);
int nfq_unfused_argmax_bf16(const void *logits, int T, int V, int32_t *tokens_out,
                            void *stream);

/*
 * Tuning hooks (process-wide, not thread-safe; for benchmarks and tests).
 * nfq_stage1_plan: the stage-1 launch plan for (T, H, k) on a GPU with
 *   num_sms SMs: out7 = {cluster CTAs per row, 16-byte vectors per thread,
 *   active consumer threads, block threads, ring slots, shared bytes,
 *   inputs per ring slot}.
 * nfq_stage1_tune: force the cluster size, vectors per thread, ring slots and
 *   inputs per slot of later stage-1 launches (0 = automatic; invalid choices
 *   fall back).
 * nfq_lm_head_small_batch: 1 (default) runs the FP8 LM head on the token-major
 *   kernels (up to 256 tokens per launch); 0 forces the weight-major kernel for
 *   every batch size.
 * nfq_lm_head_pair: 1 (default) runs 129..256 tokens of the FP8 and the NVFP4
 *   LM heads on CTA pairs that issue cta_group::2 MMAs (M = 256 tokens, each
 *   CTA holding half of the weight tile); 0 runs them as two independent
 *   128-token groups over one weight stream.  The results are the same either
 *   way.
 * nfq_lm_head_nvfp4_tune: pipeline stages of later NVFP4 LM-head launches
 *   (0 = as many as fit, at most 5; values below 2, or below 4 for the CTA-pair
 *   form of 129..256 tokens, or above what fits fall back).
 * nfq_stage1_grid: at most max_ctas CTAs for later stage-1 launches, each then
 *   taking several rows in turn (0 = one CTA per SM at most).
 * nfq_stage1_split: batches of at most max_tokens rows (-1 = the default
 *   limit, 0 = no batch) run on the small-batch stage-1 kernel, one row per
 *   cluster of ctas_per_row CTAs (0 = automatic) with vpt 16-byte vectors per
 *   thread (0 = automatic), its inputs loaded into registers (tma = 0) or
 *   copied into shared memory by bulk copies (tma = 1; -1 = automatic);
 *   larger batches run on the persistent kernel that nfq_stage1_plan
 *   describes.  The results are the same bits either way.
 * nfq_probe_fp8_mma: a measurement kernel, not part of the path.  `ctas`
 *   CTAs (pair != 0: `ctas` CTA pairs issuing cta_group::2 MMAs) each issue
 *   `iters` K blocks of four back-to-back tcgen05.mma kind::f8f6f4 from zeroed
 *   shared-memory tiles, M = 128 (pairs: 256) x N = 256 x K = 32 each, into
 *   TMEM; 2 * M * 256 * 128 * iters flops per CTA (per pair).  K block i reads
 *   the tiles of set i % stages (1..4 sets: with more than one, every K block
 *   reads operands the previous one did not).  stages = 0 (one CTA, not
 *   pairs): one operand set, while 16 other warps of the CTA read TMEM with
 *   the LM head epilogue's pattern until the MMAs are done.  Asynchronous on
 *   `stream`; time it with events.  NFQ_ERR_SHAPE for ctas outside 1..4096,
 *   iters outside 1..2^20, stages outside 0..4, or pairs with stages = 0.
 * nfq_probe_nvfp4_mma: a measurement kernel, not part of the path.  As
 *   nfq_probe_fp8_mma (one operand set) with the NVFP4 LM head's block-scaled
 *   MMA: `iters` K steps of four tcgen05.mma kind::mxf4nvf4.block_scale
 *   .scale_vec::4X, M = 128 (pairs: 256) x N = 256 x K = 64 each, block scales
 *   of 1.0 in TMEM; 2 * M * 256 * 256 * iters flops per CTA (per pair).
 *   Asynchronous on `stream`; NFQ_ERR_SHAPE for ctas outside 1..4096 or iters
 *   outside 1..2^20.
 * nfq_probe_fp8_mma_shape: a measurement kernel, not part of the path.  As
 *   nfq_probe_fp8_mma with one operand set and single CTAs, for MMAs of
 *   M = m x N = n x K = 32 (m 64 or 128; n in 16..256, a multiple of 8 for
 *   m = 64 and of 16 for m = 128): 2 * m * n * 128 * iters flops per CTA.
 *   NFQ_ERR_SHAPE for other shapes, ctas outside 1..4096 or iters outside
 *   1..2^20.
 * nfq_probe_handoff: a measurement kernel, not part of the path: `iters`
 *   round trips of a barrier hand-off between two threads, each waiting
 *   (bounded) on its own mbarrier for the other's signal.  mode 0: two warps
 *   of one CTA, local arrivals; 1: the two CTAs of a cluster, remote arrivals
 *   at CTA scope; 2: the same with release at cluster scope; 3: the same by
 *   st.async of one word counted on the peer's barrier.  Asynchronous on
 *   `stream`; time it with events.  NFQ_ERR_SHAPE for mode outside 0..3 or
 *   iters outside 1..2^20.
 * nfq_probe_tmem_ld: a measurement kernel, not part of the path.  `ctas` CTAs
 *   of 16 warps each read a 128-lane x 256-column TMEM accumulator into
 *   registers `iters` times, in the LM head epilogue's pattern (each warp 32
 *   lanes x 64 columns as four 16-column loads; batched != 0: one wait for
 *   the four instead of one each): 128 KiB per CTA per iteration.
 *   Asynchronous on `stream`; NFQ_ERR_SHAPE as for nfq_probe_fp8_mma.
 * nfq_probe_handshake: a measurement kernel, not part of the path: the FP8
 *   LM head's accumulator hand-off with no data to stream.  `ctas` CTAs
 *   (pair != 0: `ctas` CTA pairs, cta_group::2, M = 256) run `iters` K blocks;
 *   one thread issues each K block as buffers / 2 groups of four MMAs of
 *   M = 128 x N = 512 / buffers x K = 32, each group into its own TMEM buffer
 *   (buffers = 2, 4 or 8 fill the 512 columns; pairs: 2 or 4), and 16
 *   epilogue warps per CTA wait for each buffer and release it, after
 *   reading their N / 4 columns 16 at a time (mode 1) or without reading
 *   (mode 0); mode 2: no epilogue, the issuing thread waits for each group to
 *   complete before the next; mode 3 (buffers = 4): each 128-column buffer
 *   has its own half of the epilogue warps, which read 64 columns each, so
 *   the two halves of a K block are handed off independently.  Asynchronous
 *   on `stream`; time it with events: the time per K block is what one K
 *   block of the LM head's K loop costs before any data moves.  NFQ_ERR_SHAPE
 *   for ctas outside 1..4096, iters outside 1..2^20, mode outside 0..3,
 *   buffers other than 2, 4, 8, pairs with 8 buffers, or mode 3 without 4.
 * nfq_check_fp8_quotient: a verification kernel, not part of the path.  Stage
 *   1 forms each group's FP8 scale RN(amax / 448) and codes e4m3(RN(hidden /
 *   scale)) without IEEE divisions: the scale from the constant RN(1 / 448)
 *   and a correction FMA, the scale's reciprocal from the hardware
 *   approximation and one Newton step, each code from that reciprocal and
 *   two FMAs (where the scale lies in [2^-40, 2^40); IEEE division
 *   elsewhere).  This runs through every bf16 group maximum amax from 0 to
 *   +inf, and for each every bf16 hidden value y with |y| <= amax and every
 *   NaN, and counts in mismatches[0] the scales that differ from IEEE
 *   amax / 448, in mismatches[1] the reciprocals that differ from the IEEE
 *   reciprocal, in mismatches[2] the codes that differ from those of IEEE
 *   y / scale.  `mismatches` (device, 3 counters, 8-byte aligned) must be
 *   zeroed and `first_bad` (device, 4-byte aligned) set to 0xFFFFFFFF by the
 *   caller; it receives (amax bits << 16) | y bits of one difference (y bits
 *   0 for a scale or reciprocal).  Asynchronous on `stream`.  NFQ_ERR_NULL /
 *   NFQ_ERR_ALIGN for bad pointers.
 * nfq_check_fp4_quotient: a verification kernel, not part of the path.  The
 *   NVFP4 stage 1 forms each 16-element block's e4m3 scale code
 *   e4m3(RN(ab / d)), d = RN(6 g), g = RN(amax_row / 2688), and each e2m1 code
 *   e2m1(RN(y / eff)), eff = RN(value(scale code) g), without IEEE divisions
 *   (a reciprocal from the hardware approximation and one Newton step, then
 *   two FMAs per quotient, where the divisor lies in [2^-40, 2^40); IEEE
 *   division elsewhere).  This runs through every bf16 row maximum from 0 to
 *   +inf and every finite e4m3 block scale and counts: mismatches[0] the
 *   reciprocals of d, mismatches[1] the block-scale codes (every bf16 block
 *   maximum ab <= amax_row), mismatches[2] the reciprocals of eff,
 *   mismatches[3] the e2m1 codes (every bf16 y with |y| <= amax_row, and every
 *   NaN) that differ from IEEE arithmetic's.  `mismatches` (device, 4
 *   counters) must be zeroed and `first_bad` (device, one 64-bit word) set to
 *   all ones by the caller; it receives (scale code << 32) | (amax_row bits
 *   << 16) | value bits of one difference.  Both 8-byte aligned.
 *   Asynchronous on `stream`.  NFQ_ERR_NULL / NFQ_ERR_ALIGN for bad pointers.
 * nfq_probe_wait_timeout: a failure-detection check, not part of the path.
 *   One thread waits, with the bounded wait every kernel of the path uses, on
 *   a barrier nothing arrives on; after the wait's time limit (2 s) it sets the
 *   device error word, which nfq_device_error then reports as
 *   NFQ_ERR_TIMEOUT, and the kernel returns.  Asynchronous on `stream`.
 * nfq_probe_stage1_reads: a measurement kernel, not part of the path: the
 *   loads of the small-batch stage-1 kernel alone (the k partials and the
 *   residual, BF16 [T][H]) in the grid that kernel uses at this size, without
 *   arithmetic or stores; the floor under stage 1's time.  Asynchronous on
 *   `stream`.
 * nfq_stage1_split_plan: the small-batch plan for (T, H, k) on num_sms SMs:
 *   out5 = {CTAs per row (0: the persistent kernel runs), vectors per thread,
 *   active threads, block threads, 1 if the inputs go through shared memory}.
 */
int nfq_stage1_plan(int T, int H, int k, int num_sms, int *out7);
void nfq_stage1_tune(int cluster, int vpt, int slots, int per_slot);
void nfq_lm_head_small_batch(int enabled);
void nfq_lm_head_pair(int enabled);
void nfq_lm_head_nvfp4_tune(int stages);
void nfq_stage1_grid(int max_ctas);
void nfq_stage1_split(int max_tokens, int ctas_per_row, int vpt, int tma);
int nfq_probe_fp8_mma(int pair, int ctas, int iters, int stages, void *stream);
int nfq_probe_nvfp4_mma(int pair, int ctas, int iters, void *stream);
int nfq_probe_handoff(int mode, int iters, void *stream);
int nfq_probe_fp8_mma_shape(int m, int n, int ctas, int iters, void *stream);
int nfq_probe_tmem_ld(int batched, int ctas, int iters, void *stream);
int nfq_probe_handshake(int pair, int buffers, int mode, int ctas, int iters, void *stream);
int nfq_check_fp8_quotient(unsigned long long *mismatches, unsigned *first_bad, void *stream);
int nfq_probe_wait_timeout(void *stream);
int nfq_check_fp4_quotient(unsigned long long *mismatches, unsigned long long *first_bad,
                           void *stream);
int nfq_probe_stage1_reads(const void *const *partials, int k, const void *residual, int T,
                           int H, void *stream);
int nfq_stage1_split_plan(int T, int H, int k, int num_sms, int *out5);

#ifdef __cplusplus
}
#endif

#endif /* NFQ_H_ */
