/*
 * beam.h -- C ABI of libbeam.so: the forward pass (decode and prefill) of a Beam-style
 * hybrid-attention MoE decoder layer, as hand-written CUDA for sm_103a (GB300).
 *
 * The layer is the one described in the vLLM blog post "Reflection Beam 1.0 on vLLM: day-0
 * serving, agent-optimised kernels, DFlash2 speculative decoding" (cited below as "Beam page"),
 * sections "Beam model architecture", "Attention: sliding-window layers and NoPE
 * full-attention layers", "MoE and residual stream: FP32 router, sandwich norm,
 * depth-scaled residual", and the list of seven kernel changes under "Agent-driven
 * optimisation speeds up batch-1 decode 2.71x".
 *
 * Conventions for every call
 *  - Pointers marked (device) are CUDA device (or managed) memory; (host) are host memory.
 *  - bf16 tensors are raw bfloat16 bit patterns (uint16_t). Matrices are row-major,
 *    weights are [out][in] so each output row is contiguous along the reduction axis.
 *  - The caller owns every buffer: weights, activations, caches and the workspace. The
 *    library allocates no device memory and keeps no state between calls except one
 *    status word per device (beam_get_device_status) and the fixed scratch array of
 *    beam_route_noalloc.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default stream). Argument
 *    checks on sizes, enum values and pointer alignment are synchronous: a call that fails
 *    them returns BEAM_ERR_INVALID_ARG (bad argument) or BEAM_ERR_UNSUPPORTED (valid but
 *    not built, e.g. an odd head dim) and launches nothing. A kernel launch failure returns
 *    BEAM_ERR_CUDA. Values only the device sees (positions, sequence ids, expert indices)
 *    are checked on the device: an out-of-range entry is skipped and a bit is set in the
 *    device status word.
 *  - Vector-streamed pointers (all weights, activations, caches, workspace) must be
 *    16-byte aligned, and the reduction lengths (hidden, head_dim, d_ff) multiples of 8.
 *  - `ws` is caller-provided scratch of at least beam_workspace_bytes(...) bytes (device,
 *    256-byte aligned); its contents are undefined between calls. Two calls that share a
 *    workspace must be ordered on one stream.
 *  - T is the number of tokens in the call. Decode is T = number of sequences with one new
 *    token each; prefill is T = the chunk's tokens. The same entry points serve both.
 */
#ifndef BEAM_H_
#define BEAM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* beam_stream_t; /* a cudaStream_t */
typedef uint16_t beam_bf16;                /* bfloat16 bit pattern */

typedef enum {
  BEAM_OK = 0,
  BEAM_ERR_INVALID_ARG = 1,
  BEAM_ERR_UNSUPPORTED = 2,
  BEAM_ERR_CUDA = 3,
  BEAM_ERR_TIMEOUT = 4
} beam_status;

/* Bits of the device status word. */
#define BEAM_DEV_BAD_POSITION 0x1u  /* pos < 1, or a key slot beyond the cache */
#define BEAM_DEV_BAD_SEQ 0x2u       /* seq_id outside [0, num_seqs) */
#define BEAM_DEV_BAD_EXPERT 0x4u    /* expert index outside [0, n_experts) */
#define BEAM_DEV_TIMEOUT 0x8u       /* a bounded on-device wait expired (result invalid) */

typedef enum { BEAM_KV_BF16 = 0, BEAM_KV_FP8_E4M3 = 1 } beam_kv_dtype;

/* Sliding-window layers rotate Q and K (RoPE); NoPE full-attention layers scale Q by the
 * SSMax factor (1 + p/2048)^0.1 (Beam page, Attention section). */
typedef enum { BEAM_ATTN_SWA_ROPE = 0, BEAM_ATTN_NOPE_SSMAX = 1 } beam_attn_kind;

/* One layer's KV cache (Beam page, Attention section: only full-attention layers keep the
 * whole sequence; sliding-window layers need the last `window` keys).
 *  k, v      (device) [num_seqs][n_kv][capacity][head_dim], bf16 or e4m3 codes (1 byte).
 *  k_scale, v_scale   FP8 only: stored code = e4m3_satfinite(x / scale), value = code * scale.
 *  capacity  slots per sequence and head; position p (1-based) lives in slot (p-1) % capacity.
 *            A sliding-window layer needs capacity >= window + (tokens per sequence in one
 *            call) - 1; a full-attention layer needs capacity >= the largest position.
 *  window    0 for full attention, else the sliding window W (keys p-W+1 .. p). */
typedef struct {
  void* k;
  void* v;
  int32_t dtype; /* beam_kv_dtype */
  float k_scale;
  float v_scale;
  int32_t num_seqs;
  int32_t capacity;
  int32_t window;
} beam_kv_cache;

/* Shape and constants of one layer. Beam: hidden 5120, n_q 48, n_kv 8, head_dim 128,
 * window 512, rope_theta 10000, ssmax 2048 / 0.1, 256 experts in 8 groups, top-4 groups,
 * top-8 experts, d_ff_expert 2560, d_ff_dense 20480, route_scale 2.5. */
typedef struct {
  int32_t hidden;
  int32_t n_q;
  int32_t n_kv;
  int32_t head_dim;
  int32_t kind; /* beam_attn_kind */
  float rope_theta;
  float ssmax_base;
  float ssmax_exp;
  float eps; /* RMSNorm epsilon */
  int32_t n_experts;
  int32_t n_groups;
  int32_t topk_groups;
  int32_t topk;
  int32_t d_ff_expert;
  int32_t d_ff_dense;
  float route_scale;
} beam_layer_cfg;

/* Sublayer boundary: sandwich RMSNorm and depth-scaled residual (Beam page, MoE/residual
 * section; change 1 fuses post-norm, residual and next pre-norm into one kernel):
 *   y = RMSNorm(x) * w_post;  h <- sqrt((n-1)/n) * h + y / sqrt(n);  u = RMSNorm(h) * w_pre
 * FP32 math; y, h and u are stored as bf16.
 *  x      (device) [T][H] sublayer output, or NULL at the first boundary (h = embedding,
 *         n = 1: only the pre-norm runs).
 *  h      (device) [T][H] residual stream, updated in place.
 *  u_out  (device) [T][H] next sublayer's input, or NULL after the last sublayer.
 *  w_post, w_pre (device) [H] gains; w_pre may be NULL only if u_out is NULL.
 *  n      residual term index >= 1 (the embedding is 1; layer l adds 2l+2 and 2l+3). */
beam_status beam_boundary_norm(const beam_bf16* x, beam_bf16* h, beam_bf16* u_out,
                               const beam_bf16* w_post, const beam_bf16* w_pre, int T, int H,
                               int n, float eps, beam_stream_t stream);

/* Packed QKV + gate projection with per-head Q/K RMSNorm, RoPE (sliding-window layers) or
 * the SSMax query scale (NoPE layers), and the KV-cache write (Beam page, Attention section;
 * changes 2, 5 and 6).
 *  u        (device) [T][H] bf16 pre-normed input.
 *  w_qkvg   (device) [2*n_q*D + 2*n_kv*D][H] bf16, rows Q | K | V | gate, head-major.
 *  q_norm_w, k_norm_w (device) [D] bf16 gains, shared by all heads.
 *  seq_id, pos (device) [T] int32: sequence and 1-based position of each token.
 *  q_out    (device) [T][n_q][D] bf16: normed and rotated (or SSMax-scaled) queries.
 *  g_out    (device) [T][n_q*D] bf16: gate pre-activations.
 *  cache    (host struct, device arrays): K and V of all T tokens are written at their
 *           positions before the call's work ends; K is normed and rotated, V as projected.
 * RoPE: half-split pairs (i, i+D/2), angle (p-1) * theta^(-2i/D). */
beam_status beam_qkv_gate(const beam_layer_cfg* cfg, const beam_bf16* u,
                          const beam_bf16* w_qkvg, const beam_bf16* q_norm_w,
                          const beam_bf16* k_norm_w, const int32_t* seq_id, const int32_t* pos,
                          int T, beam_bf16* q_out, beam_bf16* g_out, const beam_kv_cache* cache,
                          void* ws, size_t ws_bytes, beam_stream_t stream);

/* GQA attention over the cache, sigmoid output gate and o_proj (Beam page, Attention section;
 * change 2). Query head i reads KV head i / (n_q/n_kv). Token at position p attends to keys
 * max(1, p-W+1) .. p (sliding window, cache->window = W) or 1 .. p (full attention), with
 * logits q'.k / sqrt(D) and an FP32 softmax. Then o <- bf16(o) * sigmoid(g + gate_bias[head]),
 * rounded to bf16, and out = o W_o^T.
 *  q, g      (device) outputs of beam_qkv_gate for the same tokens.
 *  gate_bias (device) [n_q] bf16.
 *  max_pos   host-side upper bound of pos[] (sizes the key split); larger pos are flagged.
 *  max_q_per_seq  host-side upper bound of the number of the call's tokens that belong to one
 *            sequence (1 for a decode batch). Up to 4 -- and up to 16 (the verification
 *            batches of speculative decoding) while the call holds fewer than two
 *            (sequence, KV head) pairs per SM -- the keys are split across SMs: per token,
 *            or, for a bound of 2 or more over a full-attention BF16 cache (head_dim 128, at
 *            least 2048 keys, T <= 1024), per group of up to max_q_per_seq consecutive tokens
 *            of one sequence that read each K/V block once; otherwise tokens are taken in
 *            tiles of consecutive tokens that share K/V tiles. Both sharing forms expect the
 *            tokens of a sequence to be consecutive in the call (any order is still computed
 *            correctly, only more slowly).
 *  w_o       (device) [H][n_q*D] bf16.   out (device) [T][H] bf16. */
beam_status beam_attn(const beam_layer_cfg* cfg, const beam_bf16* q, const beam_bf16* g,
                      const beam_bf16* gate_bias, const beam_kv_cache* cache,
                      const int32_t* seq_id, const int32_t* pos, int T, int max_pos,
                      int max_q_per_seq, const beam_bf16* w_o, beam_bf16* out, void* ws,
                      size_t ws_bytes, beam_stream_t stream);

/* FP32 router, DeepSeek-V3 style (Beam page, MoE section; change 4): logits = u W_r^T in
 * FP32, s = sigmoid(logits), b = s + corr_bias. Experts form n_groups contiguous groups;
 * a group scores the sum of its two largest b; the topk_groups best groups are kept; the
 * topk experts with the largest b among them are selected (ties: lower index).
 * w_j = s_j / sum(s_selected) * route_scale.
 *  u (device) [T][H] bf16;  w_router (device) [E][H] fp32;  corr_bias (device) [E] fp32.
 *  logits (device) [T][E] fp32 or NULL;  topk_idx (device) [T][topk] int32, in order of
 *  descending b;  topk_w (device) [T][topk] fp32. */
beam_status beam_route(const beam_layer_cfg* cfg, const beam_bf16* u, const float* w_router,
                       const float* corr_bias, int T, float* logits, int32_t* topk_idx,
                       float* topk_w, void* ws, size_t ws_bytes, beam_stream_t stream);

/* Allocation-free variant of beam_route, for callers that cannot provide device scratch: for
 * example a serving engine that has given all free device memory to its KV-cache pool, or a
 * runtime that must not call cudaMalloc (or any allocating library) once it is running.
 * (The Beam pages have no counterpart; this is an interface convenience.)
 * Same arguments and results as beam_route without logits, ws and ws_bytes. The router's
 * logits go to a fixed scratch array inside the library: 65536 floats (256 KiB) of device
 * memory that every GPU loading the library holds until the process exits, so it needs
 * T <= 256 and T * n_experts <= 65536 (256 tokens at 256 experts); larger calls return
 * BEAM_ERR_INVALID_ARG and launch nothing. Within that range it runs the same kernels as
 * beam_route and gives the same results. The call allocates nothing. The first call on a
 * device looks up the array's device address on that device (once, with it current) and
 * keeps it for the life of the process: this assumes the device's primary context lives as
 * long (no cudaDeviceReset between calls). Make that first call before any stream capture.
 * All calls on a device share the one array and
 * leave their logits in it; each call overwrites the whole T x E block it reads, so nothing
 * needs clearing, but calls whose kernels overlap on the GPU (different streams, no ordering)
 * race on the array and give undefined results. */
beam_status beam_route_noalloc(const beam_layer_cfg* cfg, const beam_bf16* u,
                               const float* w_router, const float* corr_bias, int T,
                               int32_t* topk_idx, float* topk_w, beam_stream_t stream);

/* Routed SwiGLU experts with the weighted combine (Beam page, MoE section: 256 experts,
 * d_ff 2560, no shared expert; change 3 combines the top-8 outputs). Only the selected
 * experts' weights are read. a = bf16(silu(u Wg^T) * (u Wu^T)); y = a Wd^T kept in FP32;
 * out = bf16(sum_j w_j y_j) in slot order.
 *  topk_idx, topk_w (device) [T][topk] from beam_route.
 *  w_gate_up (device) [E][2F][H] bf16, rows gate (F) then up (F);  w_down (device) [E][H][F].
 *  out (device) [T][H] bf16. */
beam_status beam_moe(const beam_layer_cfg* cfg, const beam_bf16* u, const int32_t* topk_idx,
                     const float* topk_w, const beam_bf16* w_gate_up, const beam_bf16* w_down,
                     int T, beam_bf16* out, void* ws, size_t ws_bytes, beam_stream_t stream);

/* NVFP4 expert weights (the format the Beam and Flint pages name for the shipped
 * checkpoints; the pages do not print its layout, so this is NVIDIA's published definition):
 * FP4 e2m1 elements, two per byte with the even element in the low nibble; one e4m3 scale per
 * 16 consecutive elements of a row; one FP32 scale per expert matrix. Element value =
 * e2m1 * block scale * matrix scale. All pointers are device pointers, 16-byte aligned.
 *  gate_up [E][2F][H/2], gate_up_scale [E][2F][H/16], gate_up_global [E] (rows gate, then up)
 *  down [E][H][F/2], down_scale [E][H][F/16], down_global [E]. */
typedef struct {
  const uint8_t* gate_up;
  const uint8_t* gate_up_scale;
  const float* gate_up_global;
  const uint8_t* down;
  const uint8_t* down_scale;
  const float* down_global;
} beam_nvfp4_experts;

/* beam_moe with NVFP4 expert weights (weight-only quantisation: activations stay BF16, FP32
 * accumulation of products of exactly dequantised weights). Same arguments and results as beam_moe otherwise. Below 32 tokens the products run on
 * mma.sync in f16 (the caller's u is rounded to f16: exact for BF16 values of magnitude
 * 2^-14 .. 65504); from 32 tokens the selected experts' weights are expanded to BF16 (exact:
 * e2m1 times its e4m3 scale has at most 6 significant bits), 16 experts at a time, and the
 * grouped BF16 tensor-core GEMMs of beam_moe run on them with the matrix scales applied to
 * the FP32 products. H or d_ff not a multiple of 128 returns BEAM_ERR_UNSUPPORTED. The
 * workspace is the one beam_workspace_bytes gives for T. */
beam_status beam_moe_nvfp4(const beam_layer_cfg* cfg, const beam_bf16* u,
                           const int32_t* topk_idx, const float* topk_w,
                           const beam_nvfp4_experts* w, int T, beam_bf16* out, void* ws,
                           size_t ws_bytes, beam_stream_t stream);

/* Block-scaled FP8 expert weights (the AREX feed article on the Day-0 support says the weights
 * ship in BF16, FP8 and NVFP4 without printing a layout; this is the block-scaled e4m3 format of
 * the DeepSeek-V3 release, whose routing the Beam page's MoE section names): e4m3fn codes, one
 * byte per element, row-major like the BF16 experts; one FP32 scale per 128 x 128 block of
 * each expert matrix. Element value = code * block scale. Device pointers, 16-byte aligned.
 *  gate_up [E][2F][H] (rows gate, then up), gate_up_scale [E][2F/128][H/128]
 *  down [E][H][F], down_scale [E][H/128][F/128]. */
typedef struct {
  const uint8_t* gate_up;
  const float* gate_up_scale;
  const uint8_t* down;
  const float* down_scale;
} beam_fp8_experts;

/* beam_moe with FP8 expert weights (weight-only: activations stay BF16, FP32 accumulation).
 * Same arguments and results as beam_moe otherwise. Below 32 tokens the codes become f16
 * exactly in registers and the products run on mma.sync in f16, each 128-element block's sum
 * multiplied by its FP32 scale (u is rounded to f16: exact for BF16 values of magnitude
 * 2^-14 .. 65504). From 32 tokens each selected weight code x scale is expanded to two BF16
 * parts, hi = bf16(w) and lo = bf16(w - hi) (~16 significant bits), 8 experts at a time, and
 * the grouped BF16 tensor-core GEMMs of beam_moe run over both parts. H or d_ff not a
 * multiple of 128 returns BEAM_ERR_UNSUPPORTED. The workspace is the one
 * beam_workspace_bytes gives for T. */
beam_status beam_moe_fp8(const beam_layer_cfg* cfg, const beam_bf16* u, const int32_t* topk_idx,
                         const float* topk_w, const beam_fp8_experts* w, int T, beam_bf16* out,
                         void* ws, size_t ws_bytes, beam_stream_t stream);

/* Dense SwiGLU MLP of layers 0-2 (Beam page, MoE section: d_ff 20480; change 7 runs the
 * activation in one kernel). w_gate_up (device) [2*Fd][H], w_down (device) [H][Fd]. */
beam_status beam_dense_mlp(const beam_layer_cfg* cfg, const beam_bf16* u,
                           const beam_bf16* w_gate_up, const beam_bf16* w_down, int T,
                           beam_bf16* out, void* ws, size_t ws_bytes, beam_stream_t stream);

/* The BF16 tensor-core GEMM behind the prefill projections (the packed QKV+gate projection,
 * o_proj and the dense MLP of the Beam page's change list use it once T >= 64):
 *   C[M][N] = A[M][K] . B[N][K]^T, FP32 accumulation.
 *  A (device) bf16, row stride lda;  B (device) bf16, row stride ldb (weights [out][in]).
 *  C (device) row stride ldc; out_bf16 != 0: bf16 (rounded to nearest even), else fp32.
 *  A, B 16-byte aligned; lda, ldb, K multiples of 8; M, N, K >= 1. */
beam_status beam_gemm_bf16(const beam_bf16* A, int M, int K, int lda, const beam_bf16* B, int N,
                           int ldb, void* C, int ldc, int out_bf16, beam_stream_t stream);

/* LM head with the logit softcap (AREX feed article on vLLM's Day-0 support of
 * Reflection-Beam-1.0, paragraph on the output side: logits pass through 30 * tanh(z / 30)):
 *   z[t][v] = u[t] . w_lm[v] (FP32 accumulation),  logits[t][v] = c * tanh(z[t][v] / c),
 * c = softcap (30 for Beam; softcap <= 0 leaves z uncapped).
 *  u (device) [T][H] bf16: the final-normed hidden state (beam_boundary_norm's pre-norm output
 *  with the final norm's gains after the last layer);  w_lm (device) [V][H] bf16, the
 *  vocabulary rows;  logits (device) [T][V] fp32. u, w_lm and logits 16-byte aligned, H a
 *  multiple of 8; otherwise (or a NaN softcap) BEAM_ERR_INVALID_ARG and nothing is launched.
 *  No workspace; T = 0 launches nothing. */
beam_status beam_lm_head(const beam_bf16* u, const beam_bf16* w_lm, int T, int H, int V,
                         float softcap, float* logits, beam_stream_t stream);

/* Workspace bytes that every call above needs for T tokens and positions up to max_pos. */
size_t beam_workspace_bytes(const beam_layer_cfg* cfg, int T, int max_pos);

/* Bytes of one layer's K+V cache: 2 * num_seqs * n_kv * capacity * head_dim * elem size. */
size_t beam_kv_cache_bytes(int num_seqs, int n_kv, int capacity, int head_dim, int dtype);

/* Reads and clears the current device's status word (BEAM_DEV_* bits); synchronises
 * `stream` first. */
beam_status beam_get_device_status(beam_stream_t stream, uint32_t* bits);

/* Diagnostic of the on-device timeout path: launches one thread that waits, with the bounded
 * mbarrier wait every tensor-core and TMA kernel of the library uses, on a shared-memory barrier
 * that nothing completes (no copy or MMA is issued). The wait gives up after its poll limit
 * (of the order of a second) and records BEAM_DEV_TIMEOUT in the status word, which
 * beam_get_device_status then reports; the context stays usable. Asynchronous on `stream`. */
beam_status beam_selftest_wait_timeout(beam_stream_t stream);

/* Number of CUDA kernels the library has launched in this process (host-side counter,
 * thread-safe; for benchmarks that report their own launches). */
uint64_t beam_launch_count(void);

/* Static description of a status code. */
const char* beam_status_string(beam_status s);

/* Name of the last CUDA runtime error behind a BEAM_ERR_CUDA returned to the calling thread
 * ("cudaSuccess" if there was none); a static string, valid for the process lifetime. */
const char* beam_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif /* BEAM_H_ */
