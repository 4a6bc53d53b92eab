// Long-context decode attention fed by TMA (attn_dec.cu), used by beam_attn for few tokens per
// sequence over many cached keys.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "beam.h"

namespace beam {
namespace adec {

// Whether this kernel handles the call: head_dim 128, G = n_q / n_kv <= 8 query heads per KV
// head, at least kMinKeys keys to attend to (max_keys), a ring cache (window > 0) whose
// capacity is a multiple of the key block (64 slots BF16, 128 FP8), 16-byte aligned cache.
constexpr int kMinKeys = 2048;
bool supported(int D, int G, int window, int cap, bool fp8, const void* k, const void* v,
               int max_keys);

// Workspace bytes for T tokens (partials of the pairs split between CTAs).
size_t ws_bytes(int T, int n_kv, int window, int max_pos, bool fp8);

// og[t][h][:] = bf16(bf16(softmax(q'k^T/sqrt(D)) v * v_scale) * sigmoid(g + gate_bias[h])) for
// all T tokens; sl2 = log2(e) / sqrt(D) * k_scale. Enqueues the attention kernel and, when a
// pair is split between CTAs, the merge kernel.
cudaError_t decode(const uint16_t* q, const uint16_t* g, const uint16_t* gate_bias,
                   const int32_t* seq_id, const int32_t* pos, int T, int max_pos, int n_q,
                   int n_kv, const beam_kv_cache& kc, float sl2, float v_scale, uint16_t* og,
                   void* ws, size_t ws_len, cudaStream_t st);

// Verification batches (several new tokens per sequence) over a full-attention BF16 cache:
// the tokens of one sequence that are consecutive in the call (up to a group of max_q_per_seq,
// and no more than 96 query rows) share every K/V block, which is read once per group instead
// of once per token. Same output as decode(); head_dim 128, G <= 8, at least kMinKeys keys,
// 1 <= T <= kVerifyMaxT, max_q_per_seq >= 2.
constexpr int kVerifyMaxT = 1024;
bool verify_supported(int D, int G, int window, bool fp8, const void* k, const void* v,
                      int max_keys, int T, int max_q_per_seq);
size_t verify_ws_bytes(int T, int G, int max_q_per_seq);
size_t verify_ws_bytes_max(int T);   // over every G and max_q_per_seq
cudaError_t verify(const uint16_t* q, const uint16_t* g, const uint16_t* gate_bias,
                   const int32_t* seq_id, const int32_t* pos, int T, int max_pos,
                   int max_q_per_seq, int n_q, int n_kv, const beam_kv_cache& kc, float sl2,
                   uint16_t* og, void* ws, size_t ws_len, cudaStream_t st);

}  // namespace adec
}  // namespace beam
