// Tensor-core (tcgen05) prefill attention over a BF16 KV cache, used by beam_attn when many
// tokens of a sequence are processed at once.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "beam.h"

namespace beam {
namespace atc {

// Whether the tensor-core prefill kernel handles this call: BF16 cache, head_dim 128,
// G = n_q / n_kv <= 128 query heads per KV head, a ring cache (window > 0) whose capacity is a
// multiple of 128 slots, 16-byte aligned q and cache.
bool prefill_supported(int D, int G, int window, int cap, bool fp8, const void* q, const void* k,
                       const void* v);

// Workspace bytes for T tokens (the job list).
size_t ws_bytes(int T);

// og[t][h][:] = bf16(bf16(softmax(q'k^T/sqrt(D)) v) * sigmoid(g + gate_bias[h])) for all T
// tokens (q already carries RoPE or SSMax). sl2 = log2(e) / sqrt(D).
cudaError_t prefill(const uint16_t* q, const uint16_t* g, const uint16_t* gate_bias,
                    const int32_t* seq_id, const int32_t* pos, int T, int n_q, int n_kv, int D,
                    const beam_kv_cache& kc, float sl2, uint16_t* og, void* ws, size_t ws_len,
                    cudaStream_t st);

}  // namespace atc
}  // namespace beam
