// Tensor-core (tcgen05 + TMA) BF16 GEMM used by the prefill paths: C = A . B^T.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/beam.h"

namespace beam {
namespace tc {

// A [M][K] (row stride lda), B [N][K] (row stride ldb), both bf16 and 16-byte aligned with
// lda, ldb, K multiples of 8. C [M][N] (row stride ldc) is FP32, or BF16 if out_bf16.
cudaError_t gemm_bf16(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int N, int ldb,
                      void* C, int ldc, bool out_bf16, cudaStream_t st);

bool gemm_supported(const void* A, int lda, const void* B, int ldb, int K);

// FP32 C[M][N] = A . B^T, or C += A . B^T when accumulate (each element read and rewritten
// once by the CTA that owns it).
cudaError_t gemm_f32_acc(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int N,
                         int ldb, float* C, int ldc, bool accumulate, cudaStream_t st);

// Epilogue modes of the grouped GEMM.
enum GemmMode { kF32 = 0, kBF16 = 1, kSwiGLU = 2, kF32Add = 3, kQKV = 4 };

// Epilogue of the packed QKV+gate projection (head dim 128): the output columns are the heads
// Q (n_q) | K (n_kv) | V (n_kv) | gate (n_q). Per token row: round to bf16; Q and K heads
// RMS-normalised over the head with one shared [128] gain each, then rotated by the token's
// (cos, sin) table row (sliding-window layers) or, for Q on NoPE layers, scaled by
// (1 + p / ss_base)^ss_exp; q' and g stored in bf16, k and v written into the cache slot
// (p - 1) % capacity (bf16, or e4m3 codes of value / scale). Positions and sequence ids out of
// range set the device status bits and skip the cache write.
struct QkvEpilogue {
  uint16_t* q_out;          // [T][n_q][128]
  uint16_t* g_out;          // [T][n_q * 128]
  beam_kv_cache cache;
  const int32_t* seq_id;
  const int32_t* pos;
  const uint16_t* q_norm;   // [128]
  const uint16_t* k_norm;   // [128]
  const float2* rope;       // [T][64] (cos, sin); nullptr on NoPE layers
  int n_q, n_kv, nope;
  float ss_base, ss_exp, eps;
};

// The projection A . B^T (B = w_qkvg, N = (2 n_q + 2 n_kv) * 128 rows) with the QKV epilogue.
cudaError_t gemm_qkv(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int N, int ldb,
                     const QkvEpilogue& e, cudaStream_t st);

// C[M][F] = bf16(silu(A . Bg^T) * (A . Bu^T)), B = [gate rows F; up rows F] x K.
cudaError_t gemm_swiglu(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int F,
                        int ldb, uint16_t* C, int ldc, cudaStream_t st);

// Grouped GEMM over a device job list: job j = {g, a_row0, rows, -} multiplies A rows
// [a_row0, a_row0 + rows) (at most 128) by the B rows of group g, which start at row
// g * b_stride of B (a 2-D matrix of b_rows rows: all experts stacked). Output column count N
// (units for kSwiGLU, whose up half starts up_off rows after the gate half). The output row
// of A row r is row_map[r] if given. The grid covers max_jobs jobs; jobs at index >= *n_jobs
// return at once. group_scale (optional, device): group g's products are multiplied by
// group_scale[g] in FP32 before the epilogue (kSwiGLU: both gate and up). a_twice: A has K/2
// columns and every B row holds two parts of K/2 (a weight split into BF16 high and low
// parts), each multiplied by A, so the sum runs over both (K a multiple of 128).
cudaError_t gemm_grouped(int mode, const uint16_t* A, int M, int K, int lda, const uint16_t* B,
                         int b_rows, int b_stride, int ldb, const int4* jobs, const int* n_jobs,
                         int max_jobs, int N, int up_off, const int* row_map, void* C, int ldc,
                         cudaStream_t st, const float* group_scale = nullptr,
                         bool a_twice = false);

}  // namespace tc
}  // namespace beam
