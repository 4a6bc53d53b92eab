// Weight-streaming matrix-vector products for small token counts (decode).
//
// At batch 1-8 every projection of the layer is bound by reading its weights from HBM once.
// A warp owns NR weight rows; its 32 lanes walk the row in 16-byte chunks (lane, lane+32, ...),
// keeping U chunks per row in flight, and multiply each chunk with the matching chunk of NT
// activation rows (read through L1, where they stay resident). Partial sums are reduced with
// warp shuffles at the end. FP32 accumulation throughout.
#pragma once

#include "common.cuh"

namespace beam {

// acc[r][t] = sum_k W_r[k] * X_t[k] for rows w[0..NR) and activations x[0..NT), length K
// (a multiple of 8). Activations t >= nt are skipped. Result is complete in every lane.
template <int NR, int NT, int U>
__device__ __forceinline__ void warp_dot(const uint16_t* const (&w)[NR],
                                         const uint16_t* const (&x)[NT], int nt, int K,
                                         float (&acc)[NR][NT]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
  const int nchunk = K >> 3;
  int c = lane;
  for (; c + 32 * (U - 1) < nchunk; c += 32 * U) {
    uint4 wv[U][NR];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int r = 0; r < NR; ++r) wv[u][r] = ld_stream(w[r] + size_t(c + 32 * u) * 8);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float wf[NR][8];
#pragma unroll
      for (int r = 0; r < NR; ++r) unpack8(wv[u][r], wf[r]);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < nt) {
          float xf[8];
          unpack8(__ldg(reinterpret_cast<const uint4*>(x[t] + size_t(c + 32 * u) * 8)), xf);
#pragma unroll
          for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[r][t] = fmaf(wf[r][e], xf[e], acc[r][t]);
        }
      }
    }
  }
  for (; c < nchunk; c += 32) {
    float wf[NR][8];
#pragma unroll
    for (int r = 0; r < NR; ++r) unpack8(ld_stream(w[r] + size_t(c) * 8), wf[r]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nt) {
        float xf[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(x[t] + size_t(c) * 8)), xf);
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r][t] = fmaf(wf[r][e], xf[e], acc[r][t]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = warp_sum(acc[r][t]);
}

enum GemvOut { kOutF32 = 0, kOutBF16 = 1, kOutSwiGLU = 2 };

// Y[t][row] = X[t] . W[row] for rows [0, N), tokens [0, T) of blockIdx.y's tile of NT.
//  kOutF32   : yf[t*ldy + row] = acc
//  kOutBF16  : yb[t*ldy + row] = bf16(acc)
//  kOutSwiGLU: N = F units; unit f reads rows f (gate) and F+f (up);
//              yb[t*ldy + f] = bf16(silu(gate) * up)
template <int NT, int NR, int U, int MODE>
__global__ void __launch_bounds__(256) gemv_kernel(const uint16_t* __restrict__ W, int N, int K,
                                                   const uint16_t* __restrict__ X, int T,
                                                   float* __restrict__ yf,
                                                   uint16_t* __restrict__ yb, int ldy) {
  pdl_trigger();
  constexpr int ROWS = (MODE == kOutSwiGLU) ? 2 * NR : NR;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int unit0 = warp * NR;
  if (unit0 >= N) return;
  const int t0 = blockIdx.y * NT;
  const uint16_t* w[ROWS];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    const int unit = min(unit0 + r, N - 1);
    if (MODE == kOutSwiGLU) {
      w[2 * r] = W + size_t(unit) * K;
      w[2 * r + 1] = W + size_t(N + unit) * K;
    } else {
      w[r] = W + size_t(unit) * K;
    }
  }
  // the weights are no predecessor's output: start them towards L2 before waiting -- the
  // first 64 MB of matrices up to 160 MB (QKV+gate, o_proj). Measured: prefetching the
  // 419 MB dense gate/up matrix, whole or in part, slowed it (the prefetches evict each other
  // and the demand loads from the 129 MB L2).
  constexpr size_t kPrefetchBudget = size_t(64) << 20, kPrefetchMaxMatrix = size_t(160) << 20;
  const size_t matrix_bytes = size_t(MODE == kOutSwiGLU ? 2 * N : N) * size_t(K) * 2;
  if (lane == 0 && blockIdx.y == 0 && (K & 7) == 0 && matrix_bytes <= kPrefetchMaxMatrix &&
      size_t(warp) * ROWS * size_t(K) * 2 < kPrefetchBudget) {
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
      if ((reinterpret_cast<uintptr_t>(w[r]) & 15) == 0) l2_prefetch(w[r], uint32_t(K) * 2);
  }
  pdl_wait();
  const int nt = min(NT, T - t0);
  const uint16_t* x[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) x[t] = X + size_t(t0 + min(t, nt - 1)) * K;
  float acc[ROWS][NT];
  warp_dot<ROWS, NT, U>(w, x, nt, K, acc);
  // lanes write distinct (r, t) outputs
#pragma unroll
  for (int r = 0; r < NR; ++r) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (lane == (r * NT + t) % 32 && unit0 + r < N && t < nt) {
        const size_t o = size_t(t0 + t) * ldy + unit0 + r;
        if (MODE == kOutF32) {
          yf[o] = acc[r][t];
        } else if (MODE == kOutBF16) {
          yb[o] = f2bf(acc[r][t]);
        } else {
          yb[o] = f2bf(siluf_(acc[2 * r][t]) * acc[2 * r + 1][t]);
        }
      }
    }
  }
}

// Host launcher: the register-pipelined kernel with the token tile, rows per warp and chunks in
// flight picked from T.
template <int MODE>
inline cudaError_t launch_gemv(const uint16_t* W, int N, int K, const uint16_t* X, int T,
                               float* yf, uint16_t* yb, int ldy, cudaStream_t st) {
  if (T <= 0 || N <= 0) return cudaSuccess;
  auto go = [&](auto kern, int nt, int nr) {
    const int warps = (N + nr - 1) / nr;
    dim3 grid((warps + 7) / 8, (T + nt - 1) / nt);
    launch_pdl(kern, dim3(grid), dim3(256), 0, st, W, N, K, X, T, yf, yb, ldy);
  };
  if (T == 1) {
    // three rows per warp when that fits the matrix into one wave of 4 CTAs per SM while
    // still giving every SM at least two CTAs
    const int ctas3 = (N + 23) / 24;
    if (MODE != kOutSwiGLU && ctas3 <= 4 * num_sms_cached() && ctas3 >= 2 * num_sms_cached())
      go(gemv_kernel<1, 3, 4, MODE>, 1, 3);
    else
      go(gemv_kernel<1, 2, 8, MODE>, 1, 2);
  }
  else if (T == 2)
    go(gemv_kernel<2, 2, 4, MODE>, 2, 2);
  else if (T <= 4)
    go(gemv_kernel<4, 2, 2, MODE>, 4, 2);
  else
    go(gemv_kernel<8, 2, 2, MODE>, 8, 2);
  return cudaGetLastError();
}

}  // namespace beam
