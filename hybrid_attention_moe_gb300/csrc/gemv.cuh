// Weight-streaming matrix-vector products for small token counts (decode).
//
// At batch 1-8 every projection of the layer is bound by reading its weights from HBM once.
// A warp owns NR weight rows; its 32 lanes walk the row in 16-byte chunks (lane, lane+32, ...),
// keeping U chunks per row in flight, and multiply each chunk with the matching chunk of NT
// activation rows (read through L1, where they stay resident). Partial sums are reduced with
// warp shuffles at the end. FP32 accumulation throughout.
#pragma once

#include "common.cuh"
#include "gemv_flat.cuh"

namespace beam {

// acc[r][t] = sum_k W_r[k] * X_t[k] for rows w[0..NR) and activations x[0..NT), length K
// (a multiple of 8). Activations t >= nt are skipped. Result is complete in every lane.
// MIXED: the products run as mixed-precision bf16 FMAs (fma_bf16x2) instead of FP32 FMAs on
// unpacked operands -- the same sums bit for bit, about half the instructions, but the compiler
// then keeps every requested chunk in registers (the one-token expert kernels went from 72 to
// 148 registers at 5 chunks per row), so each caller sizes its chunks for its occupancy: the
// one-token plain GEMV as before (measured inside the 6-layer decode step: the attention call
// with its o_proj GEMV 29.1 -> 26.0 us, the QKV projection unchanged), the one-token expert
// kernels at 3 chunks per row and three CTAs per SM (mlp.cu).
template <int NR, int NT, int U, bool MIXED = false>
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
      if (MIXED) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nt) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x[t] + size_t(c + 32 * u) * 8));
#pragma unroll
            for (int r = 0; r < NR; ++r) {
              acc[r][t] = fma_bf16x2(wv[u][r].x, xv.x, acc[r][t]);
              acc[r][t] = fma_bf16x2(wv[u][r].y, xv.y, acc[r][t]);
              acc[r][t] = fma_bf16x2(wv[u][r].z, xv.z, acc[r][t]);
              acc[r][t] = fma_bf16x2(wv[u][r].w, xv.w, acc[r][t]);
            }
          }
        }
        continue;
      }
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
    if (MIXED) {
      uint4 wv[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) wv[r] = ld_stream(w[r] + size_t(c) * 8);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < nt) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x[t] + size_t(c) * 8));
#pragma unroll
          for (int r = 0; r < NR; ++r) {
            acc[r][t] = fma_bf16x2(wv[r].x, xv.x, acc[r][t]);
            acc[r][t] = fma_bf16x2(wv[r].y, xv.y, acc[r][t]);
            acc[r][t] = fma_bf16x2(wv[r].z, xv.z, acc[r][t]);
            acc[r][t] = fma_bf16x2(wv[r].w, xv.w, acc[r][t]);
          }
        }
      }
      continue;
    }
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
  warp_dot<ROWS, NT, U, NT == 1>(w, x, nt, K, acc);
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

// The same products on the tensor cores (mma.sync m16n8k16, bf16 in, FP32 accumulate) for 2 to
// 64 tokens: a 16-row block of W is the A operand and NTL tiles of 8 tokens are the columns of
// B, so each 16-byte weight chunk, loaded once, costs a few instructions instead of 8 FMAs per
// token.
// The k axis is permuted inside every 32-element block (a sum does not depend on its order):
// lane (g, c) loads elements 8c..8c+7 of the block from rows g and g+8 of the row block and
// from token g, and uses elements {0,1,2,3} as the fragments of the block's first k16 step
// and {4,5,6,7} as those of the second -- one 16-byte load per row instead of four 4-byte
// ones, and the same permutation on both operands. KS warps of a CTA split the K blocks of one
// row block and add their partial tiles in order through shared memory; a CTA holds 8 / KS row
// blocks. SwiGLU: a row block is 8 gate rows f0..f0+7 and the 8 matching up rows, so one
// thread ends with both the gate and the up value of its unit.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Three CTAs per SM for 1-2 token tiles (measured: dense MLP at 8 tokens 133.8 -> 120.4 us
// against one CTA at the compiler's own 213 registers), two for 4, one for 8.
constexpr int gemv_mma_min_ctas(int ntl) { return ntl <= 2 ? 3 : (ntl == 4 ? 2 : 1); }
template <int MODE, int KS, int NTL, int U>
__global__ void __launch_bounds__(256, gemv_mma_min_ctas(NTL)) gemv_mma_kernel(const uint16_t* __restrict__ W, int N,
                                                       int K, const uint16_t* __restrict__ X,
                                                       int T, float* __restrict__ yf,
                                                       uint16_t* __restrict__ yb, int ldy) {
  pdl_trigger();
  constexpr int RB = 8 / KS;
  __shared__ float red[8][32][4 * NTL];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int rb = blockIdx.x * RB + warp / KS, ks = warp % KS;
  // the two weight rows of this lane (clamped for loads; outputs past N are not written)
  const uint16_t* w0;
  const uint16_t* w1;
  int n_lo, n_hi;
  if (MODE == kOutSwiGLU) {
    n_lo = rb * 8 + g;
    const int f = min(n_lo, N - 1);
    w0 = W + size_t(f) * K;
    w1 = W + size_t(N + f) * K;
    n_hi = n_lo;
  } else {
    n_lo = rb * 16 + g;
    n_hi = n_lo + 8;
    w0 = W + size_t(min(n_lo, N - 1)) * K;
    w1 = W + size_t(min(n_hi, N - 1)) * K;
  }
  const int nb = K >> 5;
  const int b0 = ks * nb / KS, b1 = (ks + 1) * nb / KS;
  // weights are no predecessor's output: start this warp's slice towards L2 before waiting
  // (matrices up to 160 MB, their first 64 MB, as in gemv_kernel)
  {
    constexpr size_t kPrefetchBudget = size_t(64) << 20, kPrefetchMaxMatrix = size_t(160) << 20;
    const size_t rows = MODE == kOutSwiGLU ? 2 * size_t(N) : size_t(N);
    const size_t first_row = MODE == kOutSwiGLU ? size_t(rb) * 8 : size_t(rb) * 16;
    if (rows * size_t(K) * 2 <= kPrefetchMaxMatrix && first_row * K * 2 < kPrefetchBudget &&
        b1 > b0 && lane < 16) {
      // lane l < 16 takes row l of the block (SwiGLU: gate rows, then the up rows)
      size_t r;
      if (MODE == kOutSwiGLU) r = (lane < 8 ? 0 : size_t(N)) + size_t(min(rb * 8 + (lane & 7), N - 1));
      else r = size_t(min(rb * 16 + lane, N - 1));
      l2_prefetch(W + r * K + size_t(b0) * 32, uint32_t(b1 - b0) * 64);
    }
  }
  pdl_wait();
  // n-tile j holds tokens 8j .. 8j+7; lane g loads token 8j + g
  const uint16_t* xr[NTL];
  bool tok[NTL];
#pragma unroll
  for (int j = 0; j < NTL; ++j) {
    tok[j] = 8 * j + g < T;
    xr[j] = X + size_t(tok[j] ? 8 * j + g : 0) * K + 8 * c;
  }
  w0 += 8 * c;
  w1 += 8 * c;
  // one accumulator per n-tile; a single tile alternates two (shorter dependency chains)
  float acc[NTL][4], acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NTL; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  auto step = [&](const uint4& a, const uint4& h, const uint4 (&x)[NTL]) {
#pragma unroll
    for (int j = 0; j < NTL; ++j) {
      mma16816(acc[j], a.x, h.x, a.y, h.y, x[j].x, x[j].y);
      if (NTL == 1) mma16816(acc2, a.z, h.z, a.w, h.w, x[j].z, x[j].w);
      else mma16816(acc[j], a.z, h.z, a.w, h.w, x[j].z, x[j].w);
    }
  };
  int b = b0;
  for (; b + U <= b1; b += U) {
    uint4 a[U], h[U], x[U][NTL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      a[u] = ld_stream(w0 + size_t(b + u) * 32);
      h[u] = ld_stream(w1 + size_t(b + u) * 32);
#pragma unroll
      for (int j = 0; j < NTL; ++j)
        x[u][j] = tok[j] ? __ldg(reinterpret_cast<const uint4*>(xr[j] + size_t(b + u) * 32))
                         : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) step(a[u], h[u], x[u]);
  }
  for (; b < b1; ++b) {
    const uint4 a = ld_stream(w0 + size_t(b) * 32), h = ld_stream(w1 + size_t(b) * 32);
    uint4 x[NTL];
#pragma unroll
    for (int j = 0; j < NTL; ++j)
      x[j] = tok[j] ? __ldg(reinterpret_cast<const uint4*>(xr[j] + size_t(b) * 32)) : make_uint4(0, 0, 0, 0);
    step(a, h, x);
  }
  if (NTL == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[0][i] += acc2[i];
  }
  if (KS > 1) {
#pragma unroll
    for (int j = 0; j < NTL; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[warp][lane][4 * j + i] = acc[j][i];
    __syncthreads();
    if (ks != 0) return;
#pragma unroll
    for (int j = 0; j < NTL; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = red[warp][lane][4 * j + i];
#pragma unroll
        for (int w = 1; w < KS; ++w) v += red[warp + w][lane][4 * j + i];
        acc[j][i] = v;
      }
  }
  // C fragment of tile j: acc[j][0], acc[j][1] = (row g; tokens 8j+2c, 8j+2c+1), acc[j][2],
  // acc[j][3] = (row g + 8; the same tokens)
#pragma unroll
  for (int j = 0; j < NTL; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 8 * j + 2 * c + e;
      if (t >= T) continue;
      if (MODE == kOutSwiGLU) {
        if (n_lo < N) yb[size_t(t) * ldy + n_lo] = f2bf(siluf_(acc[j][e]) * acc[j][2 + e]);
      } else if (MODE == kOutF32) {
        if (n_lo < N) yf[size_t(t) * ldy + n_lo] = acc[j][e];
        if (n_hi < N) yf[size_t(t) * ldy + n_hi] = acc[j][2 + e];
      } else {
        if (n_lo < N) yb[size_t(t) * ldy + n_lo] = f2bf(acc[j][e]);
        if (n_hi < N) yb[size_t(t) * ldy + n_hi] = f2bf(acc[j][2 + e]);
      }
    }
}

// Host launcher: the register-pipelined kernel with the token tile, rows per warp and chunks in
// flight picked from T.
// Tensor-core form for 2..64 tokens (K a multiple of 32): KS, the warps sharing a row block,
// is the smallest power of two that gives at least 16 warps per SM; NTL tiles of 8 tokens per
// pass over the weights, fewer weight chunks in flight as the token tiles grow.
constexpr int kGemvMmaMinT = 2, kGemvMmaMaxT = 64;
template <int MODE, int NTL, int U>
inline cudaError_t launch_gemv_mma_t(const uint16_t* W, int N, int K, const uint16_t* X, int T,
                                     float* yf, uint16_t* yb, int ldy, cudaStream_t st) {
  const int units = MODE == kOutSwiGLU ? (N + 7) / 8 : (N + 15) / 16;
  const int want = 16 * num_sms_cached();
  int ks = 1;
  while (ks < 8 && units * ks < want && (K / 32) >= 2 * ks) ks *= 2;
  const dim3 grid((units * ks + 7) / 8);
  switch (ks) {
    case 1: return launch_pdl(gemv_mma_kernel<MODE, 1, NTL, U>, grid, dim3(256), 0, st, W, N, K, X, T, yf, yb, ldy);
    case 2: return launch_pdl(gemv_mma_kernel<MODE, 2, NTL, U>, grid, dim3(256), 0, st, W, N, K, X, T, yf, yb, ldy);
    case 4: return launch_pdl(gemv_mma_kernel<MODE, 4, NTL, U>, grid, dim3(256), 0, st, W, N, K, X, T, yf, yb, ldy);
    default: return launch_pdl(gemv_mma_kernel<MODE, 8, NTL, U>, grid, dim3(256), 0, st, W, N, K, X, T, yf, yb, ldy);
  }
}
template <int MODE>
inline cudaError_t launch_gemv_mma(const uint16_t* W, int N, int K, const uint16_t* X, int T,
                                   float* yf, uint16_t* yb, int ldy, cudaStream_t st) {
  if (T <= 8) return launch_gemv_mma_t<MODE, 1, 4>(W, N, K, X, T, yf, yb, ldy, st);
  if (T <= 16) return launch_gemv_mma_t<MODE, 2, 2>(W, N, K, X, T, yf, yb, ldy, st);
  if (T <= 32) return launch_gemv_mma_t<MODE, 4, 1>(W, N, K, X, T, yf, yb, ldy, st);
  return launch_gemv_mma_t<MODE, 8, 1>(W, N, K, X, T, yf, yb, ldy, st);
}

// flat_one_token: at T = 1 the product runs on the balanced one-CTA-per-SM kernel of
// gemv_flat.cuh when its shape allows. Measured per call at one token (graph replays, 152 SMs):
// the dense MLP's 419 MB gate/up 74.9 -> 67.2 us and 210 MB down 42.2 -> 34.7 us; the QKV
// projection (147 MB) 22.7 -> 26.3 us and o_proj (63 MB) no better inside the layer, so only
// the dense MLP passes true. The mma.sync form at one token (one valid token column) timed
// alone is faster still (dense MLP call 119.8 -> 107.5 us) but inside the step's CUDA graph
// the 6-layer decode went from 175 to 184 us per token per layer, so it stays at 2+ tokens.
template <int MODE>
inline cudaError_t launch_gemv(const uint16_t* W, int N, int K, const uint16_t* X, int T,
                               float* yf, uint16_t* yb, int ldy, cudaStream_t st,
                               bool flat_one_token = false) {
  if (T <= 0 || N <= 0) return cudaSuccess;
  if (T == 1 && flat_one_token && flat::supported(K)) {
    flat::Args a{};
    a.W = W;
    a.x = X;
    a.N = N;
    a.K = K;
    a.F = N;
    a.yf = yf;
    a.yb = yb;
    const cudaError_t e = MODE == kOutF32    ? flat::launch<flat::kPlainF32>(a, st)
                          : MODE == kOutBF16 ? flat::launch<flat::kPlainBF16>(a, st)
                                             : flat::launch<flat::kSwiGLU>(a, st);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  if (T >= kGemvMmaMinT && T <= kGemvMmaMaxT && (K & 31) == 0) {
    const cudaError_t e = launch_gemv_mma<MODE>(W, N, K, X, T, yf, yb, ldy, st);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
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
