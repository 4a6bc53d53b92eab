// Streamed GEMV for decode (T <= 4 tokens): weight rows flow from HBM into shared memory by
// bulk copies (cp.async.bulk, the untiled TMA path), so the bytes in flight per SM are set by
// the size of the shared-memory rings, not by registers.
//
// Persistent grid, one CTA of 8 warps per SM. Every warp owns a contiguous share of the rows
// and a private ring of kRing stages; lane 0 keeps the ring full (one bulk copy per row
// segment of <= 8 KB), all lanes consume: each lane multiplies its 16-byte chunks of the
// segment with the matching chunks of the token activations (read through L1) and accumulates
// in FP32; at the end of a row the warp reduces with shuffles and writes the epilogue.
// Waits on the ring's mbarriers are bounded (BEAM_DEV_TIMEOUT on expiry).
#pragma once

#include "bulk.cuh"
#include "common.cuh"

namespace beam {
namespace sg {

constexpr int kWarps = 8;
constexpr int kRing = 3;                    // stages per warp
constexpr int kSegMax = 8192;               // bytes per stage
constexpr int kSmem = kWarps * kRing * kSegMax + kWarps * kRing * 8 + 64;
constexpr int kMaxT = 4;

// Segments per row: the fewest that keep a segment <= kSegMax and a whole number of 512-byte
// warp steps. Needs row_bytes % 512 == 0.
__host__ __device__ inline int n_segments(int row_bytes) {
  int n = (row_bytes + kSegMax - 1) / kSegMax;
  while ((row_bytes / 512) % n != 0) ++n;
  return n;
}

// One weight row (or a gate/up pair of rows) and the activations it meets.
struct RowJob {
  const uint16_t* w[2];    // row pointers (second only for paired rows)
  const uint16_t* x[kMaxT];
  int pid[kMaxT];          // caller's tag per activation (token or pair index)
  int nt;                  // activations to use
};

// Streams the rows [r0, r1) of a warp through its ring and calls epi(r, acc) per row with
// acc[part][t] reduced over the warp (valid in every lane). job(r) describes row r.
// PREFETCH: the rows do not depend on earlier kernels, so the first kRing copies are issued
// before the programmatic-launch wait and overlap the previous kernel's tail.
template <int NP, bool PREFETCH, class JobFn, class EpiFn>
__device__ __forceinline__ bool stream_rows(int r0, int r1, int K, uint8_t* ring, uint64_t* full,
                                            JobFn job, EpiFn epi) {
  const int lane = threadIdx.x & 31;
  const int row_bytes = K * 2;
  const int nseg = n_segments(row_bytes);
  const int seg = row_bytes / nseg;          // bytes, multiple of 512
  const int per_row = NP * nseg;             // loads per row
  const int n_loads = (r1 - r0) * per_row;
  // lane 0: issue load i into stage i % kRing
  auto issue = [&](int i) {
    const int r = r0 + i / per_row, rem = i % per_row;
    const int part = rem / nseg, s = rem % nseg;
    const RowJob jb = job(r);
    const int st = i % kRing;
    bar_expect_tx(&full[st], seg);
    bulk_g2s(ring + st * kSegMax, reinterpret_cast<const uint8_t*>(jb.w[part]) + size_t(s) * seg,
             seg, &full[st]);
  };
  if (!PREFETCH) pdl_wait();
  if (lane == 0)
    for (int i = 0; i < kRing && i < n_loads; ++i) issue(i);
  if (PREFETCH) pdl_wait();
  bool ok = true;
  int done = 0;
  for (int r = r0; r < r1 && ok; ++r) {
    const RowJob jb = job(r);
    float acc[NP][kMaxT];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) acc[p][t] = 0.f;
#pragma unroll
    for (int part = 0; part < NP; ++part) {
      for (int s = 0; s < nseg && ok; ++s, ++done) {
        const int st = done % kRing;
        if (!bar_wait(&full[st], (done / kRing) & 1)) {
          ok = false;
          break;
        }
        const uint4* ws = reinterpret_cast<const uint4*>(ring + st * kSegMax);
        const int cbase = s * (seg / 16);      // chunk index of the segment within the row
        const int steps = seg / 512;
#pragma unroll 2
        for (int i = 0; i < steps; ++i) {
          const int c = i * 32 + lane;
          float wf[8];
          unpack8(ws[c], wf);
#pragma unroll
          for (int t = 0; t < kMaxT; ++t) {
            if (t < jb.nt) {
              float xf[8];
              unpack8(__ldg(reinterpret_cast<const uint4*>(jb.x[t]) + cbase + c), xf);
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[part][t] = fmaf(wf[e], xf[e], acc[part][t]);
            }
          }
        }
        __syncwarp();
        if (lane == 0 && done + kRing < n_loads) issue(done + kRing);
      }
    }
    if (!ok) break;
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) acc[p][t] = warp_sum(acc[p][t]);
    epi(r, jb, acc);
  }
  if (!ok) {
    // let copies still in flight land before the shared memory is released
    if (lane == 0)
      for (int i = done; i < n_loads && i < done + kRing; ++i) bar_wait(&full[i % kRing], (i / kRing) & 1);
    if (lane == 0) flag(BEAM_DEV_TIMEOUT);
  }
  return ok;
}

// Ring and barriers of the calling warp inside the CTA's dynamic shared memory.
__device__ __forceinline__ void warp_ring(uint8_t* smem, uint8_t*& ring, uint64_t*& full) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ring = smem + warp * kRing * kSegMax;
  full = reinterpret_cast<uint64_t*>(smem + kWarps * kRing * kSegMax) + warp * kRing;
  if (lane == 0) {
    for (int s = 0; s < kRing; ++s) bar_init(&full[s], 1);
    bar_fence_init();
  }
  __syncwarp();
}

// Contiguous share [r0, r1) of n rows for global warp gw of nw.
__device__ __forceinline__ void warp_share(int n, int& r0, int& r1) {
  const int nw = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
  r0 = int((long long)n * gw / nw);
  r1 = int((long long)n * (gw + 1) / nw);
}

// Dense rows: Y[t][r] = X[t] . W[r] (MODE 0: FP32, 1: BF16), or for MODE 2 (SwiGLU pairs)
// Y[t][r] = bf16(silu(X[t] . W[r]) * (X[t] . W[N + r])), r < N.
template <int MODE>
__global__ void __launch_bounds__(kWarps * 32, 1)
    dense_kernel(const uint16_t* __restrict__ W, int N, int K, const uint16_t* __restrict__ X,
                 int T, void* __restrict__ Y, int ldy) {
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring;
  uint64_t* full;
  warp_ring(smem, ring, full);
  int r0, r1;
  warp_share(N, r0, r1);
  const int lane = threadIdx.x & 31;
  constexpr int NP = MODE == 2 ? 2 : 1;
  auto job = [&](int r) {
    RowJob j;
    j.w[0] = W + size_t(r) * K;
    j.w[1] = W + size_t(MODE == 2 ? N + r : r) * K;
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      j.x[t] = X + size_t(t < T ? t : 0) * K;
      j.pid[t] = t;
    }
    j.nt = T;
    return j;
  };
  auto epi = [&](int r, const RowJob& jb, const float (&acc)[NP][kMaxT]) {
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      if (lane == t && t < T) {
        const size_t o = size_t(t) * ldy + r;
        if (MODE == 0) static_cast<float*>(Y)[o] = acc[0][t];
        else if (MODE == 1) static_cast<uint16_t*>(Y)[o] = f2bf(acc[0][t]);
        else static_cast<uint16_t*>(Y)[o] = f2bf(siluf_(acc[0][t]) * acc[NP - 1][t]);
      }
    }
  };
  stream_rows<NP, true>(r0, r1, K, ring, full, job, epi);
}

}  // namespace sg
}  // namespace beam
