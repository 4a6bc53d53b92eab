// Balanced weight streaming for one token (batch-1 decode).
//
// At one token every projection of the layer reads its weight matrix from HBM once and does
// 2 FLOPs per weight, so its time is the matrix bytes over the bandwidth the launch sustains.
// That needs every SM streaming the same number of bytes for the whole kernel: a grid of
// row-sized work items leaves some SMs with one item more than others (5120 rows over 152 SMs
// is 33.7 per SM) and the kernel lasts as long as the busiest SM.
//
// Here the grid is one CTA of 16 warps per SM. The outputs ("groups": a row, or a gate row and
// its up row) are split into
// contiguous runs, one per CTA, whose sizes differ by at most one group. Inside a CTA the run's
// rows are cut into steps of 32 chunks (16 bytes, 8 elements; one chunk per lane) -- rows hold
// whole steps (K a multiple of 256) -- and the steps into 16 equal contiguous ranges, one per
// warp, which may start and end inside a row. A step never straddles two rows, so the row a
// warp works on changes only between steps and is the same for all its lanes. A warp keeps two
// batches of U steps of loads in flight (the next batch is requested before the current one
// is multiplied); a batch inside one row is addressed from one base pointer. When a row ends,
// the warp reduces its running sum with shuffles and adds it to its own partial sum of the
// row's group in shared memory (one slot per group and warp, so no two
// writers meet). After a barrier one thread per group adds the 16 warps' partials in warp
// order and writes the group's output. The order of every sum is fixed: results are
// deterministic. The activation vector is staged in shared memory once per CTA, as bf16.
#pragma once

#include "common.cuh"

namespace beam {
namespace flat {

enum Mode {
  kPlainF32 = 0,   // y[r] = W[r] . x                       (FP32 out)
  kPlainBF16 = 1,  // y[r] = bf16(W[r] . x)
  kSwiGLU = 2,     // a[f] = bf16(silu(W[f] . x) * (W[F + f] . x)), f < F
};

constexpr int kWarps = 16, kGroupTile = 160, kU = 8;

struct Args {
  const uint16_t* W;
  const uint16_t* x;    // [K]
  int N;                // groups: rows, or units F
  int K;                // row length (elements)
  int F;                // kSwiGLU: units (gate rows f, up rows F + f)
  float* yf;
  uint16_t* yb;
};

template <int MODE>
__host__ __device__ constexpr int rows_per_group() {
  return MODE == kSwiGLU ? 2 : 1;
}

struct RowInfo {
  const uint16_t* w;   // start of the row
  int s;               // which of the group's two sums it feeds
};

// Row r of the product (groups of rows_per_group rows, in order).
template <int MODE>
__device__ __forceinline__ RowInfo row_info(const Args& a, long r, long nrows) {
  r = r < nrows ? r : nrows - 1;   // rows past the end are never loaded; keep the address valid
  RowInfo ri{nullptr, 0};
  const size_t K = size_t(a.K);
  if (MODE == kSwiGLU) {
    const long g = r >> 1;
    ri.s = int(r & 1);
    ri.w = a.W + size_t(ri.s ? a.F + g : g) * K;
  } else {
    ri.w = a.W + size_t(r) * K;
  }
  return ri;
}

// The 8 products of a weight chunk and the matching activation chunk (both bf16), summed in
// element order: one mixed-precision FMA per element. Bit for bit the FP32 chain over widened
// operands, at about half the instructions (measured: the dense MLP call at one token
// 119.5 -> 106.8 us inside the 6-layer decode step, against the FP32 form with the activations
// staged in FP32).
__device__ __forceinline__ float dot8(const uint4& w, const uint16_t* xs) {
  const uint4 x = *reinterpret_cast<const uint4*>(xs);
  float s = fma_bf16x2(w.x, x.x, 0.f);
  s = fma_bf16x2(w.y, x.y, s);
  s = fma_bf16x2(w.z, x.z, s);
  s = fma_bf16x2(w.w, x.w, s);
  return s;
}

// Shared memory of one CTA: the group partials, then the staged activations (bf16).
inline size_t smem_bytes(int xlen, int warps = kWarps) {
  return size_t(kGroupTile) * warps * 2 * 4 + size_t(xlen) * 2;
}

template <int MODE, int U, int kWarps = flat::kWarps>
__global__ void __launch_bounds__(kWarps * 32, 1) flat_gemv_kernel(Args a) {
  constexpr int kThreads = kWarps * 32;
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  float* part = reinterpret_cast<float*>(smem);   // [kGroupTile][kWarps][2]
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + size_t(kGroupTile) * kWarps * 2 * 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int R = rows_per_group<MODE>();
  const int KS = a.K >> 8;   // steps (32 chunks of 8 elements, one per lane) per row
  const long G = a.N;
  const long g0 = long(blockIdx.x) * G / gridDim.x, g1 = long(blockIdx.x + 1) * G / gridDim.x;
  const long nrows_all = G * R;

  // cursors of this warp in the current tile: the issue cursor runs one batch ahead of the
  // compute cursor; both hold (row relative to the tile, step in the row, step in the range).
  // Every step lies inside one row, so all of this is warp-uniform.
  long t0 = g0, rbase = g0 * R, sb = 0, se = 0;
  int ng = 0;
  long irow = 0, crow = 0, is = 0, cs = 0;
  int ik = 0, ck = 0;
  const uint16_t* iptr = nullptr;
  RowInfo cri{};
  float acc0 = 0.f, acc1 = 0.f;
  auto start_tile = [&]() {
    ng = int(min(long(kGroupTile), g1 - t0));
    rbase = t0 * R;
    const long nsteps = long(ng) * R * KS;
    sb = long(warp) * nsteps / kWarps;
    se = long(warp + 1) * nsteps / kWarps;
    irow = crow = sb / KS;
    ik = ck = int(sb - irow * KS);
    is = cs = sb;
    iptr = row_info<MODE>(a, rbase + irow, nrows_all).w;
    acc0 = acc1 = 0.f;
  };
  auto next_issue_row = [&]() {
    ik = 0;
    ++irow;
    iptr = row_info<MODE>(a, rbase + irow, nrows_all).w;
  };
  auto flush_row = [&]() {   // the compute cursor's row is done (or its range ended)
    const float t = warp_sum(acc0 + acc1);
    if (lane == 0) part[(size_t(crow / R) * kWarps + warp) * 2 + cri.s] += t;
    acc0 = acc1 = 0.f;
  };
  auto next_compute_row = [&]() {
    flush_row();
    ck = 0;
    ++crow;
    cri = row_info<MODE>(a, rbase + crow, nrows_all);
  };
  auto issue = [&](uint4 (&buf)[U]) {
    if (ik + U <= KS && is + U <= se) {   // the whole batch in one row and in range
      const uint16_t* p = iptr + 8 * (32 * size_t(ik) + lane);
#pragma unroll
      for (int u = 0; u < U; ++u) buf[u] = ld_stream(p + 256 * u);
      ik += U;
      is += U;
      if (ik == KS) next_issue_row();
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (is < se) {
          buf[u] = ld_stream(iptr + 8 * (32 * size_t(ik) + lane));
          ++is;
          if (++ik == KS) next_issue_row();
        } else {
          buf[u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  };
  auto consume = [&](const uint4 (&buf)[U]) {
    if (ck + U <= KS && cs + U <= se) {
      const uint16_t* xp = xs + 8 * (32 * ck + lane);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u & 1) acc1 += dot8(buf[u], xp + 256 * u);
        else acc0 += dot8(buf[u], xp + 256 * u);
      }
      ck += U;
      cs += U;
      if (ck == KS) next_compute_row();
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (cs < se) {
          acc0 += dot8(buf[u], xs + 8 * (32 * ck + lane));
          ++cs;
          if (++ck == KS) next_compute_row();
        }
      }
    }
  };

  uint4 ba[U], bb[U];
  if (g0 < g1) {
    // the weights are no predecessor's output: the first batch is requested before waiting
    start_tile();
    if (sb < se) issue(ba);
  }
  pdl_wait();
  for (int i = threadIdx.x; i < (a.K >> 3); i += kThreads) {
    reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
  }
  for (; t0 < g1; t0 += kGroupTile) {
    if (t0 != g0) {
      start_tile();
      if (sb < se) issue(ba);
    }
    for (int i = threadIdx.x; i < ng * kWarps * 2; i += kThreads) part[i] = 0.f;
    __syncthreads();
    if (sb < se) {
      cri = row_info<MODE>(a, rbase + crow, nrows_all);
      // two batches in flight: the next batch is requested before the current one is used
      while (true) {
        issue(bb);
        consume(ba);
        if (cs >= se) break;
        issue(ba);
        consume(bb);
        if (cs >= se) break;
      }
      if (ck > 0) flush_row();   // the range ended inside a row
    }
    __syncthreads();
    for (int t = threadIdx.x; t < ng; t += kThreads) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        s0 += part[(t * kWarps + w) * 2];
        s1 += part[(t * kWarps + w) * 2 + 1];
      }
      const long g = t0 + t;
      if (MODE == kPlainF32) a.yf[g] = s0;
      else if (MODE == kPlainBF16) a.yb[g] = f2bf(s0);
      else a.yb[g] = f2bf(siluf_(s0) * s1);
    }
    __syncthreads();
  }
}

// Whether the one-token product of this shape runs here: rows of whole 32-chunk steps (K a
// multiple of 256), at least U of them, and activations that fit the shared-memory stage.
inline bool supported(int K) {
  return (K & 255) == 0 && (K >> 8) >= kU && smem_bytes(K) <= 200 * 1024;
}

template <int MODE>
inline cudaError_t launch(const Args& a, cudaStream_t st) {
  const int xlen = a.K;
  static bool attr_set = false;   // per instantiation; setting it twice is harmless
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(flat_gemv_kernel<MODE, kU>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               200 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(flat_gemv_kernel<MODE, kU>, dim3(num_sms_cached()), dim3(kWarps * 32),
                    smem_bytes(xlen), st, a);
}

}  // namespace flat
}  // namespace beam
