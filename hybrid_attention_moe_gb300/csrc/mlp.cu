// Routed SwiGLU experts with the weighted top-k combine, and the dense SwiGLU MLP.
// Beam page, MoE section (256 experts of d_ff 2560, no shared expert; layers 0-2 dense SwiGLU
// with d_ff 20480) and changes 3 and 7 of the optimisation list (the top-8 combine fused into
// a neighbouring kernel; the dense activation in one kernel). The Flint page's small-batch MoE
// kernels ("router and expert GEMV read only the selected experts") motivate reading only
// the experts some token selected.
//
// beam_moe runs three kernels:
//   plan      : one CTA buckets the T*k (token, slot) pairs by expert -> active expert list
//   gate_up   : warp per (active expert, f): rows f (gate) and F+f (up) of that expert, dotted
//               with every pair's token; a[pair][f] = bf16(silu(gate) * up)
//   down      : warp per output row h: row h of every active expert's W_down dotted with its
//               pairs' activations (FP32 y in shared memory), then out[t][h] =
//               bf16(sum_j w[t][j] y[t*k+j]) in slot order -- the combine needs no extra pass.
// Each weight byte of a selected expert is read from HBM once per call.
#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"


namespace beam {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPairTile = 4;        // pairs per weight pass in the gate_up / down warps
constexpr int kFusedMaxPairs = 1024;  // down+combine in shared memory up to this many pairs

constexpr int kMoeGemmMinT = 32;   // from here the experts run as grouped tensor-core GEMMs
// Weight chunks in flight per lane in the single-token gate/up and down kernels. The down kernel
// takes 4 rows of 2560 per warp, the gate/up kernel 2 (gate, up) row pairs of 5120 (with the
// FP32 products: 4 rows x 5 chunks measured 8-10 us faster than 2 rows x 8 chunks for the
// down kernel, 2 pairs x 5 chunks 5 us faster than one pair x 4 for gate/up). Both multiply
// with mixed-precision bf16 FMAs (warp_dot's MIXED form); that form keeps every requested chunk
// in registers, so they run 3 chunks per row at three CTAs per SM (80 registers, no spills):
// measured in the 6-layer decode step 164.3 -> 162.9 us per token per layer, against 5 chunks
// with the FP32 products (72 registers) and 5 chunks with the mixed form capped at three CTAs
// (80 registers and spills, 163.1).
constexpr int kDecodeGateUpU = 3;
constexpr int kDecodeGateUpFPW = 2;   // gate/up row pairs per warp in the one-token kernel
constexpr int kDecodeDownU = 3;
constexpr int kDecodeDownNR = 4;   // rows per warp in the one-token down kernel

struct MoePlan {
  int* n_active;   // [1]
  int* active;     // [E] expert ids, increasing
  int* act_off;    // [E+1] offsets into pairs
  int* pairs;      // [P] pair ids t*k + j grouped by expert
  int4* jobs;      // grouped GEMM only: {expert, first sorted row, rows <= 128,
                   //  the expert's first job | its job count << 20}
  int* n_jobs;     // [1]
};

// Exclusive scan over the block of one int per thread; *total gets the sum. ws: 32 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  __syncthreads();
  if (lane == 31) ws[wid] = inc;
  __syncthreads();
  if (wid == 0) {
    const int nw = blockDim.x >> 5;
    int t = lane < nw ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    if (lane < nw) ws[lane] = t;               // inclusive prefix of warp totals
  }
  __syncthreads();
  const int before = wid > 0 ? ws[wid - 1] : 0;
  *total = ws[(blockDim.x >> 5) - 1];
  return before + inc - v;
}

// Buckets the P = T*k (token, slot) pairs by expert. One CTA of kPlanThreads threads, each
// owning kPlanItems consecutive experts (E <= 4096).
constexpr int kPlanItems = 4;
__global__ void __launch_bounds__(kPlanThreads) moe_plan_kernel(const int32_t* __restrict__ idx,
                                                                int P, int E, MoePlan pl) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ int sh[];
  int* cnt = sh;               // [E]
  int* off = sh + E;           // [E]
  int* fill = sh + 2 * E;      // [E]
  __shared__ int scan_ws[32];
  for (int e = threadIdx.x; e < E; e += blockDim.x) { cnt[e] = 0; fill[e] = 0; }
  __syncthreads();
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    const int e = idx[i];
    if (e < 0 || e >= E) { flag(BEAM_DEV_BAD_EXPERT); continue; }
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  const int e0 = threadIdx.x * kPlanItems;
  int c_sum = 0, a_sum = 0;
#pragma unroll
  for (int j = 0; j < kPlanItems; ++j) {
    const int e = e0 + j;
    if (e < E) { c_sum += cnt[e]; a_sum += cnt[e] > 0; }
  }
  int c_tot, a_tot;
  int c_off = block_excl_scan(c_sum, scan_ws, &c_tot);
  int a_off = block_excl_scan(a_sum, scan_ws, &a_tot);
#pragma unroll
  for (int j = 0; j < kPlanItems; ++j) {
    const int e = e0 + j;
    if (e < E) {
      off[e] = c_off;
      if (cnt[e] > 0) {
        pl.active[a_off] = e;
        pl.act_off[a_off] = c_off;
        ++a_off;
      }
      c_off += cnt[e];
    }
  }
  if (threadIdx.x == 0) {
    pl.act_off[a_tot] = c_tot;
    *pl.n_active = a_tot;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    const int e = idx[i];
    if (e < 0 || e >= E) continue;
    const int slot = atomicAdd(&fill[e], 1);
    pl.pairs[off[e] + slot] = i;
  }
  if (pl.jobs != nullptr) {
    __threadfence_block();
    __syncthreads();
    if (threadIdx.x == 0) {
      int nj = 0;
      for (int a = 0; a < a_tot; ++a) {
        const int e = pl.active[a], o0 = pl.act_off[a], c = pl.act_off[a + 1] - o0;
        // w: the expert's first job and its job count, for the GEMM's tile order
        const int first = nj, n = (c + 127) / 128;
        for (int r = 0; r < c; r += 128)
          pl.jobs[nj++] = make_int4(e, o0 + r, min(128, c - r), first | (n << 20));
      }
      *pl.n_jobs = nj;
    }
  }
}

// Expert and pair range of active slot `ai`: from the plan, or -- when one token's k slots are
// taken as the active list directly (`direct` = that token's expert indices) -- slot ai is
// expert direct[ai] with the single pair ai. Returns false for an expert index out of range.
struct ExpertSlot {
  int e, p0, p1;
};
__device__ __forceinline__ bool expert_slot(const MoePlan& pl, const int32_t* direct, int E,
                                            int ai, ExpertSlot& s) {
  if (direct != nullptr) {
    s.e = direct[ai];
    s.p0 = ai;
    s.p1 = ai + 1;
    return s.e >= 0 && s.e < E;
  }
  s.e = pl.active[ai];
  s.p0 = pl.act_off[ai];
  s.p1 = pl.act_off[ai + 1];
  return true;
}
__device__ __forceinline__ int pair_at(const MoePlan& pl, const int32_t* direct, int i) {
  return direct != nullptr ? i : pl.pairs[i];
}

// grid (ceil(F / 8), max active experts); warp per (active expert, f): gate row f and up
// row F+f, dotted with up to NT of the expert's pairs per weight pass. CTA (0, 0) also clears
// the n_cnt completion counters of the down kernel that follows.
template <int U, int NT, int FPW>
__global__ void __launch_bounds__(256, NT == 1 ? 3 : 1) moe_gate_up_kernel(
    const uint16_t* __restrict__ u, const uint16_t* __restrict__ w_gu, int H, int F, int k,
    MoePlan pl, const int32_t* __restrict__ direct, int E, int* __restrict__ cnt, int n_cnt,
    uint16_t* __restrict__ a) {
  pdl_trigger();
  pdl_wait();
  if (cnt != nullptr && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
  const int ai = blockIdx.y;
  if (ai >= (direct != nullptr ? k : *pl.n_active)) return;
  const int f0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * FPW;
  if (f0 >= F) return;
  const int lane = threadIdx.x & 31;
  ExpertSlot es;
  if (!expert_slot(pl, direct, E, ai, es)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(BEAM_DEV_BAD_EXPERT);
    return;
  }
  const uint16_t* base = w_gu + size_t(es.e) * 2 * F * H;
  const uint16_t* w[2 * FPW];
#pragma unroll
  for (int j = 0; j < FPW; ++j) {
    const int f = min(f0 + j, F - 1);
    w[2 * j] = base + size_t(f) * H;
    w[2 * j + 1] = base + size_t(F + f) * H;
  }
  for (int pp = es.p0; pp < es.p1; pp += NT) {
    const int nt = min(NT, es.p1 - pp);
    int pid[NT];
    const uint16_t* x[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      pid[i] = pair_at(pl, direct, pp + min(i, nt - 1));
      x[i] = u + size_t(pid[i] / k) * H;
    }
    float acc[2 * FPW][NT];
    warp_dot<2 * FPW, NT, U, NT == 1>(w, x, nt, H, acc);
#pragma unroll
    for (int j = 0; j < FPW; ++j)
#pragma unroll
      for (int i = 0; i < NT; ++i)
        if (i < nt && lane == j * NT + i && f0 + j < F)
          a[size_t(pid[i]) * F + f0 + j] = f2bf(siluf_(acc[2 * j][i]) * acc[2 * j + 1][i]);
  }
}

// Fused down projection + combine. grid ceil(H / 8); warp per output row h.
// dynamic smem: 8 warps x P floats.
template <int U>
__global__ void __launch_bounds__(256) moe_down_combine_kernel(
    const uint16_t* __restrict__ a, const uint16_t* __restrict__ w_dn,
    const float* __restrict__ topk_w, int T, int H, int F, int k, MoePlan pl,
    uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float ysh[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 8 + warp;
  if (h >= H) return;
  const int P = T * k;
  float* y = ysh + size_t(warp) * P;
  for (int i = lane; i < P; i += 32) y[i] = 0.f;
  __syncwarp();
  const int na = *pl.n_active;
  for (int ai = 0; ai < na; ++ai) {
    const int e = pl.active[ai];
    const int p0 = pl.act_off[ai], p1 = pl.act_off[ai + 1];
    const uint16_t* w[1] = {w_dn + (size_t(e) * H + h) * F};
    for (int pp = p0; pp < p1; pp += kPairTile) {
      const int nt = min(kPairTile, p1 - pp);
      int pid[kPairTile];
      const uint16_t* x[kPairTile];
#pragma unroll
      for (int i = 0; i < kPairTile; ++i) {
        pid[i] = pl.pairs[pp + min(i, nt - 1)];
        x[i] = a + size_t(pid[i]) * F;
      }
      float acc[1][kPairTile];
      warp_dot<1, kPairTile, U>(w, x, nt, F, acc);
#pragma unroll
      for (int i = 0; i < kPairTile; ++i)
        if (i < nt && lane == i) y[pid[i]] = acc[0][i];
    }
  }
  __syncwarp();
  for (int t = lane; t < T; t += 32) {
    float s = 0.f;
    for (int j = 0; j < k; ++j) s = fmaf(topk_w[size_t(t) * k + j], y[t * k + j], s);
    out[size_t(t) * H + h] = f2bf(s);
  }
}

// Warp per (active expert, NR consecutive rows h); y[pair][h] (FP32) to the workspace. With
// completion counters (one per CTA column, cleared by the gate/up kernel), the last CTA of a
// column to finish also combines its 8*NR rows: out[t][h] = bf16(sum_j w[t][j] y[t*k+j][h]),
// slots in order, skipping slots whose expert index is out of range. Without counters a
// separate combine pass follows.
template <int U, int NT, int NR>
__global__ void __launch_bounds__(256, NT == 1 ? 3 : 1) moe_down_kernel(
    const uint16_t* __restrict__ a, const uint16_t* __restrict__ w_dn, int H, int F, MoePlan pl,
    const int32_t* __restrict__ direct, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, int T, int k, int E, int* __restrict__ cnt,
    float* __restrict__ y, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int na = direct != nullptr ? k : *pl.n_active;
  const int ai = blockIdx.y;
  if (ai >= max(na, 1)) return;   // uniform over the CTA
  const int h0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * NR;
  const int lane = threadIdx.x & 31;
  ExpertSlot es;
  const bool work = ai < na && h0 < H && expert_slot(pl, direct, E, ai, es);
  if (work) {
    const uint16_t* w[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) w[r] = w_dn + (size_t(es.e) * H + min(h0 + r, H - 1)) * F;
    for (int pp = es.p0; pp < es.p1; pp += NT) {
      const int nt = min(NT, es.p1 - pp);
      int pid[NT];
      const uint16_t* x[NT];
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        pid[i] = pair_at(pl, direct, pp + min(i, nt - 1));
        x[i] = a + size_t(pid[i]) * F;
      }
      float acc[NR][NT];
      warp_dot<NR, NT, U, NT == 1>(w, x, nt, F, acc);
#pragma unroll
      for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int i = 0; i < NT; ++i)
          if (i < nt && lane == r * NT + i && h0 + r < H)
            y[size_t(pid[i]) * H + h0 + r] = acc[r][i];
    }
  }
  if (cnt == nullptr) return;   // uniform over the grid
  __shared__ int s_last;
  // the CTA barrier orders every thread's y stores before thread 0's device-scope fence,
  // which releases them with the counter increment
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(cnt + blockIdx.x, 1) == max(na, 1) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int hb = blockIdx.x * 8 * NR;
  const int nh = min(8 * NR, H - hb);
  for (int i = threadIdx.x; i < T * nh; i += blockDim.x) {
    const int t = i / nh, h = hb + (i - t * nh);
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[size_t(t) * k + j];
      if (e < 0 || e >= E) continue;
      s = fmaf(topk_w[size_t(t) * k + j], __ldcg(y + (size_t(t) * k + j) * H + h), s);
    }
    out[size_t(t) * H + h] = f2bf(s);
  }
}

// Tensor-core forms of the expert products for 2..31 tokens, after the plan: as in
// gemv_mma_kernel (gemv.cuh), a warp's 16-row block of one expert's weights is the A operand of
// mma.sync m16n8k16 and up to 8 of the expert's (token, slot) pairs are the columns of B (more
// pairs: further passes over the rows), with the k axis permuted inside each 32-element block
// so that every lane loads whole 16-byte chunks. Gate/up: a warp takes 8 units (8 gate rows and
// the matching 8 up rows) and writes bf16(silu(gate) * up) per pair; CTA (0, 0) also clears the
// down kernel's completion counters. Down: a warp takes 16 rows h and writes y[pair][h] in
// FP32; the last CTA of each 128-row column to finish combines its rows for every token:
// out[t][h] = bf16(sum_j w[t][j] y[t*k+j][h]), slots in order, slots with an expert index out
// of range skipped.
constexpr int kMmaU = 4;
constexpr int kMmaRowsDown = 128;   // rows h per down CTA (8 warps x 16)

__device__ __forceinline__ void expert_rows_mma(const uint16_t* w0, const uint16_t* w1,
                                                const uint16_t* xr, bool tok, int K,
                                                float (&acc)[4]) {
  float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0.f;
  const int nb = K >> 5;
  int b = 0;
  for (; b + kMmaU <= nb; b += kMmaU) {
    uint4 a[kMmaU], h[kMmaU], x[kMmaU];
#pragma unroll
    for (int u = 0; u < kMmaU; ++u) {
      a[u] = ld_stream(w0 + size_t(b + u) * 32);
      h[u] = ld_stream(w1 + size_t(b + u) * 32);
      x[u] = tok ? __ldg(reinterpret_cast<const uint4*>(xr + size_t(b + u) * 32)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kMmaU; ++u) {
      mma16816(acc, a[u].x, h[u].x, a[u].y, h[u].y, x[u].x, x[u].y);
      mma16816(acc2, a[u].z, h[u].z, a[u].w, h[u].w, x[u].z, x[u].w);
    }
  }
  for (; b < nb; ++b) {
    const uint4 a = ld_stream(w0 + size_t(b) * 32), h = ld_stream(w1 + size_t(b) * 32);
    const uint4 x = tok ? __ldg(reinterpret_cast<const uint4*>(xr + size_t(b) * 32)) : make_uint4(0, 0, 0, 0);
    mma16816(acc, a.x, h.x, a.y, h.y, x.x, x.y);
    mma16816(acc2, a.z, h.z, a.w, h.w, x.z, x.w);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
}

// grid (ceil(F / 64), max active experts). Two CTAs per SM (at most 128 registers): measured
// 4% faster than one CTA at the compiler's own 213 registers.
__global__ void __launch_bounds__(256, 2) moe_gate_up_mma_kernel(
    const uint16_t* __restrict__ u, const uint16_t* __restrict__ w_gu, int H, int F, int k,
    MoePlan pl, int* __restrict__ cnt, int n_cnt, uint16_t* __restrict__ a) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
  const int ai = blockIdx.y;
  if (ai >= *pl.n_active) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int f0 = (blockIdx.x * 8 + warp) * 8;
  if (f0 >= F) return;
  const int e = pl.active[ai], p0 = pl.act_off[ai], p1 = pl.act_off[ai + 1];
  const int f = min(f0 + g, F - 1);
  const uint16_t* w0 = w_gu + (size_t(e) * 2 * F + f) * H + 8 * c;
  const uint16_t* w1 = w_gu + (size_t(e) * 2 * F + F + f) * H + 8 * c;
  for (int pp = p0; pp < p1; pp += 8) {
    const int np = min(8, p1 - pp);
    const bool tok = g < np;
    const uint16_t* xr = u + size_t(tok ? pl.pairs[pp + g] / k : 0) * H + 8 * c;
    float acc[4];
    expert_rows_mma(w0, w1, xr, tok, H, acc);
    // (row g = gate of unit f0+g, row g+8 = its up) x (pairs pp+2c, pp+2c+1)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int col = 2 * c + j;
      if (col < np && f0 + g < F)
        a[size_t(pl.pairs[pp + col]) * F + f0 + g] = f2bf(siluf_(acc[j]) * acc[2 + j]);
    }
  }
}

// grid (ceil(H / 128), max active experts); two CTAs per SM as above
__global__ void __launch_bounds__(256, 2) moe_down_mma_kernel(
    const uint16_t* __restrict__ a, const uint16_t* __restrict__ w_dn, int H, int F, MoePlan pl,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int T, int k, int E,
    int* __restrict__ cnt, float* __restrict__ y, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int na = *pl.n_active;
  const int ai = blockIdx.y;
  if (ai >= max(na, 1)) return;   // uniform over the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int h0 = blockIdx.x * kMmaRowsDown + warp * 16;
  if (ai < na && h0 < H) {
    const int e = pl.active[ai], p0 = pl.act_off[ai], p1 = pl.act_off[ai + 1];
    const uint16_t* w0 = w_dn + (size_t(e) * H + min(h0 + g, H - 1)) * F + 8 * c;
    const uint16_t* w1 = w_dn + (size_t(e) * H + min(h0 + g + 8, H - 1)) * F + 8 * c;
    for (int pp = p0; pp < p1; pp += 8) {
      const int np = min(8, p1 - pp);
      const bool tok = g < np;
      const uint16_t* xr = a + size_t(tok ? pl.pairs[pp + g] : 0) * F + 8 * c;
      float acc[4];
      expert_rows_mma(w0, w1, xr, tok, F, acc);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 2 * c + j;
        if (col < np) {
          const size_t yo = size_t(pl.pairs[pp + col]) * H;
          if (h0 + g < H) y[yo + h0 + g] = acc[j];
          if (h0 + g + 8 < H) y[yo + h0 + g + 8] = acc[2 + j];
        }
      }
    }
  }
  __shared__ int s_last;
  // the CTA barrier orders every thread's y stores before thread 0's device-scope fence,
  // which releases them with the counter increment
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(cnt + blockIdx.x, 1) == max(na, 1) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int hb = blockIdx.x * kMmaRowsDown;
  const int nh = min(kMmaRowsDown, H - hb);
  for (int i = threadIdx.x; i < T * nh; i += blockDim.x) {
    const int t = i / nh, h = hb + (i - t * nh);
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[size_t(t) * k + j];
      if (e < 0 || e >= E) continue;
      s = fmaf(topk_w[size_t(t) * k + j], __ldcg(y + (size_t(t) * k + j) * H + h), s);
    }
    out[size_t(t) * H + h] = f2bf(s);
  }
}

// NVFP4 expert weights (beam_moe_nvfp4). The expert products run on mma.sync in f16: an e2m1
// weight times its e4m3 block scale has at most 6 significant bits and lies in [2^-10, 2688],
// so it is exact in f16, and so are the BF16 activations of normal f16 magnitude; the FP32
// matrix scale multiplies the FP32 accumulator. A warp's 16 weight rows are the A operand and up
// to 8 of the expert's pairs the columns of B. Lane (g, c) loads, per 128-element block of a
// row, the 16 bytes holding elements [32c, 32c + 32) and their two block scales (a 2-byte load);
// the k order inside the block is permuted the same way for the token side, so the 32
// elements serve the block's 8 k16 steps (step s takes elements 4s .. 4s+3).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Eight e2m1 codes (four bytes, even element in the low nibble) -> four f16x2 words, exactly.
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t* r) {
  asm("{.reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4; cvt.rn.f16x2.e2m1x2 %0, b0;"
      " cvt.rn.f16x2.e2m1x2 %1, b1; cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3;}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}
// Two e4m3 codes -> f16x2 (exact), then each broadcast to both halves.
__device__ __forceinline__ void e4m3x2_scales(uint16_t codes, uint32_t& lo2, uint32_t& hi2) {
  uint32_t h2;
  asm("{.reg .b16 c; mov.b16 c, %1; cvt.rn.f16x2.e4m3x2 %0, c;}" : "=r"(h2) : "h"(codes));
  lo2 = __byte_perm(h2, 0, 0x1010);
  hi2 = __byte_perm(h2, 0, 0x3232);
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

constexpr int kFp4U = 2;   // 128-element blocks per load group; two groups are in flight
struct Fp4Group {
  uint4 q[kFp4U][2];
  uint16_t sc[kFp4U][2];
};
__device__ __forceinline__ void fp4_load_group(Fp4Group& G, const uint8_t* w0, const uint8_t* w1,
                                               const uint8_t* s0, const uint8_t* s1, int b0,
                                               int nb) {
#pragma unroll
  for (int u = 0; u < kFp4U; ++u) {
    const int b = min(b0 + u, nb - 1);
    G.q[u][0] = ld_stream(w0 + size_t(b) * 64);
    G.q[u][1] = ld_stream(w1 + size_t(b) * 64);
    G.sc[u][0] = __ldg(reinterpret_cast<const uint16_t*>(s0 + size_t(b) * 8));
    G.sc[u][1] = __ldg(reinterpret_cast<const uint16_t*>(s1 + size_t(b) * 8));
  }
}
__device__ __forceinline__ void fp4_block_mma(const uint4 (&q)[2], const uint16_t (&sc)[2],
                                              const uint16_t* xb, bool tok, float (&acc)[4],
                                              float (&acc2)[4]) {
  uint32_t xv[16];
  if (tok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t = *reinterpret_cast<const uint4*>(xb + 8 * i);
      xv[4 * i] = t.x;
      xv[4 * i + 1] = t.y;
      xv[4 * i + 2] = t.z;
      xv[4 * i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = 0u;
  }
  uint32_t w[2][16];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    uint32_t slo, shi;
    e4m3x2_scales(sc[r], slo, shi);
    const uint32_t qw[4] = {q[r].x, q[r].y, q[r].z, q[r].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e2m1x8_to_f16(qw[i], &w[r][4 * i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) w[r][4 * i + e] = hmul2(w[r][4 * i + e], i < 2 ? slo : shi);
    }
  }
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    if (st & 1)
      mma_f16_16816(acc2, w[0][2 * st], w[1][2 * st], w[0][2 * st + 1], w[1][2 * st + 1],
                    xv[2 * st], xv[2 * st + 1]);
    else
      mma_f16_16816(acc, w[0][2 * st], w[1][2 * st], w[0][2 * st + 1], w[1][2 * st + 1],
                    xv[2 * st], xv[2 * st + 1]);
  }
}

// acc (rows g, g+8; columns = pairs 2c, 2c+1) = W[rows] . X^T over the 128-element blocks
// [bb, nb); w0 / w1: the two rows' codes (bytes, already offset by 16c), s0 / s1: their block
// scales (offset by 2c), xr: the lane's token (f16, offset by 32c), tok: whether the lane has a
// token. The loads of the next group of blocks are issued before the current group is
// converted and multiplied.
__device__ __forceinline__ void fp4_rows_mma(const uint8_t* w0, const uint8_t* w1,
                                             const uint8_t* s0, const uint8_t* s1,
                                             const uint16_t* xr, bool tok, int bb, int nb,
                                             float (&acc)[4]) {
  float acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0.f;
  // blocks [bb, nb) of the rows
  Fp4Group cur, nxt;
  fp4_load_group(cur, w0, w1, s0, s1, bb, nb);
  for (int b0 = bb; b0 < nb; b0 += kFp4U) {
    if (b0 + kFp4U < nb) fp4_load_group(nxt, w0, w1, s0, s1, b0 + kFp4U, nb);
#pragma unroll
    for (int u = 0; u < kFp4U; ++u)
      if (b0 + u < nb) fp4_block_mma(cur.q[u], cur.sc[u], xr + size_t(b0 + u) * 128, tok, acc, acc2);
    cur = nxt;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] += acc2[i];
}

// With KS > 1, KS warps share a row block, each taking a 1/KS share of its K blocks, and add
// their partial tiles in order through shared memory: a warp's chain of dependent weight loads
// is KS times shorter and the grid has KS times the CTAs, which few tokens (few active experts,
// a grid under one wave) need; with many tokens the grid is large enough without it.
constexpr int kFp4KSMaxT = 4;   // K split up to this many tokens, else KS = 1
template <int KS>
__device__ __forceinline__ bool fp4_reduce_ks(float (&acc)[4], float (*red)[32][4]) {
  if (KS == 1) return true;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) red[warp][lane][i] = acc[i];
  __syncthreads();
  if (warp % KS != 0) return false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v = red[warp][lane][i];
#pragma unroll
    for (int j = 1; j < KS; ++j) v += red[warp + j][lane][i];
    acc[i] = v;
  }
  return true;
}

// u (bf16) -> u16 (f16) for the expert products; zeroes the down kernel's completion counters.
__global__ void __launch_bounds__(256) fp4_prep_kernel(const uint16_t* __restrict__ u, int n,
                                                       uint16_t* __restrict__ u16,
                                                       int* __restrict__ cnt, int n_cnt) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_cnt) cnt[i] = 0;
  if (i < n) u16[i] = f32_to_f16_bits(bf2f(u[i]));
}

// grid (ceil(F / (64 / KS)), max active experts); a row block is 8 units (gate rows f0..f0+7
// and the matching up rows), KS warps per row block. a16[pair][f] = f16(bf16(silu(gate) * up)).
template <int KS>
__global__ void __launch_bounds__(256, 3) moe_gate_up_fp4_kernel(
    const uint16_t* __restrict__ u16, beam_nvfp4_experts W, int H, int F, int k, MoePlan pl,
    const int32_t* __restrict__ direct, int E, uint16_t* __restrict__ a16) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8][32][4];
  const int ai = blockIdx.y;
  if (ai >= (direct != nullptr ? k : *pl.n_active)) return;   // uniform over the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int ks = warp % KS;
  const int f0 = (blockIdx.x * (8 / KS) + warp / KS) * 8;
  ExpertSlot es;
  if (!expert_slot(pl, direct, E, ai, es)) {   // uniform over the CTA
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(BEAM_DEV_BAD_EXPERT);
    return;
  }
  const int f = min(f0 + g, F - 1);
  const size_t rg = size_t(es.e) * 2 * F + f, ru = rg + F;
  const uint8_t* w0 = W.gate_up + rg * (H / 2) + 16 * c;
  const uint8_t* w1 = W.gate_up + ru * (H / 2) + 16 * c;
  const uint8_t* s0 = W.gate_up_scale + rg * (H / 16) + 2 * c;
  const uint8_t* s1 = W.gate_up_scale + ru * (H / 16) + 2 * c;
  const float gs = W.gate_up_global[es.e];
  const int nb = H >> 7, bb = ks * nb / KS, be = (ks + 1) * nb / KS;
  for (int pp = es.p0; pp < es.p1; pp += 8) {
    const int np = min(8, es.p1 - pp);
    const bool tok = g < np;
    const uint16_t* xr = u16 + size_t(tok ? pair_at(pl, direct, pp + g) / k : 0) * H + 32 * c;
    float acc[4];
    fp4_rows_mma(w0, w1, s0, s1, xr, tok, bb, be, acc);
    if (fp4_reduce_ks<KS>(acc, red)) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 2 * c + j;
        if (col < np && f0 + g < F) {
          const float a = round_bf(siluf_(acc[j] * gs) * (acc[2 + j] * gs));
          a16[size_t(pair_at(pl, direct, pp + col)) * F + f0 + g] = f32_to_f16_bits(a);
        }
      }
    }
    if (KS > 1) __syncthreads();   // the reduction buffer is free for the next pass
  }
}

// grid (ceil(H / (128 / KS)), max active experts); a row block is 16 rows h, KS warps per row
// block; y[pair][h] in FP32; the last CTA of each column of rows combines them for every token,
// slots in order.
template <int KS>
__global__ void __launch_bounds__(256, 3) moe_down_fp4_kernel(
    const uint16_t* __restrict__ a16, beam_nvfp4_experts W, int H, int F, MoePlan pl,
    const int32_t* __restrict__ direct, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, int T, int k, int E, int* __restrict__ cnt,
    float* __restrict__ y, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8][32][4];
  const int na = direct != nullptr ? k : *pl.n_active;
  const int ai = blockIdx.y;
  if (ai >= max(na, 1)) return;   // uniform over the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  constexpr int kRows = 128 / KS;   // rows h per CTA
  const int ks = warp % KS;
  const int h0 = blockIdx.x * kRows + (warp / KS) * 16;
  ExpertSlot es;
  if (ai < na && expert_slot(pl, direct, E, ai, es)) {   // uniform over the CTA
    const size_t r0 = size_t(es.e) * H + min(h0 + g, H - 1);
    const size_t r1 = size_t(es.e) * H + min(h0 + g + 8, H - 1);
    const uint8_t* w0 = W.down + r0 * (F / 2) + 16 * c;
    const uint8_t* w1 = W.down + r1 * (F / 2) + 16 * c;
    const uint8_t* s0 = W.down_scale + r0 * (F / 16) + 2 * c;
    const uint8_t* s1 = W.down_scale + r1 * (F / 16) + 2 * c;
    const float gs = W.down_global[es.e];
    const int nb = F >> 7, bb = ks * nb / KS, be = (ks + 1) * nb / KS;
    for (int pp = es.p0; pp < es.p1; pp += 8) {
      const int np = min(8, es.p1 - pp);
      const bool tok = g < np;
      const uint16_t* xr = a16 + size_t(tok ? pair_at(pl, direct, pp + g) : 0) * F + 32 * c;
      float acc[4];
      fp4_rows_mma(w0, w1, s0, s1, xr, tok, bb, be, acc);
      if (fp4_reduce_ks<KS>(acc, red)) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int col = 2 * c + j;
          if (col < np) {
            const size_t yo = size_t(pair_at(pl, direct, pp + col)) * H;
            if (h0 + g < H) y[yo + h0 + g] = acc[j] * gs;
            if (h0 + g + 8 < H) y[yo + h0 + g + 8] = acc[2 + j] * gs;
          }
        }
      }
      if (KS > 1) __syncthreads();   // the reduction buffer is free for the next pass
    }
  }
  __shared__ int s_last;
  // the CTA barrier orders every thread's y stores before thread 0's device-scope fence,
  // which releases them with the counter increment
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(cnt + blockIdx.x, 1) == max(na, 1) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int hb = blockIdx.x * kRows;
  const int nh = min(kRows, H - hb);
  for (int i = threadIdx.x; i < T * nh; i += blockDim.x) {
    const int t = i / nh, h = hb + (i - t * nh);
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[size_t(t) * k + j];
      if (e < 0 || e >= E) continue;
      s = fmaf(topk_w[size_t(t) * k + j], __ldcg(y + (size_t(t) * k + j) * H + h), s);
    }
    out[size_t(t) * H + h] = f2bf(s);
  }
}

// ------------------------------------------------------------------------------------------
// NVFP4 experts from kMoeGemmMinT tokens: the grouped BF16 tensor-core GEMMs on dequantised
// weights. An e2m1 value times its e4m3 block scale has at most 6 significant bits and lies
// in [2^-10, 2688], so it is exact in BF16: the selected experts' weights are expanded to BF16
// kFp4Chunk experts at a time into workspace scratch, and the grouped GEMMs run over that
// chunk's jobs with each expert's FP32 matrix scale applied to the FP32 accumulators (the
// same products as the oracle's exact dequantisation; activations stay BF16).
// ------------------------------------------------------------------------------------------
constexpr int kFp4Chunk = 16;   // experts dequantised per pass

// Chunk `chunk` of the active experts: expert a = chunk * kFp4Chunk + blockIdx.y. Each thread
// expands 32 elements of one row (16 code bytes and their two block scales) to BF16.
__global__ void __launch_bounds__(256) fp4_dequant_kernel(beam_nvfp4_experts W, int H, int F,
                                                          MoePlan pl, int chunk,
                                                          uint16_t* __restrict__ gu_bf,
                                                          uint16_t* __restrict__ dn_bf) {
  pdl_trigger();
  pdl_wait();   // the previous chunk's GEMMs have finished reading the scratch
  const int g = blockIdx.y, a = chunk * kFp4Chunk + g;
  if (a >= *pl.n_active) return;
  const int e = pl.active[a];
  const size_t n_gu = size_t(2) * F * (H / 32), n_dn = size_t(H) * (F / 32);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_gu + n_dn;
       i += size_t(gridDim.x) * blockDim.x) {
    const bool gu = i < n_gu;
    const size_t j = gu ? i : i - n_gu;
    const int K = gu ? H : F;
    const size_t row = j / (K / 32), c32 = j - row * (K / 32);   // 32-element group in the row
    const size_t erow = (gu ? size_t(e) * 2 * F : size_t(e) * H) + row;
    const uint8_t* codes = (gu ? W.gate_up : W.down) + erow * (K / 2) + c32 * 16;
    const uint8_t* scl = (gu ? W.gate_up_scale : W.down_scale) + erow * (K / 16) + c32 * 2;
    const uint4 q = *reinterpret_cast<const uint4*>(codes);
    uint32_t slo, shi;
    e4m3x2_scales(*reinterpret_cast<const uint16_t*>(scl), slo, shi);
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
    uint32_t o[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t h[4];
      e2m1x8_to_f16(qw[k], h);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t v = hmul2(h[t], k < 2 ? slo : shi);   // exact in f16
        float lo, hi;
        asm("{.reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b;}"
            : "=f"(lo), "=f"(hi)
            : "r"(v));
        o[4 * k + t] = pack_bf2(lo, hi);   // exact in BF16
      }
    }
    uint4* dst = reinterpret_cast<uint4*>((gu ? gu_bf + size_t(g) * 2 * F * H
                                              : dn_bf + size_t(g) * H * F) +
                                          row * K + c32 * 32);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
  }
}

// The jobs of chunk `chunk` of `csize` active experts (the plan's jobs, in active-expert order,
// are contiguous per expert): group = the expert's place in the chunk, the tile-order field
// recomputed for the chunk's list; and, when given, the chunk's FP32 matrix scales.
__global__ void moe_chunk_jobs_kernel(MoePlan pl, int chunk, int csize,
                                      const float* __restrict__ gu_global,
                                      const float* __restrict__ dn_global,
                                      int4* __restrict__ cj, int* __restrict__ cn,
                                      float* __restrict__ sgu, float* __restrict__ sdn) {
  pdl_trigger();
  pdl_wait();   // the previous chunk's GEMMs have finished reading the chunk's list
  if (threadIdx.x != 0) return;
  const int na = *pl.n_active, nj = *pl.n_jobs;
  const int a0 = chunk * csize, a1 = min(a0 + csize, na);
  int n = 0, a = -1, prev_e = -1, j_local_first = 0;
  for (int j = 0; j < nj; ++j) {
    const int4 jb = pl.jobs[j];
    if (jb.x != prev_e) {   // next active expert (jobs follow the active list)
      ++a;
      prev_e = jb.x;
      j_local_first = n;
    }
    if (a < a0) continue;
    if (a >= a1) break;
    const int cnt = jb.w >> 20;
    cj[n++] = make_int4(a - a0, jb.y, jb.z, j_local_first | (cnt << 20));
  }
  for (int g = 0; gu_global != nullptr && g < a1 - a0; ++g) {
    const int e = pl.active[a0 + g];
    sgu[g] = gu_global[e];
    sdn[g] = dn_global[e];
  }
  *cn = n;
}

// ------------------------------------------------------------------------------------------
// FP8 (e4m3, one FP32 scale per 128 x 128 block) expert weights, decode: the NVFP4 kernels'
// layout with one byte per element. Lane (g, c) loads, per 128-element block of each of its
// two rows, the 32 bytes of elements [32c, 32c + 32) (two 16-byte loads); cvt.rn.f16x2.e4m3x2
// turns each code pair into f16 exactly; the block's 8 k16 steps accumulate into a fresh FP32
// partial, which the block's scale (one per MMA row half: the gate/up kernel's upper and lower
// 8 rows are gate and up rows with their own scale blocks) multiplies into the accumulator.
// ------------------------------------------------------------------------------------------
// Four e4m3 codes (one word, first code in the low byte) -> two f16x2 words, exactly.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{.reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b;}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

struct Fp8Block {
  uint4 q[2][2];   // [row][half]: 32 codes per row
  float sc[2];     // scale of the block for rows g and g + 8
};

__device__ __forceinline__ void fp8_load_block(Fp8Block& B, const uint8_t* w0, const uint8_t* w1,
                                               const float* s0, const float* s1, int b, int nb) {
  b = min(b, nb - 1);
  B.q[0][0] = ld_stream(w0 + size_t(b) * 128);
  B.q[0][1] = ld_stream(w0 + size_t(b) * 128 + 16);
  B.q[1][0] = ld_stream(w1 + size_t(b) * 128);
  B.q[1][1] = ld_stream(w1 + size_t(b) * 128 + 16);
  B.sc[0] = __ldg(s0 + b);
  B.sc[1] = __ldg(s1 + b);
}

__device__ __forceinline__ void fp8_block_mma(const Fp8Block& B, const uint16_t* xb, bool tok,
                                              float (&acc)[4]) {
  uint32_t xv[16];
  if (tok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t = *reinterpret_cast<const uint4*>(xb + 8 * i);
      xv[4 * i] = t.x;
      xv[4 * i + 1] = t.y;
      xv[4 * i + 2] = t.z;
      xv[4 * i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) xv[i] = 0u;
  }
  uint32_t w[2][16];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t qw[8] = {B.q[r][0].x, B.q[r][0].y, B.q[r][0].z, B.q[r][0].w,
                            B.q[r][1].x, B.q[r][1].y, B.q[r][1].z, B.q[r][1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) e4m3x4_to_f16(qw[i], w[r][2 * i], w[r][2 * i + 1]);
  }
  float p[4] = {0.f, 0.f, 0.f, 0.f}, p2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int st = 0; st < 8; ++st) {
    if (st & 1)
      mma_f16_16816(p2, w[0][2 * st], w[1][2 * st], w[0][2 * st + 1], w[1][2 * st + 1],
                    xv[2 * st], xv[2 * st + 1]);
    else
      mma_f16_16816(p, w[0][2 * st], w[1][2 * st], w[0][2 * st + 1], w[1][2 * st + 1],
                    xv[2 * st], xv[2 * st + 1]);
  }
  acc[0] = fmaf(B.sc[0], p[0] + p2[0], acc[0]);
  acc[1] = fmaf(B.sc[0], p[1] + p2[1], acc[1]);
  acc[2] = fmaf(B.sc[1], p[2] + p2[2], acc[2]);
  acc[3] = fmaf(B.sc[1], p[3] + p2[3], acc[3]);
}

// acc (rows g, g+8; columns = pairs 2c, 2c+1) over the 128-element blocks [bb, be); w0 / w1:
// the two rows' codes (offset by 32c), s0 / s1: their scale rows (one FP32 per block), xr: the
// lane's token in f16 (offset by 32c). The next block's loads are issued before the current
// block is converted and multiplied.
__device__ __forceinline__ void fp8_rows_mma(const uint8_t* w0, const uint8_t* w1,
                                             const float* s0, const float* s1,
                                             const uint16_t* xr, bool tok, int bb, int be,
                                             float (&acc)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0.f;
  if (bb >= be) return;
  Fp8Block cur, nxt;
  fp8_load_block(cur, w0, w1, s0, s1, bb, be);
  for (int b = bb; b < be; ++b) {
    if (b + 1 < be) fp8_load_block(nxt, w0, w1, s0, s1, b + 1, be);
    fp8_block_mma(cur, xr + size_t(b) * 128, tok, acc);
    cur = nxt;
  }
}

// grid (ceil(F / (64 / KS)), max active experts); a row block is 8 units (gate rows f0..f0+7
// and the matching up rows), KS warps per row block. a16[pair][f] = f16(bf16(silu(gate) * up)).
template <int KS>
__global__ void __launch_bounds__(256, 3) moe_gate_up_fp8_kernel(
    const uint16_t* __restrict__ u16, beam_fp8_experts W, int H, int F, int k, MoePlan pl,
    const int32_t* __restrict__ direct, int E, uint16_t* __restrict__ a16) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8][32][4];
  const int ai = blockIdx.y;
  if (ai >= (direct != nullptr ? k : *pl.n_active)) return;   // uniform over the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int ks = warp % KS;
  const int f0 = (blockIdx.x * (8 / KS) + warp / KS) * 8;
  ExpertSlot es;
  if (!expert_slot(pl, direct, E, ai, es)) {   // uniform over the CTA
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(BEAM_DEV_BAD_EXPERT);
    return;
  }
  const int f = min(f0 + g, F - 1);
  const size_t rg = size_t(es.e) * 2 * F + f, ru = rg + F;
  const int nb = H >> 7;
  const uint8_t* w0 = W.gate_up + rg * H + 32 * c;
  const uint8_t* w1 = W.gate_up + ru * H + 32 * c;
  // scale rows: expert e's [2F/128][H/128] grid, the row block of the gate and of the up row
  const float* s0 = W.gate_up_scale + (size_t(es.e) * (2 * F / 128) + f / 128) * nb;
  const float* s1 = W.gate_up_scale + (size_t(es.e) * (2 * F / 128) + (F + f) / 128) * nb;
  const int bb = ks * nb / KS, be = (ks + 1) * nb / KS;
  for (int pp = es.p0; pp < es.p1; pp += 8) {
    const int np = min(8, es.p1 - pp);
    const bool tok = g < np;
    const uint16_t* xr = u16 + size_t(tok ? pair_at(pl, direct, pp + g) / k : 0) * H + 32 * c;
    float acc[4];
    fp8_rows_mma(w0, w1, s0, s1, xr, tok, bb, be, acc);
    if (fp4_reduce_ks<KS>(acc, red)) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 2 * c + j;
        if (col < np && f0 + g < F) {
          const float a = round_bf(siluf_(acc[j]) * acc[2 + j]);
          a16[size_t(pair_at(pl, direct, pp + col)) * F + f0 + g] = f32_to_f16_bits(a);
        }
      }
    }
    if (KS > 1) __syncthreads();   // the reduction buffer is free for the next pass
  }
}

// grid (ceil(H / (128 / KS)), max active experts); a row block is 16 rows h, KS warps per row
// block; y[pair][h] in FP32; the last CTA of each column of rows combines them for every token,
// slots in order.
template <int KS>
__global__ void __launch_bounds__(256, 3) moe_down_fp8_kernel(
    const uint16_t* __restrict__ a16, beam_fp8_experts W, int H, int F, MoePlan pl,
    const int32_t* __restrict__ direct, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, int T, int k, int E, int* __restrict__ cnt,
    float* __restrict__ y, uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8][32][4];
  const int na = direct != nullptr ? k : *pl.n_active;
  const int ai = blockIdx.y;
  if (ai >= max(na, 1)) return;   // uniform over the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  constexpr int kRows = 128 / KS;   // rows h per CTA
  const int ks = warp % KS;
  const int h0 = blockIdx.x * kRows + (warp / KS) * 16;
  ExpertSlot es;
  if (ai < na && expert_slot(pl, direct, E, ai, es)) {   // uniform over the CTA
    const int hr0 = min(h0 + g, H - 1), hr1 = min(h0 + g + 8, H - 1);
    const size_t r0 = size_t(es.e) * H + hr0, r1 = size_t(es.e) * H + hr1;
    const int nb = F >> 7;
    const uint8_t* w0 = W.down + r0 * F + 32 * c;
    const uint8_t* w1 = W.down + r1 * F + 32 * c;
    const float* s0 = W.down_scale + (size_t(es.e) * (H / 128) + hr0 / 128) * nb;
    const float* s1 = W.down_scale + (size_t(es.e) * (H / 128) + hr1 / 128) * nb;
    const int bb = ks * nb / KS, be = (ks + 1) * nb / KS;
    for (int pp = es.p0; pp < es.p1; pp += 8) {
      const int np = min(8, es.p1 - pp);
      const bool tok = g < np;
      const uint16_t* xr = a16 + size_t(tok ? pair_at(pl, direct, pp + g) : 0) * F + 32 * c;
      float acc[4];
      fp8_rows_mma(w0, w1, s0, s1, xr, tok, bb, be, acc);
      if (fp4_reduce_ks<KS>(acc, red)) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int col = 2 * c + j;
          if (col < np) {
            const size_t yo = size_t(pair_at(pl, direct, pp + col)) * H;
            if (h0 + g < H) y[yo + h0 + g] = acc[j];
            if (h0 + g + 8 < H) y[yo + h0 + g + 8] = acc[2 + j];
          }
        }
      }
      if (KS > 1) __syncthreads();   // the reduction buffer is free for the next pass
    }
  }
  __shared__ int s_last;
  // the CTA barrier orders every thread's y stores before thread 0's device-scope fence,
  // which releases them with the counter increment
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(cnt + blockIdx.x, 1) == max(na, 1) - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int hb = blockIdx.x * kRows;
  const int nh = min(kRows, H - hb);
  for (int i = threadIdx.x; i < T * nh; i += blockDim.x) {
    const int t = i / nh, h = hb + (i - t * nh);
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[size_t(t) * k + j];
      if (e < 0 || e >= E) continue;
      s = fmaf(topk_w[size_t(t) * k + j], __ldcg(y + (size_t(t) * k + j) * H + h), s);
    }
    out[size_t(t) * H + h] = f2bf(s);
  }
}

__global__ void moe_combine_kernel(const float* __restrict__ y, const float* __restrict__ topk_w,
                                   const int32_t* __restrict__ idx, int T, int H, int k, int E,
                                   uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= size_t(T) * H) return;
  const int t = int(i / H), h = int(i - size_t(t) * H);
  float s = 0.f;
  for (int j = 0; j < k; ++j) {
    const int e = idx[size_t(t) * k + j];
    if (e < 0 || e >= E) continue;
    s = fmaf(topk_w[size_t(t) * k + j], y[(size_t(t) * k + j) * H + h], s);
  }
  out[i] = f2bf(s);
}

// moe_combine_kernel four columns at a time (H % 4 == 0): 16-byte loads of the FP32 rows.
__global__ void __launch_bounds__(256) moe_combine4_kernel(const float* __restrict__ y,
                                                           const float* __restrict__ topk_w,
                                                           const int32_t* __restrict__ idx, int T,
                                                           int H, int k, int E,
                                                           uint16_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int hq = H >> 2;
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= size_t(T) * hq) return;
  const int t = int(i / hq), h = int(i - size_t(t) * hq) * 4;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int e = idx[size_t(t) * k + j];
    if (e < 0 || e >= E) continue;
    const float w = topk_w[size_t(t) * k + j];
    const float4 v = __ldcs(reinterpret_cast<const float4*>(y + (size_t(t) * k + j) * H + h));
    s.x = fmaf(w, v.x, s.x);
    s.y = fmaf(w, v.y, s.y);
    s.z = fmaf(w, v.z, s.z);
    s.w = fmaf(w, v.w, s.w);
  }
  *reinterpret_cast<uint2*>(out + size_t(t) * H + h) =
      make_uint2(pack_bf2(s.x, s.y), pack_bf2(s.z, s.w));
}

// Rows of u in expert-sorted pair order: us[i] = u[pairs[i] / k].
__global__ void gather_rows_kernel(const uint16_t* __restrict__ u, int H, int k, MoePlan pl,
                                   int P, uint16_t* __restrict__ us) {
  pdl_trigger();
  pdl_wait();
  const int nv = H / 8;
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= size_t(P) * nv) return;
  const int r = int(i / nv), c = int(i - size_t(r) * nv);
  const int tok = pl.pairs[r] / k;
  reinterpret_cast<uint4*>(us + size_t(r) * H)[c] =
      reinterpret_cast<const uint4*>(u + size_t(tok) * H)[c];
}

int max_jobs(int P, int E) { return (P + 127) / 128 + (P < E ? P : E); }

// Decode form for up to kMoeSmallT tokens (every expert then meets at most kMoeSmallT pairs).
constexpr int kMoeSmallT = 4;

MoePlan carve_plan(Carver& cv, int E, int P, bool grouped) {
  MoePlan pl;
  pl.n_active = cv.take<int>(1);
  pl.active = cv.take<int>(E);
  pl.act_off = cv.take<int>(E + 1);
  pl.pairs = cv.take<int>(P);
  pl.jobs = grouped ? cv.take<int4>(max_jobs(P, E)) : nullptr;
  pl.n_jobs = grouped ? cv.take<int>(1) : nullptr;
  return pl;
}


// FP8 experts from kMoeGemmMinT tokens. A code times its FP32 block scale is not a BF16 number
// in general, so each weight is stored as two BF16 parts, hi = bf16(w) and lo = bf16(w - hi)
// (w to ~16 significant bits), side by side in a row of 2K columns, and the grouped GEMMs
// run over K twice against the same activations (gemm_grouped's a_twice). kFp4Chunk / 2
// experts per pass fill the same scratch as the NVFP4 path.
constexpr int kFp8Chunk = kFp4Chunk / 2;

__global__ void __launch_bounds__(256) fp8_dequant_kernel(beam_fp8_experts W, int H, int F,
                                                          MoePlan pl, int chunk,
                                                          uint16_t* __restrict__ gu_bf,
                                                          uint16_t* __restrict__ dn_bf) {
  pdl_trigger();
  pdl_wait();   // the previous chunk's GEMMs have finished reading the scratch
  const int g = blockIdx.y, a = chunk * kFp8Chunk + g;
  if (a >= *pl.n_active) return;
  const int e = pl.active[a];
  const size_t n_gu = size_t(2) * F * (H / 16), n_dn = size_t(H) * (F / 16);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_gu + n_dn;
       i += size_t(gridDim.x) * blockDim.x) {
    const bool gu = i < n_gu;
    const size_t j = gu ? i : i - n_gu;
    const int K = gu ? H : F, R = gu ? 2 * F : H;
    const size_t row = j / (K / 16), c16 = j - row * (K / 16);   // 16-element group in the row
    const uint8_t* codes = (gu ? W.gate_up : W.down) + (size_t(e) * R + row) * K + c16 * 16;
    const float sc = (gu ? W.gate_up_scale : W.down_scale)[(size_t(e) * (R / 128) + row / 128) *
                                                               (K / 128) + (c16 * 16) / 128];
    const uint4 q = *reinterpret_cast<const uint4*>(codes);
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
      uint32_t h2[2];
      e4m3x4_to_f16(qw[k2], h2[0], h2[1]);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float x0, x1;
        asm("{.reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b;}"
            : "=f"(x0), "=f"(x1)
            : "r"(h2[t]));
        const float w0 = x0 * sc, w1 = x1 * sc;
        const uint32_t hh = pack_bf2(w0, w1);
        hi[2 * k2 + t] = hh;
        lo[2 * k2 + t] = pack_bf2(w0 - __uint_as_float(hh << 16), w1 - __uint_as_float(hh & 0xFFFF0000u));
      }
    }
    uint16_t* rowp = (gu ? gu_bf + size_t(g) * 2 * F * 2 * H : dn_bf + size_t(g) * H * 2 * F) +
                     row * 2 * K;
    uint4* dh = reinterpret_cast<uint4*>(rowp + c16 * 16);
    uint4* dl = reinterpret_cast<uint4*>(rowp + K + c16 * 16);
    dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
}

}  // namespace

size_t moe_ws_bytes(const beam_layer_cfg* c, int T) {
  const size_t P = size_t(T) * c->topk, E = c->n_experts;
  size_t b = 256 + align_up(E * 4, 256) + align_up((E + 1) * 4, 256) + align_up(P * 4, 256);
  b += align_up(P * c->d_ff_expert * 2, 256);
  const bool grouped = T >= kMoeGemmMinT;
  if (grouped) {
    b += align_up(size_t(max_jobs(int(P), int(E))) * 16, 256) + 256;
    b += align_up(P * c->hidden * 2, 256);                       // gathered inputs
    // NVFP4 experts: BF16 weights of kFp4Chunk experts, the chunk's jobs and matrix scales
    const size_t H = c->hidden, F = c->d_ff_expert;
    b += align_up(size_t(kFp4Chunk) * 2 * F * H * 2, 256) + align_up(size_t(kFp4Chunk) * H * F * 2, 256);
    b += align_up(size_t(max_jobs(int(P), int(E))) * 16, 256) + 3 * 256;
  }
  // FP32 per-pair rows and the down kernel's completion counters (decode forms)
  if (grouped || P > size_t(kFusedMaxPairs) || T < kMoeGemmMinT)
    b += align_up(P * c->hidden * 4, 256);
  if (T < kMoeGemmMinT) b += align_up(size_t(c->hidden / 8 + 1) * 4, 256);
  if (T < kMoeGemmMinT) b += align_up(size_t(T) * c->hidden * 2, 256);   // f16 tokens (NVFP4)
  return b;
}

size_t dense_ws_bytes(const beam_layer_cfg* c, int T) {
  return align_up(size_t(T) * c->d_ff_dense * 2, 256);
}

}  // namespace beam

extern "C" beam_status beam_moe(const beam_layer_cfg* cfg, const beam_bf16* u,
                                const int32_t* topk_idx, const float* topk_w,
                                const beam_bf16* w_gate_up, const beam_bf16* w_down, int T,
                                beam_bf16* out, void* ws, size_t ws_bytes, beam_stream_t stream) {
  using namespace beam;
  if (!cfg || T < 0 || !u || !topk_idx || !topk_w || !w_gate_up || !w_down || !out)
    return BEAM_ERR_INVALID_ARG;
  const int H = cfg->hidden, F = cfg->d_ff_expert, E = cfg->n_experts, k = cfg->topk;
  if (H <= 0 || (H & 7) || F <= 0 || (F & 7) || E <= 0 || k <= 0) return BEAM_ERR_INVALID_ARG;
  if (E > 4096) return BEAM_ERR_UNSUPPORTED;
  if (!aligned16(u) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(ws))
    return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  const int P = T * k;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carver cv{static_cast<char*>(ws), ws_bytes};
  const bool grouped = T >= kMoeGemmMinT && tc::gemm_supported(u, H, w_gate_up, H, H) &&
                       tc::gemm_supported(u, F, w_down, F, F);
  MoePlan pl = carve_plan(cv, E, P, grouped);
  uint16_t* act = cv.take<uint16_t>(size_t(P) * F);
  uint16_t* us = grouped ? cv.take<uint16_t>(size_t(P) * H) : nullptr;
  // 2..31 tokens: the tensor-core expert products (H and F multiples of 32)
  const bool mma = !grouped && T >= 2 && T < kMoeGemmMinT && (H & 31) == 0 && (F & 31) == 0;
  const bool small = !grouped && !mma && T <= kMoeSmallT;
  float* y = (grouped || small || mma || P > kFusedMaxPairs) ? cv.take<float>(size_t(P) * H) : nullptr;
  int* cnt = (small || mma) ? cv.take<int>(size_t(H / 8 + 1)) : nullptr;
  if (!cv.ok) return BEAM_ERR_INVALID_ARG;
  const int max_active = P < E ? P : E;
  if (grouped) {
    // plan -> gather -> grouped gate/up GEMM with the SwiGLU epilogue (sorted rows) -> grouped
    // down GEMM writing each row back to its (token, slot) pair -> weighted combine
    launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
    const size_t nv = size_t(P) * (H / 8);
    launch_pdl(gather_rows_kernel, dim3(unsigned((nv + 255) / 256)), dim3(256), 0, st, u, H, k, pl, P, us);
    const int mj = max_jobs(P, E);
    if (const cudaError_t err_ = tc::gemm_grouped(tc::kSwiGLU, us, P, H, H, w_gate_up, E * 2 * F, 2 * F, H, pl.jobs,
                         pl.n_jobs, mj, F, F, nullptr, act, F, st); err_ != cudaSuccess)
      return cuda_status(err_);
    if (const cudaError_t err_ = tc::gemm_grouped(tc::kF32, act, P, F, F, w_down, E * H, H, F, pl.jobs, pl.n_jobs, mj, H,
                         0, pl.pairs, y, H, st); err_ != cudaSuccess)
      return cuda_status(err_);
    if ((H & 3) == 0 && aligned16(out)) {
      const size_t n4 = size_t(T) * (H / 4);
      launch_pdl(moe_combine4_kernel, dim3(unsigned((n4 + 255) / 256)), dim3(256), 0, st, y,
                 topk_w, topk_idx, T, H, k, E, out);
    } else {
      const size_t n = size_t(T) * H;
      launch_pdl(moe_combine_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, y,
                 topk_w, topk_idx, T, H, k, E, out);
    }
    return launch_status();
  }
  if (mma) {
    const int n_cnt = (H + kMmaRowsDown - 1) / kMmaRowsDown;
    launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
    launch_pdl(moe_gate_up_mma_kernel, dim3((F + 63) / 64, max_active), dim3(256), 0, st, u,
               w_gate_up, H, F, k, pl, cnt, n_cnt, act);
    launch_pdl(moe_down_mma_kernel, dim3(n_cnt, max_active), dim3(256), 0, st, act, w_down, H, F,
               pl, topk_idx, topk_w, T, k, E, cnt, y, out);
    return launch_status();
  }
  if (small) {
    // decode: [plan] -> gate/up (SwiGLU) -> down rows per (expert, h) with the combine done by
    // the last CTA of each row block. One token needs no plan: its k slots are the active list.
    const bool direct = T == 1;
    const int32_t* dix = direct ? topk_idx : nullptr;
    const int na = direct ? k : max_active;
    const int nr = direct ? kDecodeDownNR : 1;
    const int n_cnt = (H + 8 * nr - 1) / (8 * nr);
    if (!direct)
      launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
    if (direct)
      launch_pdl(moe_gate_up_kernel<kDecodeGateUpU, 1, kDecodeGateUpFPW>,
                 dim3((F + 8 * kDecodeGateUpFPW - 1) / (8 * kDecodeGateUpFPW), na), dim3(256), 0, st,
                 u, w_gate_up, H, F, k, pl, dix, E, cnt, n_cnt, act);
    else
      launch_pdl(moe_gate_up_kernel<4, 4, 1>, dim3((F + 7) / 8, na), dim3(256), 0, st, u,
                 w_gate_up, H, F, k, pl, dix, E, cnt, n_cnt, act);
    if (direct)
      launch_pdl(moe_down_kernel<kDecodeDownU, 1, kDecodeDownNR>, dim3(n_cnt, na), dim3(256), 0, st, act,
                 w_down, H, F, pl, dix, topk_idx, topk_w, T, k, E, cnt, y, out);
    else
      launch_pdl(moe_down_kernel<8, 4, 1>, dim3(n_cnt, na), dim3(256), 0, st, act, w_down, H,
                 F, pl, dix, topk_idx, topk_w, T, k, E, cnt, y, out);
    return launch_status();
  }
  launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
  launch_pdl(moe_gate_up_kernel<4, 4, 1>, dim3((F + 7) / 8, max_active), dim3(256), 0, st, u,
             w_gate_up, H, F, k, pl, static_cast<const int32_t*>(nullptr), E,
             static_cast<int*>(nullptr), 0, act);
  if (P <= kFusedMaxPairs) {
    const int smem = 8 * P * int(sizeof(float));
    if (smem > 48 * 1024) {
      const cudaError_t err_ = cudaFuncSetAttribute(
          moe_down_combine_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (err_ != cudaSuccess) return cuda_status(err_);
    }
    launch_pdl(moe_down_combine_kernel<8>, dim3((H + 7) / 8), dim3(256), smem, st, act, w_down, topk_w, T, H, F, k,
                                                              pl, out);
  } else {
    launch_pdl(moe_down_kernel<8, 4, 1>, dim3((H + 7) / 8, max_active), dim3(256), 0, st, act,
               w_down, H, F, pl, static_cast<const int32_t*>(nullptr), topk_idx, topk_w, T, k, E,
               static_cast<int*>(nullptr), y, out);
    const size_t n = size_t(T) * H;
    launch_pdl(moe_combine_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, y, topk_w, topk_idx, T, H, k,
                                                                  E, out);
  }
  return launch_status();
}

extern "C" beam_status beam_dense_mlp(const beam_layer_cfg* cfg, const beam_bf16* u,
                                      const beam_bf16* w_gate_up, const beam_bf16* w_down, int T,
                                      beam_bf16* out, void* ws, size_t ws_bytes,
                                      beam_stream_t stream) {
  using namespace beam;
  if (!cfg || T < 0 || !u || !w_gate_up || !w_down || !out) return BEAM_ERR_INVALID_ARG;
  const int H = cfg->hidden, Fd = cfg->d_ff_dense;
  if (H <= 0 || (H & 7) || Fd <= 0 || (Fd & 7)) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(out) ||
      !aligned16(ws))
    return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carver cv{static_cast<char*>(ws), ws_bytes};
  uint16_t* act = cv.take<uint16_t>(size_t(T) * Fd);
  if (!cv.ok) return BEAM_ERR_INVALID_ARG;
  const bool tcore = T >= kGemmMinT && tc::gemm_supported(u, H, w_gate_up, H, H) &&
                     tc::gemm_supported(act, Fd, w_down, Fd, Fd);
  if (tcore) {
    if (const cudaError_t err_ = tc::gemm_swiglu(u, T, H, H, w_gate_up, Fd, H, act, Fd, st); err_ != cudaSuccess)
      return cuda_status(err_);
    if (const cudaError_t err_ = tc::gemm_bf16(act, T, Fd, Fd, w_down, H, Fd, out, H, true, st); err_ != cudaSuccess)
      return cuda_status(err_);
    return BEAM_OK;
  }
  if (const cudaError_t err_ = launch_gemv<kOutSwiGLU>(w_gate_up, Fd, H, u, T, nullptr, act, Fd, st, true); err_ != cudaSuccess)
    return cuda_status(err_);
  if (const cudaError_t err_ = launch_gemv<kOutBF16>(w_down, H, Fd, act, T, nullptr, out, H, st, true); err_ != cudaSuccess)
    return cuda_status(err_);
  return BEAM_OK;
}

extern "C" beam_status beam_moe_nvfp4(const beam_layer_cfg* cfg, const beam_bf16* u,
                                      const int32_t* topk_idx, const float* topk_w,
                                      const beam_nvfp4_experts* w, int T, beam_bf16* out,
                                      void* ws, size_t ws_bytes, beam_stream_t stream) {
  using namespace beam;
  if (!cfg || T < 0 || !u || !topk_idx || !topk_w || !w || !out) return BEAM_ERR_INVALID_ARG;
  const int H = cfg->hidden, F = cfg->d_ff_expert, E = cfg->n_experts, k = cfg->topk;
  if (H <= 0 || F <= 0 || E <= 0 || k <= 0) return BEAM_ERR_INVALID_ARG;
  if (!w->gate_up || !w->gate_up_scale || !w->gate_up_global || !w->down || !w->down_scale ||
      !w->down_global)
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(ws) || !aligned16(w->gate_up) || !aligned16(w->down) ||
      !aligned16(w->gate_up_scale) || !aligned16(w->down_scale))
    return BEAM_ERR_INVALID_ARG;
  if (E > 4096 || (H & 127) || (F & 127)) return BEAM_ERR_UNSUPPORTED;
  if (T == 0) return BEAM_OK;
  const int P = T * k;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carver cv{static_cast<char*>(ws), ws_bytes};
  if (T >= kMoeGemmMinT) {
    // plan -> gather -> per chunk of kFp4Chunk active experts: BF16 weights, the chunk's job
    // list, grouped gate/up and down GEMMs (matrix scales on the accumulators) -> combine
    if (!tc::gemm_supported(u, H, w->gate_up, H, H) || !tc::gemm_supported(u, F, w->down, F, F))
      return BEAM_ERR_UNSUPPORTED;
    MoePlan pl = carve_plan(cv, E, P, true);
    uint16_t* act = cv.take<uint16_t>(size_t(P) * F);
    uint16_t* us = cv.take<uint16_t>(size_t(P) * H);
    float* y = cv.take<float>(size_t(P) * H);
    const int mj = max_jobs(P, E);
    uint16_t* gu_bf = cv.take<uint16_t>(size_t(kFp4Chunk) * 2 * F * H);
    uint16_t* dn_bf = cv.take<uint16_t>(size_t(kFp4Chunk) * H * F);
    int4* cj = cv.take<int4>(size_t(mj));
    int* cn = cv.take<int>(1);
    float* sgu = cv.take<float>(kFp4Chunk);
    float* sdn = cv.take<float>(kFp4Chunk);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
    const size_t nv = size_t(P) * (H / 8);
    launch_pdl(gather_rows_kernel, dim3(unsigned((nv + 255) / 256)), dim3(256), 0, st, u, H, k, pl, P, us);
    const int max_active = P < E ? P : E;
    const int n_chunks = (max_active + kFp4Chunk - 1) / kFp4Chunk;
    const size_t per_expert = size_t(2) * F * (H / 32) + size_t(H) * (F / 32);
    const size_t want = (per_expert + 255) / 256;
    const unsigned dq_blocks = unsigned(want < 64 ? want : 64);
    for (int c = 0; c < n_chunks; ++c) {
      launch_pdl(fp4_dequant_kernel, dim3(dq_blocks, kFp4Chunk), dim3(256), 0, st, *w, H, F, pl,
                 c, gu_bf, dn_bf);
      launch_pdl(moe_chunk_jobs_kernel, dim3(1), dim3(32), 0, st, pl, c, kFp4Chunk,
                 w->gate_up_global, w->down_global, cj, cn, sgu, sdn);
      if (const cudaError_t err_ = tc::gemm_grouped(tc::kSwiGLU, us, P, H, H, gu_bf, kFp4Chunk * 2 * F,
                                                    2 * F, H, cj, cn, mj, F, F, nullptr, act, F, st, sgu);
          err_ != cudaSuccess)
        return cuda_status(err_);
      if (const cudaError_t err_ = tc::gemm_grouped(tc::kF32, act, P, F, F, dn_bf, kFp4Chunk * H, H, F,
                                                    cj, cn, mj, H, 0, pl.pairs, y, H, st, sdn);
          err_ != cudaSuccess)
        return cuda_status(err_);
    }
    if ((H & 3) == 0 && aligned16(out)) {
      const size_t n4 = size_t(T) * (H / 4);
      launch_pdl(moe_combine4_kernel, dim3(unsigned((n4 + 255) / 256)), dim3(256), 0, st, y,
                 topk_w, topk_idx, T, H, k, E, out);
    } else {
      const size_t n1 = size_t(T) * H;
      launch_pdl(moe_combine_kernel, dim3(unsigned((n1 + 255) / 256)), dim3(256), 0, st, y,
                 topk_w, topk_idx, T, H, k, E, out);
    }
    return launch_status();
  }
  MoePlan pl = carve_plan(cv, E, P, false);
  uint16_t* a16 = cv.take<uint16_t>(size_t(P) * F);
  float* y = cv.take<float>(size_t(P) * H);
  int* cnt = cv.take<int>(size_t(H / 8 + 1));
  uint16_t* u16 = cv.take<uint16_t>(size_t(T) * H);
  if (!cv.ok) return BEAM_ERR_INVALID_ARG;
  // one token: its k slots are the active list directly; more: the plan groups the pairs
  const bool direct = T == 1;
  const int32_t* dix = direct ? topk_idx : nullptr;
  const int na = direct ? k : (P < E ? P : E);
  // up to 4 tokens the gate/up rows are split four ways; the down rows (half as many K blocks)
  // four ways for one token, two ways for 2-4 (measured fastest each)
  const bool split = T <= kFp4KSMaxT;
  const int rows_down = !split ? 128 : T == 1 ? 32 : 64, units_up = split ? 16 : 64;
  const int n_cnt = (H + rows_down - 1) / rows_down;
  const int n = T * H;
  launch_pdl(fp4_prep_kernel, dim3((max(n, n_cnt) + 255) / 256), dim3(256), 0, st, u, n, u16, cnt,
             n_cnt);
  if (!direct)
    launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
  const dim3 gu((F + units_up - 1) / units_up, na), gd(n_cnt, na);
  if (split) {
    launch_pdl(moe_gate_up_fp4_kernel<4>, gu, dim3(256), 0, st, u16, *w, H, F, k, pl, dix, E, a16);
    if (T == 1)
      launch_pdl(moe_down_fp4_kernel<4>, gd, dim3(256), 0, st, a16, *w, H, F, pl, dix, topk_idx,
                 topk_w, T, k, E, cnt, y, out);
    else
      launch_pdl(moe_down_fp4_kernel<2>, gd, dim3(256), 0, st, a16, *w, H, F, pl, dix, topk_idx,
                 topk_w, T, k, E, cnt, y, out);
  } else {
    launch_pdl(moe_gate_up_fp4_kernel<1>, gu, dim3(256), 0, st, u16, *w, H, F, k, pl, dix, E, a16);
    launch_pdl(moe_down_fp4_kernel<1>, gd, dim3(256), 0, st, a16, *w, H, F, pl, dix, topk_idx,
               topk_w, T, k, E, cnt, y, out);
  }
  return launch_status();
}

extern "C" beam_status beam_moe_fp8(const beam_layer_cfg* cfg, const beam_bf16* u,
                                    const int32_t* topk_idx, const float* topk_w,
                                    const beam_fp8_experts* w, int T, beam_bf16* out, void* ws,
                                    size_t ws_bytes, beam_stream_t stream) {
  using namespace beam;
  if (!cfg || T < 0 || !u || !topk_idx || !topk_w || !w || !out || !w->gate_up ||
      !w->gate_up_scale || !w->down || !w->down_scale)
    return BEAM_ERR_INVALID_ARG;
  const int H = cfg->hidden, F = cfg->d_ff_expert, E = cfg->n_experts, k = cfg->topk;
  if (H <= 0 || F <= 0 || E <= 0 || k <= 0) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(ws) || !aligned16(w->gate_up) || !aligned16(w->down))
    return BEAM_ERR_INVALID_ARG;
  if (E > 4096 || (H & 127) || (F & 127)) return BEAM_ERR_UNSUPPORTED;
  if (T == 0) return BEAM_OK;
  const int P = T * k;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carver cv{static_cast<char*>(ws), ws_bytes};
  if (T >= kMoeGemmMinT) {
    // plan -> gather -> per chunk of kFp8Chunk active experts: BF16 high and low parts of the
    // weights, the chunk's job list, grouped gate/up and down GEMMs over K twice -> combine
    if (!tc::gemm_supported(u, H, w->gate_up, 2 * H, 2 * H) ||
        !tc::gemm_supported(u, F, w->down, 2 * F, 2 * F))
      return BEAM_ERR_UNSUPPORTED;
    MoePlan pl = carve_plan(cv, E, P, true);
    uint16_t* act = cv.take<uint16_t>(size_t(P) * F);
    uint16_t* us = cv.take<uint16_t>(size_t(P) * H);
    float* y = cv.take<float>(size_t(P) * H);
    const int mj = max_jobs(P, E);
    uint16_t* gu_bf = cv.take<uint16_t>(size_t(kFp4Chunk) * 2 * F * H);   // kFp8Chunk x 2 parts
    uint16_t* dn_bf = cv.take<uint16_t>(size_t(kFp4Chunk) * H * F);
    int4* cj = cv.take<int4>(size_t(mj));
    int* cn = cv.take<int>(1);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
    const size_t nv = size_t(P) * (H / 8);
    launch_pdl(gather_rows_kernel, dim3(unsigned((nv + 255) / 256)), dim3(256), 0, st, u, H, k, pl, P, us);
    const int max_active = P < E ? P : E;
    const int n_chunks = (max_active + kFp8Chunk - 1) / kFp8Chunk;
    const size_t per_expert = size_t(2) * F * (H / 16) + size_t(H) * (F / 16);
    const size_t want = (per_expert + 255) / 256;
    const unsigned dq_blocks = unsigned(want < 128 ? want : 128);
    for (int c = 0; c < n_chunks; ++c) {
      launch_pdl(fp8_dequant_kernel, dim3(dq_blocks, kFp8Chunk), dim3(256), 0, st, *w, H, F, pl,
                 c, gu_bf, dn_bf);
      launch_pdl(moe_chunk_jobs_kernel, dim3(1), dim3(32), 0, st, pl, c, kFp8Chunk,
                 static_cast<const float*>(nullptr), static_cast<const float*>(nullptr), cj, cn,
                 static_cast<float*>(nullptr), static_cast<float*>(nullptr));
      if (const cudaError_t err_ = tc::gemm_grouped(tc::kSwiGLU, us, P, 2 * H, H, gu_bf,
                                                    kFp8Chunk * 2 * F, 2 * F, 2 * H, cj, cn, mj, F,
                                                    F, nullptr, act, F, st, nullptr, true);
          err_ != cudaSuccess)
        return cuda_status(err_);
      if (const cudaError_t err_ = tc::gemm_grouped(tc::kF32, act, P, 2 * F, F, dn_bf, kFp8Chunk * H,
                                                    H, 2 * F, cj, cn, mj, H, 0, pl.pairs, y, H, st,
                                                    nullptr, true);
          err_ != cudaSuccess)
        return cuda_status(err_);
    }
    if ((H & 3) == 0 && aligned16(out)) {
      const size_t n4 = size_t(T) * (H / 4);
      launch_pdl(moe_combine4_kernel, dim3(unsigned((n4 + 255) / 256)), dim3(256), 0, st, y,
                 topk_w, topk_idx, T, H, k, E, out);
    } else {
      const size_t n1 = size_t(T) * H;
      launch_pdl(moe_combine_kernel, dim3(unsigned((n1 + 255) / 256)), dim3(256), 0, st, y,
                 topk_w, topk_idx, T, H, k, E, out);
    }
    return launch_status();
  }
  MoePlan pl = carve_plan(cv, E, P, false);
  uint16_t* a16 = cv.take<uint16_t>(size_t(P) * F);
  float* y = cv.take<float>(size_t(P) * H);
  int* cnt = cv.take<int>(size_t(H / 8 + 1));
  uint16_t* u16 = cv.take<uint16_t>(size_t(T) * H);
  if (!cv.ok) return BEAM_ERR_INVALID_ARG;
  // one token: its k slots are the active list directly; more: the plan groups the pairs
  const bool direct = T == 1;
  const int32_t* dix = direct ? topk_idx : nullptr;
  const int na = direct ? k : (P < E ? P : E);
  // up to 4 tokens four warps split each row block's K blocks (the grid is under a wave
  // otherwise); from 5 tokens a warp takes a whole row block
  const bool split = T <= kFp4KSMaxT;
  const int rows_down = split ? 32 : 128, units_up = split ? 16 : 64;
  const int n_cnt = (H + rows_down - 1) / rows_down;
  const int n = T * H;
  launch_pdl(fp4_prep_kernel, dim3((max(n, n_cnt) + 255) / 256), dim3(256), 0, st, u, n, u16, cnt,
             n_cnt);
  if (!direct)
    launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 3 * E * sizeof(int), st, topk_idx, P, E, pl);
  const dim3 gu((F + units_up - 1) / units_up, na), gd(n_cnt, na);
  if (split) {
    launch_pdl(moe_gate_up_fp8_kernel<4>, gu, dim3(256), 0, st, u16, *w, H, F, k, pl, dix, E, a16);
    launch_pdl(moe_down_fp8_kernel<4>, gd, dim3(256), 0, st, a16, *w, H, F, pl, dix, topk_idx,
               topk_w, T, k, E, cnt, y, out);
  } else {
    launch_pdl(moe_gate_up_fp8_kernel<1>, gu, dim3(256), 0, st, u16, *w, H, F, k, pl, dix, E, a16);
    launch_pdl(moe_down_fp8_kernel<1>, gd, dim3(256), 0, st, a16, *w, H, F, pl, dix, topk_idx,
               topk_w, T, k, E, cnt, y, out);
  }
  return launch_status();
}
