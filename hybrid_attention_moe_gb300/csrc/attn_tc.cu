// Prefill attention on the 5th-generation tensor cores (tcgen05), BF16 KV cache.
// Beam page, Attention section: 48 query heads share 8 KV heads of dim 128 (GQA); sliding-window
// layers see the last 512 keys, NoPE layers the whole context (SSMax is already applied to q by
// the projection epilogue); the output of each head is gated by sigmoid(gate + per-head bias).
//
// Work item = (KV head, job), job = up to 2 TPT consecutive tokens of one sequence, TPT =
// floor(128 / G). The G query heads of TPT tokens form the 128 rows of one MMA tile (row =
// token * G + head); a job holds two such query tiles, A and B, so every K/V tile brought on
// chip serves 2 TPT tokens of the whole KV group. A persistent grid walks the items; per item
// the key axis is streamed in tiles of 128 keys, and for each query tile:
//   S = Q . K^T           tcgen05.mma, A = Q (shared memory), B = K tile, FP32 in TMEM
//   P = exp2(S * c - m)   softmax warps, thread per row (TMEM lane), online max with lazy
//                         rescaling of O (only when a row max grows by more than 2^8)
//   O += P . V            tcgen05.mma, A = P from TMEM, B = V tile (MN-major)
// P is written back over its S columns as BF16 hi and lo parts (P = hi + lo to ~16 bits), and
// both are multiplied by V, so the P.V product keeps FP32-level accuracy.
//
// Warps: 0 TMA (Q per item, K and V rings), 1 MMA issue (+ zeroing V rows outside the item's
// key range, which may be uninitialised cache memory), 2-5 softmax and epilogue of tile A, 6-9
// of tile B: while one warpgroup turns its S into P, the tensor pipe works on the other tile.
// TMEM columns: S_A [0, 128), S_B [128, 256), O_A [256, 384), O_B [384, 512). Every wait is
// bounded: on expiry the CTA records BEAM_DEV_TIMEOUT, lets issued copies land, frees TMEM and
// returns.
#include <cuda.h>
#include <math.h>

#include "attn_tc.cuh"
#include "common.cuh"
#include "mma.cuh"
#include "tcgen05.cuh"

namespace beam {
namespace atc {
namespace {

using namespace beam::tc;

constexpr int KT = 128;          // keys per tile
constexpr int ROWS = 128;        // MMA rows
constexpr int KSTAGES = 2, VSTAGES = 2;
// warp 0 TMA, warp 1 MMA, warps 2-17 softmax: query tile u = (warp - 2) / 8, column half
// (warp - 2) / 4 % 2, TMEM lane quarter warp % 4 -- two threads per row, 64 columns each
constexpr int THREADS = 576;
constexpr float kRescale = 8.f;  // log2 units
// The tensor pipe's FP32 accumulation drops about 2^-24 of the running sum per MMA (measured:
// 1.8e-5 relative over 320 accumulating MMAs). O of a 100K-key row would take ~12.5K of them,
// so every kFlushTiles key tiles (~2K MMAs) the softmax warps add O from TMEM into an FP32 scratch row
// (round-to-nearest adds) and the next P.V starts a fresh TMEM accumulator.
constexpr int kFlushTiles = 128;
constexpr int kMaxGrid = 256;    // persistent CTAs at most (scratch is sized for this many)
constexpr float kNegInf = -INFINITY;

struct Job {
  int t0, n, seq, key_a, key_b, pad0, pad1, pad2;
};

// Shared memory (offsets from a 1024-aligned base). A 64-column half of a 128-row bf16 tile is
// 128 rows x 128 B = 16 KB (128-byte swizzle atoms of 8 rows).

template <int D>
struct Smem {
  static constexpr int NH = D / 64;
  static constexpr int HALF = ROWS * 128;
  static constexpr int TILE = NH * KT * 128;   // K or V tile
  static constexpr int Q = 0;                  // query tiles A and B
  static constexpr int K0 = 2 * NH * HALF;
  static constexpr int V0 = K0 + KSTAGES * TILE;
  static constexpr int BAR = V0 + VSTAGES * TILE;
  static constexpr int NBAR = 2 + 2 * KSTAGES + 2 * VSTAGES + 10;
  // row max (slots 0-1, by key-tile parity) and row sum (slots 2-3, by item parity) exchange
  // between the two threads of a row: [slot][query tile][row][half] floats
  static constexpr int XCH = BAR + NBAR * 8 + 16;
  static constexpr int BYTES = XCH + 4 * 2 * 128 * 2 * 4 + 1024;
};

struct Params {
  const Job* jobs;
  const int* n_jobs;
  const int32_t* pos;
  const uint16_t* gpre;
  const uint16_t* gate_bias;
  uint16_t* og;
  float* oacc;   // per CTA [2][128][128] FP32: O of the chunks already flushed
  int T, n_q, n_kv, G, TPT, window, cap;
  float sl2;
};

// Keys of an item, walked in tiles of KT slots. Tile i covers keys key_first + i*KT + c
// (c < KT) at cache slots (first_slot + i*KT + c) mod cap; a ring cache (window > 0) has
// cap % KT == 0 and tiles aligned to KT slots, so no tile crosses the end of the ring.
struct Walk {
  int n, first_slot, key_first;
};
__device__ __forceinline__ Walk walk_of(const Job& J, int window, int cap) {
  Walk w{0, 0, 1};
  if (J.key_b < J.key_a) return w;
  const int s_a = (J.key_a - 1) % cap;
  const int t_s = window > 0 ? (s_a / KT) * KT : s_a;
  w.first_slot = t_s;
  w.key_first = J.key_a - (s_a - t_s);
  w.n = (J.key_b - w.key_first + KT) / KT;
  return w;
}

// 2^x by the SFU's approximate exp2 instruction (relative error below 2^-22; subnormal results
// flush to zero, far below what a softmax row sum can notice).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of FP32 values (one 64-bit register pair) and the paired FMA / add / subtract:
// each lane of the pair rounds exactly as the scalar instruction would.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ bool row_pos_ok(int p, int window, int cap) {
  return p >= 1 && !(window == 0 && p > cap);
}

// ------------------------------------------------------------------------------------------
// Job plan: runs of consecutive tokens with the same seq_id, cut into jobs of <= TPT tokens;
// per job the union [key_a, key_b] of its tokens' key ranges. One CTA of 1024 threads.
// ------------------------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int block_scan_max_incl(int v, int* ws) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = max(v, n);
  }
  __syncthreads();
  if (lane == 31) ws[wid] = v;
  __syncthreads();
  if (wid == 0) {
    int t = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t = max(t, n);
    }
    ws[lane] = t;
  }
  __syncthreads();
  return wid > 0 ? max(v, ws[wid - 1]) : v;
}

__device__ __forceinline__ int block_scan_sum_excl(int v, int* ws, int* total) {
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
    int t = ws[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    ws[lane] = t;
  }
  __syncthreads();
  *total = ws[31];
  return (wid > 0 ? ws[wid - 1] : 0) + inc - v;
}

__global__ void __launch_bounds__(kPlanThreads) attn_tc_plan_kernel(
    const int32_t* __restrict__ seq_id, const int32_t* __restrict__ pos, int T, int TPT,
    int window, int cap, int num_seqs, Job* __restrict__ jobs, int* __restrict__ n_jobs) {
  pdl_trigger();
  pdl_wait();
  __shared__ int ws[32];
  __shared__ int s_njobs;
  int carry_start = 0, carry_jobs = 0;
  for (int base = 0; base < T; base += kPlanThreads) {
    const int t = base + threadIdx.x;
    const bool valid = t < T;
    const int sq = valid ? seq_id[t] : 0;
    const bool run_start = valid && (t == 0 || seq_id[t - 1] != sq);
    const int rs = max(carry_start, block_scan_max_incl(run_start ? t : -1, ws));
    const bool job_start = valid && ((t - rs) % TPT) == 0;
    int total;
    const int jpos = carry_jobs + block_scan_sum_excl(job_start ? 1 : 0, ws, &total);
    if (job_start) jobs[jpos].t0 = t;
    // the last thread's run start carries into the next chunk
    __syncthreads();
    if (threadIdx.x == kPlanThreads - 1) ws[0] = rs;
    __syncthreads();
    carry_start = ws[0];
    carry_jobs += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) s_njobs = carry_jobs;
  __threadfence_block();
  __syncthreads();
  const int nj = s_njobs;
  for (int jb = threadIdx.x; jb < nj; jb += kPlanThreads) {
    const int t0 = jobs[jb].t0;
    const int t1 = jb + 1 < nj ? jobs[jb + 1].t0 : T;
    Job J;
    J.t0 = t0;
    J.n = t1 - t0;
    J.seq = seq_id[t0];
    J.key_a = 0x7fffffff;
    J.key_b = 0;
    J.pad0 = J.pad1 = J.pad2 = 0;
    const bool seq_ok = J.seq >= 0 && J.seq < num_seqs;
    if (!seq_ok) flag(BEAM_DEV_BAD_SEQ);
    for (int t = t0; t < t1 && seq_ok; ++t) {
      const int p = pos[t];
      if (!row_pos_ok(p, window, cap)) {
        flag(BEAM_DEV_BAD_POSITION);
        continue;
      }
      J.key_a = min(J.key_a, window > 0 ? max(1, p - window + 1) : 1);
      J.key_b = max(J.key_b, p);
    }
    if (J.key_b < J.key_a) J.key_a = 1, J.key_b = 0;
    jobs[jb + T] = J;   // written to the second half: first-half t0 values are still read
  }
  __threadfence_block();
  __syncthreads();
  for (int jb = threadIdx.x; jb < nj; jb += kPlanThreads) jobs[jb] = jobs[jb + T];
  if (threadIdx.x == 0) *n_jobs = nj;
}

// ------------------------------------------------------------------------------------------
// The attention kernel
// ------------------------------------------------------------------------------------------
template <int D>
// 18 warps share the register file of 4 SM sub-partitions (16K registers each); two of them
// hold 5 warps, so a thread gets at most 16384 / (5 * 32) -> 96 registers
__global__ void __maxnreg__(96) attn_prefill_tc_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
    const __grid_constant__ CUtensorMap tv, Params p) {
  pdl_trigger();
  pdl_wait();
  using S = Smem<D>;
  constexpr uint32_t IDESC_QK = idesc_bf16(ROWS, KT, false);
  constexpr uint32_t IDESC_PV = idesc_bf16(ROWS, D, true);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::BAR);
  const uint32_t b0 = smem_u32(bars);
  const uint32_t q_full = b0, q_empty = b0 + 8;
  const uint32_t k_full = b0 + 16, k_empty = k_full + 8 * KSTAGES;
  const uint32_t v_full = k_empty + 8 * KSTAGES, v_empty = v_full + 8 * VSTAGES;
  // per query tile u: s_full[u], p_full[u], s_free[u], o_full[u], o_empty[u]
  const uint32_t s_full = v_empty + 8 * VSTAGES, p_full = s_full + 16, s_free = p_full + 16;
  const uint32_t o_full = s_free + 16, o_empty = o_full + 16;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + S::BAR + S::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int njobs = *p.n_jobs;
  const int n_work = njobs * p.n_kv;
  const int G = p.G;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < KSTAGES; ++s) {
      mbar_init(k_full + 8 * s, 1);
      mbar_init(k_empty + 8 * s, 1);
    }
    for (int s = 0; s < VSTAGES; ++s) {
      mbar_init(v_full + 8 * s, 1);
      mbar_init(v_empty + 8 * s, 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(s_full + 8 * u, 1);
      mbar_init(p_full + 8 * u, 256);
      mbar_init(s_free + 8 * u, 1);
      mbar_init(o_full + 8 * u, 1);
      mbar_init(o_empty + 8 * u, 256);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  {   // Q rows past G * TPT are never written by TMA: keep them zero
    const int q0 = G * p.TPT;
    const int n16 = (ROWS - q0) * 8;   // 16-byte chunks per half
    for (int i = threadIdx.x; i < n16 * S::NH * 2; i += THREADS) {
      const int h = i / n16, c = i - h * n16;   // h: tile * NH + half
      *reinterpret_cast<uint4*>(smem + S::Q + h * S::HALF + q0 * 128 + c * 16) =
          make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;   // S of tile u at column 128 u, O of tile u at 256 + 128 u

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t kc = 0, vc = 0;
      int item = 0;
      int last_k[KSTAGES], last_v[VSTAGES], last_q = -1;
      for (int s = 0; s < KSTAGES; ++s) last_k[s] = -1;
      for (int s = 0; s < VSTAGES; ++s) last_v[s] = -1;
      for (int w = blockIdx.x; w < n_work; w += gridDim.x, ++item) {
        if (*abort_flag) break;
        const int hk = w / njobs;
        const Job J = p.jobs[w - hk * njobs];
        if (!mbar_wait(q_empty, (item & 1) ^ 1)) { *abort_flag = 1; break; }
        mbar_expect_tx(q_full, uint32_t(2 * S::NH * 128 * G * p.TPT));
        for (int u = 0; u < 2; ++u)
          for (int h = 0; h < S::NH; ++h)
            tma_load_3d(sb + S::Q + (u * S::NH + h) * S::HALF, &tq, 64 * h, hk * G,
                        J.t0 + u * p.TPT, q_full);
        last_q = item;
        const Walk wk = walk_of(J, p.window, p.cap);
        const int zidx = J.seq * p.n_kv + hk;
        bool bad = false;
        for (int i = 0; i < wk.n; ++i) {
          int slot = wk.first_slot + i * KT;
          if (p.window > 0) slot %= p.cap;
          const int ks = int(kc % KSTAGES);
          if (!mbar_wait(k_empty + 8 * ks, ((kc / KSTAGES) & 1) ^ 1)) { bad = true; break; }
          mbar_expect_tx(k_full + 8 * ks, uint32_t(S::TILE));
          for (int h = 0; h < S::NH; ++h)
            tma_load_3d(sb + S::K0 + ks * S::TILE + h * KT * 128, &tk, 64 * h, slot, zidx, k_full + 8 * ks);
          last_k[ks] = int(kc);
          ++kc;
          const int vs = int(vc % VSTAGES);
          if (!mbar_wait(v_empty + 8 * vs, ((vc / VSTAGES) & 1) ^ 1)) { bad = true; break; }
          mbar_expect_tx(v_full + 8 * vs, uint32_t(S::TILE));
          for (int h = 0; h < S::NH; ++h)
            tma_load_3d(sb + S::V0 + vs * S::TILE + h * KT * 128, &tv, 64 * h, slot, zidx, v_full + 8 * vs);
          last_v[vs] = int(vc);
          ++vc;
        }
        if (bad) { *abort_flag = 1; break; }
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA's shared memory goes away
        for (int s = 0; s < KSTAGES; ++s)
          if (last_k[s] >= 0) mbar_wait(k_full + 8 * s, (uint32_t(last_k[s]) / KSTAGES) & 1);
        for (int s = 0; s < VSTAGES; ++s)
          if (last_v[s] >= 0) mbar_wait(v_full + 8 * s, (uint32_t(last_v[s]) / VSTAGES) & 1);
        if (last_q >= 0) mbar_wait(q_full, uint32_t(last_q) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    // Issue order per key tile j: PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1). Each P.V waits for
    // its softmax warpgroup; the next S of the same query tile follows it at once. tcgen05.mma
    // operations issued by one thread execute in issue order (an implicitly pipelined pair in
    // the PTX memory model), so QK_u(j+1) overwrites the TMEM columns holding P_u(j) only after
    // PV_u(j) has read them, and while one warpgroup computes its P the tensor pipe works
    // through the other tile's P.V and the next S.
    uint32_t kc = 0, vc = 0, pt = 0;   // pt: key tiles of earlier items (per query tile)
    uint32_t ostart = 0;                // fresh O accumulations started so far (per query tile)
    int item = 0;
    bool ok = true;
    auto all = [&](bool v) { return __all_sync(0xffffffffu, v) && !*abort_flag; };
    // In the key-tile loop the abort flag is not read: a shared-memory load takes ~130 cycles
    // while the tensor pipe streams operands, and the pipe holds under 200 cycles of queued
    // MMAs. A role that gave up stops arriving, so the next wait here expires instead.
    auto all_fast = [&](bool v) { return __all_sync(0xffffffffu, v); };
    // descriptors of stage 0 / query tile 0; others differ only in the start address field,
    // (address >> 4) in the low 14 bits, which no offset below carries out of
    const uint64_t dq0 = smem_desc(sb + S::Q), dk0 = smem_desc(sb + S::K0);
    const uint64_t dv0 = smem_desc_mn(sb + S::V0, KT * 128, 1024);
    // The tensor pipe queues only ~3 MMAs of these shapes (~170 cycles of work), so the issue
    // path is kept short: descriptors are stepped in their low word (the address field) only.
    const uint32_t dq0_hi = uint32_t(dq0 >> 32), dk0_hi = uint32_t(dk0 >> 32);
    auto qk = [&](int u, int ks) {
      const uint32_t qlo = uint32_t(dq0) + uint32_t((u * S::NH * S::HALF) >> 4);
      const uint32_t klo = uint32_t(dk0) + uint32_t((ks * S::TILE) >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk & 3) * 32) >> 4;
        umma_ss_e(tmem + 128 * u, qlo + ((kk >> 2) * S::HALF >> 4) + off, dq0_hi,
                  klo + ((kk >> 2) * KT * 128 >> 4) + off, dk0_hi, IDESC_QK, kk > 0 ? 1u : 0u);
      }
      umma_commit_e(s_full + 8 * u);
    };
    const uint32_t dv0_hi = uint32_t(dv0 >> 32);
    auto pv = [&](int u, int vs, bool first) {
      const uint32_t blo = uint32_t(dv0) + uint32_t((vs * S::TILE) >> 4);
      const uint32_t ts = tmem + 128 * u, to = tmem + 256 + 128 * u;
      umma_ts_e(to, ts, blo, dv0_hi, IDESC_PV, first ? 0u : 1u);
      umma_ts_e(to, ts + 16, blo, dv0_hi, IDESC_PV, 1u);
#pragma unroll
      for (int kk = 1; kk < KT / 16; ++kk) {
        const uint32_t b = blo + uint32_t((kk * 16 * 128) >> 4);
        const uint32_t a_hi = ts + 32 * (kk >> 1) + 8 * (kk & 1);
        umma_ts_e(to, a_hi, b, dv0_hi, IDESC_PV, 1u);
        umma_ts_e(to, a_hi + 16, b, dv0_hi, IDESC_PV, 1u);
      }
      umma_commit_e(s_free + 8 * u);
    };
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x, ++item) {
      const int hk = w / njobs;
      const Job J = p.jobs[w - hk * njobs];
      const Walk wk = walk_of(J, p.window, p.cap);
      if (!all(mbar_wait(q_full, uint32_t(item) & 1))) { ok = false; break; }
      tc_fence_after();
      if (wk.n == 0) {
        // no keys: release Q; O is never written, the epilogue stores zeros
        const uint32_t oph = (ostart & 1) ^ 1;
        if (!all(mbar_wait(o_empty, oph) && mbar_wait(o_empty + 8, oph))) { ok = false; break; }
        ++ostart;
        umma_commit_e(q_empty);
        umma_commit_e(o_full);
        umma_commit_e(o_full + 8);
        continue;
      }
      int ks = int(kc % KSTAGES);
      if (!all(mbar_wait(k_full + 8 * ks, (kc / KSTAGES) & 1))) { ok = false; break; }
      tc_fence_after();
      qk(0, ks);
      qk(1, ks);
      umma_commit_e(k_empty + 8 * ks);
      if (wk.n == 1) umma_commit_e(q_empty);
      ++kc;
      uint32_t gt_i = 0;   // key tiles of this item done
      for (int i = 0; i < wk.n; ++i) {
        const int vs = int(vc % VSTAGES);
        const bool more = i + 1 < wk.n;
        // a fresh O accumulation at the item's first tile and after each flush; it waits until
        // the softmax warps have taken the previous one out of TMEM
        const bool fresh = i % kFlushTiles == 0;
        const uint32_t oph = (ostart & 1) ^ 1;
        // ---- query tile A: P.V of tile i, then S of tile i + 1
        if (more) ks = int(kc % KSTAGES);
        // the tile's barriers polled together (their latencies overlap), then waited for one by
        // one only if one was not yet complete
        const bool r_v = mbar_try(v_full + 8 * vs, (vc / VSTAGES) & 1);
        const bool r_p = mbar_try(p_full, (pt + gt_i) & 1);
        const bool r_k = !more || mbar_try(k_full + 8 * ks, (kc / KSTAGES) & 1);
        const bool r_o = !fresh || mbar_try(o_empty, oph);
        bool w_ok = r_v && r_p && r_k && r_o;
        if (!w_ok) {
          w_ok = mbar_wait(v_full + 8 * vs, (vc / VSTAGES) & 1) &&
                 mbar_wait(p_full, (pt + gt_i) & 1) && (!fresh || mbar_wait(o_empty, oph)) &&
                 (!more || mbar_wait(k_full + 8 * ks, (kc / KSTAGES) & 1));
        }
        if (!all_fast(w_ok)) { ok = false; break; }
        const int kb = wk.key_first + i * KT;
        const int r0 = max(0, J.key_a - kb), r1 = min(KT, J.key_b - kb + 1);
        if (r0 > 0 || r1 < KT) {
          // V rows outside [key_a, key_b] may hold uninitialised memory: zero them
          uint8_t* vt = smem + S::V0 + vs * S::TILE;
          const int nz = (r0 + (KT - r1)) * 8;   // 16-byte chunks per half
          for (int c = lane; c < nz * S::NH; c += 32) {
            const int h = c / nz, e = c - h * nz;
            const int row = e / 8 < r0 ? e / 8 : r1 + (e / 8 - r0);
            *reinterpret_cast<uint4*>(vt + h * KT * 128 + row * 128 + (e % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        pv(0, vs, fresh);
        if (!more) umma_commit_e(o_full);
        const bool r_pb = mbar_test(p_full + 8, (pt + gt_i) & 1);   // answered while QK_A issues
        if (more) qk(0, ks);
        // ---- query tile B
        w_ok = r_pb || mbar_wait(p_full + 8, (pt + gt_i) & 1);
        if (fresh) w_ok = w_ok && mbar_wait(o_empty + 8, oph);
        if (!all_fast(w_ok)) { ok = false; break; }
        if (fresh) ++ostart;
        tc_fence_after();
        pv(1, vs, fresh);
        umma_commit_e(v_empty + 8 * vs);
        if (!more) umma_commit_e(o_full + 8);
        ++vc;
        if (more) {
          qk(1, ks);
          umma_commit_e(k_empty + 8 * ks);
          if (i + 1 == wk.n - 1) umma_commit_e(q_empty);
          ++kc;
        }
        ++gt_i;
      }
      if (!ok) break;
      pt += uint32_t(wk.n);
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    const int u = (warp - 2) >> 3;           // query tile
    const int half = ((warp - 2) >> 2) & 1;  // columns [64 half, 64 half + 64) of S and O
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lrow = uint32_t(q4 * 32) << 16;
    const uint32_t ts = tmem + 128 * u + 64 * half + lrow;
    const uint32_t to = tmem + 256 + 128 * u + 64 * half + lrow;
    const uint32_t my_s_full = s_full + 8 * u, my_p_full = p_full + 8 * u;
    const uint32_t my_s_free = s_free + 8 * u, my_o_full = o_full + 8 * u;
    const uint32_t my_o_empty = o_empty + 8 * u;
    // the two threads of a row meet at a named barrier of their two warps
    const uint32_t pair_bar = 1 + u * 4 + q4;
    float* xch = reinterpret_cast<float*>(smem + S::XCH);   // [parity][u][row][half]
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory"); };
    // every exit decision is taken by both threads of a row together, so neither can leave
    // while the other waits at their barrier
    auto pair_all = [&](bool v) {
      uint32_t res;
      asm volatile(
          "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; bar.red.and.pred po, %2, 64, pi; selp.u32 %0, 1, 0, po; }"
          : "=r"(res)
          : "r"(uint32_t(v)), "r"(pair_bar)
          : "memory");
      return res != 0;
    };
    const int tl = r / G, hj = r - tl * G;
    uint32_t gt = 0;
    int item = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x, ++item) {
      const int hk = w / njobs;
      const Job J = p.jobs[w - hk * njobs];
      const Walk wk = walk_of(J, p.window, p.cap);
      const int tj = u * p.TPT + tl;           // token index within the job
      const bool row_ok = tl < p.TPT && tj < J.n;
      int pr = 0, lo = 1;
      if (row_ok) {
        const int pp = p.pos[J.t0 + tj];
        if (row_pos_ok(pp, p.window, p.cap)) {
          pr = min(pp, J.key_b);
          lo = p.window > 0 ? max(1, pp - p.window + 1) : 1;
        }
      }
      float m_ref = kNegInf, l = 0.f;
      bool flushed = false;   // oacc holds earlier chunks of this item
      float* oacc = p.oacc + ((size_t(blockIdx.x) * 2 + u) * 128 + r) * 128 + 64 * half;
      for (int i = 0; i < wk.n; ++i) {
        const uint32_t G_ = gt + uint32_t(i);
        if (!pair_all(mbar_wait(my_s_full, G_ & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kb = wk.key_first + i * KT + 64 * half;
        const int c_lo = lo - kb, c_hi = pr - kb;   // valid columns [c_lo, c_hi] of this half
        float mh;
        {
          // row max of this half, 32 columns at a time; columns outside the row's keys become
          // -inf, in TMEM too, so P below needs no mask
          const bool full = __all_sync(0xffffffffu, c_lo <= 0 && c_hi >= 63);
          float mx[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = kNegInf;
#pragma unroll 1
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t sv[32];
            tmem_ld32_nowait(ts + 32 * c2, sv);
            tmem_wait_ld();
            if (!full) {
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (32 * c2 + c < c_lo || 32 * c2 + c > c_hi) sv[c] = __float_as_uint(kNegInf);
              tmem_st32(ts + 32 * c2, sv);
              tmem_wait_st();
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(sv[c]));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], mx[k + 4]);
          mh = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        }
        float* xm = xch + ((G_ & 1) * 2 + u) * 256;
        xm[r * 2 + half] = mh;
        pair_sync();
        const float mt = fmaxf(mh, xm[r * 2 + (half ^ 1)]) * p.sl2;
        const bool need = m_ref != kNegInf && mt > m_ref + kRescale;
        if (__any_sync(0xffffffffu, need)) {
          // O holds the earlier tiles' P.V of this item: wait for the last one, then rescale
          if (!pair_all(mbar_wait(my_s_free, (G_ - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = need ? exp2f(m_ref - mt) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32_nowait(to + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(to + 32 * c, o);
          }
          tmem_wait_st();
          if (flushed && need) {
#pragma unroll 4
            for (int c = 0; c < 64; c += 4) {
              float4 a = *reinterpret_cast<float4*>(oacc + c);
              a.x *= f;
              a.y *= f;
              a.z *= f;
              a.w *= f;
              *reinterpret_cast<float4*>(oacc + c) = a;
            }
          }
          if (need) {
            l *= f;
            m_ref = mt;
          }
        }
        if (m_ref == kNegInf) m_ref = mt;   // first keys of the row: O row is still zero
        const float nmref = m_ref == kNegInf ? 0.f : -m_ref;
        // P two columns at a time: one paired FMA for s * c - m, the SFU's exp2 per column,
        // paired row sums and a paired subtract for the lo parts
        const uint64_t sl2x2 = f2(p.sl2, p.sl2), nm2 = f2(nmref, nmref);
        uint64_t ls2[4] = {0, 0, 0, 0};
#pragma unroll 1
        for (int c4 = 0; c4 < 2; ++c4) {
          uint32_t v[32], pk[32];
          tmem_ld32_nowait(ts + 32 * c4, v);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            float x0, x1;
            f2_split(fma2(f2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1])), sl2x2, nm2),
                     x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const uint64_t pp = f2(p0, p1);
            ls2[q & 3] = add2(ls2[q & 3], pp);
            const uint32_t hi = pack_bf16x2(p0, p1);
            float d0, d1;
            f2_split(sub2(pp, f2(bf_lo(hi), bf_hi(hi))), d0, d1);
            pk[q] = hi;
            pk[16 + q] = pack_bf16x2(d0, d1);
          }
          tmem_st32(ts + 32 * c4, pk);
        }
        {
          float a0, a1, b0, b1;
          f2_split(add2(ls2[0], ls2[1]), a0, a1);
          f2_split(add2(ls2[2], ls2[3]), b0, b1);
          l += (a0 + b0) + (a1 + b1);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(my_p_full);
        if ((i + 1) % kFlushTiles == 0 && i + 1 < wk.n) {
          // flush: once this tile's P.V has completed, add O into the FP32 scratch row and
          // hand TMEM back for a fresh accumulation
          if (!pair_all(mbar_wait(my_s_free, G_ & 1) && !*abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t ov[32];
            tmem_ld32_nowait(to + 32 * c2, ov);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              float4 a = make_float4(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1]),
                                     __uint_as_float(ov[c + 2]), __uint_as_float(ov[c + 3]));
              if (flushed) {
                const float4 b = *reinterpret_cast<const float4*>(oacc + 32 * c2 + c);
                a.x += b.x;
                a.y += b.y;
                a.z += b.z;
                a.w += b.w;
              }
              *reinterpret_cast<float4*>(oacc + 32 * c2 + c) = a;
            }
          }
          tc_fence_before();
          mbar_arrive(my_o_empty);
          flushed = true;
        }
      }
      if (!ok) break;
      gt += uint32_t(wk.n);
      // epilogue: o = O / l, rounded, gated, rounded; l is the sum of the row's two halves
      if (!pair_all(mbar_wait(my_o_full, uint32_t(item) & 1) && !*abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float* xl = xch + ((2 + (item & 1)) * 2 + u) * 256;
      xl[r * 2 + half] = l;
      pair_sync();
      const float lt = l + xl[r * 2 + (half ^ 1)];
      const float inv = (wk.n > 0 && lt > 0.f) ? 1.f / lt : 0.f;
      const int t = J.t0 + tj, hq = hk * G + hj;
      const size_t oi = (size_t(row_ok ? t : 0) * p.n_q + hq) * D + 64 * half;
      const float gb = row_ok ? bf2f(p.gate_bias[hq]) : 0.f;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t ov[32];
        tmem_ld32_nowait(to + 32 * c2, ov);
        tmem_wait_ld();
        if (flushed) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            ov[c] = __float_as_uint(__uint_as_float(ov[c]) + oacc[32 * c2 + c]);
        }
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const size_t oc = oi + 32 * c2 + 8 * c;
            const uint4 gv = *reinterpret_cast<const uint4*>(p.gpre + oc);
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t q[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float o0 = inv > 0.f ? round_bf(__uint_as_float(ov[8 * c + 2 * e]) * inv) : 0.f;
              const float o1 = inv > 0.f ? round_bf(__uint_as_float(ov[8 * c + 2 * e + 1]) * inv) : 0.f;
              const float g0 = sigmoidf_(bf_lo(gw[e]) + gb), g1 = sigmoidf_(bf_hi(gw[e]) + gb);
              q[e] = pack_bf16x2(o0 * g0, o1 * g1);
            }
            *reinterpret_cast<uint4*>(p.og + oc) = make_uint4(q[0], q[1], q[2], q[3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(my_o_empty);
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag(BEAM_DEV_TIMEOUT);
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                 : "memory");
  }
}

}  // namespace

bool prefill_supported(int D, int G, int window, int cap, bool fp8, const void* q,
                       const void* k, const void* v) {
  if (fp8 || D != 128 || G < 1 || G > ROWS) return false;
  if (window > 0 && cap % KT != 0) return false;
  return aligned16(q) && aligned16(k) && aligned16(v) && tensor_map_encoder_ready();
}

size_t ws_bytes(int T) {
  return align_up(size_t(2 * T + 1) * sizeof(Job), 256) + 256 +
         size_t(kMaxGrid) * 2 * 128 * 128 * sizeof(float);
}

cudaError_t prefill(const uint16_t* q, const uint16_t* g, const uint16_t* gate_bias,
                    const int32_t* seq_id, const int32_t* pos, int T, int n_q, int n_kv, int D,
                    const beam_kv_cache& kc, float sl2, uint16_t* og, void* ws, size_t ws_len,
                    cudaStream_t st) {
  const int G = n_q / n_kv, TPT = ROWS / G;
  if (ws_len < ws_bytes(T)) return cudaErrorInvalidValue;
  Job* jobs = static_cast<Job*>(ws);
  int* n_jobs = reinterpret_cast<int*>(static_cast<char*>(ws) + align_up(size_t(2 * T + 1) * sizeof(Job), 256));
  CUtensorMap mq, mk, mv;
  {
    const uint64_t dims[3] = {uint64_t(D), uint64_t(n_q), uint64_t(T)};
    const uint64_t str[2] = {uint64_t(D) * 2, uint64_t(n_q) * D * 2};
    const uint32_t box[3] = {64, uint32_t(G), uint32_t(TPT)};
    if (!encode_tiled(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {uint64_t(D), uint64_t(kc.capacity), uint64_t(kc.num_seqs) * n_kv};
    const uint64_t str[2] = {uint64_t(D) * 2, uint64_t(kc.capacity) * D * 2};
    const uint32_t box[3] = {64, uint32_t(KT), 1};
    if (!encode_tiled(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kc.k, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kc.v, dims, str, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  launch_pdl(attn_tc_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, seq_id, pos, T, 2 * TPT,
             kc.window, kc.capacity, kc.num_seqs, jobs, n_jobs);
  float* oacc = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                        align_up(size_t(2 * T + 1) * sizeof(Job), 256) + 256);
  Params prm{jobs, n_jobs, pos, g, gate_bias, og, oacc, T, n_q, n_kv, G, TPT, kc.window, kc.capacity, sl2};
  int grid = num_sms_cached();
  if (grid > kMaxGrid) grid = kMaxGrid;
  if (int64_t(T) * n_kv < grid) grid = T * n_kv;
  cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<128>::BYTES);
  if (e != cudaSuccess) return e;
  launch_pdl(attn_prefill_tc_kernel<128>, dim3(grid), dim3(THREADS), Smem<128>::BYTES, st, mq, mk, mv, prm);
  return cudaGetLastError();
}

}  // namespace atc
}  // namespace beam
