// Long-context decode attention: TMA-fed, warp-specialised split-K flash decoding.
// Beam page, Attention section: 48 query heads share 8 KV heads of dim 128 (GQA); sliding-window
// layers see the last 512 keys, NoPE layers the whole context (q already carries RoPE or the
// SSMax scale); the cache holds BF16 or FP8-e4m3 K/V; each head's output is multiplied by
// sigmoid(gate + per-head bias) before o_proj.
//
// The (token, KV head) pairs are cut into blocks of BK keys, and the flattened (pair, block)
// space into equal contiguous ranges, one per CTA (one CTA per SM): every SM streams the same
// number of K/V bytes whatever the batch, and a range may end inside one pair and start the
// next. Per CTA one producer warp issues TMA loads of whole key blocks (K and V, 128-byte
// swizzle) into a ring of NST stages; NCW consumer warps each take 16 keys of every block.
// With G <= 8 query heads per KV head the tiles are computed transposed, so the heads are the
// 8-wide N side of mma.sync m16n8k16 and no MMA row is padding:
//   S^T[16 keys x 8 heads]  = K[16 x 128] . Q^T           A = K rows, B = q fragments
//   O^T[128 x 8 heads]     += V^T[128 x 16 keys] . P^T    A = V (transposed), B = P^T
// movmatrix (8x8 transposes in registers) turns the accumulator layout of P^T into the B
// layout. P is split into hi and lo halves, so P carries ~16 significant bits; the running
// max is rescaled lazily (only when it grows by more than 2^8). At the end of a pair's range
// the consumer warps combine their partials: a pair that one CTA covers whole is finished in
// place, otherwise the partial (max, sum, O) goes to the workspace and a small second kernel
// (programmatic dependent launch) merges the partials of each such pair. The finish
// normalises, rounds to BF16, gates and rounds again.
// FP8 cache: K and V bytes become f16 in registers (every e4m3 value is exact in f16) and the
// MMAs run in f16 with q converted to f16 once. The d axis is permuted the same way in q and K
// (and undone on the output for V) so that each thread's bytes are contiguous in shared memory.
// Every wait is bounded: on expiry the CTA records BEAM_DEV_TIMEOUT, stops issuing, lets its
// issued copies land and finishes without valid results.
#include <cuda.h>
#include <math.h>

#include "attn_dec.cuh"
#include "common.cuh"
#include "mma.cuh"
#include "tcgen05.cuh"

namespace beam {
namespace adec {
namespace {

using namespace beam::tc;

constexpr float kNegInf = -INFINITY;
constexpr float kRescale = 8.f;   // log2 units
constexpr int D = 128;
constexpr int kHeads = 8;         // MMA N: query heads of one KV group (G <= 8)
constexpr int kMaxParts = 160;    // partials of one pair at most

template <bool FP8>
struct Cfg {
  static constexpr int NCW = FP8 ? 8 : 4;          // consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;   // + the TMA warp
  static constexpr int BK = 16 * NCW;              // keys per block
  static constexpr int ROWB = FP8 ? D : 2 * D;     // bytes of one cached key row
  static constexpr int KB = BK * ROWB;             // K (or V) bytes of one block
  static constexpr int STAGE = 2 * KB;
  static constexpr int NST = 4;
  static constexpr int OLD = D + 4;                // row stride of the combine buffer (floats)
  // combine area, after the stages (byte offsets)
  static constexpr int COMB = NST * STAGE;
  static constexpr int OW = COMB;                                  // [NCW][8][OLD] O partials
  static constexpr int MLW = OW + NCW * kHeads * OLD * 4;          // [NCW][8][2] (m, l)
  static constexpr int FW = MLW + NCW * kHeads * 2 * 4;            // [NCW][8] warp weights
  static constexpr int LH = FW + NCW * kHeads * 4;                 // [8] sum, [8] max
  static constexpr int MISC = LH + 2 * kHeads * 4;                 // ints: -, abort, issued
  static constexpr int BAR = (MISC + 16 + 7) / 8 * 8;
  static constexpr int BYTES = BAR + 2 * NST * 8 + 1024;           // + alignment slack
};

struct Params {
  const uint16_t* q;
  const int32_t* seq_id;
  const int32_t* pos;
  const uint16_t* gpre;
  const uint16_t* gate_bias;
  uint16_t* og;
  float* part_acc;   // [grid][2][8][D]: a CTA's partials of its first and its last pair
  float* part_ml;    // [grid][2][8][2]
  int n_q, n_kv, G, num_seqs, cap, window;
  int NB;            // blocks per pair (sized by max_pos)
  int R;             // blocks per CTA
  int total;         // pairs * NB
  float sl2, v_scale;
};

// Partial slot of CTA c for pair q: 0 when q is the first pair of c's range, else 1 (a pair
// that is neither first nor last in a range lies whole inside it and needs no partial).
__device__ __forceinline__ size_t part_slot(const Params& P, int q, int c) {
  const int first = int((int64_t(c) * P.R) / P.NB);
  return size_t(2 * c + (q == first ? 0 : 1));
}

// Pair q = token * n_kv + KV head: its valid keys are positions [lo, p]; block b holds
// positions BK*b + 1 .. BK*b + BK, at ring slots starting at (BK*b) mod cap (a ring's capacity
// is a multiple of BK, so no block crosses the end of the ring). The pair's blocks are
// blk0 .. blk0 + nbq - 1.
struct Pair {
  int t, hk, p, s, lo, blk0, nbq;
  bool ok;
  unsigned int bad;
};
template <int BK>
__device__ __forceinline__ Pair pair_of(const Params& P, int q) {
  Pair r;
  r.t = q / P.n_kv;
  r.hk = q - r.t * P.n_kv;
  r.p = P.pos[r.t];
  r.s = P.seq_id[r.t];
  r.bad = 0;
  if (r.p < 1 || (P.window == 0 && r.p > P.cap)) r.bad = BEAM_DEV_BAD_POSITION;
  else if (r.s < 0 || r.s >= P.num_seqs) r.bad = BEAM_DEV_BAD_SEQ;
  r.lo = P.window > 0 ? max(1, r.p - P.window + 1) : 1;
  r.blk0 = r.bad ? 0 : (r.lo - 1) / BK;
  r.nbq = r.bad ? 0 : (r.p - 1) / BK - r.blk0 + 1;
  if (r.nbq > P.NB) {   // a position beyond the host's bound max_pos
    r.bad = BEAM_DEV_BAD_POSITION;
    r.nbq = 0;
  }
  r.ok = r.bad == 0;
  return r;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Transpose of the warp's 8x8 b16 matrix held one 32-bit pair per thread.
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f16x2(uint32_t w, float& lo, float& hi) {
  asm("{.reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b;}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
}
// Four e4m3 codes -> two f16x2 words (bytes 0-1 -> lo, bytes 2-3 -> hi), exactly.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{.reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b;}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <int NT>
__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// O^T += V^T . P^T over the warp's 16 keys. MASK: keys outside the pair's range (whose slots
// may hold anything, NaN included) have their V values replaced by zeros, so that P = 0 there
// contributes exactly nothing; m01 / m89 select the valid halves of keys (2c, 2c+1) and
// (2c+8, 2c+9).
template <bool FP8, bool MASK>
__device__ __forceinline__ void pv_block(uint32_t vb, const uint32_t (&voff)[4], uint32_t bh0,
                                         uint32_t bh1, uint32_t bl0, uint32_t bl1, uint32_t m01,
                                         uint32_t m89, float (&acc)[8][4]) {
  using C = Cfg<FP8>;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int w = threadIdx.x >> 5;
  if constexpr (!FP8) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t a[4];
      ldsm_x4_t(vb + (mt >> 2) * (C::KB / 2) + voff[mt & 3], a[0], a[1], a[2], a[3]);
      if (MASK) {
        a[0] &= m01;
        a[1] &= m01;
        a[2] &= m89;
        a[3] &= m89;
      }
      mma_bf16(acc[mt], a, bh0, bh1);
      mma_bf16(acc[mt], a, bl0, bl1);
    }
  } else {
    // key rows 16w + {2c, 2c+1, 2c+8, 2c+9}, bytes [16g, 16g + 16): logical row g of m-tile mt
    // is d = 16g + 2mt, row g + 8 is d = 16g + 2mt + 1
    const uint32_t rb = vb + (16 * w + 2 * c) * 128;
    const uint4 q0 = lds128(rb + ((g ^ (2 * c)) << 4));
    const uint4 q1 = lds128(rb + 128 + ((g ^ (2 * c + 1)) << 4));
    const uint4 q2 = lds128(rb + 8 * 128 + ((g ^ (2 * c)) << 4));
    const uint4 q3 = lds128(rb + 9 * 128 + ((g ^ (2 * c + 1)) << 4));
    const uint32_t r0[4] = {q0.x, q0.y, q0.z, q0.w}, r1[4] = {q1.x, q1.y, q1.z, q1.w};
    const uint32_t r2[4] = {q2.x, q2.y, q2.z, q2.w}, r3[4] = {q3.x, q3.y, q3.z, q3.w};
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
      uint32_t a[4];
      e4m3x4_to_f16(prmt(r0[mt >> 1], r1[mt >> 1], sel), a[0], a[1]);
      e4m3x4_to_f16(prmt(r2[mt >> 1], r3[mt >> 1], sel), a[2], a[3]);
      if (MASK) {
        a[0] &= m01;
        a[1] &= m01;
        a[2] &= m89;
        a[3] &= m89;
      }
      mma_f16(acc[mt], a, bh0, bh1);
      mma_f16(acc[mt], a, bl0, bl1);
    }
  }
}

// One warp's 16 keys of a staged block: S^T = K . Q^T, online softmax, O^T += V^T . P^T.
// kb / vb: shared addresses of the block's K and V; kbase: position of the warp's key row 0;
// the pair's keys are positions [lo, p].
template <bool FP8>
__device__ __forceinline__ void warp_block(uint32_t kb, uint32_t vb, const uint32_t (&qb)[8][2],
                                           const uint32_t (&koff)[4], const uint32_t (&voff)[4],
                                           int kbase, int lo, int p, float sl2, float (&m)[2],
                                           float (&l)[2], float (&acc)[8][4]) {
  using C = Cfg<FP8>;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int w = threadIdx.x >> 5;
  const int kp0 = kbase + g;
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (!FP8) {
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
      uint32_t a[4], b[4];
      ldsm_x4(kb + (kk >> 2) * (C::KB / 2) + koff[kk & 3], a[0], a[1], a[2], a[3]);
      ldsm_x4(kb + ((kk + 1) >> 2) * (C::KB / 2) + koff[(kk + 1) & 3], b[0], b[1], b[2], b[3]);
      mma_bf16(sa, a, qb[kk][0], qb[kk][1]);
      mma_bf16(sb, b, qb[kk + 1][0], qb[kk + 1][1]);
    }
  } else {
    // rows 16w + g and 16w + g + 8, bytes [32c, 32c + 32): logical k (16kk + 2c + e [+8]) is
    // byte 32c + 4kk + e [+2]
    const uint32_t r0 = kb + (16 * w + g) * 128, r1 = r0 + 8 * 128;
    const uint4 k00 = lds128(r0 + (((2 * c) ^ g) << 4)), k01 = lds128(r0 + (((2 * c + 1) ^ g) << 4));
    const uint4 k10 = lds128(r1 + (((2 * c) ^ g) << 4)), k11 = lds128(r1 + (((2 * c + 1) ^ g) << 4));
    const uint32_t w0[8] = {k00.x, k00.y, k00.z, k00.w, k01.x, k01.y, k01.z, k01.w};
    const uint32_t w1[8] = {k10.x, k10.y, k10.z, k10.w, k11.x, k11.y, k11.z, k11.w};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      e4m3x4_to_f16(w0[kk], a[0], a[2]);
      e4m3x4_to_f16(w1[kk], a[1], a[3]);
      if (kk & 1) mma_f16(sb, a, qb[kk][0], qb[kk][1]);
      else mma_f16(sa, a, qb[kk][0], qb[kk][1]);
    }
  }
  // S^T fragment: [0] (key g, head 2c), [1] (key g, head 2c+1), [2], [3] key g + 8
  const bool v0 = kp0 >= lo && kp0 <= p, v1 = kp0 + 8 >= lo && kp0 + 8 <= p;
  float x[4];
  x[0] = v0 ? (sa[0] + sb[0]) * sl2 : kNegInf;
  x[1] = v0 ? (sa[1] + sb[1]) * sl2 : kNegInf;
  x[2] = v1 ? (sa[2] + sb[2]) * sl2 : kNegInf;
  x[3] = v1 ? (sa[3] + sb[3]) * sl2 : kNegInf;
  float mh[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mh[0] = fmaxf(mh[0], __shfl_xor_sync(0xffffffffu, mh[0], o));
    mh[1] = fmaxf(mh[1], __shfl_xor_sync(0xffffffffu, mh[1], o));
  }
  if (__any_sync(0xffffffffu, mh[0] > m[0] + kRescale || mh[1] > m[1] + kRescale)) {
    float cr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(m[h], mh[h]);
      cr[h] = m[h] == kNegInf ? 0.f : ex2_approx(m[h] - mn);
      m[h] = mn;
      l[h] *= cr[h];
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc[mt][0] *= cr[0];
      acc[mt][1] *= cr[1];
      acc[mt][2] *= cr[0];
      acc[mt][3] *= cr[1];
    }
  }
  const float ms0 = m[0] == kNegInf ? 0.f : m[0], ms1 = m[1] == kNegInf ? 0.f : m[1];
  const float p0 = ex2_approx(x[0] - ms0), p1 = ex2_approx(x[1] - ms1);
  const float p2 = ex2_approx(x[2] - ms0), p3 = ex2_approx(x[3] - ms1);
  l[0] += p0 + p2;
  l[1] += p1 + p3;
  // P (key rows, head columns) as hi + lo, then transposed into the B fragments of P^T:
  // b0 = (keys 2c, 2c+1; head g), b1 = (keys 2c+8, 2c+9; head g)
  uint32_t h01, h23, l01, l23;
  if constexpr (!FP8) {
    h01 = pack_bf16x2(p0, p1);
    h23 = pack_bf16x2(p2, p3);
    l01 = pack_bf16x2(p0 - bf_lo(h01), p1 - bf_hi(h01));
    l23 = pack_bf16x2(p2 - bf_lo(h23), p3 - bf_hi(h23));
  } else {
    float f0, f1, f2, f3;
    h01 = pack_f16x2(p0, p1);
    h23 = pack_f16x2(p2, p3);
    unpack_f16x2(h01, f0, f1);
    unpack_f16x2(h23, f2, f3);
    l01 = pack_f16x2(p0 - f0, p1 - f1);
    l23 = pack_f16x2(p2 - f2, p3 - f3);
  }
  const uint32_t bh0 = movtrans(h01), bh1 = movtrans(h23);
  const uint32_t bl0 = movtrans(l01), bl1 = movtrans(l23);
  if (kbase >= lo && kbase + 15 <= p) {
    pv_block<FP8, false>(vb, voff, bh0, bh1, bl0, bl1, 0u, 0u, acc);
  } else {
    auto ok = [&](int k) { return kbase + k >= lo && kbase + k <= p; };
    const uint32_t m01 = (ok(2 * c) ? 0x0000FFFFu : 0u) | (ok(2 * c + 1) ? 0xFFFF0000u : 0u);
    const uint32_t m89 = (ok(2 * c + 8) ? 0x0000FFFFu : 0u) | (ok(2 * c + 9) ? 0xFFFF0000u : 0u);
    pv_block<FP8, true>(vb, voff, bh0, bh1, bl0, bl1, m01, m89, acc);
  }
}

template <bool FP8>
__global__ void __launch_bounds__(Cfg<FP8>::THREADS, 1) attn_decode_tma_kernel(
    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
    const Params P) {
  using C = Cfg<FP8>;
  constexpr int NCT = C::NCW * 32;   // consumer threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar_full = sbase + C::BAR, bar_empty = bar_full + 8 * C::NST;
  volatile int* misc = reinterpret_cast<volatile int*>(sm + C::MISC);   // -, abort, issued
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, C::NCW);
    }
    misc[1] = 0;
    misc[2] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  const int f_lo = blockIdx.x * P.R, f_hi = min(P.total, f_lo + P.R);

  if (warp == C::NCW) {
    // ---------------- producer: one lane issues the TMA loads of every block in range
    if (lane == 0) {
      int i = 0;
      bool run = true;
      for (int f = f_lo; f < f_hi && run;) {
        const int q = f / P.NB, j0 = f - q * P.NB, j1 = min(P.NB, j0 + (f_hi - f));
        f += j1 - j0;
        const Pair pr = pair_of<C::BK>(P, q);
        const int jl = min(j1, pr.nbq);
        const int z = pr.s * P.n_kv + pr.hk;
        for (int j = j0; j < jl; ++j) {
          const int st = i % C::NST;
          if (misc[1] != 0 ||
              (i >= C::NST && !mbar_wait(bar_empty + 8 * st, ((i / C::NST) - 1) & 1))) {
            misc[1] = 1;
            run = false;
            break;
          }
          const int b = pr.blk0 + j;
          const int slot = P.window > 0 ? (C::BK * b) % P.cap : C::BK * b;
          const uint32_t dk = sbase + st * C::STAGE, dv = dk + C::KB, fb = bar_full + 8 * st;
          mbar_expect_tx(fb, C::STAGE);
          if constexpr (FP8) {
            tma_load_3d(dk, &tk, 0, slot, z, fb);
            tma_load_3d(dv, &tv, 0, slot, z, fb);
          } else {
            tma_load_3d(dk, &tk, 0, slot, z, fb);
            tma_load_3d(dk + C::KB / 2, &tk, 64, slot, z, fb);
            tma_load_3d(dv, &tv, 0, slot, z, fb);
            tma_load_3d(dv + C::KB / 2, &tv, 64, slot, z, fb);
          }
          ++i;
        }
      }
      misc[2] = i;
    }
  } else {
    // ---------------- consumers
    const int w = warp, g = lane >> 2, c = lane & 3;
    const int ct = threadIdx.x;
    uint32_t koff[4] = {0, 0, 0, 0}, voff[4] = {0, 0, 0, 0};
    if constexpr (!FP8) {
      // ldmatrix row addresses: K (A operand, 16 keys x 16 d): matrices (keys 0-7 | 8-15) x
      // (d chunk 2kk | 2kk+1); V (A = V^T via .trans): (keys 0-7, chunk 2mt), (0-7, 2mt+1),
      // (8-15, 2mt), (8-15, 2mt+1). 128-byte swizzle: chunk ^= row % 8.
      const int rk = 16 * w + ((lane >> 3) & 1) * 8 + (lane & 7), ck = (lane >> 4) & 1;
      const int rv = 16 * w + ((lane >> 4) & 1) * 8 + (lane & 7), cv = (lane >> 3) & 1;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        koff[e] = uint32_t(rk * 128 + (((2 * e + ck) ^ (lane & 7)) << 4));
        voff[e] = uint32_t(rv * 128 + (((2 * e + cv) ^ (lane & 7)) << 4));
      }
    }
    float* Ow = reinterpret_cast<float*>(sm + C::OW);
    float* MLw = reinterpret_cast<float*>(sm + C::MLW);
    float* FWs = reinterpret_cast<float*>(sm + C::FW);
    float* LHs = reinterpret_cast<float*>(sm + C::LH);   // [0, 8) sums, [8, 16) maxima
    const int G = P.G;
    int i = 0;
    for (int f = f_lo; f < f_hi;) {
      const int q = f / P.NB, j0 = f - q * P.NB, j1 = min(P.NB, j0 + (f_hi - f));
      f += j1 - j0;
      const Pair pr = pair_of<C::BK>(P, q);
      const int jl = min(j1, pr.nbq);
      if (pr.bad && j0 == 0 && pr.hk == 0 && ct == 0) flag(pr.bad);
      // q fragments (B operand, column = head g)
      uint32_t qb[8][2];
      {
        const bool rok = g < G;
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(
            P.q + (size_t(pr.t) * P.n_q + pr.hk * G + (rok ? g : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if constexpr (!FP8) {
            qb[kk][0] = rok ? qr[8 * kk + c] : 0u;
            qb[kk][1] = rok ? qr[8 * kk + c + 4] : 0u;
          } else {
            const uint32_t x0 = rok ? qr[16 * c + 2 * kk] : 0u, x1 = rok ? qr[16 * c + 2 * kk + 1] : 0u;
            qb[kk][0] = pack_f16x2(bf_lo(x0), bf_hi(x0));
            qb[kk][1] = pack_f16x2(bf_lo(x1), bf_hi(x1));
          }
        }
      }
      float acc[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
      for (int j = j0; j < jl; ++j, ++i) {
        const int st = i % C::NST;
        bool ok = misc[1] == 0;
        if (ok) ok = mbar_wait(bar_full + 8 * st, (i / C::NST) & 1);
        if (__all_sync(0xffffffffu, ok)) {
          const uint32_t kb = sbase + st * C::STAGE;
          const int kbase = C::BK * (pr.blk0 + j) + 16 * w + 1;
          warp_block<FP8>(kb, kb + C::KB, qb, koff, voff, kbase, pr.lo, pr.p, P.sl2, m, l, acc);
        } else if (lane == 0) {
          misc[1] = 1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
      }
      // ---- combine the consumer warps' partials of pair q
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
      }
      consumer_bar<NCT>();   // the previous pair's readers of the combine area are done
      {
        float* ow = Ow + w * kHeads * C::OLD;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int da = FP8 ? 16 * g + 2 * mt : 16 * mt + g;
          const int db = FP8 ? da + 1 : da + 8;
          ow[(2 * c) * C::OLD + da] = acc[mt][0];
          ow[(2 * c + 1) * C::OLD + da] = acc[mt][1];
          ow[(2 * c) * C::OLD + db] = acc[mt][2];
          ow[(2 * c + 1) * C::OLD + db] = acc[mt][3];
        }
        if (g == 0) {
          MLw[(w * kHeads + 2 * c) * 2] = m[0];
          MLw[(w * kHeads + 2 * c) * 2 + 1] = l[0];
          MLw[(w * kHeads + 2 * c + 1) * 2] = m[1];
          MLw[(w * kHeads + 2 * c + 1) * 2 + 1] = l[1];
        }
      }
      consumer_bar<NCT>();
      if (ct < G) {
        const int h = ct;
        float M = kNegInf;
#pragma unroll
        for (int ww = 0; ww < C::NCW; ++ww) M = fmaxf(M, MLw[(ww * kHeads + h) * 2]);
        float L = 0.f;
#pragma unroll
        for (int ww = 0; ww < C::NCW; ++ww) {
          const float fw = M == kNegInf ? 0.f : ex2_approx(MLw[(ww * kHeads + h) * 2] - M);
          FWs[ww * kHeads + h] = fw;
          L += fw * MLw[(ww * kHeads + h) * 2 + 1];
        }
        LHs[h] = L;
        LHs[kHeads + h] = M;
      }
      consumer_bar<NCT>();
      const int c_first = int((int64_t(q) * P.NB) / P.R);
      const int c_last = int((int64_t(q + 1) * P.NB - 1) / P.R);
      const int ncontrib = c_last - c_first + 1;
      if (ncontrib == 1) {
        for (int idx = ct; idx < G * D; idx += NCT) {
          const int h = idx / D, d = idx - h * D;
          float O = 0.f;
#pragma unroll
          for (int ww = 0; ww < C::NCW; ++ww) O += FWs[ww * kHeads + h] * Ow[(ww * kHeads + h) * C::OLD + d];
          const float L = LHs[h];
          const float o = round_bf(O * (L > 0.f ? P.v_scale / L : 0.f));
          const int hq = pr.hk * G + h;
          const size_t oi = (size_t(pr.t) * P.n_q + hq) * D + d;
          const float gate = sigmoidf_(bf2f(P.gpre[oi]) + bf2f(P.gate_bias[hq]));
          P.og[oi] = f2bf(o * gate);
        }
      } else {
        const size_t pb = part_slot(P, q, blockIdx.x) * kHeads;
        for (int idx = ct; idx < G * D; idx += NCT) {
          const int h = idx / D, d = idx - h * D;
          float O = 0.f;
#pragma unroll
          for (int ww = 0; ww < C::NCW; ++ww) O += FWs[ww * kHeads + h] * Ow[(ww * kHeads + h) * C::OLD + d];
          P.part_acc[(pb + h) * D + d] = O;
        }
        if (ct < G) {
          P.part_ml[(pb + ct) * 2] = LHs[kHeads + ct];
          P.part_ml[(pb + ct) * 2 + 1] = LHs[ct];
        }
      }
    }
  }
  __syncthreads();
  // dependents are released only now, not at entry: launched early, the merge and the o_proj
  // GEMV behind it (which prefetches its weights into L2 before its wait) ran beside the key
  // stream and cost more than the launch latency they hide (measured: the 8-token
  // verification step 2.82 -> 2.59 ms with the grouped kernel; neutral to slightly faster
  // with the per-token one)
  pdl_trigger();
  if (warp == C::NCW && lane == 0) {
    // normally a no-op: every issued block was consumed; after an expired wait, let the
    // copies still in flight land before the CTA's shared memory is released
    const int n = misc[2];
    for (int k = n > C::NST ? n - C::NST : 0; k < n; ++k)
      mbar_wait(bar_full + 8 * (k % C::NST), (k / C::NST) & 1);
    if (misc[1]) flag(BEAM_DEV_TIMEOUT);
  }
}

// Finish of the pairs split between CTAs: merge CTA m takes the pair whose first block lies in
// CTA m's range and that runs on past it (at most one), combines the partials of the CTAs
// c_first .. c_last, normalises, rounds, gates and rounds.
constexpr int kMergeThreads = 192;
__global__ void __launch_bounds__(kMergeThreads) attn_decode_merge_kernel(const Params P) {
  pdl_trigger();
  __shared__ float wsh[kHeads][kMaxParts];   // part maxima, then their weights
  __shared__ float lsh[kHeads][kMaxParts];   // part sums
  __shared__ float inv[kHeads];
  __shared__ int sl[kMaxParts];
  const int m = blockIdx.x;
  const int f_last = int(min(int64_t(P.total), int64_t(m + 1) * P.R) - 1);
  const int q = f_last / P.NB;
  const int c_first = int((int64_t(q) * P.NB) / P.R);
  const int c_last = int((int64_t(q + 1) * P.NB - 1) / P.R);
  if (c_first != m || c_last == m) return;
  pdl_wait();
  const int n = c_last - c_first + 1, G = P.G;
  const int t = q / P.n_kv, hk = q - t * P.n_kv;
  for (int s = threadIdx.x; s < n; s += kMergeThreads) sl[s] = int(part_slot(P, q, m + s) * kHeads);
  __syncthreads();
  // every part's (max, sum) fetched at once into shared memory, then reduced per head
  for (int i = threadIdx.x; i < n * G; i += kMergeThreads) {
    const int s = i / G, h = i - s * G;
    const float2 v = __ldcg(reinterpret_cast<const float2*>(P.part_ml + (sl[s] + h) * 2));
    wsh[h][s] = v.x;
    lsh[h][s] = v.y;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = kNegInf;
    for (int s = 0; s < n; ++s) M = fmaxf(M, wsh[h][s]);
    float L = 0.f;
    for (int s = 0; s < n; ++s) {
      const float fw = M == kNegInf ? 0.f : ex2_approx(wsh[h][s] - M);
      wsh[h][s] = fw;
      L += fw * lsh[h][s];
    }
    inv[h] = L > 0.f ? P.v_scale / L : 0.f;
  }
  __syncthreads();
  // one thread per 4 consecutive outputs of a head; all parts' loads issued 8 at a time
  for (int o4 = threadIdx.x; o4 < G * (D / 4); o4 += kMergeThreads) {
    const int h = o4 / (D / 4), d = 4 * (o4 - h * (D / 4));
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 8 <= n; s += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = __ldcg(reinterpret_cast<const float4*>(P.part_acc + size_t(sl[s + u] + h) * D + d));
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float fw = wsh[h][s + u];
        O.x += fw * v[u].x;
        O.y += fw * v[u].y;
        O.z += fw * v[u].z;
        O.w += fw * v[u].w;
      }
    }
    for (; s < n; ++s) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(P.part_acc + size_t(sl[s] + h) * D + d));
      const float fw = wsh[h][s];
      O.x += fw * v.x;
      O.y += fw * v.y;
      O.z += fw * v.z;
      O.w += fw * v.w;
    }
    const int hq = hk * G + h;
    const size_t oi = (size_t(t) * P.n_q + hq) * D + d;
    const float gb = bf2f(P.gate_bias[hq]);
    const uint2 gv = *reinterpret_cast<const uint2*>(P.gpre + oi);
    const float o0 = round_bf(O.x * inv[h]), o1 = round_bf(O.y * inv[h]);
    const float o2 = round_bf(O.z * inv[h]), o3 = round_bf(O.w * inv[h]);
    const uint32_t r0 = pack_bf16x2(o0 * sigmoidf_(bf_lo(gv.x) + gb), o1 * sigmoidf_(bf_hi(gv.x) + gb));
    const uint32_t r1 = pack_bf16x2(o2 * sigmoidf_(bf_lo(gv.y) + gb), o3 * sigmoidf_(bf_hi(gv.y) + gb));
    *reinterpret_cast<uint2*>(P.og + oi) = make_uint2(r0, r1);
  }
}

// ------------------------------------------------------------------------------------------
// Verification batches (several new tokens of one sequence, full attention, BF16 cache): the
// tokens of a sequence share every K/V block. A group is a run of up to TG consecutive tokens
// of the call with the same sequence id; its query rows (token-major, then the G heads of the
// KV group) are the columns of NT n-tiles of 8, so a block loaded once serves the whole group
// instead of being read once per token. The (group, KV head) pairs take the place of the
// (token, KV head) pairs above: blocks of 64 keys, equal contiguous ranges per CTA, partials
// and a merge kernel for pairs split between CTAs. Consumer warp w takes n-tile w % NT and
// the 16-key slices w / NT, w / NT + WPT, ... of every block. Each column masks the keys past
// its own token's position; V is masked only past the group's last position (slots there may
// hold anything). The group list is built on the device from seq_id, so any token order is
// computed correctly; a sequence's tokens share blocks only where they are consecutive.
// ------------------------------------------------------------------------------------------
constexpr int kVMaxParts = 40;   // CTAs meeting one (group, KV head) pair at most

template <int NT>
struct VCfg {
  static constexpr int WPT = NT <= 3 ? 4 : (NT <= 6 ? 2 : 1);   // warps per n-tile
  static constexpr int NCW = NT * WPT;                           // consumer warps
  static constexpr int THREADS = (NCW + 1) * 32;
  static constexpr int NCOL = NT * 8;
  static constexpr int BK = 64;
  static constexpr int KB = BK * 2 * D;    // K (or V) bytes of one block
  static constexpr int STAGE = 2 * KB;
  static constexpr int NST = 4;
  static constexpr int OLD = D + 4;
  static constexpr int OW = NST * STAGE;                         // [NCW][8][OLD] O partials
  static constexpr int MLW = OW + NCW * 8 * OLD * 4;             // [NCW][8][2] (m, l)
  static constexpr int FW = MLW + NCW * 8 * 2 * 4;               // [NCW][8] warp weights
  static constexpr int LH = FW + NCW * 8 * 4;                    // [NCOL] sums, [NCOL] maxima
  static constexpr int GL = LH + 2 * NCOL * 4;                   // [kVerifyMaxT + 1] group starts
  static constexpr int MISC = GL + (kVerifyMaxT + 1) * 4;        // ints: groups, abort, issued
  static constexpr int BAR = (MISC + 16 + 7) / 8 * 8;
  static constexpr int BYTES = BAR + 2 * NST * 8 + 1024;         // + alignment slack
};
static_assert(VCfg<12>::BYTES <= 227 * 1024, "verify form exceeds shared memory");

struct VParams {
  const uint16_t* q;
  const int32_t* seq_id;
  const int32_t* pos;
  const uint16_t* gpre;
  const uint16_t* gate_bias;
  uint16_t* og;
  float* part_acc;   // [grid][2][NCOL][D]
  float* part_ml;    // [grid][2][NCOL][2]
  int* groups;       // [0] = number of groups n, [1 + i] = first token of group i, [1 + n] = T
  int T, TG, n_q, n_kv, G, num_seqs, cap;
  int NB;            // blocks per (group, KV head) pair: positions 1 .. max_pos
  int grid;
  float sl2;
};

// Blocks per CTA: an equal share of the flattened (pair, block) space, and at least enough
// that a pair meets no more than kVMaxParts CTA ranges.
__host__ __device__ __forceinline__ int verify_range(int total, int NB, int grid) {
  const int a = (total + grid - 1) / grid, b = (NB + kVMaxParts - 2) / (kVMaxParts - 1);
  const int r = a > b ? a : b;
  return r > 1 ? r : 1;
}
__device__ __forceinline__ size_t vpart_slot(int q, int c, int R, int NB) {
  const int first = int((int64_t(c) * R) / NB);
  return size_t(2 * c + (q == first ? 0 : 1));
}

// The call's group list, built by one warp: a group starts at token t when t opens a run of
// equal sequence ids or lies a multiple of TG tokens into its run. gl[i] = first token of
// group i, gl[n] = T; returns n (in every lane).
__device__ int build_groups(const VParams& P, int* gl) {
  const int lane = threadIdx.x & 31;
  int run = 0, last_s = 0, n = 0;
  for (int base = 0; base < P.T; base += 32) {
    const int t = base + lane;
    const bool valid = t < P.T;
    const int s = valid ? P.seq_id[t] : 0;
    int sp = __shfl_up_sync(0xffffffffu, s, 1);
    if (lane == 0) sp = last_s;
    const unsigned brk = __ballot_sync(0xffffffffu, valid && (t == 0 || s != sp));
    const unsigned below = brk & (0xffffffffu >> (31 - lane));   // bits 0 .. lane
    const int rs = below ? base + 31 - __clz(below) : run;        // start of t's run
    const bool start = valid && (t - rs) % P.TG == 0;
    const unsigned sm = __ballot_sync(0xffffffffu, start);
    if (start) gl[n + __popc(sm & ((1u << lane) - 1u))] = t;
    n += __popc(sm);
    run = __shfl_sync(0xffffffffu, rs, 31);
    last_s = __shfl_sync(0xffffffffu, s, 31);
  }
  if (lane == 0) gl[n] = P.T;
  __syncwarp();
  return n;
}

// Pair q = group * n_kv + KV head. A token takes part when 1 <= pos <= cap and its position
// lies within the host's bound (NB blocks); pg = the last position of the group's tokens that
// take part, nbq = the blocks covering 1 .. pg.
struct VGroup {
  int t0, cnt, s, hk, pg, nbq;
  unsigned int bad;
};
__device__ __forceinline__ bool vtoken_ok(const VParams& P, int p) {
  return p >= 1 && p <= P.cap && (p - 1) / VCfg<2>::BK < P.NB;
}
__device__ __forceinline__ VGroup group_of(const VParams& P, const int* gl, int q) {
  VGroup r;
  const int gi = q / P.n_kv;
  r.hk = q - gi * P.n_kv;
  r.t0 = gl[gi];
  r.cnt = gl[gi + 1] - r.t0;
  r.s = P.seq_id[r.t0];
  r.bad = 0;
  r.pg = 0;
  if (r.s < 0 || r.s >= P.num_seqs) {
    r.bad = BEAM_DEV_BAD_SEQ;
  } else {
    for (int i = 0; i < r.cnt; ++i) {
      const int p = P.pos[r.t0 + i];
      if (vtoken_ok(P, p)) r.pg = max(r.pg, p);
      else r.bad = BEAM_DEV_BAD_POSITION;
    }
  }
  r.nbq = r.pg >= 1 ? (r.pg - 1) / VCfg<2>::BK + 1 : 0;
  return r;
}

// One warp's 16 keys of a staged block for 8 query columns of a group (BF16 cache): as
// warp_block, with a last position per accumulator column (pc0: column 2c, pc1: column 2c+1;
// 0 = the column attends to nothing) and V masked past the group's last position pg. Keys
// start at position 1 (full attention), so kbase >= 1.
__device__ __forceinline__ void warp_block_cols(uint32_t kb, uint32_t vb,
                                                const uint32_t (&qb)[8][2],
                                                const uint32_t (&koff)[4],
                                                const uint32_t (&voff)[4], int kbase, int pc0,
                                                int pc1, int pg, float sl2, float (&m)[2],
                                                float (&l)[2], float (&acc)[8][4]) {
  using C = Cfg<false>;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int kp0 = kbase + g;
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; kk += 2) {
    uint32_t a[4], b[4];
    ldsm_x4(kb + (kk >> 2) * (C::KB / 2) + koff[kk & 3], a[0], a[1], a[2], a[3]);
    ldsm_x4(kb + ((kk + 1) >> 2) * (C::KB / 2) + koff[(kk + 1) & 3], b[0], b[1], b[2], b[3]);
    mma_bf16(sa, a, qb[kk][0], qb[kk][1]);
    mma_bf16(sb, b, qb[kk + 1][0], qb[kk + 1][1]);
  }
  // S^T fragment: [0] (key g, column 2c), [1] (key g, column 2c+1), [2], [3] key g + 8
  float x[4];
  x[0] = kp0 <= pc0 ? (sa[0] + sb[0]) * sl2 : kNegInf;
  x[1] = kp0 <= pc1 ? (sa[1] + sb[1]) * sl2 : kNegInf;
  x[2] = kp0 + 8 <= pc0 ? (sa[2] + sb[2]) * sl2 : kNegInf;
  x[3] = kp0 + 8 <= pc1 ? (sa[3] + sb[3]) * sl2 : kNegInf;
  float mh[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mh[0] = fmaxf(mh[0], __shfl_xor_sync(0xffffffffu, mh[0], o));
    mh[1] = fmaxf(mh[1], __shfl_xor_sync(0xffffffffu, mh[1], o));
  }
  if (__any_sync(0xffffffffu, mh[0] > m[0] + kRescale || mh[1] > m[1] + kRescale)) {
    float cr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(m[h], mh[h]);
      cr[h] = m[h] == kNegInf ? 0.f : ex2_approx(m[h] - mn);
      m[h] = mn;
      l[h] *= cr[h];
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc[mt][0] *= cr[0];
      acc[mt][1] *= cr[1];
      acc[mt][2] *= cr[0];
      acc[mt][3] *= cr[1];
    }
  }
  const float ms0 = m[0] == kNegInf ? 0.f : m[0], ms1 = m[1] == kNegInf ? 0.f : m[1];
  const float p0 = ex2_approx(x[0] - ms0), p1 = ex2_approx(x[1] - ms1);
  const float p2 = ex2_approx(x[2] - ms0), p3 = ex2_approx(x[3] - ms1);
  l[0] += p0 + p2;
  l[1] += p1 + p3;
  const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
  const uint32_t l01 = pack_bf16x2(p0 - bf_lo(h01), p1 - bf_hi(h01));
  const uint32_t l23 = pack_bf16x2(p2 - bf_lo(h23), p3 - bf_hi(h23));
  const uint32_t bh0 = movtrans(h01), bh1 = movtrans(h23);
  const uint32_t bl0 = movtrans(l01), bl1 = movtrans(l23);
  if (kbase + 15 <= pg) {
    pv_block<false, false>(vb, voff, bh0, bh1, bl0, bl1, 0u, 0u, acc);
  } else {
    auto ok = [&](int k) { return kbase + k <= pg; };
    const uint32_t m01 = (ok(2 * c) ? 0x0000FFFFu : 0u) | (ok(2 * c + 1) ? 0xFFFF0000u : 0u);
    const uint32_t m89 = (ok(2 * c + 8) ? 0x0000FFFFu : 0u) | (ok(2 * c + 9) ? 0xFFFF0000u : 0u);
    pv_block<false, true>(vb, voff, bh0, bh1, bl0, bl1, m01, m89, acc);
  }
}

// Two 16-key slices of a staged block for the same 8 columns (kb0/vb0: the first slice, kbase0
// its first position; kb1/vb1/kbase1 the second): both S tiles first, one max and rescale over
// the 32 keys, then both P.V products. The same arithmetic as two warp_block_cols calls up to
// the point at which the running max is updated; the two slices' MMA chains interleave.
__device__ __forceinline__ void warp_block_cols2(uint32_t kb0, uint32_t vb0, uint32_t kb1,
                                                 uint32_t vb1, const uint32_t (&qb)[8][2],
                                                 const uint32_t (&koff)[4],
                                                 const uint32_t (&voff)[4], int kbase0, int kbase1,
                                                 int pc0, int pc1, int pg, float sl2,
                                                 float (&m)[2], float (&l)[2], float (&acc)[8][4]) {
  using C = Cfg<false>;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  float s0a[4] = {0.f, 0.f, 0.f, 0.f}, s0b[4] = {0.f, 0.f, 0.f, 0.f};
  float s1a[4] = {0.f, 0.f, 0.f, 0.f}, s1b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < 8; kk += 2) {
    uint32_t a0[4], b0[4], a1[4], b1[4];
    const uint32_t o0 = (kk >> 2) * (C::KB / 2) + koff[kk & 3];
    const uint32_t o1 = ((kk + 1) >> 2) * (C::KB / 2) + koff[(kk + 1) & 3];
    ldsm_x4(kb0 + o0, a0[0], a0[1], a0[2], a0[3]);
    ldsm_x4(kb1 + o0, a1[0], a1[1], a1[2], a1[3]);
    ldsm_x4(kb0 + o1, b0[0], b0[1], b0[2], b0[3]);
    ldsm_x4(kb1 + o1, b1[0], b1[1], b1[2], b1[3]);
    mma_bf16(s0a, a0, qb[kk][0], qb[kk][1]);
    mma_bf16(s1a, a1, qb[kk][0], qb[kk][1]);
    mma_bf16(s0b, b0, qb[kk + 1][0], qb[kk + 1][1]);
    mma_bf16(s1b, b1, qb[kk + 1][0], qb[kk + 1][1]);
  }
  const int k0 = kbase0 + g, k1 = kbase1 + g;
  float x[8];
  x[0] = k0 <= pc0 ? (s0a[0] + s0b[0]) * sl2 : kNegInf;
  x[1] = k0 <= pc1 ? (s0a[1] + s0b[1]) * sl2 : kNegInf;
  x[2] = k0 + 8 <= pc0 ? (s0a[2] + s0b[2]) * sl2 : kNegInf;
  x[3] = k0 + 8 <= pc1 ? (s0a[3] + s0b[3]) * sl2 : kNegInf;
  x[4] = k1 <= pc0 ? (s1a[0] + s1b[0]) * sl2 : kNegInf;
  x[5] = k1 <= pc1 ? (s1a[1] + s1b[1]) * sl2 : kNegInf;
  x[6] = k1 + 8 <= pc0 ? (s1a[2] + s1b[2]) * sl2 : kNegInf;
  x[7] = k1 + 8 <= pc1 ? (s1a[3] + s1b[3]) * sl2 : kNegInf;
  float mh[2] = {fmaxf(fmaxf(x[0], x[2]), fmaxf(x[4], x[6])),
                 fmaxf(fmaxf(x[1], x[3]), fmaxf(x[5], x[7]))};
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mh[0] = fmaxf(mh[0], __shfl_xor_sync(0xffffffffu, mh[0], o));
    mh[1] = fmaxf(mh[1], __shfl_xor_sync(0xffffffffu, mh[1], o));
  }
  if (__any_sync(0xffffffffu, mh[0] > m[0] + kRescale || mh[1] > m[1] + kRescale)) {
    float cr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mn = fmaxf(m[h], mh[h]);
      cr[h] = m[h] == kNegInf ? 0.f : ex2_approx(m[h] - mn);
      m[h] = mn;
      l[h] *= cr[h];
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      acc[mt][0] *= cr[0];
      acc[mt][1] *= cr[1];
      acc[mt][2] *= cr[0];
      acc[mt][3] *= cr[1];
    }
  }
  const float ms0 = m[0] == kNegInf ? 0.f : m[0], ms1 = m[1] == kNegInf ? 0.f : m[1];
  float p[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) p[e] = ex2_approx(x[e] - ((e & 1) ? ms1 : ms0));
  l[0] += (p[0] + p[2]) + (p[4] + p[6]);
  l[1] += (p[1] + p[3]) + (p[5] + p[7]);
  uint32_t bh[4], bl[4];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const uint32_t h01 = pack_bf16x2(p[4 * s], p[4 * s + 1]);
    const uint32_t h23 = pack_bf16x2(p[4 * s + 2], p[4 * s + 3]);
    const uint32_t l01 = pack_bf16x2(p[4 * s] - bf_lo(h01), p[4 * s + 1] - bf_hi(h01));
    const uint32_t l23 = pack_bf16x2(p[4 * s + 2] - bf_lo(h23), p[4 * s + 3] - bf_hi(h23));
    bh[2 * s] = movtrans(h01);
    bh[2 * s + 1] = movtrans(h23);
    bl[2 * s] = movtrans(l01);
    bl[2 * s + 1] = movtrans(l23);
  }
  auto pv = [&](uint32_t vb, int kbase, int s) {
    if (kbase + 15 <= pg) {
      pv_block<false, false>(vb, voff, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1], 0u,
                             0u, acc);
    } else {
      auto ok = [&](int k) { return kbase + k <= pg; };
      const uint32_t m01 = (ok(2 * c) ? 0x0000FFFFu : 0u) | (ok(2 * c + 1) ? 0xFFFF0000u : 0u);
      const uint32_t m89 = (ok(2 * c + 8) ? 0x0000FFFFu : 0u) | (ok(2 * c + 9) ? 0xFFFF0000u : 0u);
      pv_block<false, true>(vb, voff, bh[2 * s], bh[2 * s + 1], bl[2 * s], bl[2 * s + 1], m01,
                            m89, acc);
    }
  };
  pv(vb0, kbase0, 0);
  pv(vb1, kbase1, 1);
}

template <int NT>
__global__ void __launch_bounds__(VCfg<NT>::THREADS, 1) attn_verify_tma_kernel(
    const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
    const VParams P) {
  using C = VCfg<NT>;
  constexpr int NCT = C::NCW * 32;   // consumer threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar_full = sbase + C::BAR, bar_empty = bar_full + 8 * C::NST;
  volatile int* misc = reinterpret_cast<volatile int*>(sm + C::MISC);   // groups, abort, issued
  int* gl = reinterpret_cast<int*>(sm + C::GL);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, C::NCW);
    }
    misc[1] = 0;
    misc[2] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  if (warp == C::NCW) {
    const int n = build_groups(P, gl);
    if (lane == 0) misc[0] = n;
    if (blockIdx.x == 0) {   // for the merge kernel
      for (int i = lane; i <= n; i += 32) P.groups[1 + i] = gl[i];
      if (lane == 0) P.groups[0] = n;
    }
  }
  __syncthreads();
  const int total = misc[0] * P.n_kv * P.NB;
  const int R = verify_range(total, P.NB, P.grid);
  const int f_lo = int(min(int64_t(total), int64_t(blockIdx.x) * R));
  const int f_hi = min(total, f_lo + R);

  if (warp == C::NCW) {
    // ---------------- producer: one lane issues the TMA loads of every block in range
    if (lane == 0) {
      int i = 0;
      bool run = true;
      for (int f = f_lo; f < f_hi && run;) {
        const int q = f / P.NB, j0 = f - q * P.NB, j1 = min(P.NB, j0 + (f_hi - f));
        f += j1 - j0;
        const VGroup gr = group_of(P, gl, q);
        const int jl = min(j1, gr.nbq);
        const int z = gr.s * P.n_kv + gr.hk;
        for (int j = j0; j < jl; ++j) {
          const int st = i % C::NST;
          if (misc[1] != 0 ||
              (i >= C::NST && !mbar_wait(bar_empty + 8 * st, ((i / C::NST) - 1) & 1))) {
            misc[1] = 1;
            run = false;
            break;
          }
          const int slot = C::BK * j;
          const uint32_t dk = sbase + st * C::STAGE, dv = dk + C::KB, fb = bar_full + 8 * st;
          mbar_expect_tx(fb, C::STAGE);
          tma_load_3d(dk, &tk, 0, slot, z, fb);
          tma_load_3d(dk + C::KB / 2, &tk, 64, slot, z, fb);
          tma_load_3d(dv, &tv, 0, slot, z, fb);
          tma_load_3d(dv + C::KB / 2, &tv, 64, slot, z, fb);
          ++i;
        }
      }
      misc[2] = i;
    }
  } else {
    // ---------------- consumers
    const int w = warp, g = lane >> 2, c = lane & 3;
    const int ct = threadIdx.x;
    const int nt = w % NT, sw = w / NT;   // n-tile, first key slice
    // ldmatrix row addresses of key slice 0 (slice s adds 16 rows = 2048 bytes); as in the
    // per-token kernel, 128-byte swizzle: chunk ^= row % 8
    uint32_t koff[4], voff[4];
    {
      const int rk = ((lane >> 3) & 1) * 8 + (lane & 7), ck = (lane >> 4) & 1;
      const int rv = ((lane >> 4) & 1) * 8 + (lane & 7), cv = (lane >> 3) & 1;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        koff[e] = uint32_t(rk * 128 + (((2 * e + ck) ^ (lane & 7)) << 4));
        voff[e] = uint32_t(rv * 128 + (((2 * e + cv) ^ (lane & 7)) << 4));
      }
    }
    float* Ow = reinterpret_cast<float*>(sm + C::OW);
    float* MLw = reinterpret_cast<float*>(sm + C::MLW);
    float* FWs = reinterpret_cast<float*>(sm + C::FW);
    float* LHs = reinterpret_cast<float*>(sm + C::LH);   // [0, NCOL) sums, [NCOL, 2 NCOL) maxima
    const int G = P.G;
    int i = 0;
    for (int f = f_lo; f < f_hi;) {
      const int q = f / P.NB, j0 = f - q * P.NB, j1 = min(P.NB, j0 + (f_hi - f));
      f += j1 - j0;
      const VGroup gr = group_of(P, gl, q);
      const int jl = min(j1, gr.nbq);
      if (gr.bad && j0 == 0 && gr.hk == 0 && ct == 0) flag(gr.bad);
      const int ncols = gr.cnt * G;
      const bool active = 8 * nt < ncols;   // uniform over the warp
      // last position of a column (0: a column past the group, or a token that takes no part)
      auto col_pos = [&](int col) -> int {
        if (col >= ncols || gr.bad == BEAM_DEV_BAD_SEQ) return 0;
        const int p = P.pos[gr.t0 + col / G];
        return vtoken_ok(P, p) ? p : 0;
      };
      const int pc0 = col_pos(8 * nt + 2 * c), pc1 = col_pos(8 * nt + 2 * c + 1);
      // q fragments (B operand, column 8 nt + g)
      uint32_t qb[8][2];
      {
        const int col = 8 * nt + g;
        const bool rok = col < ncols;
        const int tq = gr.t0 + (rok ? col / G : 0), hq = gr.hk * G + (rok ? col % G : 0);
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(P.q + (size_t(tq) * P.n_q + hq) * D);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qb[kk][0] = rok ? qr[8 * kk + c] : 0u;
          qb[kk][1] = rok ? qr[8 * kk + c + 4] : 0u;
        }
      }
      float acc[8][4];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
      for (int j = j0; j < jl; ++j, ++i) {
        const int st = i % C::NST;
        bool ok = misc[1] == 0;
        if (ok) ok = mbar_wait(bar_full + 8 * st, (i / C::NST) & 1);
        if (__all_sync(0xffffffffu, ok)) {
          if (active) {
            const uint32_t kb = sbase + st * C::STAGE;
            if constexpr (C::WPT == 2) {
              // this warp's two slices together (their MMA chains interleave)
              const int s0 = sw, s1 = sw + 2;
              warp_block_cols2(kb + s0 * 2048, kb + C::KB + s0 * 2048, kb + s1 * 2048,
                               kb + C::KB + s1 * 2048, qb, koff, voff, C::BK * j + 16 * s0 + 1,
                               C::BK * j + 16 * s1 + 1, pc0, pc1, gr.pg, P.sl2, m, l, acc);
            } else {
              // one slice (WPT 4), or four one after the other (WPT 1: the paired form
              // would spill at this warp count's register budget)
#pragma unroll
              for (int s = 0; s < 4 / C::WPT; ++s) {
                const int sl = sw + s * C::WPT;
                warp_block_cols(kb + sl * 2048, kb + C::KB + sl * 2048, qb, koff, voff,
                                C::BK * j + 16 * sl + 1, pc0, pc1, gr.pg, P.sl2, m, l, acc);
              }
            }
          }
        } else if (lane == 0) {
          misc[1] = 1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * st);
      }
      // ---- combine the partials of the WPT warps of each n-tile
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
      }
      consumer_bar<NCT>();   // the previous pair's readers of the combine area are done
      {
        float* ow = Ow + w * 8 * C::OLD;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int da = 16 * mt + g, db = da + 8;
          ow[(2 * c) * C::OLD + da] = acc[mt][0];
          ow[(2 * c + 1) * C::OLD + da] = acc[mt][1];
          ow[(2 * c) * C::OLD + db] = acc[mt][2];
          ow[(2 * c + 1) * C::OLD + db] = acc[mt][3];
        }
        if (g == 0) {
          MLw[(w * 8 + 2 * c) * 2] = m[0];
          MLw[(w * 8 + 2 * c) * 2 + 1] = l[0];
          MLw[(w * 8 + 2 * c + 1) * 2] = m[1];
          MLw[(w * 8 + 2 * c + 1) * 2 + 1] = l[1];
        }
      }
      consumer_bar<NCT>();
      if (ct < C::NCOL) {
        const int ntc = ct >> 3, h8 = ct & 7;
        float M = kNegInf;
#pragma unroll
        for (int jw = 0; jw < C::WPT; ++jw) M = fmaxf(M, MLw[((ntc + NT * jw) * 8 + h8) * 2]);
        float L = 0.f;
#pragma unroll
        for (int jw = 0; jw < C::WPT; ++jw) {
          const int wi = (ntc + NT * jw) * 8 + h8;
          const float fw = M == kNegInf ? 0.f : ex2_approx(MLw[wi * 2] - M);
          FWs[wi] = fw;
          L += fw * MLw[wi * 2 + 1];
        }
        LHs[ct] = L;
        LHs[C::NCOL + ct] = M;
      }
      consumer_bar<NCT>();
      const int c_first = int((int64_t(q) * P.NB) / R);
      const int c_last = int((int64_t(q + 1) * P.NB - 1) / R);
      const size_t pb = c_last > c_first ? vpart_slot(q, blockIdx.x, R, P.NB) * C::NCOL : 0;
      for (int idx = ct; idx < ncols * D; idx += NCT) {
        const int col = idx / D, d = idx - col * D;
        const int ntc = col >> 3, h8 = col & 7;
        float O = 0.f;
#pragma unroll
        for (int jw = 0; jw < C::WPT; ++jw) {
          const int wi = (ntc + NT * jw) * 8 + h8;
          O += FWs[wi] * Ow[wi * C::OLD + d];
        }
        if (c_last == c_first) {
          const float L = LHs[col];
          const float o = round_bf(O * (L > 0.f ? 1.f / L : 0.f));
          const int hq = gr.hk * G + col % G;
          const size_t oi = (size_t(gr.t0 + col / G) * P.n_q + hq) * D + d;
          const float gate = sigmoidf_(bf2f(P.gpre[oi]) + bf2f(P.gate_bias[hq]));
          P.og[oi] = f2bf(o * gate);
        } else {
          P.part_acc[(pb + col) * D + d] = O;
        }
      }
      if (c_last > c_first && ct < ncols) {
        P.part_ml[(pb + ct) * 2] = LHs[C::NCOL + ct];
        P.part_ml[(pb + ct) * 2 + 1] = LHs[ct];
      }
    }
  }
  __syncthreads();
  // dependents are released only now, not at entry: launched early, the merge and the o_proj
  // GEMV behind it (which prefetches its weights into L2 before its wait) ran beside the key
  // stream and cost more than the launch latency they hide (measured: the 8-token
  // verification step 2.82 -> 2.59 ms with the grouped kernel; neutral to slightly faster
  // with the per-token one)
  pdl_trigger();
  if (warp == C::NCW && lane == 0) {
    // normally a no-op: every issued block was consumed; after an expired wait, let the
    // copies still in flight land before the CTA's shared memory is released
    const int n = misc[2];
    for (int k = n > C::NST ? n - C::NST : 0; k < n; ++k)
      mbar_wait(bar_full + 8 * (k % C::NST), (k / C::NST) & 1);
    if (misc[1]) flag(BEAM_DEV_TIMEOUT);
  }
}

// Finish of the (group, KV head) pairs split between CTAs: merge CTA m takes the pair whose
// first block lies in CTA m's range and that runs on past it (at most one), combines the
// partials of CTAs c_first .. c_last for each of the group's columns, normalises, rounds,
// gates and rounds.
constexpr int kVMergeThreads = 256;
template <int NT>
__global__ void __launch_bounds__(kVMergeThreads) attn_verify_merge_kernel(const VParams P) {
  constexpr int NCOL = NT * 8;
  pdl_trigger();
  __shared__ float wsh[NCOL][kVMaxParts];   // part maxima, then their weights
  __shared__ float lsh[NCOL][kVMaxParts];   // part sums
  __shared__ float inv[NCOL];
  __shared__ int sl[kVMaxParts];
  pdl_wait();
  const int ng = P.groups[0];
  const int total = ng * P.n_kv * P.NB;
  const int R = verify_range(total, P.NB, P.grid);
  const int m = blockIdx.x;
  if (int64_t(m) * R >= total) return;
  const int f_last = int(min(int64_t(total), int64_t(m + 1) * R) - 1);
  const int q = f_last / P.NB;
  const int c_first = int((int64_t(q) * P.NB) / R);
  const int c_last = int((int64_t(q + 1) * P.NB - 1) / R);
  if (c_first != m || c_last == m) return;
  const int n = c_last - c_first + 1, G = P.G;
  const int gi = q / P.n_kv, hk = q - gi * P.n_kv;
  const int t0 = P.groups[1 + gi], ncols = (P.groups[2 + gi] - t0) * G;
  for (int s = threadIdx.x; s < n; s += kVMergeThreads) sl[s] = int(vpart_slot(q, m + s, R, P.NB) * NCOL);
  __syncthreads();
  for (int i = threadIdx.x; i < n * ncols; i += kVMergeThreads) {
    const int s = i / ncols, h = i - s * ncols;
    const float2 v = __ldcg(reinterpret_cast<const float2*>(P.part_ml + (sl[s] + h) * 2));
    wsh[h][s] = v.x;
    lsh[h][s] = v.y;
  }
  __syncthreads();
  if (threadIdx.x < ncols) {
    const int h = threadIdx.x;
    float M = kNegInf;
    for (int s = 0; s < n; ++s) M = fmaxf(M, wsh[h][s]);
    float L = 0.f;
    for (int s = 0; s < n; ++s) {
      const float fw = M == kNegInf ? 0.f : ex2_approx(wsh[h][s] - M);
      wsh[h][s] = fw;
      L += fw * lsh[h][s];
    }
    inv[h] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  // one thread per 4 consecutive outputs of a column
  for (int o4 = threadIdx.x; o4 < ncols * (D / 4); o4 += kVMergeThreads) {
    const int h = o4 / (D / 4), d = 4 * (o4 - h * (D / 4));
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n; ++s) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(P.part_acc + size_t(sl[s] + h) * D + d));
      const float fw = wsh[h][s];
      O.x += fw * v.x;
      O.y += fw * v.y;
      O.z += fw * v.z;
      O.w += fw * v.w;
    }
    const int hq = hk * G + h % G;
    const size_t oi = (size_t(t0 + h / G) * P.n_q + hq) * D + d;
    const float gb = bf2f(P.gate_bias[hq]);
    const uint2 gv = *reinterpret_cast<const uint2*>(P.gpre + oi);
    const float o0 = round_bf(O.x * inv[h]), o1 = round_bf(O.y * inv[h]);
    const float o2 = round_bf(O.z * inv[h]), o3 = round_bf(O.w * inv[h]);
    const uint32_t r0 = pack_bf16x2(o0 * sigmoidf_(bf_lo(gv.x) + gb), o1 * sigmoidf_(bf_hi(gv.x) + gb));
    const uint32_t r1 = pack_bf16x2(o2 * sigmoidf_(bf_lo(gv.y) + gb), o3 * sigmoidf_(bf_hi(gv.y) + gb));
    *reinterpret_cast<uint2*>(P.og + oi) = make_uint2(r0, r1);
  }
}

struct Plan {
  int NB, R, grid, total;
};

Plan make_plan(int T, int n_kv, int window, int max_pos, bool fp8) {
  const int BK = fp8 ? Cfg<true>::BK : Cfg<false>::BK;
  const int max_keys = window > 0 ? (max_pos < window ? max_pos : window) : max_pos;
  Plan pl;
  pl.NB = (max_keys + BK - 1) / BK + (window > 0 ? 1 : 0);
  pl.total = T * n_kv * pl.NB;
  const int sms = num_sms_cached();
  int grid = pl.total < sms ? pl.total : sms;
  if (grid < 1) grid = 1;
  pl.R = (pl.total + grid - 1) / grid;
  // a pair's blocks meet at most ceil(NB / R) + 1 CTA ranges
  while ((pl.NB + pl.R - 1) / pl.R + 1 > kMaxParts) ++pl.R;
  pl.grid = (pl.total + pl.R - 1) / pl.R;
  return pl;
}

}  // namespace

bool supported(int D_, int G, int window, int cap, bool fp8, const void* k, const void* v,
               int max_keys) {
  if (D_ != D || G < 1 || G > kHeads || max_keys < kMinKeys) return false;
  const int BK = fp8 ? Cfg<true>::BK : Cfg<false>::BK;
  if (window > 0 && cap % BK != 0) return false;
  return aligned16(k) && aligned16(v) && tensor_map_encoder_ready();
}

size_t ws_bytes(int T, int n_kv, int window, int max_pos, bool fp8) {
  if (T <= 0 || max_pos < 1) return 0;
  const Plan pl = make_plan(T, n_kv, window, max_pos, fp8);
  const size_t parts = size_t(pl.grid) * 2 * kHeads;
  return align_up(parts * D * 4, 256) + align_up(parts * 2 * 4, 256);
}

cudaError_t decode(const uint16_t* q, const uint16_t* g, const uint16_t* gate_bias,
                   const int32_t* seq_id, const int32_t* pos, int T, int max_pos, int n_q,
                   int n_kv, const beam_kv_cache& kc, float sl2, float v_scale, uint16_t* og,
                   void* ws, size_t ws_len, cudaStream_t st) {
  const bool fp8 = kc.dtype == BEAM_KV_FP8_E4M3;
  const Plan pl = make_plan(T, n_kv, kc.window, max_pos, fp8);
  if (ws_len < ws_bytes(T, n_kv, kc.window, max_pos, fp8)) return cudaErrorInvalidValue;
  const size_t parts = size_t(pl.grid) * 2 * kHeads;
  char* w = static_cast<char*>(ws);
  float* part_acc = reinterpret_cast<float*>(w);
  float* part_ml = reinterpret_cast<float*>(w + align_up(parts * D * 4, 256));
  CUtensorMap mk, mv;
  {
    const int rowb = fp8 ? D : 2 * D;
    const uint64_t dims[3] = {uint64_t(fp8 ? D : D), uint64_t(kc.capacity),
                              uint64_t(kc.num_seqs) * n_kv};
    const uint64_t str[2] = {uint64_t(rowb), uint64_t(kc.capacity) * rowb};
    const uint32_t box[3] = {uint32_t(fp8 ? 128 : 64), uint32_t(fp8 ? Cfg<true>::BK : Cfg<false>::BK), 1};
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_tiled(&mk, dt, 3, kc.k, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&mv, dt, 3, kc.v, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  cudaError_t e;
  Params prm{q,  seq_id, pos, g, gate_bias, og, part_acc, part_ml, n_q, n_kv, n_q / n_kv,
             kc.num_seqs, kc.capacity, kc.window, pl.NB, pl.R, pl.total, sl2, v_scale};
  if (fp8) {
    auto kern = attn_decode_tma_kernel<true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<true>::BYTES);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(pl.grid), dim3(Cfg<true>::THREADS), Cfg<true>::BYTES, st, mk, mv, prm);
  } else {
    auto kern = attn_decode_tma_kernel<false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<false>::BYTES);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(pl.grid), dim3(Cfg<false>::THREADS), Cfg<false>::BYTES, st, mk, mv, prm);
  }
  if (e != cudaSuccess) return e;
  // ranges that are whole multiples of a pair's blocks split no pair: nothing to merge
  if (pl.R % pl.NB != 0) {
    e = launch_pdl(attn_decode_merge_kernel, dim3(pl.grid), dim3(kMergeThreads), 0, st, prm);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}


namespace {

// n-tile counts compiled for the grouped form; a group's G * TG columns take the next one up
constexpr int kVerifyNT[] = {2, 3, 4, 6, 12};
constexpr int kVerifyMaxNT = 12;

int verify_tg(int G, int max_q_per_seq) {
  const int cap = kVerifyMaxNT * 8 / G;
  return max_q_per_seq < cap ? max_q_per_seq : cap;
}
int verify_nt(int G, int TG) {
  const int need = (G * TG + 7) / 8;
  for (int nt : kVerifyNT)
    if (nt >= need) return nt;
  return 0;
}
size_t verify_ws_for(int T, int nt) {
  const size_t parts = size_t(num_sms_cached()) * 2 * nt * 8;
  return align_up(parts * D * 4, 256) + align_up(parts * 2 * 4, 256) +
         align_up(size_t(T + 2) * 4, 256);
}

bool encode_kv_maps(const beam_kv_cache& kc, int n_kv, bool fp8, CUtensorMap* mk, CUtensorMap* mv) {
  const int rowb = fp8 ? D : 2 * D;
  const uint64_t dims[3] = {uint64_t(D), uint64_t(kc.capacity), uint64_t(kc.num_seqs) * n_kv};
  const uint64_t str[2] = {uint64_t(rowb), uint64_t(kc.capacity) * rowb};
  const uint32_t box[3] = {uint32_t(fp8 ? 128 : 64), uint32_t(fp8 ? Cfg<true>::BK : Cfg<false>::BK), 1};
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return encode_tiled(mk, dt, 3, kc.k, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_tiled(mv, dt, 3, kc.v, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int NT>
cudaError_t launch_verify(const CUtensorMap& mk, const CUtensorMap& mv, const VParams& prm,
                          cudaStream_t st) {
  auto kern = attn_verify_tma_kernel<NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, VCfg<NT>::BYTES);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(prm.grid), dim3(VCfg<NT>::THREADS), VCfg<NT>::BYTES, st, mk, mv, prm);
  if (e != cudaSuccess) return e;
  // whether a pair is split between CTAs is known only on the device (the group count)
  return launch_pdl(attn_verify_merge_kernel<NT>, dim3(prm.grid), dim3(kVMergeThreads), 0, st, prm);
}

}  // namespace

bool verify_supported(int D_, int G, int window, bool fp8, const void* k, const void* v,
                      int max_keys, int T, int max_q_per_seq) {
  if (D_ != D || G < 1 || G > kHeads || window != 0 || fp8 || max_keys < kMinKeys) return false;
  if (T < 1 || T > kVerifyMaxT || max_q_per_seq < 2) return false;
  return aligned16(k) && aligned16(v) && tensor_map_encoder_ready();
}

size_t verify_ws_bytes(int T, int G, int max_q_per_seq) {
  if (T <= 0 || G < 1 || G > kHeads) return 0;
  return verify_ws_for(T, verify_nt(G, verify_tg(G, max_q_per_seq)));
}

size_t verify_ws_bytes_max(int T) {
  return T > 0 && T <= kVerifyMaxT ? verify_ws_for(T, kVerifyMaxNT) : 0;
}

cudaError_t verify(const uint16_t* q, const uint16_t* g, const uint16_t* gate_bias,
                   const int32_t* seq_id, const int32_t* pos, int T, int max_pos,
                   int max_q_per_seq, int n_q, int n_kv, const beam_kv_cache& kc, float sl2,
                   uint16_t* og, void* ws, size_t ws_len, cudaStream_t st) {
  const int G = n_q / n_kv;
  const int TG = verify_tg(G, max_q_per_seq), nt = verify_nt(G, TG);
  if (nt == 0 || ws_len < verify_ws_for(T, nt)) return cudaErrorInvalidValue;
  const int grid = num_sms_cached();
  const size_t parts = size_t(grid) * 2 * nt * 8;
  char* w = static_cast<char*>(ws);
  float* part_acc = reinterpret_cast<float*>(w);
  float* part_ml = reinterpret_cast<float*>(w + align_up(parts * D * 4, 256));
  int* groups = reinterpret_cast<int*>(w + align_up(parts * D * 4, 256) + align_up(parts * 2 * 4, 256));
  CUtensorMap mk, mv;
  if (!encode_kv_maps(kc, n_kv, false, &mk, &mv)) return cudaErrorInvalidValue;
  const int NB = (max_pos + VCfg<2>::BK - 1) / VCfg<2>::BK;
  const VParams prm{q,  seq_id, pos, g,    gate_bias,   og,          part_acc, part_ml, groups,
                    T,  TG,     n_q, n_kv, G,           kc.num_seqs, kc.capacity, NB,   grid,
                    sl2};
  switch (nt) {
    case 2: return launch_verify<2>(mk, mv, prm, st);
    case 3: return launch_verify<3>(mk, mv, prm, st);
    case 4: return launch_verify<4>(mk, mv, prm, st);
    case 6: return launch_verify<6>(mk, mv, prm, st);
    default: return launch_verify<12>(mk, mv, prm, st);
  }
}

}  // namespace adec
}  // namespace beam
