// BF16 tensor-core GEMM for the prefill projections: C[M][N] = A[M][K] . B[N][K]^T, FP32
// accumulation in tensor memory, written as FP32 or BF16.
//
// Blackwell (sm_103a) structure: a persistent grid (at most one CTA per SM) walks the 128 x 256
// output tiles; a 4-stage shared-memory ring of 64-wide K slices filled by TMA (128-byte
// swizzle, no multicast) runs on across tiles, consumed by tcgen05.mma issued from one thread
// into one of two 128 x 256 FP32 accumulators in TMEM; four epilogue warps read a finished
// accumulator back with tcgen05.ld and store it while the next tile accumulates into the
// other. Warp roles:
//   warp 0 : TMA producer (one elected lane)
//   warp 1 : TMEM allocation owner and MMA issuer (one elected lane)
//   warps 2-5 : epilogue (warp w reads TMEM lanes 32*(w%4) .. +31, i.e. output rows)
// Every mbarrier wait is bounded; on expiry the CTA records BEAM_DEV_TIMEOUT in the status
// word, lets its in-flight copies land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "mma.cuh"
#include "tcgen05.cuh"

namespace beam {
namespace tc {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;   // ring, alignment, barriers
constexpr int THREADS = 192;
constexpr int kGroupM = 16;   // row tiles walked per column tile (dense grids)
constexpr uint32_t kIdesc = idesc_bf16(BM, BN, false);

// One CTA computes output columns [n0, n0 + BN) (kSwiGLU: units [n0, n0 + BN/2)) for A rows
// [a_row0, a_row0 + rows). Dense GEMMs map a 1-D grid onto (row tile, column tile) in groups
// of kGroupM row tiles; grouped GEMMs read (group, a_row0, rows) from a device-side job list
// (one job per expert row tile), blockIdx.y = job, blockIdx.x = column tile.
struct GemmParams {
  int M, N, K;           // A rows (bound), output columns (units for kSwiGLU), reduction
  void* C;
  int ldc;
  const int4* jobs;      // grouped: {group, a_row0, rows, group's first job | its jobs << 20};
                         // nullptr for a dense GEMM
  const int* n_jobs;     // grouped: number of valid jobs (device)
  int b_stride;          // grouped: B rows per group (b_row0 = group * b_stride)
  int up_off;            // kSwiGLU: B row offset of the up half from the gate half
  const int* row_map;    // optional: C row of A row r is row_map[r]
  const float* group_scale;   // grouped, optional: the accumulator of group g is multiplied by
                              // group_scale[g] before the epilogue (per-matrix weight scales)
  int a_k;               // A columns when the reduction runs over A twice (K = 2 a_k: B rows
                         // hold two parts of the weights, e.g. BF16 high and low); else 0
};

// The QKV epilogue for one token row and one 128-column head of the tile (kQKV mode).
__device__ __forceinline__ void qkv_head_epilogue(const QkvEpilogue& e, uint32_t taddr, int t,
                                                  bool tok_ok, int head, int p, int s,
                                                  bool kv_ok, float ssmax) {
  constexpr int QD = 128;
  float v[QD];
#pragma unroll
  for (int c = 0; c < QD / 16; ++c) {
    uint32_t r[16];
    tmem_ld16(taddr + uint32_t(c * 16), r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[c * 16 + i] = __uint_as_float(r[i]);
  }
  if (!tok_ok) return;
  const int nq = e.n_q, nkv = e.n_kv;
  const int kind = head < nq ? 0 : head < nq + nkv ? 1 : head < nq + 2 * nkv ? 2 : 3;
#pragma unroll
  for (int i = 0; i < QD; ++i) v[i] = round_bf(v[i]);   // the projection's bf16 output
  if (kind <= 1) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < QD; ++i) ss = fmaf(v[i], v[i], ss);
    const float rn = rsqrtf(ss / float(QD) + e.eps);
    const uint16_t* gw = kind == 0 ? e.q_norm : e.k_norm;
#pragma unroll
    for (int i = 0; i < QD; ++i) v[i] = v[i] * rn * bf2f(gw[i]);
    if (!e.nope) {
      const float2* cs = e.rope + size_t(t) * (QD / 2);
#pragma unroll
      for (int i = 0; i < QD / 2; ++i) {
        const float2 c = cs[i];
        const float a = v[i], b = v[i + QD / 2];
        v[i] = a * c.x - b * c.y;
        v[i + QD / 2] = b * c.x + a * c.y;
      }
    } else if (kind == 0) {
#pragma unroll
      for (int i = 0; i < QD; ++i) v[i] *= ssmax;
    }
  }
  if (kind == 0 || kind == 3) {
    uint16_t* dst = kind == 0 ? e.q_out + (size_t(t) * nq + head) * QD
                              : e.g_out + size_t(t) * nq * QD + size_t(head - nq - 2 * nkv) * QD;
#pragma unroll
    for (int i = 0; i < QD; i += 8)
      *reinterpret_cast<uint4*>(dst + i) =
          make_uint4(pack_bf2(v[i], v[i + 1]), pack_bf2(v[i + 2], v[i + 3]),
                     pack_bf2(v[i + 4], v[i + 5]), pack_bf2(v[i + 6], v[i + 7]));
    return;
  }
  if (!kv_ok) return;
  const beam_kv_cache& kc = e.cache;
  const int kvh = kind == 1 ? head - nq : head - nq - nkv;
  const int slot = (p - 1) % kc.capacity;
  const size_t base = ((size_t(s) * nkv + kvh) * kc.capacity + slot) * QD;
  if (kc.dtype == BEAM_KV_BF16) {
    uint16_t* dst = static_cast<uint16_t*>(kind == 1 ? kc.k : kc.v) + base;
#pragma unroll
    for (int i = 0; i < QD; i += 8)
      *reinterpret_cast<uint4*>(dst + i) =
          make_uint4(pack_bf2(v[i], v[i + 1]), pack_bf2(v[i + 2], v[i + 3]),
                     pack_bf2(v[i + 4], v[i + 5]), pack_bf2(v[i + 6], v[i + 7]));
  } else {
    uint8_t* dst = static_cast<uint8_t*>(kind == 1 ? kc.k : kc.v) + base;
    const float sc = kind == 1 ? kc.k_scale : kc.v_scale;
#pragma unroll
    for (int i = 0; i < QD; ++i)
      dst[i] = __nv_cvt_float_to_fp8(__fdiv_rn(v[i], sc), __NV_SATFINITE, __NV_E4M3);
  }
}

// Output tile t of a launch: A rows [a_row0, a_row0 + rows), B rows from b_row0, output
// columns [n0, n0 + NT). Dense GEMMs walk (row tile, column tile) in groups of kGroupM row
// tiles per column tile: the tiles the resident CTAs hold at one time cover a compact block of
// the output, so both operands' tiles are reused through L2. Grouped GEMMs walk each group's
// (expert's) tiles column by column, its jobs fastest (tile_of).
struct Tile {
  int a_row0, b_row0, rows, n0, group;
};
template <int NT>
__device__ __forceinline__ Tile tile_of(const GemmParams& p, int t, int num_m, int num_n) {
  Tile r;
  if (p.jobs == nullptr) {
    const int group = t / (kGroupM * num_n);
    const int first_m = group * kGroupM;
    const int gsize = min(num_m - first_m, kGroupM);
    const int in_group = t - group * kGroupM * num_n;
    r.a_row0 = (first_m + in_group % gsize) * BM;
    r.n0 = (in_group / gsize) * NT;
    r.b_row0 = 0;
    r.rows = BM;
    r.group = 0;
  } else {
    // An expert's tiles occupy one contiguous range of t; inside it the tiles go column by
    // column, the expert's row tiles (jobs) fastest, so the CTAs that share a column of the
    // expert's weights run side by side and read it from L2 once (job-major order split an
    // expert's columns across waves of the persistent grid: 1.39x the weight bytes from DRAM).
    int jb = t / num_n, col = t - jb * num_n;
    const int w = p.jobs[jb].w;
    const int je0 = w & 0xFFFFF, nje = w >> 20;
    if (nje > 0) {
      const int local = t - je0 * num_n;
      col = local / nje;
      jb = je0 + (local - col * nje);
    }
    const int4 j = p.jobs[jb];
    r.n0 = col * NT;
    r.b_row0 = j.x * p.b_stride;
    r.group = j.x;
    r.a_row0 = j.y;
    r.rows = j.z;
  }
  return r;
}

// Persistent: CTA c takes tiles c, c + gridDim.x, ... Two 256-column FP32 accumulators in
// TMEM (512 columns) let the epilogue of tile i run while the MMAs of tile i+1 accumulate into
// the other buffer, and the TMA ring runs on across tile boundaries, so neither the epilogue
// nor the pipeline fill of a tile leaves the tensor pipe idle.
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                   GemmParams p, QkvEpilogue qe) {
  pdl_trigger();
  pdl_wait();
  constexpr int NT = MODE == kSwiGLU ? BN / 2 : BN;   // output columns per tile
  const int num_n = (p.N + NT - 1) / NT;
  const int num_m = (p.M + BM - 1) / BM;
  const int n_tiles = p.jobs == nullptr ? num_m * num_n : *p.n_jobs * num_n;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  const uint32_t s_base = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
  const uint32_t accf0 = smem_u32(bars + 2 * STAGES), acce0 = accf0 + 16;   // [2] each
  const uint32_t mma_done = acce0 + 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf0 + 8 * a, 1);
      mbar_init(acce0 + 8 * a, 4);   // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;   // k-blocks issued, over all tiles of this CTA
      for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x) {
        const Tile tl = tile_of<NT>(p, t, num_m, num_n);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          // the abort flag is read per tile, not per k-block: under a busy tensor pipe a
          // shared-memory load takes ~130 cycles (a role that gave up stops arriving, so this
          // wait then expires)
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1)) {
            *abort_flag = 1;
            break;
          }
          mbar_expect_tx(full0 + 8 * s, STAGE_BYTES);
          const uint32_t sa = s_base + s * STAGE_BYTES;
          tma_load_2d(sa, &ta, p.a_k > 0 && kb * BK >= p.a_k ? kb * BK - p.a_k : kb * BK,
                      tl.a_row0, full0 + 8 * s);
          if (MODE == kSwiGLU) {
            tma_load_2d(sa + A_BYTES, &tb, kb * BK, tl.b_row0 + tl.n0, full0 + 8 * s);
            tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tb, kb * BK, tl.b_row0 + p.up_off + tl.n0,
                        full0 + 8 * s);
          } else {
            tma_load_2d(sa + A_BYTES, &tb, kb * BK, tl.b_row0 + tl.n0, full0 + 8 * s);
          }
        }
      }
      // normally a no-op (every issued stage was consumed); after an expired wait, let the
      // copies already issued land before the CTA's shared memory goes away
      for (int k = it - 1; k >= 0 && k >= it - STAGES; --k)
        mbar_wait(full0 + 8 * (k % STAGES), (k / STAGES) & 1);
    }
  } else if (warp == 1) {
    {
      // the whole warp runs the issue loop on warp-uniform values and elect.sync picks the
      // lane that issues each MMA and commit (lane 0: the warp stays converged)
      // descriptor of the ring's first byte: A and B tiles of every stage differ from it only
      // in the start address field (shared-memory offsets >> 4 stay below 2^14)
      const uint64_t d0 = smem_desc(s_base);
      const uint32_t d_lo0 = uint32_t(d0), d_hi = uint32_t(d0 >> 32);
      int it = 0, i = 0;
      for (int t = blockIdx.x; t < n_tiles && !*abort_flag; t += gridDim.x, ++i) {
        const int ab = i & 1;
        // the epilogue has drained this accumulator (tile i - 2)
        if (!__all_sync(0xffffffffu, mbar_wait(acce0 + 8 * ab, ((i >> 1) & 1) ^ 1))) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t acc = tmem + uint32_t(ab * BN);
        bool ok = true;
        // The tensor pipe queues only ~3 MMAs (~350 cycles of work at this shape): the issue
        // path per k-block is one barrier poll, the descriptors stepped in their low word (the
        // start address field) and the four MMAs.
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, ph))) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t alo = d_lo0 + uint32_t((s * STAGE_BYTES) >> 4);
          const uint32_t blo = alo + uint32_t(A_BYTES >> 4);
          umma_ss_e(acc, alo, d_hi, blo, d_hi, kIdesc, kb != 0 ? 1u : 0u);
#pragma unroll
          for (int k = 1; k < BK / 16; ++k)
            umma_ss_e(acc, alo + uint32_t((32 * k) >> 4), d_hi, blo + uint32_t((32 * k) >> 4), d_hi,
                      kIdesc, 1u);
          umma_commit_e(empty0 + 8 * s);
        }
        umma_commit_e(accf0 + 8 * ab);   // arrives once every MMA issued above has completed
        if (!ok) {
          if (lane == 0) *abort_flag = 1;
          break;
        }
      }
      // every MMA of this CTA has completed before TMEM is released (after an early exit the
      // epilogue may not have waited for them)
      umma_commit_e(mma_done);
      mbar_wait(mma_done, 0);
    }
  } else {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
      const int ab = i & 1;
      const bool ok = !*abort_flag && mbar_wait(accf0 + 8 * ab, (i >> 1) & 1);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // tcgen05.ld is warp-collective: the decision is taken once for the whole warp
      if (!__all_sync(0xffffffffu, ok)) {
        *abort_flag = 1;
        break;
      }
      const Tile tl = tile_of<NT>(p, t, num_m, num_n);
      const int arow = tl.a_row0 + r;
      const bool row_ok = r < tl.rows && arow < p.M;
      const int crow = row_ok ? (p.row_map ? p.row_map[arow] : arow) : 0;
      const int n0 = tl.n0;
      const float gsc = p.group_scale != nullptr ? p.group_scale[tl.group] : 1.f;
      const uint32_t tbase = tmem + uint32_t(ab * BN) + (uint32_t(quad * 32) << 16);
      if (MODE == kQKV) {
        // per token row: two 128-column heads of the packed projection
        int pp = 0, sq = 0;
        bool kv_ok = false;
        float ssmax = 1.f;
        if (row_ok) {
          pp = qe.pos[arow];
          sq = qe.seq_id[arow];
          const beam_kv_cache& kc = qe.cache;
          const bool bad_p = pp < 1 || (kc.window == 0 && pp > kc.capacity);
          const bool bad_s = sq < 0 || sq >= kc.num_seqs;
          if (n0 == 0 && bad_p) flag(BEAM_DEV_BAD_POSITION);
          if (n0 == 0 && bad_s) flag(BEAM_DEV_BAD_SEQ);
          kv_ok = !bad_p && !bad_s;
          if (qe.nope) ssmax = ssmax_scale(pp, qe.ss_base, qe.ss_exp);
        }
#pragma unroll 1
        for (int hh = 0; hh < BN / 128; ++hh) {
          const int head = n0 / 128 + hh;
          if (head * 128 >= p.N) break;   // uniform over the CTA
          qkv_head_epilogue(qe, tbase + uint32_t(hh * 128), arow, row_ok, head, pp, sq, kv_ok,
                            ssmax);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < NT / 16; ++c) {
          uint32_t v[16];
          tmem_ld16(tbase + uint32_t(c * 16), v);
          const int col = n0 + c * 16;
          if (MODE == kSwiGLU) {
            uint32_t up[16];
            tmem_ld16(tbase + uint32_t(BN / 2 + c * 16), up);
            if (row_ok && col < p.N) {
              uint16_t* dst = static_cast<uint16_t*>(p.C) + size_t(crow) * p.ldc + col;
              float a[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                a[e] = siluf_(__uint_as_float(v[e]) * gsc) * (__uint_as_float(up[e]) * gsc);
              if (col + 16 <= p.N && (p.ldc & 7) == 0) {
                uint32_t q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) q[e] = pack_bf2(a[2 * e], a[2 * e + 1]);
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(q[0], q[1], q[2], q[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(q[4], q[5], q[6], q[7]);
              } else {
                for (int e = 0; e < 16 && col + e < p.N; ++e) dst[e] = f2bf(a[e]);
              }
            }
          } else if (row_ok && col < p.N) {
            if (p.group_scale != nullptr) {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * gsc);
            }
            if (MODE == kF32 || MODE == kF32Add) {
              float* dst = static_cast<float*>(p.C) + size_t(crow) * p.ldc + col;
              if (col + 16 <= p.N && (p.ldc & 3) == 0) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float4 o = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                         __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                  if (MODE == kF32Add) {
                    const float4 cc = reinterpret_cast<const float4*>(dst)[e];
                    o.x += cc.x;
                    o.y += cc.y;
                    o.z += cc.z;
                    o.w += cc.w;
                  }
                  reinterpret_cast<float4*>(dst)[e] = o;
                }
              } else {
                for (int e = 0; e < 16 && col + e < p.N; ++e)
                  dst[e] = MODE == kF32Add ? dst[e] + __uint_as_float(v[e]) : __uint_as_float(v[e]);
              }
            } else {
              uint16_t* dst = static_cast<uint16_t*>(p.C) + size_t(crow) * p.ldc + col;
              if (col + 16 <= p.N && (p.ldc & 7) == 0) {
                uint32_t q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  q[e] = pack_bf2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(q[0], q[1], q[2], q[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(q[4], q[5], q[6], q[7]);
              } else {
                for (int e = 0; e < 16 && col + e < p.N; ++e) dst[e] = f2bf(__uint_as_float(v[e]));
              }
            }
          }
        }
      }
      // this warp's TMEM reads are done: release the accumulator to the MMA issuer
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * ab);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag(BEAM_DEV_TIMEOUT);
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN)
                 : "memory");
  }
}

// 2-D bf16 map over rows x inner (row stride ld elements), box box_rows x 64, 128 B swizzle.
bool make_map(CUtensorMap* m, const void* base, int inner, int rows, int ld, int box_rows) {
  const uint64_t d[2] = {uint64_t(inner), uint64_t(rows)};
  const uint64_t st[1] = {uint64_t(ld) * 2};
  const uint32_t bx[2] = {uint32_t(BK), uint32_t(box_rows)};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, d, st, bx,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

bool tensor_map_encoder_ready() {
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return true;
}

bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swz) {
  if (!tensor_map_encoder_ready() || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return g_encode(m, dt, cuuint32_t(rank), const_cast<void*>(base), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_supported(const void* A, int lda, const void* B, int ldb, int K) {
  return aligned16(A) && aligned16(B) && (lda % 8) == 0 && (ldb % 8) == 0 && (K % 8) == 0 &&
         K > 0;
}

namespace {

// tiles: the number of output tiles (an upper bound for grouped GEMMs); one CTA per SM at most
template <int MODE>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int tiles,
                   cudaStream_t st, const QkvEpilogue& qe = QkvEpilogue{}) {
  const int sms = num_sms_cached();
  const dim3 grid(tiles < sms ? tiles : sms);
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  launch_pdl(gemm_tc_kernel<MODE>, grid, dim3(THREADS), SMEM_BYTES, st, ta, tb, p, qe);
  return cudaGetLastError();
}

}  // namespace

cudaError_t gemm_bf16(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int N, int ldb,
                      void* C, int ldc, bool out_bf16, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (!gemm_supported(A, lda, B, ldb, K)) return cudaErrorInvalidValue;
  if (!tensor_map_encoder_ready()) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, K, M, lda, BM) || !make_map(&tb, B, K, N, ldb, BN))
    return cudaErrorInvalidValue;
  GemmParams p{M, N, K, C, ldc, nullptr, nullptr, 0, 0, nullptr};
  const int tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
  return out_bf16 ? launch<kBF16>(ta, tb, p, tiles, st) : launch<kF32>(ta, tb, p, tiles, st);
}

cudaError_t gemm_f32_acc(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int N,
                         int ldb, float* C, int ldc, bool accumulate, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (!gemm_supported(A, lda, B, ldb, K)) return cudaErrorInvalidValue;
  if (!tensor_map_encoder_ready()) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, K, M, lda, BM) || !make_map(&tb, B, K, N, ldb, BN))
    return cudaErrorInvalidValue;
  GemmParams p{M, N, K, C, ldc, nullptr, nullptr, 0, 0, nullptr};
  const int tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
  return accumulate ? launch<kF32Add>(ta, tb, p, tiles, st) : launch<kF32>(ta, tb, p, tiles, st);
}

cudaError_t gemm_qkv(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int N, int ldb,
                     const QkvEpilogue& qe, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (!gemm_supported(A, lda, B, ldb, K) || N % 128 != 0) return cudaErrorInvalidValue;
  if (!tensor_map_encoder_ready()) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, K, M, lda, BM) || !make_map(&tb, B, K, N, ldb, BN))
    return cudaErrorInvalidValue;
  GemmParams p{M, N, K, nullptr, 0, nullptr, nullptr, 0, 0, nullptr};
  const int tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
  return launch<kQKV>(ta, tb, p, tiles, st, qe);
}

cudaError_t gemm_swiglu(const uint16_t* A, int M, int K, int lda, const uint16_t* B, int F,
                        int ldb, uint16_t* C, int ldc, cudaStream_t st) {
  if (M <= 0 || F <= 0) return cudaSuccess;
  if (!gemm_supported(A, lda, B, ldb, K)) return cudaErrorInvalidValue;
  if (!tensor_map_encoder_ready()) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, K, M, lda, BM) || !make_map(&tb, B, K, 2 * F, ldb, BN / 2))
    return cudaErrorInvalidValue;
  GemmParams p{M, F, K, C, ldc, nullptr, nullptr, 0, F, nullptr};
  const int tiles = ((F + BN / 2 - 1) / (BN / 2)) * ((M + BM - 1) / BM);
  return launch<kSwiGLU>(ta, tb, p, tiles, st);
}

cudaError_t gemm_grouped(int mode, const uint16_t* A, int M, int K, int lda, const uint16_t* B,
                         int b_rows, int b_stride, int ldb, const int4* jobs, const int* n_jobs,
                         int max_jobs, int N, int up_off, const int* row_map, void* C, int ldc,
                         cudaStream_t st, const float* group_scale, bool a_twice) {
  if (M <= 0 || N <= 0 || max_jobs <= 0) return cudaSuccess;
  // a_twice: B rows are [part 0 | part 1] of K/2 columns each, both multiplied by A's K/2
  const int a_k = a_twice ? K / 2 : 0;
  if (a_twice && (K % (2 * BK)) != 0) return cudaErrorInvalidValue;
  if (!gemm_supported(A, lda, B, ldb, K)) return cudaErrorInvalidValue;
  if (!tensor_map_encoder_ready()) return cudaErrorNotSupported;
  CUtensorMap ta, tb;
  const int bbox = mode == kSwiGLU ? BN / 2 : BN;
  if (!make_map(&ta, A, a_twice ? a_k : K, M, lda, BM) || !make_map(&tb, B, K, b_rows, ldb, bbox))
    return cudaErrorInvalidValue;
  GemmParams p{M, N, K, C, ldc, jobs, n_jobs, b_stride, up_off, row_map, group_scale, a_k};
  const int nt = mode == kSwiGLU ? BN / 2 : BN;
  const int tiles = ((N + nt - 1) / nt) * max_jobs;
  if (mode == kSwiGLU) return launch<kSwiGLU>(ta, tb, p, tiles, st);
  if (mode == kBF16) return launch<kBF16>(ta, tb, p, tiles, st);
  return launch<kF32>(ta, tb, p, tiles, st);
}

}  // namespace tc
}  // namespace beam

extern "C" beam_status beam_gemm_bf16(const beam_bf16* A, int M, int K, int lda,
                                      const beam_bf16* B, int N, int ldb, void* C, int ldc,
                                      int out_bf16, beam_stream_t stream) {
  using namespace beam;
  if (!A || !B || !C || M < 1 || N < 1 || K < 1 || ldc < N || lda < K || ldb < K)
    return BEAM_ERR_INVALID_ARG;
  if (!tc::gemm_supported(A, lda, B, ldb, K)) return BEAM_ERR_INVALID_ARG;
  const cudaError_t e = tc::gemm_bf16(A, M, K, lda, B, N, ldb, C, ldc, out_bf16 != 0,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BEAM_OK : BEAM_ERR_CUDA;
}
