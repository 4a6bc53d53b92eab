// GQA attention over the KV cache, sigmoid output gate, o_proj.
// Beam page, Attention section: 48 query heads share 8 KV heads (dim 128); sliding-window
// layers attend to the last 512 keys, NoPE layers to the whole context; each head's output is
// multiplied by sigmoid(gate + per-head bias) before o_proj. Change 2 of the optimisation list
// keeps the gate as its own step; here it is fused into the attention epilogue.
//
// Decode (few tokens): split-K flash decoding. A CTA takes one (token, KV head, key range);
// the G query heads of the KV group form the rows of a 16-row tensor-core tile, so every K/V
// byte read from HBM serves all G heads. Each of the 4 warps streams its own 32-key tiles
// through a 2-stage cp.async pipeline. With at most 8 splits the split CTAs of a (token, KV
// head) form one thread-block cluster and merge their partial (max, sum, P.V) through
// distributed shared memory, each CTA finishing a slice of the outputs; with more splits the
// partials go to the workspace and the last split CTA to finish merges them. The merge
// normalises, applies the output gate and writes o.
// Prefill (many tokens): a CTA takes 16 consecutive tokens and one KV group; warp w computes
// query head w of the group for those 16 tokens, all warps sharing each staged K/V tile.
//
// P is split into bf16 hi + lo parts for the P.V product, so P carries ~16 significant bits;
// the logits Q.K^T are exact products of bf16 inputs accumulated in FP32.
#include <cooperative_groups.h>
#include <math.h>

#include "attn_dec.cuh"
#include "attn_tc.cuh"
#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"
#include "mma.cuh"

namespace beam {
namespace {

constexpr float kNegInf = -INFINITY;
constexpr int kDecWarps = 4;
// Keys per warp tile (decode): 32 when 2-8 split CTAs of a (token, KV head) form a cluster;
// 16 with a single split or with many splits merged through the workspace, which fits two
// CTAs on an SM -- twice the tiles in flight (measured: NoPE batch 1 at 100K keys 180 -> 124
// us, batch-128 stack layer 1350 -> 1140 us; clusters of 5 at batch 8 were 7% faster at 32).
constexpr int kDecKTCluster = 32, kDecKTSplit = 16;
// cp.async stages per warp with 16-key tiles: three keep two CTAs on an SM with two tiles in
// flight per warp
constexpr int kDecStagesSplit = 3;
constexpr int kPreKT = 64;   // keys per CTA tile (prefill)
constexpr int kRows = 16;    // tensor-core tile rows

template <int D, bool FP8, int KT>
struct TileGeom {
  static constexpr int ROWB = D * 2;          // bf16 row bytes
  static constexpr int RAWROW = FP8 ? D : D * 2;
  static constexpr int RAWCH = RAWROW / 16;   // 16-byte chunks per stored row
  static constexpr int TILEB = KT * ROWB;     // one bf16 tile
  static constexpr int RAWB = KT * RAWROW;    // one stored tile
  // 2 stages of raw K and V, plus (fp8 only) one converted K and V tile
  static constexpr int BYTES = 4 * RAWB + (FP8 ? 2 * TILEB : 0);
};

// Issue the copies of `rows` keys starting at cache slot chain s0 (slot of row r is
// (s0 + r) mod cap) into raw tile `dst`; rows >= nvalid are zero-filled. Threads
// [tid0, tid0 + nthr) share the work. bf16 tiles are stored swizzled, fp8 tiles plainly.
template <int D, bool FP8, int KT>
__device__ __forceinline__ void issue_tile(uint8_t* dst, const uint8_t* src_base, int s0, int cap,
                                           int nvalid, int tid, int nthr) {
  using Gm = TileGeom<D, FP8, KT>;
  const uint32_t d0 = smem_u32(dst);
  for (int q = tid; q < KT * Gm::RAWCH; q += nthr) {
    const int r = q / Gm::RAWCH, ch = q - r * Gm::RAWCH;
    int sl = s0 + r;
    while (sl >= cap) sl -= cap;
    const bool ok = r < nvalid;
    const uint8_t* src = src_base + (ok ? size_t(sl) * Gm::RAWROW + ch * 16 : 0);
    const uint32_t off = FP8 ? uint32_t(r * Gm::RAWROW + ch * 16) : swz(r, ch, Gm::ROWB);
    cp_async16(d0 + off, src, ok ? 16 : 0);
  }
}

// fp8 raw tile -> swizzled bf16 tile (exact conversion).
template <int D, int KT>
__device__ __forceinline__ void convert_tile(const uint8_t* raw, uint8_t* out, int tid, int nthr) {
  using Gm = TileGeom<D, true, KT>;
  for (int q = tid; q < KT * Gm::RAWCH; q += nthr) {
    const int r = q / Gm::RAWCH, c16 = q - r * Gm::RAWCH;
    const uint4 v = *reinterpret_cast<const uint4*>(raw + r * Gm::RAWROW + c16 * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = e4m3x2_to_bf16x2(uint16_t(w[i] & 0xFFFF));
      o[2 * i + 1] = e4m3x2_to_bf16x2(uint16_t(w[i] >> 16));
    }
    *reinterpret_cast<uint4*>(out + swz(r, 2 * c16, Gm::ROWB)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(out + swz(r, 2 * c16 + 1, Gm::ROWB)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// S[16 x KT] = Q (fragments qa) . K_tile^T
template <int D, int KT>
__device__ __forceinline__ void qk_tile(const uint32_t (&qa)[D / 16][4], const uint8_t* ktile,
                                        float (&s)[KT / 8][4]) {
  constexpr int ROWB = D * 2;
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3, rr = lane & 7;
  const uint32_t base = smem_u32(ktile);
#pragma unroll
  for (int j = 0; j < KT / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int nb = 0; nb < KT / 16; ++nb) {
      const int row = nb * 16 + ((mi >> 1) << 3) + rr;
      const int ch = 2 * kk + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(base + swz(row, ch, ROWB), b0, b1, b2, b3);
      mma_bf16(s[2 * nb], qa[kk], b0, b1);
      mma_bf16(s[2 * nb + 1], qa[kk], b2, b3);
    }
  }
}

// acc[16 x D] += P[16 x KT] . V_tile; P given as C fragments p (already exponentiated).
template <int D, int KT, bool SPLITP>
__device__ __forceinline__ void pv_tile(const float (&p)[KT / 8][4], const uint8_t* vtile,
                                        float (&acc)[D / 8][4]) {
  constexpr int ROWB = D * 2;
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3, rr = lane & 7;
  const uint32_t base = smem_u32(vtile);
#pragma unroll
  for (int ks = 0; ks < KT / 16; ++ks) {
    uint32_t hi[4], lo[4];
    const float* p0 = p[2 * ks];
    const float* p1 = p[2 * ks + 1];
    hi[0] = pack_bf16x2(p0[0], p0[1]);
    hi[1] = pack_bf16x2(p0[2], p0[3]);
    hi[2] = pack_bf16x2(p1[0], p1[1]);
    hi[3] = pack_bf16x2(p1[2], p1[3]);
    if (SPLITP) {
      lo[0] = pack_bf16x2(p0[0] - bf_lo(hi[0]), p0[1] - bf_hi(hi[0]));
      lo[1] = pack_bf16x2(p0[2] - bf_lo(hi[1]), p0[3] - bf_hi(hi[1]));
      lo[2] = pack_bf16x2(p1[0] - bf_lo(hi[2]), p1[1] - bf_hi(hi[2]));
      lo[3] = pack_bf16x2(p1[2] - bf_lo(hi[3]), p1[3] - bf_hi(hi[3]));
    }
#pragma unroll
    for (int db = 0; db < D / 16; ++db) {
      const int row = ks * 16 + ((mi & 1) << 3) + rr;
      const int ch = 2 * db + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(base + swz(row, ch, ROWB), b0, b1, b2, b3);
      mma_bf16(acc[2 * db], hi, b0, b1);
      mma_bf16(acc[2 * db + 1], hi, b2, b3);
      if (SPLITP) {
        mma_bf16(acc[2 * db], lo, b0, b1);
        mma_bf16(acc[2 * db + 1], lo, b2, b3);
      }
    }
  }
}

// Online-softmax update of one tile. s holds raw logits; keys whose `valid` bit is clear
// are masked. On return s holds P = exp2(s * sl2 - m).
template <int KT, int DN>
__device__ __forceinline__ void softmax_update(float (&s)[KT / 8][4], const bool (&valid)[KT / 8][4],
                                               float sl2, float (&m)[2], float (&l)[2],
                                               float (&acc)[DN][4]) {
  float mx[2] = {kNegInf, kNegInf};
#pragma unroll
  for (int j = 0; j < KT / 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = valid[j][e] ? s[j][e] * sl2 : kNegInf;
      s[j][e] = x;
      mx[e >> 1] = fmaxf(mx[e >> 1], x);
    }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
    const float mnew = fmaxf(m[h], mx[h]);
    const float corr = (mnew == kNegInf) ? 1.f : exp2f(m[h] - mnew);
    m[h] = mnew;
    l[h] *= corr;
#pragma unroll
    for (int n = 0; n < DN; ++n) {
      acc[n][2 * h] *= corr;
      acc[n][2 * h + 1] *= corr;
    }
  }
#pragma unroll
  for (int j = 0; j < KT / 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float mm = m[e >> 1];
      const float pv = (s[j][e] == kNegInf) ? 0.f : exp2f(s[j][e] - mm);
      s[j][e] = pv;
      l[e >> 1] += pv;
    }
}

// Query fragments of 16 rows; row r is query head (head0 + r*hstride) of token (tok0 + r*tstride),
// rows with r >= nrows are zero.
template <int D>
__device__ __forceinline__ void load_q(const uint16_t* q, uint32_t (&qa)[D / 16][4],
                                       const int (&rowoff)[2], const bool (&rowok)[2]) {
  const int lane = threadIdx.x & 31;
  const int c = lane & 3;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(q + rowoff[h] + kk * 16 + 2 * c);
      qa[kk][h] = rowok[h] ? src[0] : 0u;       // a0 / a1: cols 2c..2c+1
      qa[kk][h + 2] = rowok[h] ? src[4] : 0u;   // a2 / a3: cols 2c+8..
    }
  }
}

// Merge the splits of one (token, KV head), normalise, round, gate, round. Run by the last
// split CTA of the pair to finish; the partials of the other CTAs are read through L2. The
// per-split (max, sum) pairs are staged in shared memory first, so each output element then
// needs one pass of independent loads over the splits.
constexpr int kMergeMaxSplits = 64;
__device__ __forceinline__ void merge_gate(const float* part_acc, const float* part_ml,
                                           int n_splits, int n_q, int n_kv, int D, float v_scale,
                                           const uint16_t* __restrict__ gpre,
                                           const uint16_t* __restrict__ gate_bias,
                                           uint16_t* __restrict__ og, int t, int hk, float* sh) {
  const int G = n_q / n_kv;
  const size_t pbase = (size_t(t) * n_kv + hk) * n_splits;
  float* w = sh;                              // [kRows][n_splits]: exp2(m_s - M)
  float* inv = sh + kRows * kMergeMaxSplits;  // [kRows]: 1 / sum_s w_s l_s
  for (int i = threadIdx.x; i < G * n_splits; i += blockDim.x) {
    const int row = i / n_splits, sp = i - row * n_splits;
    w[row * kMergeMaxSplits + sp] = __ldcg(part_ml + ((pbase + sp) * kRows + row) * 2);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int row = threadIdx.x;
    float M = kNegInf;
    for (int sp = 0; sp < n_splits; ++sp) M = fmaxf(M, w[row * kMergeMaxSplits + sp]);
    float L = 0.f;
    for (int sp = 0; sp < n_splits; ++sp) {
      const float f = M == kNegInf ? 0.f : exp2f(w[row * kMergeMaxSplits + sp] - M);
      w[row * kMergeMaxSplits + sp] = f;
      L += f * __ldcg(part_ml + ((pbase + sp) * kRows + row) * 2 + 1);
    }
    inv[row] = L > 0.f ? v_scale / L : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int row = idx / D, d = idx - row * D;
    float O = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < n_splits; ++sp)
      O += w[row * kMergeMaxSplits + sp] * __ldcg(part_acc + ((pbase + sp) * kRows + row) * D + d);
    const float o = round_bf(O * inv[row]);
    const int hq = hk * G + row;
    const size_t oi = (size_t(t) * n_q + hq) * D + d;
    const float gate = sigmoidf_(bf2f(gpre[oi]) + bf2f(gate_bias[hq]));
    og[oi] = f2bf(o * gate);
  }
}

// Row `row`, column d of the CTA's 4 warp partials: the common max M, the rescaled P.V sum O
// and the rescaled softmax denominator L.
__device__ __forceinline__ void combine_warps(const float* sacc_all, const float* sml, int ld,
                                              int row, int d, float& M, float& O, float& L) {
  M = kNegInf;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sml[(w * kRows + row) * 2]);
  O = 0.f;
  L = 0.f;
  if (M != kNegInf) {
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float f = exp2f(sml[(w * kRows + row) * 2] - M);
      O += f * sacc_all[(w * kRows + row) * ld + d];
      L += f * sml[(w * kRows + row) * 2 + 1];
    }
  }
}

// The cluster form of merge_gate: split s's partial lives in the shared memory of cluster CTA
// s; CTA `rank` finishes outputs [rank * chunk, (rank + 1) * chunk) of the G x D block.
constexpr int kClusterMaxSplits = 8;
__device__ __forceinline__ void merge_gate_cluster(
    cooperative_groups::cluster_group& cl, float* cO, float* cML, int n_splits, int n_q,
    int n_kv, int D, float v_scale, const uint16_t* __restrict__ gpre,
    const uint16_t* __restrict__ gate_bias, uint16_t* __restrict__ og, int t, int hk, float* sh) {
  const int G = n_q / n_kv;
  float* w = sh;                                // [kRows][kClusterMaxSplits]: exp2(m_s - M)
  float* inv = sh + kRows * kClusterMaxSplits;  // [kRows]
  const float* peerO[kClusterMaxSplits];
  const float* peerML[kClusterMaxSplits];
#pragma unroll
  for (int sp = 0; sp < kClusterMaxSplits; ++sp) {
    const int r = sp < n_splits ? sp : 0;
    peerO[sp] = cl.map_shared_rank(cO, r);
    peerML[sp] = cl.map_shared_rank(cML, r);
  }
  if (threadIdx.x < G) {
    const int row = threadIdx.x;
    float m[kClusterMaxSplits], l[kClusterMaxSplits];
    float M = kNegInf;
#pragma unroll
    for (int sp = 0; sp < kClusterMaxSplits; ++sp) {
      if (sp < n_splits) {
        m[sp] = peerML[sp][row * 2];
        l[sp] = peerML[sp][row * 2 + 1];
        M = fmaxf(M, m[sp]);
      }
    }
    float L = 0.f;
#pragma unroll
    for (int sp = 0; sp < kClusterMaxSplits; ++sp) {
      if (sp < n_splits) {
        const float f = M == kNegInf ? 0.f : exp2f(m[sp] - M);
        w[row * kClusterMaxSplits + sp] = f;
        L += f * l[sp];
      }
    }
    inv[row] = L > 0.f ? v_scale / L : 0.f;
  }
  __syncthreads();
  const int total = G * D;
  const int chunk = (total + n_splits - 1) / n_splits;
  const int i0 = int(cl.block_rank()) * chunk, i1 = min(total, i0 + chunk);
  for (int idx = i0 + threadIdx.x; idx < i1; idx += blockDim.x) {
    const int row = idx / D, d = idx - row * D;
    float O = 0.f;
#pragma unroll
    for (int sp = 0; sp < kClusterMaxSplits; ++sp)
      if (sp < n_splits) O += w[row * kClusterMaxSplits + sp] * peerO[sp][row * D + d];
    const float o = round_bf(O * inv[row]);
    const int hq = hk * G + row;
    const size_t oi = (size_t(t) * n_q + hq) * D + d;
    const float gate = sigmoidf_(bf2f(gpre[oi]) + bf2f(gate_bias[hq]));
    og[oi] = f2bf(o * gate);
  }
}

// Dynamic shared memory of the decode kernel: the 4 warps' tile pipelines, reused for the
// cross-warp combine, then (cluster form) the CTA's partial for its peers.
// Per-warp pipeline of the decode kernel: ST stages of raw K and V tiles, plus (fp8 only) one
// converted K and V tile.
template <int D, bool FP8, int KT, int ST>
__host__ __device__ constexpr int dec_warp_bytes() {
  return 2 * ST * TileGeom<D, FP8, KT>::RAWB + (FP8 ? 2 * TileGeom<D, FP8, KT>::TILEB : 0);
}

template <int D, bool FP8, int KT, int ST>
struct DecodeSmem {
  static constexpr int kTiles = kDecWarps * dec_warp_bytes<D, FP8, KT, ST>();
  static constexpr int kComb = (kDecWarps * kRows * (D + 4) + kDecWarps * kRows * 2) * 4;
  static constexpr int kPartOff = ((kTiles > kComb ? kTiles : kComb) + 127) / 128 * 128;
  static constexpr int kBytes = kPartOff + (kRows * D + kRows * 2) * 4;
};

// ------------------------------------------------------------------------------------------
// Decode: split-K partials
// ------------------------------------------------------------------------------------------
template <int D, bool FP8, bool CLUSTER, int KT, int ST>
__global__ void __launch_bounds__(kDecWarps * 32) attn_decode_split_kernel(
    const uint16_t* __restrict__ q, const int32_t* __restrict__ seq_id,
    const int32_t* __restrict__ pos, int n_q, int n_kv, beam_kv_cache kc, int kps, int n_splits,
    float sl2, float* __restrict__ part_acc, float* __restrict__ part_ml, int* __restrict__ done,
    float v_scale, const uint16_t* __restrict__ gpre, const uint16_t* __restrict__ gate_bias,
    uint16_t* __restrict__ og) {
  pdl_trigger();
  pdl_wait();
  using Gm = TileGeom<D, FP8, KT>;
  constexpr int DN = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, hk = blockIdx.y, t = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = n_q / n_kv;
  const int p = pos[t], s = seq_id[t];
  bool ok = p >= 1 && s >= 0 && s < kc.num_seqs && !(kc.window == 0 && p > kc.capacity);
  if (!ok && split == 0 && hk == 0 && threadIdx.x == 0)
    flag((p < 1 || (kc.window == 0 && p > kc.capacity)) ? BEAM_DEV_BAD_POSITION : BEAM_DEV_BAD_SEQ);
  const int lo = kc.window > 0 ? max(1, p - kc.window + 1) : 1;
  const int nkeys = ok ? p - lo + 1 : 0;
  const int k_begin = split * kps;
  const int k_end = min(nkeys, k_begin + kps);
  const int ntiles = k_end > k_begin ? (k_end - k_begin + KT - 1) / KT : 0;
  const int my_tiles = ntiles > warp ? (ntiles - warp + kDecWarps - 1) / kDecWarps : 0;

  uint32_t qa[D / 16][4];
  {
    const int rows[2] = {g, g + 8};
    int off[2];
    bool rok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      rok[h] = rows[h] < G;
      off[h] = (t * n_q + hk * G + (rok[h] ? rows[h] : 0)) * D;
    }
    load_q<D>(q, qa, off, rok);
  }

  float acc[DN][4];
#pragma unroll
  for (int n = 0; n < DN; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};

  uint8_t* wbase = smem + warp * dec_warp_bytes<D, FP8, KT, ST>();
  const size_t head_off = (size_t(ok ? s : 0) * n_kv + hk) * kc.capacity;
  const uint8_t* kbase = static_cast<const uint8_t*>(kc.k) + head_off * Gm::RAWROW;
  const uint8_t* vbase = static_cast<const uint8_t*>(kc.v) + head_off * Gm::RAWROW;
  const int slot_lo = ok ? (lo - 1) % kc.capacity : 0;

  auto issue = [&](int i, int stage) {
    const int key0 = k_begin + (warp + i * kDecWarps) * KT;
    const int s0 = (slot_lo + key0) % kc.capacity;
    uint8_t* kd = wbase + stage * 2 * Gm::RAWB;
    issue_tile<D, FP8, KT>(kd, kbase, s0, kc.capacity, k_end - key0, lane, 32);
    issue_tile<D, FP8, KT>(kd + Gm::RAWB, vbase, s0, kc.capacity, k_end - key0, lane, 32);
  };
  // ST-stage cp.async pipeline: tiles i+1 .. i+ST-1 are in flight while tile i is computed
#pragma unroll
  for (int s = 0; s < ST - 1; ++s) {
    if (s < my_tiles) issue(s, s);
    cp_async_commit();
  }
  for (int i = 0; i < my_tiles; ++i) {
    if (i + ST - 1 < my_tiles) issue(i + ST - 1, (i + ST - 1) % ST);
    cp_async_commit();
    cp_async_wait<ST - 1>();
    __syncwarp();
    const uint8_t* kt = wbase + (i % ST) * 2 * Gm::RAWB;
    const uint8_t* vt = kt + Gm::RAWB;
    if (FP8) {
      uint8_t* cvt = wbase + 2 * ST * Gm::RAWB;
      convert_tile<D, KT>(kt, cvt, lane, 32);
      convert_tile<D, KT>(vt, cvt + Gm::TILEB, lane, 32);
      __syncwarp();
      kt = cvt;
      vt = cvt + Gm::TILEB;
    }
    float sacc[KT / 8][4];
    qk_tile<D, KT>(qa, kt, sacc);
    const int key0 = k_begin + (warp + i * kDecWarps) * KT;
    bool valid[KT / 8][4];
#pragma unroll
    for (int j = 0; j < KT / 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) valid[j][e] = key0 + 8 * j + 2 * c + (e & 1) < k_end;
    softmax_update<KT, DN>(sacc, valid, sl2, m, l, acc);
    pv_tile<D, KT, true>(sacc, vt, acc);
    __syncwarp();
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }

  // combine the 4 warps of the CTA through shared memory
  cp_async_wait<0>();
  __syncthreads();
  constexpr int ACC_LD = D + 4;
  float* sacc_all = reinterpret_cast<float*>(smem);                       // [warps][16][ACC_LD]
  float* sml = sacc_all + kDecWarps * kRows * ACC_LD;                     // [warps][16][2]
  {
    float* a = sacc_all + warp * kRows * ACC_LD;
#pragma unroll
    for (int n = 0; n < DN; ++n) {
      a[g * ACC_LD + 8 * n + 2 * c] = acc[n][0];
      a[g * ACC_LD + 8 * n + 2 * c + 1] = acc[n][1];
      a[(g + 8) * ACC_LD + 8 * n + 2 * c] = acc[n][2];
      a[(g + 8) * ACC_LD + 8 * n + 2 * c + 1] = acc[n][3];
    }
    if (c == 0) {
      sml[(warp * kRows + g) * 2] = m[0];
      sml[(warp * kRows + g) * 2 + 1] = l[0];
      sml[(warp * kRows + g + 8) * 2] = m[1];
      sml[(warp * kRows + g + 8) * 2 + 1] = l[1];
    }
  }
  __syncthreads();
  if constexpr (CLUSTER) {
    // this CTA's partial to its own shared memory, above the tile and combine buffers
    float* cO = reinterpret_cast<float*>(smem + DecodeSmem<D, FP8, KT, ST>::kPartOff);   // [16][D]
    float* cML = cO + kRows * D;                                                 // [16][2]
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int row = idx / D, d = idx - row * D;
      float M, O, L;
      combine_warps(sacc_all, sml, ACC_LD, row, d, M, O, L);
      cO[row * D + d] = O;
      if (d == 0) {
        cML[row * 2] = M;
        cML[row * 2 + 1] = L;
      }
    }
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    merge_gate_cluster(cl, cO, cML, n_splits, n_q, n_kv, D, v_scale, gpre, gate_bias, og, t, hk,
                       reinterpret_cast<float*>(smem));
    cl.sync();   // peers may still be reading this CTA's partial
    return;
  } else {
    const size_t pbase = (size_t(t) * n_kv + hk) * n_splits + split;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int row = idx / D, d = idx - row * D;
      float M, O, L;
      combine_warps(sacc_all, sml, ACC_LD, row, d, M, O, L);
      part_acc[(pbase * kRows + row) * D + d] = O;
      if (d == 0) {
        part_ml[(pbase * kRows + row) * 2] = M;
        part_ml[(pbase * kRows + row) * 2 + 1] = L;
      }
    }
    // the last split CTA of this (token, KV head) merges all splits
    __shared__ int s_last;
    // the CTA barrier orders every thread's partial stores before thread 0's device-scope
    // fence, which releases them with the counter increment
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      s_last = atomicAdd(done + t * n_kv + hk, 1) == n_splits - 1;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      // the tile buffers are free now: stage the merge weights there
      merge_gate(part_acc, part_ml, n_splits, n_q, n_kv, D, v_scale, gpre, gate_bias, og, t, hk,
                 reinterpret_cast<float*>(smem));
    }
  }
}

// ------------------------------------------------------------------------------------------
// Prefill: query tiles of 16 tokens x one KV group
// ------------------------------------------------------------------------------------------
template <int D, bool FP8>
__global__ void __launch_bounds__(256) attn_prefill_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ gpre,
    const uint16_t* __restrict__ gate_bias, const int32_t* __restrict__ seq_id,
    const int32_t* __restrict__ pos, int T, int n_q, int n_kv, beam_kv_cache kc, float sl2,
    uint16_t* __restrict__ og) {
  pdl_trigger();
  pdl_wait();
  using Gm = TileGeom<D, FP8, kPreKT>;
  constexpr int KT = kPreKT;
  constexpr int DN = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_seq[kRows], s_lo[kRows], s_hi[kRows];
  const int t0 = blockIdx.x * kRows, hk = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = n_q / n_kv;
  const int hq = hk * G + warp;

  if (threadIdx.x < kRows) {
    const int t = t0 + threadIdx.x;
    int sq = -1, lo = 1, hi = 0;
    if (t < T) {
      const int p = pos[t], s = seq_id[t];
      const bool badp = p < 1 || (kc.window == 0 && p > kc.capacity);
      const bool bads = s < 0 || s >= kc.num_seqs;
      if (badp) flag(BEAM_DEV_BAD_POSITION);
      if (bads) flag(BEAM_DEV_BAD_SEQ);
      if (!badp && !bads) {
        sq = s;
        hi = p;
        lo = kc.window > 0 ? max(1, p - kc.window + 1) : 1;
      }
    }
    s_seq[threadIdx.x] = sq;
    s_lo[threadIdx.x] = lo;
    s_hi[threadIdx.x] = hi;
  }
  __syncthreads();

  uint32_t qa[D / 16][4];
  {
    int off[2];
    bool rok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + g + 8 * h;
      rok[h] = t < T && s_seq[g + 8 * h] >= 0;
      off[h] = ((rok[h] ? t : 0) * n_q + hq) * D;
    }
    load_q<D>(q, qa, off, rok);
  }
  const int rseq[2] = {s_seq[g], s_seq[g + 8]};
  const int rlo[2] = {s_lo[g], s_lo[g + 8]};
  const int rhi[2] = {s_hi[g], s_hi[g + 8]};

  float acc[DN][4];
#pragma unroll
  for (int n = 0; n < DN; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};

  int cur = -1;
  while (true) {
    // next sequence present in the tile
    int nxt = 0x7fffffff;
    for (int r = 0; r < kRows; ++r)
      if (s_seq[r] > cur) nxt = min(nxt, s_seq[r]);
    if (nxt == 0x7fffffff) break;
    cur = nxt;
    int kmin = 0x7fffffff, kmax = 0;
    for (int r = 0; r < kRows; ++r)
      if (s_seq[r] == cur) { kmin = min(kmin, s_lo[r]); kmax = max(kmax, s_hi[r]); }
    const int nkeys = kmax - kmin + 1;
    const int ntiles = (nkeys + KT - 1) / KT;
    const size_t head_off = (size_t(cur) * n_kv + hk) * kc.capacity;
    const uint8_t* kbase = static_cast<const uint8_t*>(kc.k) + head_off * Gm::RAWROW;
    const uint8_t* vbase = static_cast<const uint8_t*>(kc.v) + head_off * Gm::RAWROW;
    const int slot_lo = (kmin - 1) % kc.capacity;
    auto issue = [&](int i, int stage) {
      const int key0 = i * KT;
      const int s0 = (slot_lo + key0) % kc.capacity;
      uint8_t* kd = smem + stage * 2 * Gm::RAWB;
      issue_tile<D, FP8, KT>(kd, kbase, s0, kc.capacity, nkeys - key0, threadIdx.x, blockDim.x);
      issue_tile<D, FP8, KT>(kd + Gm::RAWB, vbase, s0, kc.capacity, nkeys - key0, threadIdx.x,
                             blockDim.x);
    };
    issue(0, 0);
    cp_async_commit();
    for (int i = 0; i < ntiles; ++i) {
      if (i + 1 < ntiles) issue(i + 1, (i + 1) & 1);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      const uint8_t* kt = smem + (i & 1) * 2 * Gm::RAWB;
      const uint8_t* vt = kt + Gm::RAWB;
      if (FP8) {
        uint8_t* cvt = smem + 4 * Gm::RAWB;
        convert_tile<D, KT>(kt, cvt, threadIdx.x, blockDim.x);
        convert_tile<D, KT>(vt, cvt + Gm::TILEB, threadIdx.x, blockDim.x);
        __syncthreads();
        kt = cvt;
        vt = cvt + Gm::TILEB;
      }
      const int kp0 = kmin + i * KT;   // position of the tile's first key
      bool any = false;
      bool valid[KT / 8][4];
#pragma unroll
      for (int j = 0; j < KT / 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const int kp = kp0 + 8 * j + 2 * c + (e & 1);
          valid[j][e] = rseq[h] == cur && kp >= rlo[h] && kp <= rhi[h];
          any |= valid[j][e];
        }
      if (__any_sync(0xffffffffu, any)) {
        float sacc[KT / 8][4];
        qk_tile<D, KT>(qa, kt, sacc);
        softmax_update<KT, DN>(sacc, valid, sl2, m, l, acc);
        pv_tile<D, KT, true>(sacc, vt, acc);
      }
      __syncthreads();
    }
    cp_async_wait<0>();
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
  }
  const float vs = FP8 ? kc.v_scale : 1.f;
  const float gb = bf2f(gate_bias[hq]);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = t0 + g + 8 * h;
    if (t >= T) continue;
    const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
    const size_t ob = (size_t(t) * n_q + hq) * D;
#pragma unroll
    for (int n = 0; n < DN; ++n) {
      const int d = 8 * n + 2 * c;
      const float o0 = round_bf(acc[n][2 * h] * inv * vs);
      const float o1 = round_bf(acc[n][2 * h + 1] * inv * vs);
      const uint32_t gg = *reinterpret_cast<const uint32_t*>(gpre + ob + d);
      const float r0 = o0 * sigmoidf_(bf_lo(gg) + gb);
      const float r1 = o1 * sigmoidf_(bf_hi(gg) + gb);
      *reinterpret_cast<uint32_t*>(og + ob + d) = pack_bf16x2(r0, r1);
    }
  }
}

int g_num_sms = 0;
int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 152;
  }
  return g_num_sms;
}

constexpr int kDecodeMaxQ = 4;   // split-K per token up to this many tokens per sequence
// Verification batches of speculative decoding (up to kVerifyMaxQ tokens per sequence): the
// query-tile prefill form walks one sequence's keys per (KV head, job) item without splitting
// them, so with fewer items than SMs most SMs idle (one sequence at 100K keys and 8 tokens:
// 2.8 ms for the NoPE layer); the split-K decode form reads the keys once per token but keeps
// every SM busy (345 us). The decode form is taken while the call has fewer (sequence, KV
// head) items than two per SM.
constexpr int kVerifyMaxQ = 16;
bool decode_form(int T, int max_q_per_seq, int n_kv) {
  if (max_q_per_seq <= kDecodeMaxQ) return true;
  const long seqs = (long(T) + max_q_per_seq - 1) / max_q_per_seq;   // at least this many
  return max_q_per_seq <= kVerifyMaxQ && seqs * n_kv < 2L * num_sms();
}

struct DecodePlan {
  int kps, n_splits;
};

DecodePlan decode_plan(int T, int n_kv, int max_keys) {
  const int per = T * n_kv;
  // CTAs resident at once (two per SM); the split count fills whole waves of them: the
  // smallest multiple (up to 4) of the resident slots that the (token, KV head) count divides
  const int slots = 2 * num_sms();
  int splits = 1;
  if (per < slots) {
    int w = 1;
    while (w < 4 && (slots * w) % per != 0) ++w;
    splits = (slots * w + per - 1) / per;
  }
  const int max_splits = (max_keys + 127) / 128;
  splits = splits < 1 ? 1 : (splits > max_splits ? max_splits : splits);
  if (splits > kMergeMaxSplits) splits = kMergeMaxSplits;
  int kps = (max_keys + splits - 1) / splits;
  kps = (kps + 127) / 128 * 128;
  splits = (max_keys + kps - 1) / kps;
  if (splits < 1) splits = 1;
  if (splits > kMergeMaxSplits) {   // keep within the merge's staging (never hit in practice)
    kps = (max_keys + kMergeMaxSplits - 1) / kMergeMaxSplits;
    kps = (kps + 127) / 128 * 128;
    splits = (max_keys + kps - 1) / kps;
  }
  return {kps, splits};
}

int max_keys_of(int window, int max_pos) {
  return window > 0 ? (max_pos < window ? max_pos : window) : max_pos;
}

template <class K>
cudaError_t set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int D, bool FP8>
cudaError_t launch_decode(const uint16_t* q, const int32_t* seq_id, const int32_t* pos, int T,
                          int n_q, int n_kv, const beam_kv_cache& kc, DecodePlan pl, float sl2,
                          float* pacc, float* pml, int* done, float v_scale, const uint16_t* g,
                          const uint16_t* gb, uint16_t* og, cudaStream_t st) {
  const dim3 grid(pl.n_splits, n_kv, T), block(kDecWarps * 32);
  if (pl.n_splits == 1) {
    // one split per (token, KV head): many small CTAs, two per SM
    using Sm = DecodeSmem<D, FP8, kDecKTSplit, kDecStagesSplit>;
    auto kern = attn_decode_split_kernel<D, FP8, true, kDecKTSplit, kDecStagesSplit>;
    cudaError_t e = set_smem(kern, Sm::kBytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl_cluster(kern, grid, block, Sm::kBytes, st, 1, q, seq_id, pos, n_q, n_kv, kc,
                           pl.kps, pl.n_splits, sl2, pacc, pml, done, v_scale, g, gb, og);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  if (pl.n_splits <= kClusterMaxSplits) {
    using Sm = DecodeSmem<D, FP8, kDecKTCluster, 2>;
    auto kern = attn_decode_split_kernel<D, FP8, true, kDecKTCluster, 2>;
    cudaError_t e = set_smem(kern, Sm::kBytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl_cluster(kern, grid, block, Sm::kBytes, st, pl.n_splits, q, seq_id, pos, n_q,
                           n_kv, kc, pl.kps, pl.n_splits, sl2, pacc, pml, done, v_scale, g, gb, og);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  using Sm = DecodeSmem<D, FP8, kDecKTSplit, kDecStagesSplit>;
  auto kern = attn_decode_split_kernel<D, FP8, false, kDecKTSplit, kDecStagesSplit>;
  cudaError_t e = set_smem(kern, Sm::kPartOff);
  if (e != cudaSuccess) return e;
  launch_pdl(kern, grid, block, Sm::kPartOff, st, q, seq_id, pos, n_q, n_kv, kc, pl.kps,
             pl.n_splits, sl2, pacc, pml, done, v_scale, g, gb, og);
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_prefill(const uint16_t* q, const uint16_t* g, const uint16_t* gb,
                           const int32_t* seq_id, const int32_t* pos, int T, int n_q, int n_kv,
                           const beam_kv_cache& kc, float sl2, uint16_t* og, cudaStream_t st) {
  using Gm = TileGeom<D, FP8, kPreKT>;
  const int bytes = Gm::BYTES;
  auto kern = attn_prefill_kernel<D, FP8>;
  cudaError_t e = set_smem(kern, bytes);
  if (e != cudaSuccess) return e;
  dim3 grid((T + kRows - 1) / kRows, n_kv);
  launch_pdl(kern, dim3(grid), dim3(32 * (n_q / n_kv)), bytes, st, q, g, gb, seq_id, pos, T, n_q, n_kv, kc, sl2, og);
  return cudaGetLastError();
}

}  // namespace

size_t attn_ws_bytes(const beam_layer_cfg* c, int T, int max_pos, int window) {
  size_t b = align_up(size_t(T) * c->n_q * c->head_dim * 2, 256);
  {   // the split-K decode form may be chosen for any T (decode_form)
    // partials only when the splits merge through the workspace (more than a cluster)
    const DecodePlan pl = decode_plan(T, c->n_kv, max_keys_of(window, max_pos > 0 ? max_pos : 1));
    const size_t parts =
        pl.n_splits > kClusterMaxSplits ? size_t(T) * c->n_kv * pl.n_splits * kRows : 0;
    b += align_up(parts * c->head_dim * 4, 256) + align_up(parts * 2 * 4, 256);
    b += align_up(size_t(T) * c->n_kv * 4, 256);     // split completion counters
  }
  // or the TMA decode kernel's partials (BF16 or FP8 cache), or the tensor-core prefill's job list
  size_t alt = atc::ws_bytes(T);
  const int mp = max_pos > 0 ? max_pos : 1;
  const size_t d16 = adec::ws_bytes(T, c->n_kv, window, mp, false);
  const size_t d8 = adec::ws_bytes(T, c->n_kv, window, mp, true);
  if (d16 > alt) alt = d16;
  if (d8 > alt) alt = d8;
  if (window == 0) {   // or the grouped verification form's partials and group list
    const size_t dv = adec::verify_ws_bytes_max(T);
    if (dv > alt) alt = dv;
  }
  const size_t dec = b - align_up(size_t(T) * c->n_q * c->head_dim * 2, 256);
  if (alt > dec) b += alt - dec;
  return b;
}

}  // namespace beam

extern "C" beam_status beam_attn(const beam_layer_cfg* cfg, const beam_bf16* q,
                                 const beam_bf16* g, const beam_bf16* gate_bias,
                                 const beam_kv_cache* cache, const int32_t* seq_id,
                                 const int32_t* pos, int T, int max_pos, int max_q_per_seq,
                                 const beam_bf16* w_o, beam_bf16* out, void* ws, size_t ws_bytes,
                                 beam_stream_t stream) {
  using namespace beam;
  beam_status stt = check_cfg_attn(cfg);
  if (stt != BEAM_OK) return stt;
  if ((stt = check_cache(cache, cfg)) != BEAM_OK) return stt;
  if (T < 0 || max_pos < 1 || max_q_per_seq < 1 || !q || !g || !gate_bias || !seq_id || !pos ||
      !w_o || !out)
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(g) || !aligned16(w_o) || !aligned16(out) || !aligned16(ws))
    return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  const int D = cfg->head_dim, H = cfg->hidden, HD = cfg->n_q * D;
  const bool fp8 = cache->dtype == BEAM_KV_FP8_E4M3;
  const float sl2 = float(1.4426950408889634 / sqrt(double(D))) * (fp8 ? cache->k_scale : 1.f);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carver cv{static_cast<char*>(ws), ws_bytes};
  uint16_t* og = cv.take<uint16_t>(size_t(T) * HD);
  cudaError_t e;
  const int G = cfg->n_q / cfg->n_kv;
  const bool dec = decode_form(T, max_q_per_seq, cfg->n_kv);
  if (dec && adec::verify_supported(D, G, cache->window, fp8, cache->k, cache->v,
                                    max_keys_of(cache->window, max_pos), T, max_q_per_seq)) {
    // several tokens of a sequence: each K/V block is read once for all of them
    const size_t vb = adec::verify_ws_bytes(T, G, max_q_per_seq);
    void* vw = cv.take<char>(vb);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    e = adec::verify(q, g, gate_bias, seq_id, pos, T, max_pos, max_q_per_seq, cfg->n_q,
                     cfg->n_kv, *cache, sl2, og, vw, vb, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else if (dec &&
      adec::supported(D, G, cache->window, cache->capacity, fp8, cache->k, cache->v,
                      max_keys_of(cache->window, max_pos))) {
    const size_t db = adec::ws_bytes(T, cfg->n_kv, cache->window, max_pos, fp8);
    void* dw = cv.take<char>(db);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    e = adec::decode(q, g, gate_bias, seq_id, pos, T, max_pos, cfg->n_q, cfg->n_kv, *cache, sl2,
                     fp8 ? cache->v_scale : 1.f, og, dw, db, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else if (dec) {
    const DecodePlan pl = decode_plan(T, cfg->n_kv, max_keys_of(cache->window, max_pos));
    const size_t parts =
        pl.n_splits > kClusterMaxSplits ? size_t(T) * cfg->n_kv * pl.n_splits * kRows : 0;
    float* pacc = cv.take<float>(parts * D);
    float* pml = cv.take<float>(parts * 2);
    int* done = cv.take<int>(size_t(T) * cfg->n_kv);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    // the cluster form merges on chip; the other counts finished splits from zero
    if (pl.n_splits > kClusterMaxSplits) {
      const cudaError_t err_ = cudaMemsetAsync(done, 0, size_t(T) * cfg->n_kv * sizeof(int), st);
      if (err_ != cudaSuccess) return cuda_status(err_);
    }
    const float vs = fp8 ? cache->v_scale : 1.f;
    if (D == 128)
      e = fp8 ? launch_decode<128, true>(q, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, pl, sl2, pacc, pml, done, vs, g, gate_bias, og, st)
              : launch_decode<128, false>(q, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, pl, sl2, pacc, pml, done, vs, g, gate_bias, og, st);
    else
      e = fp8 ? launch_decode<64, true>(q, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, pl, sl2, pacc, pml, done, vs, g, gate_bias, og, st)
              : launch_decode<64, false>(q, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, pl, sl2, pacc, pml, done, vs, g, gate_bias, og, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else if (atc::prefill_supported(D, cfg->n_q / cfg->n_kv, cache->window, cache->capacity, fp8,
                                     q, cache->k, cache->v)) {
    const size_t tcb = atc::ws_bytes(T);
    void* jw = cv.take<char>(tcb);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    e = atc::prefill(q, g, gate_bias, seq_id, pos, T, cfg->n_q, cfg->n_kv, D, *cache, sl2, og, jw,
                     tcb, st);
    if (e != cudaSuccess) return cuda_status(e);
  } else {
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    if (cfg->n_q / cfg->n_kv * 32 > 256) return BEAM_ERR_UNSUPPORTED;
    if (D == 128)
      e = fp8 ? launch_prefill<128, true>(q, g, gate_bias, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, sl2, og, st)
              : launch_prefill<128, false>(q, g, gate_bias, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, sl2, og, st);
    else
      e = fp8 ? launch_prefill<64, true>(q, g, gate_bias, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, sl2, og, st)
              : launch_prefill<64, false>(q, g, gate_bias, seq_id, pos, T, cfg->n_q, cfg->n_kv, *cache, sl2, og, st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  const cudaError_t ge =
      T >= kGemmMinT && tc::gemm_supported(og, HD, w_o, HD, HD)
          ? tc::gemm_bf16(og, T, HD, HD, w_o, H, HD, out, H, true, st)
          : launch_gemv<kOutBF16>(w_o, H, HD, og, T, nullptr, out, H, st);
  if (ge != cudaSuccess) return cuda_status(ge);
  return BEAM_OK;
}
