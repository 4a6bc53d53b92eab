// Packed QKV + gate projection, per-head Q/K RMSNorm, RoPE or SSMax, KV-cache write.
// Beam page, Attention section (48 query / 8 KV heads of 128, Q and K RMS-normalised per head
// before RoPE or SSMax (1 + p/2048)^0.1) and changes 2, 5 and 6 of the optimisation list
// (one packed projection; norm, rotation and cache write in one kernel).
#include <math.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"

namespace beam {
namespace {

constexpr int kMaxHalf = 64;  // D/2 for D = 128

// theta^(-2i/D), i < D/2, computed on the host in double and passed by value.
struct RopeTab {
  double inv[kMaxHalf];
};

// Grid (token, slot group of 8): z holds the projection (fp32) of the token, rows
// Q | K | V | gate. Each warp takes one (kind, head) slot: n_q query heads, n_kv key heads,
// n_kv value heads and n_q gate heads. Lane l holds elements l, l+32, ... of the head (VPL = D/32 values), so the
// RoPE partner i + D/2 of element l + 32j is element j + VPL/2 of the same lane.
template <int VPL>
__global__ void __launch_bounds__(256) qkv_epilogue_kernel(
    const float* __restrict__ z, int rows, const uint16_t* __restrict__ qnw,
    const uint16_t* __restrict__ knw, const int32_t* __restrict__ seq_id,
    const int32_t* __restrict__ pos, int n_q, int n_kv, int nope, RopeTab rope, float ss_base,
    float ss_exp, float eps, uint16_t* __restrict__ q_out, uint16_t* __restrict__ g_out,
    beam_kv_cache kc) {
  pdl_trigger();
  pdl_wait();
  constexpr int D = VPL * 32;
  constexpr int HALF = D / 2;
  __shared__ float cs[kMaxHalf], sn[kMaxHalf];
  __shared__ float s_ssmax;
  const int t = blockIdx.x;
  const int p = pos[t];
  const int s = seq_id[t];
  bool ok_kv = true;
  if (p < 1) { if (threadIdx.x == 0) flag(BEAM_DEV_BAD_POSITION); ok_kv = false; }
  if (s < 0 || s >= kc.num_seqs) { if (threadIdx.x == 0) flag(BEAM_DEV_BAD_SEQ); ok_kv = false; }
  if (kc.window == 0 && p > kc.capacity) {
    if (threadIdx.x == 0) flag(BEAM_DEV_BAD_POSITION);
    ok_kv = false;
  }
  if (!nope) {
    // angle (p-1) * theta^(-2i/D), formed in double precision and reduced modulo 2*pi so
    // that positions around 1e5 keep full single-precision accuracy in cos/sin
    for (int i = threadIdx.x; i < HALF; i += blockDim.x) {
      float sv, cv;
      sincosf(rope_angle(p, rope.inv[i]), &sv, &cv);
      cs[i] = cv;
      sn[i] = sv;
    }
  } else if (threadIdx.x == 0) {
    s_ssmax = ssmax_scale(p, ss_base, ss_exp);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int nslots = 2 * n_q + 2 * n_kv;
  const float* zt = z + size_t(t) * rows;
  for (int slot = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5); slot < nslots;
       slot += gridDim.y * (blockDim.x >> 5)) {
    int kind, head, row0;
    if (slot < n_q) { kind = 0; head = slot; row0 = head * D; }
    else if (slot < n_q + n_kv) { kind = 1; head = slot - n_q; row0 = (n_q + head) * D; }
    else if (slot < n_q + 2 * n_kv) { kind = 2; head = slot - n_q - n_kv; row0 = (n_q + n_kv + head) * D; }
    else { kind = 3; head = slot - n_q - 2 * n_kv; row0 = (n_q + 2 * n_kv + head) * D; }
    float v[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) v[j] = round_bf(zt[row0 + lane + 32 * j]);  // projection out
    if (kind == 3) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) g_out[size_t(t) * n_q * D + head * D + lane + 32 * j] = f2bf(v[j]);
      continue;
    }
    if (kind <= 1) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j) ss = fmaf(v[j], v[j], ss);
      const float r = rsqrtf(warp_sum(ss) / float(D) + eps);
      const uint16_t* gw = kind == 0 ? qnw : knw;
#pragma unroll
      for (int j = 0; j < VPL; ++j) v[j] = v[j] * r * bf2f(gw[lane + 32 * j]);
      if (!nope) {
#pragma unroll
        for (int j = 0; j < VPL / 2; ++j) {
          const int i = lane + 32 * j;  // < HALF
          const float a = v[j], b = v[j + VPL / 2];
          v[j] = a * cs[i] - b * sn[i];
          v[j + VPL / 2] = b * cs[i] + a * sn[i];
        }
      } else if (kind == 0) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) v[j] *= s_ssmax;
      }
    }
    if (kind == 0) {
#pragma unroll
      for (int j = 0; j < VPL; ++j) q_out[(size_t(t) * n_q + head) * D + lane + 32 * j] = f2bf(v[j]);
      continue;
    }
    if (!ok_kv) continue;
    const int slotk = (p - 1) % kc.capacity;
    const size_t base = ((size_t(s) * n_kv + head) * kc.capacity + slotk) * D;
    if (kc.dtype == BEAM_KV_BF16) {
      uint16_t* dst = static_cast<uint16_t*>(kind == 1 ? kc.k : kc.v) + base;
#pragma unroll
      for (int j = 0; j < VPL; ++j) dst[lane + 32 * j] = f2bf(v[j]);
    } else {
      uint8_t* dst = static_cast<uint8_t*>(kind == 1 ? kc.k : kc.v) + base;
      const float sc = kind == 1 ? kc.k_scale : kc.v_scale;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        dst[lane + 32 * j] = __nv_cvt_float_to_fp8(__fdiv_rn(v[j], sc), __NV_SATFINITE, __NV_E4M3);
    }
  }
}

// (cos, sin) of angle (p - 1) * theta^(-2i/D) for each token's position, i < D/2: the RoPE
// rows the tensor-core projection's epilogue reads (same angle reduction as above).
__global__ void __launch_bounds__(256) rope_table_kernel(const int32_t* __restrict__ pos, int T,
                                                         int half, RopeTab rope,
                                                         float2* __restrict__ tab) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * half) return;
  const int t = i / half, j = i - t * half;
  float sv, cv;
  sincosf(rope_angle(pos[t], rope.inv[j]), &sv, &cv);
  tab[i] = make_float2(cv, sv);
}

}  // namespace

size_t qkv_ws_bytes(const beam_layer_cfg* c, int T) {
  const size_t rows = size_t(2 * c->n_q + 2 * c->n_kv) * c->head_dim;
  return align_up(size_t(T) * rows * sizeof(float), 256);
}

}  // namespace beam

extern "C" beam_status beam_qkv_gate(const beam_layer_cfg* cfg, const beam_bf16* u,
                                     const beam_bf16* w_qkvg, const beam_bf16* q_norm_w,
                                     const beam_bf16* k_norm_w, const int32_t* seq_id,
                                     const int32_t* pos, int T, beam_bf16* q_out,
                                     beam_bf16* g_out, const beam_kv_cache* cache, void* ws,
                                     size_t ws_bytes, beam_stream_t stream) {
  using namespace beam;
  beam_status st = check_cfg_attn(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_cache(cache, cfg)) != BEAM_OK) return st;
  if (T < 0 || !u || !w_qkvg || !q_norm_w || !k_norm_w || !seq_id || !pos || !q_out || !g_out)
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_qkvg) || !aligned16(ws)) return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  const int D = cfg->head_dim, H = cfg->hidden;
  const int rows = (2 * cfg->n_q + 2 * cfg->n_kv) * D;
  Carver cv{static_cast<char*>(ws), ws_bytes};
  float* z = cv.take<float>(size_t(T) * rows);
  if (!cv.ok) return BEAM_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int nope = cfg->kind == BEAM_ATTN_NOPE_SSMAX;
  RopeTab rope;
  for (int i = 0; i < D / 2; ++i)
    rope.inv[i] = pow(double(cfg->rope_theta), -2.0 * double(i) / double(D));
  if (T >= kGemmMinT && D == 128 && tc::gemm_supported(u, H, w_qkvg, H, H) && aligned16(q_out) &&
      aligned16(g_out) && aligned16(cache->k) && aligned16(cache->v)) {
    // prefill: the projection's epilogue does the norms, RoPE/SSMax and the cache write
    float2* tab = reinterpret_cast<float2*>(z);   // the FP32 projection buffer is unused here
    if (!nope)
      launch_pdl(rope_table_kernel, dim3((T * (D / 2) + 255) / 256), dim3(256), 0, s, pos, T,
                 D / 2, rope, tab);
    tc::QkvEpilogue e{q_out, g_out, *cache, seq_id, pos, q_norm_w, k_norm_w,
                      nope ? nullptr : tab, cfg->n_q, cfg->n_kv, nope, cfg->ssmax_base,
                      cfg->ssmax_exp, cfg->eps};
    return cuda_status(tc::gemm_qkv(u, T, H, H, w_qkvg, rows, H, e, s));
  }
  const cudaError_t ge =
      T >= kGemmMinT && tc::gemm_supported(u, H, w_qkvg, H, H)
          ? tc::gemm_bf16(u, T, H, H, w_qkvg, rows, H, z, rows, false, s)
          : launch_gemv<kOutF32>(w_qkvg, rows, H, u, T, z, nullptr, rows, s);
  if (ge != cudaSuccess) return cuda_status(ge);
  if (D == 128)
    launch_pdl(qkv_epilogue_kernel<4>, dim3(T, (2 * cfg->n_q + 2 * cfg->n_kv + 7) / 8), dim3(256), 0, s, z, rows, q_norm_w, k_norm_w, seq_id, pos, cfg->n_q,
                                             cfg->n_kv, nope, rope, cfg->ssmax_base,
                                             cfg->ssmax_exp, cfg->eps, q_out, g_out, *cache);
  else
    launch_pdl(qkv_epilogue_kernel<2>, dim3(T, (2 * cfg->n_q + 2 * cfg->n_kv + 7) / 8), dim3(256), 0, s, z, rows, q_norm_w, k_norm_w, seq_id, pos, cfg->n_q,
                                             cfg->n_kv, nope, rope, cfg->ssmax_base,
                                             cfg->ssmax_exp, cfg->eps, q_out, g_out, *cache);
  return launch_status();
}
