// FP32 router, DeepSeek-V3 style group-limited top-k.
// Beam page, MoE section (sigmoid scores plus a correction bias pick the best 4 of 8 expert
// groups, then the top-8 experts; the renormalised weights are scaled by 2.5; the 5120 x 256
// router weights, accumulation and logits are FP32) and change 4 of the optimisation list
// (a dedicated small-batch FP32 router kernel).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "gemm_tc.cuh"

namespace beam {
namespace {

constexpr int kRouteMaxT = 8;  // tokens per CTA pass in the GEMV form
constexpr int kRouteBatch = 3; // weight chunks in flight per thread in the GEMV form
// Above kRouteGemvMaxT tokens the logits run on the tensor cores: every FP32 router weight is split
// exactly into three BF16 parts, w = hi + mid + lo (hi = bf16(w), mid = bf16(w - hi),
// lo = w - hi - mid, each step exact), the BF16 activations times each part are exact FP32
// products, and one BF16 GEMM against the stacked [hi; mid; lo] rows accumulates them in FP32;
// logit = (u.hi + u.mid) + u.lo. Up to kRouteGemvMaxT tokens (decode, and every size the
// allocation-free router accepts: it refuses more) the FP32 SIMT GEMV runs, one CTA per
// expert row.
constexpr int kRouteTcMinT = 257;
constexpr int kRouteGemvMaxT = 256;   // up to here the GEMV form (the allocation-free router's range)
constexpr int kRouteKChunks = 8;   // K chains of the tensor-core logits (640 at hidden 5120)

// Small T: one CTA per expert row; its warps split the hidden axis; every token of a pass
// reuses the row held in registers/L1.
__global__ void __launch_bounds__(256) router_gemv_kernel(const uint16_t* __restrict__ u,
                                                          const float* __restrict__ wr, int T,
                                                          int H, int E,
                                                          float* __restrict__ logits) {
  pdl_trigger();
  __shared__ float red[8][kRouteMaxT];
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* row = wr + size_t(e) * H;
  // the router weights are no predecessor's output: start the row towards L2 before waiting
  if (threadIdx.x == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0)
    l2_prefetch(row, uint32_t(H) * 4);
  pdl_wait();
  for (int t0 = 0; t0 < T; t0 += kRouteMaxT) {
    const int nt = min(kRouteMaxT, T - t0);
    float acc[kRouteMaxT];
#pragma unroll
    for (int t = 0; t < kRouteMaxT; ++t) acc[t] = 0.f;
    // kRouteBatch chunks of 8 weights per thread are requested before any is used, so a
    // 5120-wide row arrives in one round trip
    for (int i0 = threadIdx.x; i0 < H / 8; i0 += kRouteBatch * blockDim.x) {
      float4 w0[kRouteBatch], w1[kRouteBatch];
#pragma unroll
      for (int b = 0; b < kRouteBatch; ++b) {
        const int i = i0 + b * blockDim.x;
        if (i < H / 8) {
          w0[b] = ld_stream_f4(row + i * 8);
          w1[b] = ld_stream_f4(row + i * 8 + 4);
        }
      }
#pragma unroll
      for (int b = 0; b < kRouteBatch; ++b) {
        const int i = i0 + b * blockDim.x;
        if (i >= H / 8) break;
#pragma unroll
        for (int t = 0; t < kRouteMaxT; ++t) {
          if (t < nt) {
            float x[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(u + size_t(t0 + t) * H + i * 8)), x);
            acc[t] = fmaf(w0[b].x, x[0], acc[t]); acc[t] = fmaf(w0[b].y, x[1], acc[t]);
            acc[t] = fmaf(w0[b].z, x[2], acc[t]); acc[t] = fmaf(w0[b].w, x[3], acc[t]);
            acc[t] = fmaf(w1[b].x, x[4], acc[t]); acc[t] = fmaf(w1[b].y, x[5], acc[t]);
            acc[t] = fmaf(w1[b].z, x[6], acc[t]); acc[t] = fmaf(w1[b].w, x[7], acc[t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kRouteMaxT; ++t) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) red[warp][t] = v;
    }
    __syncthreads();
    if (threadIdx.x < nt) {
      float s = 0.f;
      for (int w = 0; w < int(blockDim.x >> 5); ++w) s += red[w][threadIdx.x];
      logits[size_t(t0 + threadIdx.x) * E + e] = s;
    }
    __syncthreads();
  }
}

// Large T: 64 x 64 output tiles, FP32 SIMT, bf16 activations widened on the fly.
// FP32 SIMT tiles of TILE tokens x TILE experts, each thread an R x R block of outputs. Every
// logit is one FMA chain over k = 0 .. H-1 in order, whatever the tile size, so the tile size
// changes the parallelism, not the result (64 x 64 tiles, used where the tensor-core form
// does not apply).
constexpr int kTK = 32;
template <int TILE, int R>
__global__ void __launch_bounds__((TILE / R) * (TILE / R)) router_gemm_kernel(
    const uint16_t* __restrict__ u, const float* __restrict__ wr, int T, int H, int E,
    float* __restrict__ logits) {
  pdl_trigger();
  pdl_wait();
  constexpr int NT = (TILE / R) * (TILE / R), TW = TILE / R;
  __shared__ float As[kTK][TILE + 4];
  __shared__ float Bs[kTK][TILE + 4];
  const int tm = blockIdx.y * TILE, tn = blockIdx.x * TILE;
  const int tx = threadIdx.x % TW, ty = threadIdx.x / TW;
  float acc[R][R] = {};
  for (int k0 = 0; k0 < H; k0 += kTK) {
    for (int i = threadIdx.x; i < TILE * kTK; i += NT) {
      const int r = i / kTK, k = i - r * kTK;
      const int t = tm + r;
      As[k][r] = (t < T && k0 + k < H) ? bf2f(u[size_t(t) * H + k0 + k]) : 0.f;
      const int e = tn + r;
      Bs[k][r] = (e < E && k0 + k < H) ? wr[size_t(e) * H + k0 + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kTK; ++k) {
      float a[R], b[R];
#pragma unroll
      for (int i = 0; i < R; ++i) { a[i] = As[k][ty * R + i]; b[i] = Bs[k][tx * R + i]; }
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < R; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int t = tm + ty * R + i, e = tn + tx * R + j;
      if (t < T && e < E) logits[size_t(t) * E + e] = acc[i][j];
    }
}

// w3 = [hi; mid; lo] of the n FP32 weights (three stacked copies of the E x H matrix).
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ w, size_t n,
                                                           uint16_t* __restrict__ w3) {
  pdl_trigger();
  pdl_wait();
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float x = w[i];
  const uint16_t hi = f2bf(x);
  const float r1 = x - bf2f(hi);
  const uint16_t mid = f2bf(r1);
  w3[i] = hi;
  w3[n + i] = mid;
  w3[2 * n + i] = f2bf(r1 - bf2f(mid));
}

// logits[t][e] = (c[t][e] + c[t][E + e]) + c[t][2E + e], c = u . [hi; mid; lo]^T
__global__ void __launch_bounds__(256) router_sum3_kernel(const float* __restrict__ c, int T,
                                                          int E, float* __restrict__ logits) {
  pdl_trigger();
  pdl_wait();
  const size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= size_t(T) * E) return;
  const size_t t = i / E, e = i - t * E;
  const float* ct = c + t * 3 * E;
  logits[i] = (ct[e] + ct[E + e]) + ct[2 * E + e];
}

// Warp-wide argmax of (value, index), ties to the lower index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
  }
}

constexpr int kMaxE = 1024, kMaxG = 32, kMaxK = 32;

// One CTA of 256 threads per token. s = sigmoid(logit), b = s + bias (FP32); group score =
// sum of the group's two largest b; keep the kG best groups; select the k best b among their
// experts; every choice breaks ties towards the lower index.
constexpr int kTopkThreads = 256;
__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(
    const float* __restrict__ logits, const float* __restrict__ corr_bias, int T, int E, int G,
    int kG, int k, float scale, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sb[kMaxE], ss[kMaxE], sg[kMaxG];
  __shared__ int kept[kMaxG];
  __shared__ int sel_i[kMaxK];
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float z = logits[size_t(t) * E + e];
    const float sv = 1.0f / (1.0f + expf(-z));
    ss[e] = sv;
    sb[e] = sv + corr_bias[e];
  }
  __syncthreads();
  const int per = E / G;
  if (threadIdx.x < G) {
    float m1 = -INFINITY, m2 = -INFINITY;
    for (int j = 0; j < per; ++j) {
      const float v = sb[threadIdx.x * per + j];
      if (v > m1) { m2 = m1; m1 = v; } else if (v > m2) { m2 = v; }
    }
    sg[threadIdx.x] = m1 + m2;
  }
  __syncthreads();
  if (warp != 0) return;
  // kG best groups, listed in increasing group order
  unsigned keep = 0u;
  for (int r = 0; r < kG; ++r) {
    float v = (lane < G && !((keep >> lane) & 1u)) ? sg[lane] : -INFINITY;
    int i = lane < G ? lane : 0x7fffffff;
    warp_argmax(v, i);
    keep |= 1u << i;
  }
  if (lane == 0) {
    int n = 0;
    for (int g = 0; g < G; ++g)
      if ((keep >> g) & 1u) kept[n++] = g;
  }
  __syncwarp();
  // candidates c = lane + 32 j over the kept groups' experts
  const int ncand = kG * per;
  unsigned taken = 0u;
  for (int r = 0; r < k; ++r) {
    float v = -INFINITY;
    int best = 0x7fffffff;
    for (int j = 0; lane + 32 * j < ncand; ++j) {
      if ((taken >> j) & 1u) continue;
      const int c = lane + 32 * j;
      const int e = kept[c / per] * per + c % per;
      const float be = sb[e];
      if (be > v || (be == v && e < best)) { v = be; best = e; }
    }
    warp_argmax(v, best);
    for (int j = 0; lane + 32 * j < ncand; ++j) {
      const int c = lane + 32 * j;
      if (kept[c / per] * per + c % per == best) taken |= 1u << j;
    }
    if (lane == 0) sel_i[r] = best;
  }
  __syncwarp();
  if (lane < k) {
    float ssum = 0.f;
    for (int r = 0; r < k; ++r) ssum += ss[sel_i[r]];   // selection order, as every lane
    const int e = sel_i[lane];
    topk_idx[size_t(t) * k + lane] = e;
    topk_w[size_t(t) * k + lane] = ss[e] / ssum * scale;
  }
}

// Warp per token (8 tokens per CTA), every decision in registers. Lane l holds experts
// [l*EPL, (l+1)*EPL); a group of `per` experts spans LPG = per/EPL lanes (a power of two), so
// the group's top-2 merges across those lanes with xor shuffles. Every lane then sees all G
// group scores and ranks its own group; the k experts are taken in k rounds of a warp argmax
// over each lane's best remaining candidate. Same arithmetic and tie rules as
// router_topk_kernel (sigmoid via expf, group score m1 + m2, ties to the lower index,
// weights s / sum(s in selection order) * scale).
template <int EPL>
__global__ void __launch_bounds__(256) router_topk_warp_kernel(
    const float* __restrict__ logits, const float* __restrict__ corr_bias, int T, int E, int G,
    int LPG, int kG, int k, float scale, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int e0 = lane * EPL;
  const bool active = e0 < E;
  float b[EPL], sv[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const float z = active ? logits[size_t(t) * E + e0 + j] : 0.f;
    sv[j] = 1.0f / (1.0f + expf(-z));
    b[j] = active ? sv[j] + corr_bias[e0 + j] : -INFINITY;
  }
  // group score: the two largest b of the group (equal values count twice)
  float m1 = -INFINITY, m2 = -INFINITY;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    if (b[j] > m1) { m2 = m1; m1 = b[j]; } else if (b[j] > m2) { m2 = b[j]; }
  }
  for (int o = 1; o < LPG; o <<= 1) {
    const float o1 = __shfl_xor_sync(0xffffffffu, m1, o);
    const float o2 = __shfl_xor_sync(0xffffffffu, m2, o);
    const float hi = fmaxf(m1, o1), lo = fmaxf(fminf(m1, o1), fmaxf(m2, o2));
    m1 = hi;
    m2 = lo;
  }
  const float gs = m1 + m2;
  // rank of this lane's group among the G groups (ties to the lower group index)
  const int my_g = lane / LPG;
  int rank = 0;
  for (int g = 0; g < G; ++g) {
    const float o = __shfl_sync(0xffffffffu, gs, g * LPG);
    rank += (o > gs || (o == gs && g < my_g)) ? 1 : 0;
  }
  const bool kept = active && rank < kG;
  unsigned taken = kept ? 0u : 0xffffffffu;
  int sel_e = 0;
  float sel_s = 0.f;
  for (int r = 0; r < k; ++r) {
    float v = -INFINITY, vs = 0.f;
    int best = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      if (!((taken >> j) & 1u) && (b[j] > v || best == 0x7fffffff)) {
        v = b[j];
        vs = sv[j];
        best = e0 + j;
      }
    }
    const int mine = best;
    warp_argmax(v, best);
    const float s_best = __shfl_sync(0xffffffffu, vs, best / EPL);
    if (mine == best) taken |= 1u << (best - e0);
    if (lane == r) { sel_e = best; sel_s = s_best; }
  }
  float ssum = 0.f;
  for (int r = 0; r < k; ++r) ssum += __shfl_sync(0xffffffffu, sel_s, r);   // selection order
  if (lane < k) {
    topk_idx[size_t(t) * k + lane] = sel_e;
    topk_w[size_t(t) * k + lane] = sel_s / ssum * scale;
  }
}

// Experts per lane for the warp-per-token top-k, or 0 when the shape does not fit it.
int topk_epl(int E, int G, int k) {
  const int per = E / G;
  if (k > 32) return 0;
  for (int epl = 1; epl <= 16; epl <<= 1) {
    if (E > 32 * epl || per % epl != 0) continue;
    const int lpg = per / epl;
    if ((lpg & (lpg - 1)) != 0 || lpg > 32) return 0;
    return epl;
  }
  return 0;
}

beam_status launch_topk(const beam_layer_cfg* cfg, const float* lg, const float* corr_bias,
                        int T, int32_t* topk_idx, float* topk_w, cudaStream_t st) {
  const int E = cfg->n_experts, G = cfg->n_groups;
  const int epl = topk_epl(E, G, cfg->topk);
  const dim3 grid((T + 7) / 8), block(256);
  const int lpg = epl > 0 ? E / G / epl : 0;
  switch (epl) {
    case 1: launch_pdl(router_topk_warp_kernel<1>, grid, block, 0, st, lg, corr_bias, T, E, G, lpg, cfg->topk_groups, cfg->topk, cfg->route_scale, topk_idx, topk_w); break;
    case 2: launch_pdl(router_topk_warp_kernel<2>, grid, block, 0, st, lg, corr_bias, T, E, G, lpg, cfg->topk_groups, cfg->topk, cfg->route_scale, topk_idx, topk_w); break;
    case 4: launch_pdl(router_topk_warp_kernel<4>, grid, block, 0, st, lg, corr_bias, T, E, G, lpg, cfg->topk_groups, cfg->topk, cfg->route_scale, topk_idx, topk_w); break;
    case 8: launch_pdl(router_topk_warp_kernel<8>, grid, block, 0, st, lg, corr_bias, T, E, G, lpg, cfg->topk_groups, cfg->topk, cfg->route_scale, topk_idx, topk_w); break;
    case 16: launch_pdl(router_topk_warp_kernel<16>, grid, block, 0, st, lg, corr_bias, T, E, G, lpg, cfg->topk_groups, cfg->topk, cfg->route_scale, topk_idx, topk_w); break;
    default:
      router_topk_kernel<<<T, kTopkThreads, 0, st>>>(lg, corr_bias, T, E, G, cfg->topk_groups,
                                                      cfg->topk, cfg->route_scale, topk_idx,
                                                      topk_w);
      note_launches(1);
  }
  return launch_status();
}

// logits[T][E] = float(u) . w_router^T
beam_status launch_logits(const uint16_t* u, const float* w_router, int T, int H, int E,
                          float* lg, cudaStream_t st) {
  if (T <= kRouteGemvMaxT)
    launch_pdl(router_gemv_kernel, dim3(E), dim3(256), 0, st, u, w_router, T, H, E, lg);
  else
    launch_pdl(router_gemm_kernel<64, 4>, dim3((E + 63) / 64, (T + 63) / 64), dim3(256), 0, st,
               u, w_router, T, H, E, lg);
  return launch_status();
}

}  // namespace

size_t route_ws_bytes(const beam_layer_cfg* c, int T) {
  size_t b = align_up(size_t(T) * c->n_experts * sizeof(float), 256);
  if (T >= kRouteTcMinT)
    b += align_up(size_t(3) * c->n_experts * c->hidden * 2, 256) +
         align_up(size_t(T) * 3 * c->n_experts * sizeof(float), 256);
  return b;
}

}  // namespace beam

extern "C" beam_status beam_route(const beam_layer_cfg* cfg, const beam_bf16* u,
                                  const float* w_router, const float* corr_bias, int T,
                                  float* logits, int32_t* topk_idx, float* topk_w, void* ws,
                                  size_t ws_bytes, beam_stream_t stream) {
  using namespace beam;
  if (!cfg || T < 0 || !u || !w_router || !corr_bias || !topk_idx || !topk_w)
    return BEAM_ERR_INVALID_ARG;
  const int E = cfg->n_experts, G = cfg->n_groups, H = cfg->hidden;
  if (H <= 0 || (H & 7) || E <= 0 || G <= 0 || E % G != 0 || cfg->topk_groups < 1 ||
      cfg->topk_groups > G || cfg->topk < 1 || cfg->topk > cfg->topk_groups * (E / G) ||
      E / G < 2)
    return BEAM_ERR_INVALID_ARG;
  if (E > kMaxE || G > kMaxG || cfg->topk > kMaxK) return BEAM_ERR_UNSUPPORTED;
  if (!aligned16(u) || !aligned16(w_router) || !aligned16_or_null(logits) || !aligned16(ws))
    return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  Carver cv{static_cast<char*>(ws), ws_bytes};
  float* lg = logits;
  if (lg == nullptr) lg = cv.take<float>(size_t(T) * E);
  if (!cv.ok) return BEAM_ERR_INVALID_ARG;
  if (T >= kRouteTcMinT && tc::gemm_supported(u, H, u, H, H)) {
    const size_t n = size_t(E) * H;
    uint16_t* w3 = cv.take<uint16_t>(3 * n);
    float* c3 = cv.take<float>(size_t(T) * 3 * E);
    if (!cv.ok) return BEAM_ERR_INVALID_ARG;
    launch_pdl(router_split_kernel, dim3(unsigned((n + 255) / 256)), dim3(256), 0, st, w_router, n, w3);
    // the tensor pipe's FP32 accumulation loses about 2^-24 of the running sum per K step of
    // 16, so the reduction runs as kRouteKChunks chains summed in FP32 memory
    const int kc = (H % (8 * kRouteKChunks) == 0) ? H / kRouteKChunks : H;
    for (int k0 = 0; k0 < H; k0 += kc) {
      if (const cudaError_t e = tc::gemm_f32_acc(u + k0, T, kc, H, w3 + k0, 3 * E, H, c3, 3 * E,
                                                 k0 > 0, st);
          e != cudaSuccess)
        return cuda_status(e);
    }
    const size_t nl = size_t(T) * E;
    launch_pdl(router_sum3_kernel, dim3(unsigned((nl + 255) / 256)), dim3(256), 0, st, c3, T, E, lg);
    return launch_topk(cfg, lg, corr_bias, T, topk_idx, topk_w, st);
  }
  const beam_status ls = launch_logits(u, w_router, T, H, E, lg, st);
  if (ls != BEAM_OK) return ls;
  return launch_topk(cfg, lg, corr_bias, T, topk_idx, topk_w, st);
}

// ------------------------------------------------------------------------------------------
// Allocation-free router
//
// Some callers cannot hand the library any scratch memory: a serving engine that has given all
// free device memory to its KV-cache pool, or a runtime whose device memory is partitioned up
// front and that may not call cudaMalloc (or any allocating library) afterwards. For them the
// router's one piece of scratch -- the FP32 logits when the caller does not want them back --
// lives in a fixed array in the library's own device memory instead of a caller workspace.
// ------------------------------------------------------------------------------------------
namespace beam {
namespace {

// Logits scratch of the allocation-free router: 65536 floats (256 KiB), i.e. up to
// T * n_experts <= 65536 (256 tokens at 256 experts). Every GPU that loads the library holds
// one copy of it until the process exits.
constexpr int kNoAllocLogits = 65536;
static __device__ __align__(256) float g_route_scratch[kNoAllocLogits];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_dev[kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device, with that device
// current, and cached for the life of the process (the device's primary context is assumed
// to live as long: after a cudaDeviceReset the cached address would be stale).
float* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_dev[dev] = static_cast<float*>(p);
  }
  return g_scratch_dev[dev];
}

}  // namespace
}  // namespace beam

extern "C" beam_status beam_route_noalloc(const beam_layer_cfg* cfg, const beam_bf16* u,
                                          const float* w_router, const float* corr_bias, int T,
                                          int32_t* topk_idx, float* topk_w,
                                          beam_stream_t stream) {
  using namespace beam;
  if (!cfg || T < 0 || !u || !w_router || !corr_bias || !topk_idx || !topk_w)
    return BEAM_ERR_INVALID_ARG;
  const int E = cfg->n_experts, G = cfg->n_groups, H = cfg->hidden;
  if (H <= 0 || (H & 7) || E <= 0 || G <= 0 || E % G != 0 || cfg->topk_groups < 1 ||
      cfg->topk_groups > G || cfg->topk < 1 || cfg->topk > cfg->topk_groups * (E / G) ||
      E / G < 2)
    return BEAM_ERR_INVALID_ARG;
  if (E > kMaxE || G > kMaxG || cfg->topk > kMaxK) return BEAM_ERR_UNSUPPORTED;
  // beyond kRouteGemvMaxT tokens beam_route takes its tensor-core form, which needs
  // workspace; the allocation-free call stays within the range where both run the GEMV
  if (T > kRouteGemvMaxT || size_t(T) * size_t(E) > size_t(kNoAllocLogits))
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_router)) return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  float* lg = scratch_on_current_device();
  if (lg == nullptr) return BEAM_ERR_CUDA;
  // the GEMV/GEMM writes every logit of the T x E block before the top-k reads it, so the
  // scratch needs no clearing between calls
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const beam_status ls = launch_logits(u, w_router, T, H, E, lg, st);
  if (ls != BEAM_OK) return ls;
  return launch_topk(cfg, lg, corr_bias, T, topk_idx, topk_w, st);
}
