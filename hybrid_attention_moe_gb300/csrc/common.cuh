// Shared device helpers for the Beam layer kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/beam.h"

namespace beam {

// Status word of the device (BEAM_DEV_* bits). Defined once in misc.cu.
extern __device__ unsigned int g_dev_status;

__device__ __forceinline__ void flag(unsigned int bit) { atomicOr(&g_dev_status, bit); }

// ---- bf16 <-> fp32 ------------------------------------------------------------------
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ float bflo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bfhi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float round_bf(float f) { return bf2f(f2bf(f)); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return uint32_t(f2bf(lo)) | (uint32_t(f2bf(hi)) << 16);
}

// 8 bf16 held in a uint4 -> 8 floats
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  f[0] = bflo(v.x); f[1] = bfhi(v.x); f[2] = bflo(v.y); f[3] = bfhi(v.y);
  f[4] = bflo(v.z); f[5] = bfhi(v.z); f[6] = bflo(v.w); f[7] = bfhi(v.w);
}

// acc + w.lo * x.lo, then + w.hi * x.hi, for two bf16 pairs packed in 32-bit words. Each step
// is one mixed-precision FMA (fma.rn.f32.bf16: the bf16 operands widen exactly, the product
// and the sum are rounded once to FP32), so the result equals
// fmaf(bfhi(w), bfhi(x), fmaf(bflo(w), bflo(x), acc)) without the two unpacking instructions
// per element that the FP32 form spends.
__device__ __forceinline__ float fma_bf16x2(uint32_t w, uint32_t x, float acc) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(x));
  return acc;
}

// Streaming 16-byte load that does not allocate in L1 (weights are read once per call).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ float4 ld_stream_f4(const void* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// ---- reductions -----------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the block; every thread gets the result. `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float s = lane < nw ? red[lane] : 0.f;
  s = warp_sum(s);
  return s;
}

// Programmatic dependent launch: allow the next kernel to be scheduled; wait until every
// predecessor's results are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16). Used before pdl_wait
// on weights, which no kernel writes, so their stream starts while the predecessor finishes.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + __expf(-z)); }

// SSMax query scale (1 + p / base)^e in FP32 (GB300's FP64 rate is a small fraction of FP32,
// and a double pow cost several microseconds in a one-thread prologue): 1 + p / base is exact
// for base a power of two and p < 2^23, and log2 / exp2 keep the relative error near 1e-7.
__device__ __forceinline__ float ssmax_scale(int p, float base, float e) {
  return exp2f(e * log2f(1.f + float(p) / base));
}
// RoPE angle (p - 1) * inv reduced into about [-pi, pi]: the product in double (positions
// near 1e5 need more than FP32's 24 bits), the reduction by a multiply with 1 / (2 pi) rather
// than a double division (any integer multiple of 2 pi may be removed; the error of the
// removed multiple stays near 1e-11 rad).
__device__ __forceinline__ float rope_angle(int p, double inv) {
  double ang = double(p - 1) * inv;
  constexpr double kTwoPi = 6.283185307179586476925, kInvTwoPi = 0.15915494309189533576888;
  ang = fma(-kTwoPi, rint(ang * kInvTwoPi), ang);
  return float(ang);
}
__device__ __forceinline__ float siluf_(float z) { return z / (1.0f + __expf(-z)); }

// ---- host-side argument checks ------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned16_or_null(const void* p) { return p == nullptr || aligned16(p); }

// Host-side count of kernel launches (misc.cu).
void note_launches(int n);

// Number of SMs of the current device (queried once).
int num_sms_cached();

// Launch with programmatic stream serialization: the kernel may start while its predecessor
// in the stream finishes; it must execute griddepcontrol.wait (pdl_wait) before reading or
// writing anything a predecessor touches. Kernels launched this way all begin with
// pdl_trigger(), so their own successors can be scheduled as their CTAs drain.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// launch_pdl for a kernel whose grid is tiled by thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t st, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = unsigned(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Records the CUDA error behind a BEAM_ERR_CUDA for beam_last_cuda_error (per host thread).
void note_cuda_error(cudaError_t e);

inline beam_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BEAM_OK;
  note_cuda_error(e);
  return BEAM_ERR_CUDA;
}

inline beam_status launch_status() { return cuda_status(cudaGetLastError()); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carves 256-byte aligned regions out of the caller's workspace.
struct Carver {
  char* base;
  size_t cap;
  size_t off = 0;
  bool ok = true;
  template <class T>
  T* take(size_t count) {
    size_t o = align_up(off, 256);
    size_t bytes = count * sizeof(T);
    if (o + bytes > cap) { ok = false; return nullptr; }
    off = o + bytes;
    return reinterpret_cast<T*>(base + o);
  }
};

}  // namespace beam

namespace beam {

// Token count from which the projections run on the tensor-core GEMM instead of the
// weight-streaming GEMV (below it the weights' HBM read dominates and the GEMV is at roofline).
constexpr int kGemmMinT = 64;

// Attention widths this build compiles for.
inline bool head_dim_ok(int D) { return D == 64 || D == 128; }

inline beam_status check_cfg_attn(const beam_layer_cfg* c) {
  if (c == nullptr) return BEAM_ERR_INVALID_ARG;
  if (c->hidden <= 0 || (c->hidden & 7) || c->n_q <= 0 || c->n_kv <= 0 ||
      c->n_q % c->n_kv != 0 || c->head_dim <= 0 ||
      (c->kind != BEAM_ATTN_SWA_ROPE && c->kind != BEAM_ATTN_NOPE_SSMAX) || !(c->eps >= 0.f))
    return BEAM_ERR_INVALID_ARG;
  if (!head_dim_ok(c->head_dim)) return BEAM_ERR_UNSUPPORTED;
  if (c->n_q / c->n_kv > 16) return BEAM_ERR_UNSUPPORTED;
  return BEAM_OK;
}

inline beam_status check_cache(const beam_kv_cache* kc, const beam_layer_cfg* c) {
  if (kc == nullptr || kc->k == nullptr || kc->v == nullptr || kc->num_seqs <= 0 ||
      kc->capacity <= 0 || kc->window < 0)
    return BEAM_ERR_INVALID_ARG;
  if (kc->dtype != BEAM_KV_BF16 && kc->dtype != BEAM_KV_FP8_E4M3) return BEAM_ERR_INVALID_ARG;
  if (kc->dtype == BEAM_KV_FP8_E4M3 && !(kc->k_scale > 0.f && kc->v_scale > 0.f))
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(kc->k) || !aligned16(kc->v)) return BEAM_ERR_INVALID_ARG;
  if (kc->window > 0 && kc->capacity < kc->window) return BEAM_ERR_INVALID_ARG;
  (void)c;
  return BEAM_OK;
}

}  // namespace beam
