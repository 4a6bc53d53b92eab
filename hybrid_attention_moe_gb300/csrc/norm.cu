// Sublayer boundary: post-norm, depth-scaled residual, next pre-norm in one pass.
// Beam page, "MoE and residual stream" section (sandwich RMSNorm; h <- sqrt((n-1)/n) h + x/sqrt(n))
// and change 1 of the optimisation list (one kernel per boundary, FP32 math, BF16 storage).
#include <math.h>

#include "common.cuh"

namespace beam {
namespace {

constexpr int kNormMaxVec = 4;  // 16-byte vectors held per thread

// One CTA per token row. Each thread holds up to kNormMaxVec 16-byte vectors of every input;
// all loads are issued up front (the gains before the programmatic-launch wait, since no
// kernel writes them), so the row costs one memory round trip plus two block reductions.
__global__ void __launch_bounds__(512) boundary_norm_kernel(
    const uint16_t* __restrict__ x, uint16_t* __restrict__ h, uint16_t* __restrict__ u_out,
    const uint16_t* __restrict__ w_post, const uint16_t* __restrict__ w_pre, int H,
    float c_keep, float c_add, float eps) {
  pdl_trigger();
  __shared__ float red[32];
  const int nvec = H >> 3;
  const size_t row = size_t(blockIdx.x) * H;
  uint4 wpo[kNormMaxVec], wpr[kNormMaxVec], xr[kNormMaxVec], hr[kNormMaxVec];
#pragma unroll
  for (int j = 0; j < kNormMaxVec; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nvec) {
      if (x != nullptr) wpo[j] = __ldg(reinterpret_cast<const uint4*>(w_post) + i);
      if (u_out != nullptr) wpr[j] = __ldg(reinterpret_cast<const uint4*>(w_pre) + i);
    }
  }
  pdl_wait();
#pragma unroll
  for (int j = 0; j < kNormMaxVec; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    if (i < nvec) {
      hr[j] = *reinterpret_cast<const uint4*>(h + row + size_t(i) * 8);
      if (x != nullptr) xr[j] = *reinterpret_cast<const uint4*>(x + row + size_t(i) * 8);
    }
  }
  float hv[kNormMaxVec][8];
#pragma unroll
  for (int j = 0; j < kNormMaxVec; ++j)
    if (threadIdx.x + j * blockDim.x < nvec) unpack8(hr[j], hv[j]);

  if (x != nullptr) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kNormMaxVec; ++j) {
      if (threadIdx.x + j * blockDim.x < nvec) {
        float xv[8];
        unpack8(xr[j], xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(xv[e], xv[e], ss);
      }
    }
    const float r = rsqrtf(block_sum(ss, red) / float(H) + eps);
#pragma unroll
    for (int j = 0; j < kNormMaxVec; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      if (i < nvec) {
        float xv[8], wv[8];
        unpack8(xr[j], xv);
        unpack8(wpo[j], wv);
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float y = round_bf(xv[e] * r * wv[e]);                 // post-norm output (bf16)
          hv[j][e] = round_bf(fmaf(c_keep, hv[j][e], c_add * y));      // new residual (bf16)
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) packed[e] = pack_bf2(hv[j][2 * e], hv[j][2 * e + 1]);
        *reinterpret_cast<uint4*>(h + row + size_t(i) * 8) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    }
  }

  if (u_out != nullptr) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kNormMaxVec; ++j) {
      if (threadIdx.x + j * blockDim.x < nvec) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(hv[j][e], hv[j][e], ss);
      }
    }
    const float r = rsqrtf(block_sum(ss, red) / float(H) + eps);
#pragma unroll
    for (int j = 0; j < kNormMaxVec; ++j) {
      const int i = threadIdx.x + j * blockDim.x;
      if (i < nvec) {
        float wv[8];
        unpack8(wpr[j], wv);
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          packed[e] = pack_bf2(hv[j][2 * e] * r * wv[2 * e], hv[j][2 * e + 1] * r * wv[2 * e + 1]);
        *reinterpret_cast<uint4*>(u_out + row + size_t(i) * 8) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
    }
  }
}

}  // namespace
}  // namespace beam

extern "C" beam_status beam_boundary_norm(const beam_bf16* x, beam_bf16* h, beam_bf16* u_out,
                                          const beam_bf16* w_post, const beam_bf16* w_pre,
                                          int T, int H, int n, float eps,
                                          beam_stream_t stream) {
  using namespace beam;
  if (T < 0 || H <= 0 || (H & 7) || n < 1 || !(eps >= 0.f) || h == nullptr)
    return BEAM_ERR_INVALID_ARG;
  if (x != nullptr && w_post == nullptr) return BEAM_ERR_INVALID_ARG;
  if (u_out != nullptr && w_pre == nullptr) return BEAM_ERR_INVALID_ARG;
  if (!aligned16_or_null(x) || !aligned16(h) || !aligned16_or_null(u_out) ||
      !aligned16_or_null(w_post) || !aligned16_or_null(w_pre))
    return BEAM_ERR_INVALID_ARG;
  const int nvec = H / 8;
  int threads = (nvec + kNormMaxVec - 1) / kNormMaxVec;
  threads = (threads + 31) / 32 * 32;
  if (threads > 512) return BEAM_ERR_UNSUPPORTED;
  if (T == 0) return BEAM_OK;
  const double nd = double(n);
  const float c_keep = float(sqrt((nd - 1.0) / nd));
  const float c_add = float(1.0 / sqrt(nd));
  launch_pdl(boundary_norm_kernel, dim3(T), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream), 
      x, h, u_out, w_post, w_pre, H, c_keep, c_add, eps);
  return launch_status();
}
