// LM head with the logit softcap (AREX feed article on vLLM's Day-0 support of
// Reflection-Beam-1.0, the paragraph on the output side): logits = c * tanh((u W^T) / c).
// The projection runs on the library's GEMV (few tokens) or tensor-core GEMM (64 tokens and
// more) with FP32 output; the cap is a separate elementwise pass over the logits, as the page's
// own dedicated softcap kernel is.
#include <math.h>

#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"

namespace beam {
namespace {

// z <- c * tanh(z / c) over n floats in place; z 16-byte aligned (float4 body, scalar tail).
__global__ void __launch_bounds__(256) softcap_kernel(float* __restrict__ z, size_t n, float c) {
  pdl_trigger();
  pdl_wait();
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  const size_t first = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t n4 = n / 4;
  float4* z4 = reinterpret_cast<float4*>(z);
  for (size_t i = first; i < n4; i += stride) {
    float4 v = z4[i];
    v.x = c * tanhf(v.x / c);
    v.y = c * tanhf(v.y / c);
    v.z = c * tanhf(v.z / c);
    v.w = c * tanhf(v.w / c);
    z4[i] = v;
  }
  for (size_t i = 4 * n4 + first; i < n; i += stride) z[i] = c * tanhf(z[i] / c);
}

}  // namespace
}  // namespace beam

extern "C" beam_status beam_lm_head(const beam_bf16* u, const beam_bf16* w_lm, int T, int H,
                                    int V, float softcap, float* logits, beam_stream_t stream) {
  using namespace beam;
  if (!u || !w_lm || !logits || T < 0 || H <= 0 || (H & 7) || V <= 0 || !(softcap == softcap))
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_lm) || !aligned16(logits)) return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = T >= kGemmMinT
                            ? tc::gemm_bf16(u, T, H, H, w_lm, V, H, logits, V, false, st)
                            : launch_gemv<kOutF32>(w_lm, V, H, u, T, logits, nullptr, V, st);
  if (e != cudaSuccess) return cuda_status(e);
  if (softcap > 0.f) {
    const size_t n = size_t(T) * size_t(V);
    const size_t blocks = (n / 4 + 255) / 256;
    const size_t cap = size_t(4) * num_sms_cached();
    launch_pdl(softcap_kernel, dim3(unsigned(blocks == 0 ? 1 : blocks < cap ? blocks : cap)),
               dim3(256), 0, st, logits, n, softcap);
  }
  return launch_status();
}
