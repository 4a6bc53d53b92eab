// Workspace sizing, cache sizing, device status word and status strings.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "tcgen05.cuh"

namespace beam {

__device__ unsigned int g_dev_status = 0u;

static std::atomic<unsigned long long> g_launches{0};

// SM count of the current device (cached per device).
int num_sms_cached() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 152;
  }
  return cache[dev];
}
void note_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }

static thread_local cudaError_t g_last_cuda_error = cudaSuccess;
void note_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

size_t qkv_ws_bytes(const beam_layer_cfg* c, int T);
size_t attn_ws_bytes(const beam_layer_cfg* c, int T, int max_pos, int window);
size_t route_ws_bytes(const beam_layer_cfg* c, int T);
size_t moe_ws_bytes(const beam_layer_cfg* c, int T);
size_t dense_ws_bytes(const beam_layer_cfg* c, int T);

}  // namespace beam

extern "C" size_t beam_workspace_bytes(const beam_layer_cfg* cfg, int T, int max_pos) {
  using namespace beam;
  if (cfg == nullptr || T <= 0) return 256;
  size_t b = qkv_ws_bytes(cfg, T);
  // the key split grows with the key count, so full attention bounds any window
  b = std::max(b, attn_ws_bytes(cfg, T, max_pos, 0));
  b = std::max(b, route_ws_bytes(cfg, T));
  b = std::max(b, moe_ws_bytes(cfg, T));
  b = std::max(b, dense_ws_bytes(cfg, T));
  return align_up(b, 256);
}

extern "C" size_t beam_kv_cache_bytes(int num_seqs, int n_kv, int capacity, int head_dim,
                                      int dtype) {
  if (num_seqs <= 0 || n_kv <= 0 || capacity <= 0 || head_dim <= 0) return 0;
  const size_t elem = dtype == BEAM_KV_FP8_E4M3 ? 1 : 2;
  return 2 * size_t(num_seqs) * n_kv * capacity * head_dim * elem;
}

extern "C" beam_status beam_get_device_status(beam_stream_t stream, uint32_t* bits) {
  if (bits == nullptr) return BEAM_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return BEAM_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, beam::g_dev_status, sizeof(v)) != cudaSuccess) return BEAM_ERR_CUDA;
  if (cudaMemcpyToSymbol(beam::g_dev_status, &zero, sizeof(zero)) != cudaSuccess)
    return BEAM_ERR_CUDA;
  *bits = v;
  return BEAM_OK;
}

extern "C" const char* beam_status_string(beam_status s) {
  switch (s) {
    case BEAM_OK: return "ok";
    case BEAM_ERR_INVALID_ARG: return "invalid argument";
    case BEAM_ERR_UNSUPPORTED: return "unsupported shape or option";
    case BEAM_ERR_CUDA: return "CUDA launch or runtime error";
    case BEAM_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

extern "C" uint64_t beam_launch_count(void) { return beam::g_launches.load(); }

extern "C" const char* beam_last_cuda_error(void) {
  return cudaGetErrorName(beam::g_last_cuda_error);
}

namespace beam {
namespace {
// One thread waits on a barrier that expects one arrival and never gets it.
__global__ void wait_timeout_selftest_kernel() {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  tc::mbar_init(a, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!tc::mbar_wait(a, 0)) flag(BEAM_DEV_TIMEOUT);
}
}  // namespace
}  // namespace beam

extern "C" beam_status beam_selftest_wait_timeout(beam_stream_t stream) {
  using namespace beam;
  wait_timeout_selftest_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
  note_launches(1);
  return launch_status();
}
