// Blackwell (sm_103a) building blocks shared by the tensor-core kernels: mbarriers with bounded
// waits, TMA tile loads, UMMA shared-memory and instruction descriptors, tcgen05.mma with the A
// operand in shared or tensor memory, and tensor-memory loads and stores.
//
// Descriptor and fragment formats follow the PTX ISA (tcgen05 "Shared memory descriptor",
// "Instruction descriptor" for kind::f16, and the 32x32b tensor-memory access shape, in which
// thread i of a warp reads or writes TMEM lane (32 * (warp % 4) + i)).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace beam {
namespace tc {

constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase (try_wait may suspend the thread while the phase is pending).
__device__ __forceinline__ bool mbar_test(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after kWaitLimit polls (each poll may suspend the thread briefly).
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try(a, parity)) return true;
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(mbar)
      : "memory");
}

// Generic-proxy shared-memory writes made visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle. K-major operand: 8-row groups of 128 B
// stacked at 1024 B (stride byte offset); the leading byte offset is unused.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(1) << 16;             // leading byte offset (ignored), 16 B units
  d |= uint64_t(1024 >> 4) << 32;     // stride byte offset, 16 B units
  d |= uint64_t(1) << 46;             // descriptor version for tcgen05
  d |= uint64_t(2) << 61;             // swizzle: 128 B
  return d;
}
// MN-major operand, 128-byte swizzle: a 128 B row holds 64 consecutive MN elements of one K
// index; 8 K rows form a 1024 B atom. lbo = byte distance between 64-element MN blocks,
// sbo = byte distance between 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with BF16 A and B, FP32 D, shape M x N; b_mn: B is
// MN-major (A is always K-major here).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Whole-warp forms: every lane of a converged warp executes the call with the same values and
// elect.sync picks the one lane (lane 0) that issues the operation. Measured against issuing
// from a lane-0 branch: the full-size NoPE prefill attention 48.9 -> 47.0 ms, same output.
// Commits must come from the lane that issued the MMAs, which elect.sync keeps the same.
// D[tmem] (+)= A[smem] . B[smem], each descriptor passed as its two 32-bit words (callers that
// step through a tile change only the low word, the start address field); acc = 0 overwrites D.
__device__ __forceinline__ void umma_ss_e(uint32_t tmem_d, uint32_t a_lo, uint32_t a_hi,
                                          uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; .reg .b64 ad, bd; elect.sync _|e, 0xffffffff; setp.ne.b32 p, %6, 0;"
      " mov.b64 ad, {%1, %2}; mov.b64 bd, {%3, %4};"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p; }" ::"r"(tmem_d),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem], the B descriptor as its two 32-bit words.
__device__ __forceinline__ void umma_ts_e(uint32_t tmem_d, uint32_t tmem_a, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p, e; .reg .b64 bd; elect.sync _|e, 0xffffffff; setp.ne.b32 p, %5, 0;"
      " mov.b64 bd, {%2, %3}; @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p; }"
      ::"r"(tmem_d), "r"(tmem_a), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation issued so far by the elected lane completes.
__device__ __forceinline__ void umma_commit_e(uint32_t mbar) {
  asm volatile(
      "{ .reg .pred e; elect.sync _|e, 0xffffffff;"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }" ::"r"(mbar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 consecutive columns of this thread's lane, without waiting (see tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// Host: cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
bool tensor_map_encoder_ready();
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swz);

}  // namespace tc
}  // namespace beam
