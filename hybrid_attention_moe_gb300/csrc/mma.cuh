// Warp-level tensor-core tiles (mma.sync m16n8k16 bf16 -> fp32), ldmatrix and cp.async helpers
// for the attention kernels. Fragment layouts (PTX ISA, "Matrix fragments for mma.m16n8k16"):
// with g = lane/4 and c = lane%4,
//   A (16x16, row): a0 (g, 2c..2c+1)  a1 (g+8, 2c..)  a2 (g, 2c+8..)  a3 (g+8, 2c+8..)
//   B (16x8, col) : b0 (k 2c..2c+1, n g)  b1 (k 2c+8.., n g)
//   C (16x8)      : c0,c1 (g, 2c..2c+1)  c2,c3 (g+8, 2c..2c+1)
#pragma once

#include <stdint.h>

namespace beam {

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// 16-byte async copy global -> shared; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two e4m3 codes (low byte first) -> two bf16 in one word; exact (every e4m3 value is a bf16).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t codes) {
  uint32_t h2;
  asm("{.reg .b16 c; mov.b16 c, %1; cvt.rn.f16x2.e4m3x2 %0, c;}" : "=r"(h2) : "h"(codes));
  float lo, hi;
  asm("{.reg .f16 a, b; mov.b32 {a, b}, %2; cvt.f32.f16 %0, a; cvt.f32.f16 %1, b;}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return pack_bf16x2(lo, hi);
}

// Byte offset of 16-byte chunk `ch` of row `row` in a tile of rows of `row_bytes`, with the
// chunk index XOR-swizzled by the row so ldmatrix reads of 8 rows hit 8 different bank groups.
__device__ __forceinline__ uint32_t swz(int row, int ch, int row_bytes) {
  return uint32_t(row * row_bytes + ((ch ^ (row & 7)) << 4));
}

}  // namespace beam
