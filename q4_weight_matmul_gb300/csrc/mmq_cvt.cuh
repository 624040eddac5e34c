// Register-level conversions shared by the tensor-core GEMMs: BLOCK144
// header fields, and quant bytes widened to the fp16 B operand sc*q.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace q4k {
namespace cvt {

// One word of quant bytes (weights l..l+3 of the low sub-block in the low
// nibbles, of the high sub-block in the high nibbles) -> sc*q fp16 pairs in
// k order: (l, l+1), (l+2, l+3) of the low sub-block in lo0/lo1, of the high
// sub-block in hi0/hi1.  Bytes go under the fp16 exponent of 1024 (low
// nibble as 1024+q, high nibble as 1024+16q); one exact FMA removes the bias
// and applies sc.
__device__ __forceinline__ void cvt_q4x8(uint32_t w, uint32_t mlo, uint32_t alo, uint32_t mhi,
                                         uint32_t ahi, uint32_t& lo0, uint32_t& lo1, uint32_t& hi0,
                                         uint32_t& hi1) {
  asm("{\n\t.reg .b32 t01, t23, z;\n\tmov.b32 z, 0;\n\t"
      "prmt.b32 t01, %4, z, 0x4140;\n\tprmt.b32 t23, %4, z, 0x4342;\n\t"
      "lop3.b32 %0, t01, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 %1, t23, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 %2, t01, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "lop3.b32 %3, t23, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "fma.rn.f16x2 %0, %0, %5, %6;\n\tfma.rn.f16x2 %1, %1, %5, %6;\n\t"
      "fma.rn.f16x2 %2, %2, %7, %8;\n\tfma.rn.f16x2 %3, %3, %7, %8;\n\t}"
      : "=r"(lo0), "=r"(lo1), "=r"(hi0), "=r"(hi1)
      : "r"(w), "r"(mlo), "r"(alo), "r"(mhi), "r"(ahi));
}

// fp16x2 (byte b0 of w, byte b1 of w), each an integer 0..255 (exact): each
// byte under the exponent of 1024, minus 1024
__device__ __forceinline__ uint32_t bytes_h2(uint32_t w, uint32_t b0, uint32_t b1) {
  const uint32_t sel = b0 | 0x40u | (b1 << 8) | 0x4000u;   // bytes [b0, 0, b1, 0]
  uint32_t r;
  asm("{\n\t.reg .b32 t, z, k;\n\tmov.b32 z, 0;\n\tmov.b32 k, 0x64006400;\n\t"
      "prmt.b32 t, %1, z, %2;\n\tor.b32 t, t, k;\n\tsub.rn.f16x2 %0, t, k;\n\t}"
      : "=r"(r) : "r"(w), "r"(sel));
  return r;
}

// fp16x2 (v, v) of byte `bi` of w
__device__ __forceinline__ uint32_t byte_h2(uint32_t w, uint32_t bi) { return bytes_h2(w, bi, bi); }

__device__ __forceinline__ uint32_t mul_h2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// packed 6-bit scales / mins of sub-blocks 0..3 and 4..7 of a header
__device__ __forceinline__ void header_sc_m(const uint4& h, uint32_t& sc03, uint32_t& sc47, uint32_t& m03,
                                            uint32_t& m47) {
  sc03 = h.y & 0x3F3F3F3Fu;
  m03 = h.z & 0x3F3F3F3Fu;
  sc47 = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
  m47 = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
}

}  // namespace cvt
}  // namespace q4k
