// Exact widening of shifted int8 / uint8 values to fp16, shared by the operand
// pre-pass, the integer convolution's pre-pass, the fused kernel and the integer
// GEMM that converts its own operands.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace igc {
namespace prepass {

// Four packed bytes to four exact fp16 values, two per 32-bit word (byte order
// kept).  u = byte (uint8) or byte with its top bit flipped (int8: flip =
// 0x80808080, so u = value + 128); placed in the low mantissa byte of 0x6400,
// u reads as the fp16 number 1024 + u, and subtracting 1152 = 1024 + 128 leaves
// u - 128 exactly (|u - 128| <= 128).  usum += the sum of the four u.
static __device__ __forceinline__ void widen4(uint32_t word, uint32_t flip, uint32_t& lo,
                                              uint32_t& hi, uint32_t& usum) {
  const uint32_t u = word ^ flip;
  usum = __dp4a(u, 0x01010101u, usum);
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // (1024 + u0, 1024 + u1)
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);  // (1024 + u2, 1024 + u3)
  const __half2 k1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 ra = __hsub2(*reinterpret_cast<const __half2*>(&a), k1152);
  const __half2 rb = __hsub2(*reinterpret_cast<const __half2*>(&b), k1152);
  lo = *reinterpret_cast<const uint32_t*>(&ra);
  hi = *reinterpret_cast<const uint32_t*>(&rb);
}

}  // namespace prepass
}  // namespace igc
