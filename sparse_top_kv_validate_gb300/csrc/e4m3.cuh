// e4m3.cuh -- exact conversion of E4M3FN code pairs (OCP 8-bit floating
// point: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities,
// S.1111.111 is NaN).  Every E4M3 value is exactly representable in f16 and in
// f32, so the pair goes through one f16x2 conversion instruction
// (cvt.rn.f16x2.e4m3x2: the rounding mode cannot change an exact result) and
// then to f32.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace sa {

// Two codes (low byte first, in the low 16 bits) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tmov.b16 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h)
      : "h"(static_cast<uint16_t>(two)));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

}  // namespace sa
