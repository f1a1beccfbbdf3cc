// codes.cuh -- number formats shared by the index and compression kernels:
// bfloat16 rounding, exact powers of two, binary exponents and the OCP E2M1
// magnitude grid (0, 0.5, 1, 1.5, 2, 3, 4, 6).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace sa {

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// 2^e as binary32 for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

// floor(log2(m)) of a positive finite binary32 value.
__device__ __forceinline__ int floor_log2(float m) {
  const uint32_t u = __float_as_uint(m);
  const int ex = static_cast<int>((u >> 23) & 0xffu);
  if (ex) return ex - 127;
  return (31 - __clz(u & 0x7fffffu)) - 149;
}

// 2 * (nearest E2M1 magnitude to v >= 0), ties to the even code, saturating at 6.
__device__ __forceinline__ int e2m1_twice(float v) {
  if (v <= 0.25f) return 0;
  if (v < 0.75f) return 1;
  if (v <= 1.25f) return 2;
  if (v < 1.75f) return 3;
  if (v <= 2.5f) return 4;
  if (v < 3.5f) return 6;
  if (v <= 5.0f) return 8;
  return 12;
}


// E2M1 magnitude code (0..7) of a value returned by e2m1_twice.
__device__ __forceinline__ int e2m1_code(int twice) {
  return twice <= 4 ? twice : (twice == 6 ? 5 : (twice == 8 ? 6 : 7));
}

}  // namespace sa
