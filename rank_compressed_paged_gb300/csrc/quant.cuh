// Conversions of quantized coefficient codes to fp16, shared by the decode kernels and the
// prefill's page-widening pass.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace rcp {

// Two 4-bit codes (one byte: the even coefficient in the low nibble, two's complement) times
// their group's scale, as an fp16 pair.  Each nibble n becomes the fp16 1024 + (n ^ 8)
// (exponent bits 0x6400 with n ^ 8 as the low mantissa bits), minus 1032 the signed code,
// exactly; the product with the scale rounds once.
__device__ __forceinline__ uint32_t int4x2_to_half2_bits(uint32_t byte, __half2 scale) {
  const uint32_t b = ((byte & 0xFu) | ((byte & 0xF0u) << 12)) ^ 0x64086408u;
  const __half2 code = __hsub2(*reinterpret_cast<const __half2*>(&b), __float2half2_rn(1032.f));
  const __half2 v = __hmul2(code, scale);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace rcp
