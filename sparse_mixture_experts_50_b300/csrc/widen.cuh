// Exact widening of int8 weight codes to bf16 on the SM (the int8 weight-only
// experts: KerasFormers Mixtral docs, "Lower memory").  Every code lies in
// [-127, 127], which bf16 (8 significant bits) holds exactly.
#pragma once

#include <stdint.h>

#ifndef MOE_CVT_F32X2
#define MOE_CVT_F32X2 1
#endif

namespace moe {

// Four int8 codes (one 32-bit word, element 0 in the low byte) -> four bf16
// (two words: lo = elements 0, 1; hi = elements 2, 3; lower element in the
// low half).  Flipping the sign bit gives b + 128 in [0, 255] as an unsigned
// byte; placed in the low mantissa bits of the fp32 2^23 it is the fp32 value
// 2^23 + b + 128, and subtracting 2^23 + 128 leaves b exactly.  A value of at
// most 8 significant bits has zero low 16 bits in fp32, so its bf16 encoding
// is the high half of the fp32 word.
__device__ __forceinline__ void i8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
#if MOE_CVT_F32X2
  // The two subtractions of a pair as one packed fp32x2 add of -(2^23 + 128).
  constexpr unsigned long long kBias2 = 0xCB000080CB000080ull;
  unsigned long long p01 = (static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7541)) << 32) |
                           __byte_perm(u, 0x4B000000u, 0x7540);
  unsigned long long p23 = (static_cast<unsigned long long>(__byte_perm(u, 0x4B000000u, 0x7543)) << 32) |
                           __byte_perm(u, 0x4B000000u, 0x7542);
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(p01) : "l"(kBias2));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(p23) : "l"(kBias2));
  lo = __byte_perm(static_cast<uint32_t>(p01), static_cast<uint32_t>(p01 >> 32), 0x7632);
  hi = __byte_perm(static_cast<uint32_t>(p23), static_cast<uint32_t>(p23 >> 32), 0x7632);
#else
  constexpr float kBias = 8388736.0f;  // 2^23 + 128
  const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)) - kBias;
  const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541)) - kBias;
  const float f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)) - kBias;
  const float f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543)) - kBias;
  lo = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
  hi = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
#endif
}

}  // namespace moe
