// MXFP4 (OCP microscaling, e2m1 codes with one UE8M0 scale byte per 32)
// weights widened exactly to bf16 without a table: the tensor-core GEMM's
// converter (grouped_gemm.cu).  The matrix-vector decode kernels widen the
// same codes to fp32 by the hardware e2m1 -> f16 conversion instead; both
// give the exact values code * 2^(byte - 127).
#pragma once

#include "common.cuh"

namespace moe_mx {

MOE_DEVICE uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

MOE_DEVICE uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Multipliers that turn an e2m1 code placed in bf16 bits (below) into the
// weight code * 2^(s - 127) for the UE8M0 scale byte s: mul[0] = 2^(s - 1)
// and, where that exceeds the bf16 range (s > 128), 2^127 followed by
// mul[1] = 2^(s - 128).  Both replicated into the two bf16 lanes.
MOE_DEVICE void mx_multipliers(uint32_t s, uint32_t& m1, uint32_t& m2) {
  const uint32_t e1 = s <= 128u ? s + 126u : 254u;  // bf16 exponent field of mul[0]
  const uint32_t e2 = s <= 128u ? 127u : s - 1u;   // 1.0, or 2^(s - 128)
  m1 = (e1 << 7) * 0x10001u;
  m2 = (e2 << 7) * 0x10001u;
}

// Eight e2m1 codes of a word (element 2i in the low nibble of byte i) ->
// eight bf16 weights in element order.  A code (sign s, exponent e, mantissa
// m) written as the bf16 bits s<<15 | e<<7 | m<<6 is exactly the bf16 number
// code * 2^-126 (e = 0 is the bf16 subnormal 2^-127 = 0.5 * 2^-126), so one
// correctly rounded bf16 multiply by a power of two gives the weight exactly.
// Per pair: one byte permute spreads the two codes of byte i into the two
// 16-bit lanes (selector 8 copies the clear top bit of a nibble byte: a zero
// byte), one multiply by 2^6 + 2^12 puts the magnitude bits at 6..8 and the
// sign bit at 15 of each lane (the two shifted copies do not overlap), one
// mask keeps exactly those bits.
MOE_DEVICE void e2m1x8_to_bf16(uint32_t w, uint32_t m1, uint32_t m2, bool big, uint32_t* out) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = prmt(lo, hi, 0x8080u | (uint32_t)i | ((uint32_t)(4 + i) << 8));
    const uint32_t v = bf16x2_mul((x * 0x1040u) & 0x81C081C0u, m1);
    out[i] = big ? bf16x2_mul(v, m2) : v;
  }
}

}  // namespace moe_mx
