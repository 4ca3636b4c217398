// Device-side helpers shared by the W4A4 kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace w4a4 {

// fl32(1/sqrt(32)): the normalisation of the 32-point Walsh-Hadamard rotation.
__device__ __forceinline__ float c_h32() { return __uint_as_float(0x3E3504F3u); }

// ---------------------------------------------------------------------------
// int4 -> fp8 (e4m3) without a lookup table.
//
// The W4A4 product needs P = sum_j (q_w - 8) * q_a exactly, with both factors
// in -8..7.  In e4m3 (bias 7) the bytes 0x00..0x0F encode exactly b * 2^-9:
// exponent field 0 gives m * 2^-9 (subnormal), exponent field 1 gives
// (8 + m) * 2^-9.  So the sign-magnitude byte (v < 0 ? 0x80 : 0) | |v| is the
// e4m3 value v * 2^-9 for every |v| <= 15, and an fp8 tensor-core product of
// two such operands is (q_w - 8) * q_a * 2^-18, exact, with a 32-term sum of at
// most 2048 * 2^-18 that fp32 holds exactly.  The fold multiplies by 2^18 back
// (folded into the weight scale).
//
// x holds four bytes, each a 4-bit two's complement value in its low nibble
// (high nibble zero).  Returns the four e4m3 bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t s4x4_to_e4m3x4(uint32_t x) {
  // bit 3 of every byte moved to bit 7 (x's high nibbles are zero, so no byte
  // spills into the next), then prmt's sign-replicate selectors (8..11) give
  // 0xFF for negative bytes and 0x00 otherwise.
  const uint32_t neg = prmt(x << 4, 0u, 0xBA98u);
  // negative byte: 0x80 | (16 - x) = 0x90 - x (no borrow: every byte of x <= 15)
  const uint32_t mag = 0x90909090u - x;
  return (neg & mag) | (~neg & x);
}

// 8 packed activation nibbles (one 32-bit word of a block's 16 code bytes):
// lo = elements 4t..4t+3 of the block, hi = elements 16+4t..16+4t+3.
__device__ __forceinline__ void act_word_to_e4m3(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = s4x4_to_e4m3x4(w & 0x0F0F0F0Fu);
  hi = s4x4_to_e4m3x4((w >> 4) & 0x0F0F0F0Fu);
}

// 8 packed Q4_0 weight nibbles: code q stands for q - 8, and q ^ 8 read as a
// signed 4-bit value is exactly q - 8, so flip bit 3 of every nibble first.
__device__ __forceinline__ void q4_0_word_to_e4m3(uint32_t w, uint32_t& lo, uint32_t& hi) {
  act_word_to_e4m3(w ^ 0x88888888u, lo, hi);
}

// 2^18: undoes the 2^-9 * 2^-9 of the fp8 encoding above.
__device__ __forceinline__ float fp8_unscale() { return 262144.0f; }

// ---------------------------------------------------------------------------
// Round half away from zero to an integer-valued float.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float round_half_away(float v) { return roundf(v); }

}  // namespace w4a4
