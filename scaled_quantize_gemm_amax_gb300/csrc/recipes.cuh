// recipes.cuh -- the scale rules of the four recipes, as device functions.
//
// Per-tensor / blockwise (Colossal-AI FP8 "current scaling"; FP8 quantized-training
// guide, "instant scaling scheme" and "block-level scaling"):
//   scale = FMAX / amax (one IEEE binary32 division, round to nearest),
//   scale_inv = 1 / scale; amax == 0 or non-finite -> scale 1; an overflowing
//   quotient -> FLT_MAX.
// MXFP8 (guide, "MXFP8 scaling": 1x32 blocks, E8M0 power-of-two scale):
//   e = smallest integer with amax <= FMAX * 2^e, clamped to [-127, 127],
//   amax == 0 or non-finite -> 0; elements are multiplied by 2^-e; byte = e + 127.
//   (Alternate, its own recipe: e = floor(log2 amax) - floor(log2 FMAX).)
// The cast is round-to-nearest-even with saturation to +-FMAX.
#pragma once
#include <cfloat>
#include <cstdint>

namespace fp8q {

__device__ __forceinline__ float fmax_of(bool e5m2) { return e5m2 ? 57344.0f : 448.0f; }
// FMAX = 1.75 * 2^fmax_exp
__device__ __forceinline__ int fmax_exp_of(bool e5m2) { return e5m2 ? 15 : 8; }

__device__ __forceinline__ bool is_inf_or_nan(float v) {
  return (__float_as_uint(v) & 0x7F800000u) == 0x7F800000u;
}

__device__ __forceinline__ float scale_from_amax(float amax, float fmax) {
  if (!(amax > 0.0f) || is_inf_or_nan(amax)) return 1.0f;
  float s = __fdiv_rn(fmax, amax);
  if (is_inf_or_nan(s)) s = FLT_MAX;
  return s;
}

__device__ __forceinline__ float recip_rn(float s) { return __fdiv_rn(1.0f, s); }

// Smallest e with amax <= 1.75 * 2^(fmax_exp + e): write amax = m * 2^E with
// m in [1, 2); then e = E - fmax_exp, plus one when m > 1.75.
__device__ __forceinline__ int mx_exponent(float amax, int fmax_exp) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  const uint32_t ef = b >> 23, mf = b & 0x7FFFFFu;
  if (b == 0 || ef == 0xFFu) return 0;
  uint32_t m;   // significand with its leading one at bit 23
  int E;
  if (ef == 0) {
    const int lz = __clz(mf) - 8;
    m = mf << lz;
    E = -126 - lz;
  } else {
    m = mf | 0x800000u;
    E = static_cast<int>(ef) - 127;
  }
  int e = E - fmax_exp + (m > 0xE00000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// The floor convention (the alternate behind FP8_MX_1x32_FLOOR*): e = floor(log2 amax)
// - fmax_exp, the unbiased binary exponent of amax less the format's largest power-of-two
// exponent, so the block maximum scales into [2^fmax_exp, 2^(fmax_exp + 1)) and what lies
// above FMAX saturates; amax == 0 or non-finite -> 0; clamped to [-127, 127].
__device__ __forceinline__ int mx_exponent_floor(float amax, int fmax_exp) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  const uint32_t ef = b >> 23, mf = b & 0x7FFFFFu;
  if (b == 0 || ef == 0xFFu) return 0;
  const int E = ef == 0 ? -126 - (__clz(mf) - 8) : static_cast<int>(ef) - 127;
  const int e = E - fmax_exp;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as binary32, exact for e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2_neg(int e) {
  const int x = -e;
  return x >= -126 ? __uint_as_float(static_cast<uint32_t>(x + 127) << 23) : __uint_as_float(0x00400000u);
}

// bf16 pair helpers (a 32-bit word holds two bf16: low half = lower address).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// Lane-wise max of |a| and |b| on bf16 pairs; NaN inputs are ignored.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a & 0x7FFF7FFFu), "r"(b & 0x7FFF7FFFu));
  return d;
}
// Both halves of an (already absolute) bf16 pair -> the larger as binary32.
__device__ __forceinline__ float pair_max_f32(uint32_t w) { return fmaxf(bf16lo(w), bf16hi(w)); }

}  // namespace fp8q
