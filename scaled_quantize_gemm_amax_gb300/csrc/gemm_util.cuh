// gemm_util.cuh -- device helpers of the GEMM kernels (gemm.cu):
// packed binary32 pairs, shared/global vector stores, and the persistent tile walker.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fp8q {
namespace gemm_util {

// Tile raster: groups of GM M-tiles walk N together, so they share B tiles in L2 (8 for
// the blockwise kernels' 256 x 128 tiles, 16 for the 256 x 256 per-tensor and MX tiles:
// both measured side by side, per-tensor and MX 8192^3 +2 % with 16, blockwise -1 %).

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Packed pairs of binary32 (Blackwell's f32x2 arithmetic: one instruction, two lanes).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t pack_f32x2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void sts32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
// volatile: stays after the barrier wait that precedes it
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ void stg128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// a / b for a >= 0, b > 0.  Below 2^22 a binary32 estimate (relative error under 2^-23,
// so within one of the quotient) corrected by one step either way: a few instructions
// instead of an integer division, which the tile walker paid at every tile change
// (1-2 % at 8192^3, measured).
__device__ __forceinline__ int div_small(int a, int b) {
  if (a >= (1 << 22)) return a / b;
  int q = __float2int_rz(__fmul_rn(static_cast<float>(a), __frcp_rn(static_cast<float>(b))));
  const int r = a - q * b;
  q += (r >= b) - (r < 0);
  return q;
}

template <int GM>
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = GM * tiles_n;
  const int group = div_small(t, per_group);
  const int first_m = group * GM;
  const int gsize = min(tiles_m - first_m, GM);
  const int r = t - group * per_group;
  tn = div_small(r, gsize);
  tm = first_m + (r - tn * gsize);
}

}  // namespace gemm_util
}  // namespace fp8q
