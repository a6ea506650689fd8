// dequantize.cu -- FP8 -> BF16: y = RN_bf16(decode(q) * multiplier), the exact
// product rounded once to bfloat16 (ties to even).  The multiplier of element
// (r, c) is the one the quantizer stored for its block:
//   per-tensor s[0]; 1x128 s[r, c/128]; 128x128 s[r/128, c/128];
//   MXFP8 2^(e - 127) with e the E8M0 byte of block (r, c/32) (0xFF: NaN),
//   row-major or in the GEMM-ready tiled layout.
// (Search-result page: FP8 weights converted to BF16 for use elsewhere; guide,
// "block-level scaling" and "MXFP8 scaling" for the multipliers.)
//
// One rounding of an exact product without wider arithmetic: the product is
// formed rounded toward zero in binary32 and made "round to odd" (its last bit
// set when the product was inexact, which the exact FMA residual tells); a
// round-to-odd value with at least two bits beyond the target precision rounds
// to nearest exactly like the exact value (Boldo and Melquiond, "Emulation of
// FMA and correctly rounded sums: proved algorithms using rounding to odd",
// IEEE Trans. Computers 2008).  The residual is exact while the product and
// its error stay normal, which holds for every FP8 code when the multiplier is
// in [2^-100, 2^100]; other chunks (and E5M2 infinities, whose residual is
// NaN) take a path that forms the product in binary64 (exact) and rounds it to
// odd binary32 the same way.
//
// Layout: a grid-stride loop over 16-element chunks (one 16-byte load of codes,
// two 16-byte stores of bf16), four chunks in flight per thread.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

constexpr int kDqThreads = 256;
constexpr int kDqUnroll = 4;

// round-to-odd binary32 of d * m (fast path: the product and its residual are normal)
__device__ __forceinline__ float mul_odd_fast(float d, float m) {
  const float p = __fmul_rz(d, m);
  const float r = __fmaf_rn(d, m, -p);
  return __uint_as_float(__float_as_uint(p) | (r != 0.0f ? 1u : 0u));
}
// round-to-odd binary32 of d * m for any operands (the product is exact in binary64)
__device__ __forceinline__ float mul_odd_exact(float d, float m) {
  const double pd = static_cast<double>(d) * static_cast<double>(m);
  const float f = __double2float_rz(pd);
  if (f != f) return f;   // NaN
  return __uint_as_float(__float_as_uint(f) | (static_cast<double>(f) != pd ? 1u : 0u));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// 4 codes -> 4 bf16 (two 32-bit words)
template <bool FAST>
__device__ __forceinline__ uint2 deq4(uint32_t w, float m, bool e5) {
  float a, b, c, d;
  decode_pair(w & 0xFFFFu, e5, a, b);
  decode_pair(w >> 16, e5, c, d);
  uint2 r;
  if (FAST) {
    r.x = pack_bf16x2(mul_odd_fast(a, m), mul_odd_fast(b, m));
    r.y = pack_bf16x2(mul_odd_fast(c, m), mul_odd_fast(d, m));
  } else {
    r.x = pack_bf16x2(mul_odd_exact(a, m), mul_odd_exact(b, m));
    r.y = pack_bf16x2(mul_odd_exact(c, m), mul_odd_exact(d, m));
  }
  return r;
}

__device__ __forceinline__ float e8m0_value(uint32_t e) {
  if (e == 255u) return __uint_as_float(0x7FC00000u);            // the E8M0 NaN
  return e == 0u ? __uint_as_float(0x00400000u) : __uint_as_float(e << 23);   // 2^(e - 127)
}

// GEMM-ready MX layout: atom (r/128, b/4) of 512 bytes, inside it (r%32)*16 + ((r%128)/32)*4 + b%4
__device__ __forceinline__ int64_t mx_tiled_at(int64_t r, int64_t b, int64_t atoms_per_row) {
  return ((r >> 7) * atoms_per_row + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3);
}

struct DqParams {
  const uint8_t* q;
  int64_t R, C;
  int64_t nchunks;   // whole 16-element chunks (per-tensor: of the flat array)
  int64_t n;         // elements (per-tensor tail: n - 16 * nchunks)
  const void* s;
  int e5m2;
  uint16_t* y;
};

// RECIPE: kTensor, kBlock1x128, kBlock128x128, kMx; TILED: MX scales in the GEMM-ready layout
template <int RECIPE, bool TILED>
__global__ void __launch_bounds__(kDqThreads) k_dequantize(const DqParams p) {
  pdl_wait();
  pdl_launch_dependents();
  const bool e5 = p.e5m2 != 0;
  const int64_t cpr = p.C / 16;   // chunks per row (block recipes)
  const uint4* q16 = reinterpret_cast<const uint4*>(p.q);
  uint4* y16 = reinterpret_cast<uint4*>(p.y);
  const float m_tensor = RECIPE == kTensor ? *static_cast<const float*>(p.s) : 0.0f;
  auto multiplier = [&](int64_t chunk) -> float {
    if (RECIPE == kTensor) return m_tensor;
    const int64_t r = chunk / cpr, c = (chunk - r * cpr) * 16;
    if (RECIPE == kBlock1x128) return __ldg(static_cast<const float*>(p.s) + r * (p.C / 128) + c / 128);
    if (RECIPE == kBlock128x128) return __ldg(static_cast<const float*>(p.s) + (r / 128) * (p.C / 128) + c / 128);
    const uint8_t* se = static_cast<const uint8_t*>(p.s);
    const int64_t off = TILED ? mx_tiled_at(r, c / 32, p.C / 128) : r * (p.C / 32) + c / 32;
    return e8m0_value(__ldg(se + off));
  };
  auto convert = [&](uint4 w, float m, int64_t chunk) {
    // every product of this chunk normal and finite with an exact residual?
    bool fast = m >= 0x1p-100f && m <= 0x1p100f;
    if (e5) {
      // E5M2 infinity / NaN codes (exponent field all ones): their residual is NaN
      const uint32_t hi = __vcmpgeu4(w.x & 0x7F7F7F7Fu, 0x7C7C7C7Cu) | __vcmpgeu4(w.y & 0x7F7F7F7Fu, 0x7C7C7C7Cu) |
                          __vcmpgeu4(w.z & 0x7F7F7F7Fu, 0x7C7C7C7Cu) | __vcmpgeu4(w.w & 0x7F7F7F7Fu, 0x7C7C7C7Cu);
      fast = fast && hi == 0u;
    }
    uint2 a, b, c, d;
    if (fast) {
      a = deq4<true>(w.x, m, e5);
      b = deq4<true>(w.y, m, e5);
      c = deq4<true>(w.z, m, e5);
      d = deq4<true>(w.w, m, e5);
    } else {
      a = deq4<false>(w.x, m, e5);
      b = deq4<false>(w.y, m, e5);
      c = deq4<false>(w.z, m, e5);
      d = deq4<false>(w.w, m, e5);
    }
    y16[2 * chunk] = make_uint4(a.x, a.y, b.x, b.y);
    y16[2 * chunk + 1] = make_uint4(c.x, c.y, d.x, d.y);
  };
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kDqUnroll - 1) * stride < p.nchunks; i += kDqUnroll * stride) {
    uint4 w[kDqUnroll];
    float m[kDqUnroll];
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) {
      w[u] = __ldg(q16 + i + u * stride);
      m[u] = multiplier(i + u * stride);
    }
#pragma unroll
    for (int u = 0; u < kDqUnroll; ++u) convert(w[u], m[u], i + u * stride);
  }
  for (; i < p.nchunks; i += stride) convert(__ldg(q16 + i), multiplier(i), i);
  if (RECIPE == kTensor && blockIdx.x == 0) {
    // the last n % 16 elements of a per-tensor array, one per thread
    const int64_t e = p.nchunks * 16 + threadIdx.x;
    if (e < p.n) {
      float v, unused;
      decode_pair(p.q[e], e5, v, unused);
      p.y[e] = static_cast<uint16_t>(pack_bf16x2(mul_odd_exact(v, m_tensor), 0.0f) & 0xFFFFu);
    }
  }
}

template <int RECIPE, bool TILED>
cudaError_t launch_dq(const DqParams& p, int num_sms, cudaStream_t s) {
  const int64_t per_cta = static_cast<int64_t>(kDqThreads) * kDqUnroll;
  int64_t want = (p.nchunks + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
  return launch_pdl(k_dequantize<RECIPE, TILED>, dim3(grid), dim3(kDqThreads), 0, s, 1, p);
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* q, int64_t R, int64_t C, int recipe, bool mx_tiled, bool e5m2,
                              const void* s, void* y, int num_sms, cudaStream_t stream) {
  DqParams p;
  p.q = q;
  p.R = R;
  p.C = C;
  p.n = R * C;
  p.nchunks = p.n / 16;
  p.s = s;
  p.e5m2 = e5m2 ? 1 : 0;
  p.y = static_cast<uint16_t*>(y);
  switch (recipe) {
    case kTensor: return launch_dq<kTensor, false>(p, num_sms, stream);
    case kBlock1x128: return launch_dq<kBlock1x128, false>(p, num_sms, stream);
    case kBlock128x128: return launch_dq<kBlock128x128, false>(p, num_sms, stream);
    default:
      return mx_tiled ? launch_dq<kMx, true>(p, num_sms, stream) : launch_dq<kMx, false>(p, num_sms, stream);
  }
}

}  // namespace fp8q
