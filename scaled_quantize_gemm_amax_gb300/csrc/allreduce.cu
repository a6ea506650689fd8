// allreduce.cu -- FP8 gradient all-reduce with a shared scale for k
// data-parallel ranks whose gradients are the rows of g [k, n] on this device
// (FP8-LM news article, "automatic scaling": the scaling factor keeps the
// gradient within FP8's range through the all-reduce).  The ranks agree on the
// global amax A (an all-reduce MAX: here fp8_amax over all k rows), all cast
// with s = FMAX / A, and the reduction sums the decoded payloads in rank order
// in binary32 and multiplies once by 1 / s:
//   q[r, i] = encode_sat(g[r, i] * s)
//   out[i]  = ((decode(q[0, i]) + decode(q[1, i])) + ... + decode(q[k-1, i])) * (1 / s)
// For E4M3 and k <= 64 the sum is exact (every payload lies on the 2^-9 grid below
// 448), so the result does not depend on the order; for E5M2 the order is fixed.
//
// Kernel: a grid-stride loop over 8-element column chunks; a thread reads the
// chunk of every rank (coalesced across the warp per rank, four ranks' loads in
// flight), writes each rank's 8 payload bytes and keeps the 8 running sums in
// registers.
#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

constexpr int kArThreads = 256;
constexpr int kArRanksInFlight = 4;

// 8 bf16 -> 8 codes (x * s in binary32, then the saturating cast), and their decoded values
__device__ __forceinline__ uint2 cast8(uint4 w, float s, bool e5, float (&d)[8]) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t c[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    c[j] = cvt_pair(__fmul_rn(bf16lo(in[j]), s), __fmul_rn(bf16hi(in[j]), s), e5);
    decode_pair(c[j], e5, d[2 * j], d[2 * j + 1]);
  }
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__global__ void __launch_bounds__(kArThreads) k_allreduce(const uint4* __restrict__ g, int k, int64_t n8,
                                                         const float* __restrict__ amax, int e5m2,
                                                         uint2* __restrict__ q, float* __restrict__ scale_inv,
                                                         float4* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const bool e5 = e5m2 != 0;
  const float s = scale_from_amax(*amax, fmax_of(e5));
  const float si = recip_rn(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_inv = si;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    int r = 0;
    for (; r + kArRanksInFlight <= k; r += kArRanksInFlight) {
      uint4 w[kArRanksInFlight];
#pragma unroll
      for (int u = 0; u < kArRanksInFlight; ++u) w[u] = __ldg(g + static_cast<int64_t>(r + u) * n8 + i);
#pragma unroll
      for (int u = 0; u < kArRanksInFlight; ++u) {
        float d[8];
        q[static_cast<int64_t>(r + u) * n8 + i] = cast8(w[u], s, e5, d);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], d[j]);   // rank order
      }
    }
    for (; r < k; ++r) {
      float d[8];
      q[static_cast<int64_t>(r) * n8 + i] = cast8(__ldg(g + static_cast<int64_t>(r) * n8 + i), s, e5, d);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], d[j]);
    }
    out[2 * i] = make_float4(__fmul_rn(acc[0], si), __fmul_rn(acc[1], si), __fmul_rn(acc[2], si), __fmul_rn(acc[3], si));
    out[2 * i + 1] =
        make_float4(__fmul_rn(acc[4], si), __fmul_rn(acc[5], si), __fmul_rn(acc[6], si), __fmul_rn(acc[7], si));
  }
}

}  // namespace

cudaError_t launch_allreduce(const void* g, int k, int64_t n, const float* amax, bool e5m2, uint8_t* q,
                             float* scale_inv, float* out, int num_sms, cudaStream_t s) {
  const int64_t n8 = n / 8;
  int64_t want = (n8 + kArThreads - 1) / kArThreads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const int grid = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
  return launch_pdl(k_allreduce, dim3(grid), dim3(kArThreads), 0, s, 1, static_cast<const uint4*>(g), k, n8, amax,
                    e5m2 ? 1 : 0, reinterpret_cast<uint2*>(q), scale_inv, reinterpret_cast<float4*>(out));
}

}  // namespace fp8q
