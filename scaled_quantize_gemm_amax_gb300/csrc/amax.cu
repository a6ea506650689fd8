// amax.cu -- per-tensor amax reduction, per-tensor scale, and the delayed-scaling
// amax-history update.
//
// amax: the maximum of |x| over a BF16 (or binary32) tensor, NaN ignored (Colossal-AI FP8,
// "current scaling": the scale comes from the current tensor's maximum).  The
// reduction is order-free (a max), so any grid shape gives the same bits.
// History: a ring of past amaxes; the next scale comes from the window maximum
// (Colossal-AI FP8, "delayed scaling"; guide, "delayed scaling scheme").
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 8;

__device__ __forceinline__ uint32_t fold16(uint32_t m, uint4 v) {
  m = absmax_bf16x2(m, v.x);
  m = absmax_bf16x2(m, v.y);
  m = absmax_bf16x2(m, v.z);
  m = absmax_bf16x2(m, v.w);
  return m;
}

// Grid-stride max over 16-byte chunks (8 bf16 each), 8 independent loads in
// flight per thread, the last round predicated (chunks past the end read as zero,
// which leaves a max of magnitudes unchanged) so that no round has fewer loads in
// flight; the n % 8 tail is folded in by block 0.  One atomicMax per block on the
// (non-negative) float bit pattern, which orders like the value.
//
// Launched right after k_zero_f32 (programmatic launch): that kernel waits for every
// earlier kernel in the stream before it lets this one start, so x is complete and may
// be read at once; only the atomic on amax waits (griddepcontrol.wait) for the zeroing.
__global__ void __launch_bounds__(kAmaxThreads) k_amax(const uint4* __restrict__ x16, int64_t n16,
                                                      const uint16_t* __restrict__ tail, int ntail,
                                                      float* __restrict__ amax) {
  pdl_launch_dependents();
  uint32_t m = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kAmaxUnroll - 1) * stride < n16; i += kAmaxUnroll * stride) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) v[u] = __ldg(x16 + i + u * stride);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) m = fold16(m, v[u]);
  }
  if (i < n16) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) v[u] = i + u * stride < n16 ? __ldg(x16 + i + u * stride) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) m = fold16(m, v[u]);
  }
  float a = pair_max_f32(m);
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < ntail)
    a = fmaxf(a, fabsf(__uint_as_float(static_cast<uint32_t>(tail[threadIdx.x]) << 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  __shared__ float red[kAmaxThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int w = 1; w < kAmaxThreads / 32; ++w) b = fmaxf(b, red[w]);
    pdl_wait();   // the zeroing of amax is done
    if (b > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(b));
  }
}

// The same maximum over binary32 values (the FP32 master copy of a weight quantized
// with current scaling): 16-byte chunks of four values, NaN ignored by fmaxf.
__device__ __forceinline__ float fold4(float m, float4 v) {
  return fmaxf(fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fabsf(v.y)), fabsf(v.z)), fabsf(v.w));
}

// Launched right after k_zero_f32, as k_amax.
__global__ void __launch_bounds__(kAmaxThreads) k_amax_f32(const float4* __restrict__ x4, int64_t n4,
                                                          const float* __restrict__ tail, int ntail,
                                                          float* __restrict__ amax) {
  pdl_launch_dependents();
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kAmaxUnroll - 1) * stride < n4; i += kAmaxUnroll * stride) {
    float4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) v[u] = __ldg(x4 + i + u * stride);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) m = fold4(m, v[u]);
  }
  if (i < n4) {
    float4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u)
      v[u] = i + u * stride < n4 ? __ldg(x4 + i + u * stride) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) m = fold4(m, v[u]);
  }
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < ntail) m = fmaxf(m, fabsf(tail[threadIdx.x]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  __shared__ float red[kAmaxThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int w = 1; w < kAmaxThreads / 32; ++w) b = fmaxf(b, red[w]);
    pdl_wait();   // the zeroing of amax is done
    if (b > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(b));
  }
}

__global__ void k_compute_scale(const float* __restrict__ amax, int e5m2, float* __restrict__ scale,
                                float* __restrict__ scale_inv) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x != 0) return;
  const float s = scale_from_amax(*amax, fmax_of(e5m2 != 0));
  *scale = s;
  *scale_inv = recip_rn(s);
}

// hist[pos] = amax; pos = (pos + 1) mod len; m = max(hist) (NaN ignored);
// if 0 < m < inf: scale = FMAX / m (inf -> FLT_MAX), scale_inv = 1 / scale;
// otherwise the scale is left as it is.
__global__ void k_history_update(float* __restrict__ hist, int32_t len, int32_t* __restrict__ pos,
                                 const float* __restrict__ amax, int e5m2, float* __restrict__ scale,
                                 float* __restrict__ scale_inv, uint32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x != 0) return;
  const int32_t p = *pos;
  if (p < 0 || p >= len) {
    atomicOr(err, kErrBadState);
    return;
  }
  hist[p] = *amax;
  *pos = (p + 1) % len;
  float m = 0.0f;
  for (int32_t i = 0; i < len; ++i) {
    const float h = hist[i];
    if (h > m) m = h;
  }
  if (m > 0.0f && !is_inf_or_nan(m)) {
    float s = __fdiv_rn(fmax_of(e5m2 != 0), m);
    if (is_inf_or_nan(s)) s = FLT_MAX;
    *scale = s;
    *scale_inv = recip_rn(s);
  }
}

__global__ void k_reciprocal(const float* __restrict__ in, float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) *out = recip_rn(*in);
}

// One CTA waits for an mbarrier phase that never completes; the bounded wait
// must give up, report kErrTimeoutTmaLoad and let the kernel return.
__global__ void k_wait_selftest(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(b, 0, err, kErrTimeoutTmaLoad, nullptr);
  __syncthreads();
}

}  // namespace

cudaError_t launch_amax(const void* x, int64_t n, float* amax, int num_sms, cudaStream_t s) {
  const int64_t n16 = n / 8;
  const int ntail = static_cast<int>(n - n16 * 8);
  int64_t want = (n16 + static_cast<int64_t>(kAmaxThreads) * kAmaxUnroll - 1) / (kAmaxThreads * kAmaxUnroll);
  int64_t cap = static_cast<int64_t>(num_sms) * 4;
  int grid = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
  return launch_pdl(k_amax, dim3(grid), dim3(kAmaxThreads), 0, s, 1, static_cast<const uint4*>(x), n16,
                    static_cast<const uint16_t*>(x) + n16 * 8, ntail, amax);
}

cudaError_t launch_amax_f32(const float* x, int64_t n, float* amax, int num_sms, cudaStream_t s) {
  const int64_t n4 = n / 4;
  const int ntail = static_cast<int>(n - n4 * 4);
  int64_t want = (n4 + static_cast<int64_t>(kAmaxThreads) * kAmaxUnroll - 1) / (kAmaxThreads * kAmaxUnroll);
  int64_t cap = static_cast<int64_t>(num_sms) * 4;
  int grid = static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
  return launch_pdl(k_amax_f32, dim3(grid), dim3(kAmaxThreads), 0, s, 1, reinterpret_cast<const float4*>(x), n4,
                    x + n4 * 4, ntail, amax);
}

cudaError_t launch_compute_scale(const float* amax, bool e5m2, float* scale, float* scale_inv, cudaStream_t s) {
  return launch_pdl(k_compute_scale, dim3(1), dim3(32), 0, s, 1, amax, e5m2 ? 1 : 0, scale, scale_inv);
}

cudaError_t launch_history_update(float* hist, int32_t len, int32_t* pos, const float* amax, bool e5m2, float* scale,
                                  float* scale_inv, uint32_t* err, cudaStream_t s) {
  return launch_pdl(k_history_update, dim3(1), dim3(32), 0, s, 1, hist, len, pos, amax, e5m2 ? 1 : 0, scale, scale_inv,
                    err);
}

// p[0 .. n) = 0 before a kernel that folds maxima into it with atomicMax.  A kernel
// rather than a memset node: it lets its dependent start early (programmatic
// launch), whose griddepcontrol.wait then orders every access after the zeroing;
// a memset node in front of the reduction cost it ~5 us of launch gap.
__global__ void k_zero_f32(float* __restrict__ p, int n) {
  pdl_wait();   // after the previous kernel's last use of p
  pdl_launch_dependents();
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0.0f;
}

cudaError_t launch_zero_f32(float* p, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(k_zero_f32, dim3(1), dim3(n < 1024 ? ((n + 31) / 32) * 32 : 1024), 0, s, 1, p, n);
}

cudaError_t launch_reciprocal(const float* in, float* out, cudaStream_t s) {
  return launch_pdl(k_reciprocal, dim3(1), dim3(32), 0, s, 1, in, out);
}

cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

// The index check the kernels apply to their plain global accesses, on one value and
// touching no memory (it reports only in debug builds).
__global__ void k_index_selftest(int64_t index, int64_t extent, uint32_t* err) { (void)in_range(index, extent, err); }

cudaError_t launch_index_selftest(int64_t index, int64_t extent, uint32_t* err, cudaStream_t s) {
  k_index_selftest<<<1, 1, 0, s>>>(index, extent, err);
  return cudaGetLastError();
}

}  // namespace fp8q
