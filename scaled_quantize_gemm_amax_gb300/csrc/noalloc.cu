// noalloc.cu -- fp8_allreduce_sum_noalloc: the FP8 gradient all-reduce of
// fp8_allreduce_sum with its intermediate amax kept in library-owned scratch, for
// callers that cannot hand the library any device memory besides the buffers they
// reduce (a gradient-reduction hook in a runtime with no device allocator of its
// own, or a process whose device memory a caching allocator has already reserved in
// full: an allocation there fails or breaks the budget).  The entry point
// allocates nothing: the scratch is a file-scope device array.
//
//   scratch[r]  (r < k)  the amax of rank r's gradient (the contribution each rank
//                        would make to the all-reduce MAX)
//   scratch[kMaxRanks]   their maximum, the global amax the cast-and-sum pass reads
//
// Every call clears scratch[0..k) before use, so nothing has to start at zero.  All
// calls on a device share the array: calls whose executions overlap (on different
// streams or from different threads) race on it.
#include <atomic>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

constexpr int kNoAllocMaxRanks = 1024;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocMaxRanks + 1];

constexpr int kRankAmaxThreads = 256;

// Block (x, r) folds a grid-stride slice of rank r's row into scratch[r].
__global__ void __launch_bounds__(kRankAmaxThreads) k_rank_amax(const uint4* __restrict__ g, int64_t n8,
                                                               float* __restrict__ scratch) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.y;
  const uint4* row = g + static_cast<int64_t>(r) * n8;
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 v = __ldg(row + i);
    m = absmax_bf16x2(m, v.x);
    m = absmax_bf16x2(m, v.y);
    m = absmax_bf16x2(m, v.z);
    m = absmax_bf16x2(m, v.w);
  }
  float a = pair_max_f32(m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  __shared__ float red[kRankAmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int w = 1; w < kRankAmaxThreads / 32; ++w) b = fmaxf(b, red[w]);
    // non-negative floats order like their bit patterns
    if (b > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(scratch + r), __float_as_uint(b));
  }
}

// scratch[kNoAllocMaxRanks] = max over the k per-rank slots (the all-reduce MAX)
__global__ void k_max_ranks(float* __restrict__ scratch, int k) {
  pdl_wait();
  pdl_launch_dependents();
  float a = 0.0f;
  for (int r = threadIdx.x; r < k; r += blockDim.x) a = fmaxf(a, scratch[r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  if (threadIdx.x == 0) scratch[kNoAllocMaxRanks] = a;
}

// The scratch address and SM count of each device, looked up on the first call made
// with that device current.  `ready` is published with release order after the other
// fields are written, and read with acquire order, so a thread that sees it set also
// sees the address (the check outside the lock is then well defined).
struct NoAllocDevice {
  std::atomic<bool> ready{false};
  float* scratch = nullptr;
  int num_sms = 0;
};
NoAllocDevice g_noalloc_dev[kMaxDevices];
std::mutex g_noalloc_mutex;

cudaError_t noalloc_device(NoAllocDevice** out, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  NoAllocDevice& d = g_noalloc_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    // the set-up queries below are not allowed while the stream is being captured
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      int n = 0;
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      d.scratch = static_cast<float*>(p);
      d.num_sms = n;
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return cudaSuccess;
}

}  // namespace

int noalloc_max_ranks() { return kNoAllocMaxRanks; }

cudaError_t launch_allreduce_noalloc(const void* g, int k, int64_t n, bool e5m2, uint8_t* q, float* scale_inv,
                                     float* out, cudaStream_t s) {
  if (k < 1 || k > kNoAllocMaxRanks) return cudaErrorInvalidValue;
  NoAllocDevice* d = nullptr;
  cudaError_t e = noalloc_device(&d, s);
  if (e != cudaSuccess) return e;
  e = launch_zero_f32(d->scratch, k, s);
  if (e != cudaSuccess) return e;
  const int64_t n8 = n / 8;
  int64_t bx = (n8 + kRankAmaxThreads - 1) / kRankAmaxThreads;
  const int64_t cap = (static_cast<int64_t>(d->num_sms) * 8 + k - 1) / k;   // about 8 blocks per SM in all
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  e = launch_pdl(k_rank_amax, dim3(static_cast<unsigned>(bx), static_cast<unsigned>(k)), dim3(kRankAmaxThreads), 0, s,
                 1, static_cast<const uint4*>(g), n8, d->scratch);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_max_ranks, dim3(1), dim3(32), 0, s, 1, d->scratch, k);
  if (e != cudaSuccess) return e;
  return launch_allreduce(g, k, n, d->scratch + kNoAllocMaxRanks, e5m2, q, scale_inv, out, d->num_sms, s);
}

}  // namespace fp8q
