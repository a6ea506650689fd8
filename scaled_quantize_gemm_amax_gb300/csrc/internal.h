// internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8q {

enum Recipe : int { kTensor = 0, kBlock1x128 = 1, kBlock128x128 = 2, kMx = 3 };

constexpr int kMaxDevices = 64;

// Raise a kernel's dynamic shared-memory limit once per device (the setting is
// per function and device); `done` is the caller's per-kernel flag array (atomic:
// any host thread may launch; setting the attribute twice is harmless).
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel* fn, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// Launch with programmatic stream serialization: the kernel may be scheduled while the
// kernel before it in the stream drains.  Every kernel of this library executes
// griddepcontrol.wait (pdl_wait) before its first global-memory access, which returns
// once the preceding kernel has completed and its writes are visible, so stream order
// holds for all data; only launch latency and set-up (barriers, TMEM, tensor-map
// prefetch) overlap.  cluster_x > 1 adds a cluster dimension.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_x,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---- amax / scale / history (amax.cu)
cudaError_t launch_reciprocal(const float* in, float* out, cudaStream_t s);
// p[0 .. n) = 0 as a (programmatically launched) kernel, ahead of an atomicMax reduction
cudaError_t launch_zero_f32(float* p, int n, cudaStream_t s);
// The amax kernels, and the casts when amax_out is set, must be launched right after
// launch_zero_f32 of their amax: they read their inputs before griddepcontrol.wait (the
// zeroing kernel waited for every earlier kernel before letting them start) and wait
// only before the atomic.
cudaError_t launch_amax(const void* x, int64_t n, float* amax, int num_sms, cudaStream_t s);
cudaError_t launch_amax_f32(const float* x, int64_t n, float* amax, int num_sms, cudaStream_t s);
cudaError_t launch_compute_scale(const float* amax, bool e5m2, float* scale, float* scale_inv, cudaStream_t s);
cudaError_t launch_history_update(float* hist, int32_t len, int32_t* pos, const float* amax, bool e5m2, float* scale,
                                  float* scale_inv, uint32_t* err, cudaStream_t s);

// ---- quantize / cast-transpose (quantize.cu)
struct CastParams {
  int64_t R, C;          // input rows / columns (bf16, row-major)
  int recipe;
  int e5m2;
  int mx_tiled;          // MX scales in the GEMM-ready tiled layout
  int mx_floor;          // MX exponent by the floor rule (else the ceil rule)
  int do_row, do_col;
  const float* scale;    // per-tensor scale (device)
  float* amax_out;       // optional (device, zeroed by the kernel launched just before)
  uint8_t* q_row;        // [R, C] (generic path only; the tiled path stores through tensor maps)
  uint8_t* q_col;        // [C, R]
  void* s_row;
  void* s_col;
  uint32_t* err;
  int tiles_r, tiles_c;
  int col_from_row;      // set by the launcher: the column copy as the byte transpose of the row copy
  int keep_col_scales;   // set by the launcher: 1x128 column scales stored with the L2 evict-last policy
  int one_division;      // set by the launcher: a 1x128 tile's row and column scales from one division a lane
};
// Tiled TMA path; requires C % 16 == 0 and (when do_col) R % 16 == 0.
cudaError_t launch_cast_transpose_tiled(const CastParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_qrow,
                                        const CUtensorMap& tm_qcol, int num_sms, cudaStream_t s);
// Plain path for the per-tensor recipe at any shape.
cudaError_t launch_cast_generic(const CastParams& p, const void* x, cudaStream_t s);
// The same two paths for a binary32 input (quantize_f32.cu); the tiled path's tensor map
// holds the input as 32-column boxes of 128 rows.
cudaError_t launch_cast_transpose_tiled_f32(const CastParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_qrow,
                                            const CUtensorMap& tm_qcol, int num_sms, cudaStream_t s);
cudaError_t launch_cast_generic_f32(const CastParams& p, const void* x, cudaStream_t s);
// Several tiled casts in one launch: job j owns tiles [tile_start[j], tile_start[j+1]).
constexpr int kMaxCastJobs = 4;
struct CastJobMaps {
  CUtensorMap x, qrow, qcol;
};
struct CastJobs {
  CastJobMaps m[kMaxCastJobs];
  CastParams p[kMaxCastJobs];
  int tile_start[kMaxCastJobs + 1];
  int n;
};
cudaError_t launch_cast_jobs(const CastJobs& jobs, int num_sms, cudaStream_t s);

// ---- dequantize (dequantize.cu): y bf16 [R, C] = RN_bf16(decode(q) * multiplier)
cudaError_t launch_dequantize(const uint8_t* q, int64_t R, int64_t C, int recipe, bool mx_tiled, bool e5m2,
                              const void* s, void* y, int num_sms, cudaStream_t stream);

// ---- FP8 gradient all-reduce of k ranks held as rows of g [k, n] (allreduce.cu);
// *amax must hold the global amax when the kernel runs
cudaError_t launch_allreduce(const void* g, int k, int64_t n, const float* amax, bool e5m2, uint8_t* q,
                             float* scale_inv, float* out, int num_sms, cudaStream_t s);

// ---- the all-reduce with its amax in library-owned scratch (noalloc.cu)
int noalloc_max_ranks();
cudaError_t launch_allreduce_noalloc(const void* g, int k, int64_t n, bool e5m2, uint8_t* q, float* scale_inv,
                                     float* out, cudaStream_t s);

// ---- scaled GEMM (gemm.cu)
struct GemmParams {
  int64_t M, N, K;
  int kind;              // kTensor, kBlock1x128 (A 1x128), kMx
  int b_1x128;           // blockwise: B scales per (row, 128-K) instead of per (128 rows, 128-K)
  int e5m2_a, e5m2_b;
  int out_fp32;
  const void* sa;        // per-tensor: float[1]; blockwise: float[M, K/128]; MX: tiled E8M0
  const void* sb;        // per-tensor: float[1]; blockwise: float[N/128, K/128] or [N, K/128]; MX: tiled E8M0
  void* c;               // [M, N] row-major, bf16 or fp32; null: not stored
  // fused output quantization (all null: off).  y = the value stored in c (bf16-rounded
  // for bf16 output): c_amax = max |y|, cq = encode_sat(y * c_scale), c_scale_inv = 1 / c_scale
  float* c_amax;         // float[1], zeroed by the caller's stream before the launch
  const float* c_scale;  // float[1]
  uint8_t* cq;           // [M, N] row-major FP8 (format e5m2_c)
  float* c_scale_inv;    // float[1]
  int e5m2_c;
  uint32_t* err;
  // Split of the last, partial wave (per-tensor and MX on CTA pairs): the tiles from
  // tail0 on are cut into `split` K ranges computed by otherwise idle pairs; range c > 0
  // leaves its raw FP32 accumulators in ws slot (c - 1) * (tiles - tail0) + j and counts
  // its warps on ws_flags[slot]; the pair with range 0 adds the ranges in order and
  // resets the count.  split = 1: off (tail0 = the tile count).
  int split;
  int tail0;
  // Balanced division instead (streamk = 1, same kernels and workspace): the tiles' K
  // blocks in order, cut into one contiguous share per pair; a tile cut between pairs u
  // and u + 1 has its later part left in slot u + 1 by pair u + 1 (its first work) and
  // added by pair u (its last work).
  int streamk;
  float* ws;             // [slots][256][256] fp32
  int* ws_flags;         // [slots], 0 between launches
  int64_t ws_len;        // floats in ws, and
  int ws_nflags;         // counters in ws_flags (index checks of debug builds)
  // Blockwise 1x128 x 128x128 on 256 x 160 pair tiles (set by gemm_select_wide)
  int wide160;
};
// Whether the blockwise 1x128 x 128x128 GEMM these parameters describe runs on 256 x 160
// pair tiles with 128-deep stages (BF16 out, no fused output cast, M % 256 == 0, K / 128
// odd); the caller stores the answer in p.wide160 before asking for the tile shape and
// building the tensor maps.
bool gemm_select_wide(const GemmParams& p, int num_sms);
// Width (N) of one output tile of the GEMM variant these parameters select.
int gemm_block_n(const GemmParams& p);
// Whether the GEMM runs on 2-CTA pairs (256-row tiles) for these parameters.
bool gemm_uses_pair(const GemmParams& p);
// Rows of B one TMA box carries (the tile width, or half of it for a pair).
int gemm_b_box_rows(const GemmParams& p);
// Columns of C one TMA store box carries: 16 (BF16, unswizzled) for the 160-wide tiles,
// else 0: the usual 128-byte box (64 BF16 or 32 FP32 columns, 128-byte swizzle).
int gemm_c_box_cols(const GemmParams& p);
// The division of a CTA-pair launch's tiles (host logic only): whole tiles, stream-K
// shares of the tiles from tail0 on (streamk = 1), or the last wave cut into `split` K
// ranges; `launched` pairs.  Per-tensor and MX only (other kinds: whole tiles).  Both cuts
// also need the stream's workspace; without it a launch runs whole tiles.
struct PairDivision {
  int streamk;
  int split;
  int tail0;
  int64_t launched;
};
PairDivision pair_division(int kind, int64_t ntiles, int64_t pairs, int64_t k);
// What a GEMM with these parameters launches (host logic only, p.wide160 already chosen):
// kernel variant (kTensor, kBlock1x128, kMx, or the blockwise variants 4 = per-row B on
// one CTA, 5 = 256-deep stages, 6 = per-row B on pairs, 7 = 256 x 160 pair tiles), CTA
// pairs or not, tile width, tile count, and the division above.
struct GemmPlan {
  int pair;
  int variant;
  int block_n;
  int64_t ntiles;
  PairDivision div;
};
GemmPlan gemm_plan(const GemmParams& p, int num_sms, int resident_pairs);
// tm_sfa / tm_sfb: MX only (the tiled E8M0 buffers as [atoms * 2, 256] bytes, box 2 x 256).
cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_sfa,
                        const CUtensorMap& tm_sfb, const CUtensorMap& tm_c, int num_sms, cudaStream_t s);

// Bounded-wait self test: one CTA waits on an mbarrier nothing arrives on.
cudaError_t launch_wait_selftest(uint32_t* err, cudaStream_t s);
// Index-check self test: one thread checks `index` against `extent` the way the kernels
// check their accesses (no memory is touched); only debug builds report.
cudaError_t launch_index_selftest(int64_t index, int64_t extent, uint32_t* err, cudaStream_t s);

}  // namespace fp8q
