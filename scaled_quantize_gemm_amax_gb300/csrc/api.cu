// api.cu -- the C ABI (include/fp8q.h): argument checks, TMA tensor maps and
// dispatch to the kernels.  All checks run on the host before anything is
// enqueued, and before any CUDA call, so a rejected call has no effect.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "fp8q.h"
#include "internal.h"
#include "ptx.cuh"

namespace fp8q {
namespace {

// The device error word (one per device that loads the library).
__device__ uint32_t g_error_word;

// `ready` is stored with release order once the other fields are filled in and loaded
// with acquire order, so the unlocked check in device_info() is well defined.
struct DeviceInfo {
  std::atomic<bool> ready{false};
  int num_sms = 0;
  uint32_t* err = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

fp8_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8_ERR_CUDA;
  DeviceInfo& d = g_devices[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int n = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FP8_ERR_CUDA;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return FP8_ERR_CUDA;
      d.num_sms = n;
      d.err = static_cast<uint32_t*>(p);
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return FP8_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major tensor [outer, inner] of `elem` bytes, box [box_outer, box_inner].
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t elem, const void* ptr, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * elem};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_recipe(fp8_recipe r) { return r >= FP8_TENSOR && r <= FP8_MX_1x32_FLOOR_TILED; }
bool is_mx(fp8_recipe r) {
  return r == FP8_MX_1x32 || r == FP8_MX_1x32_TILED || r == FP8_MX_1x32_FLOOR || r == FP8_MX_1x32_FLOOR_TILED;
}
bool is_mx_tiled(fp8_recipe r) { return r == FP8_MX_1x32_TILED || r == FP8_MX_1x32_FLOOR_TILED; }
bool is_mx_floor(fp8_recipe r) { return r == FP8_MX_1x32_FLOOR || r == FP8_MX_1x32_FLOOR_TILED; }
bool valid_fmt(fp8_format f) { return f == FP8_E4M3 || f == FP8_E5M2; }
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;   // TMA coordinates are signed 32-bit

fp8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

// One NVTX range per C-ABI call, in the "fp8q" domain, so that a profiler's timeline
// shows which entry point enqueued which kernels.  With no tool attached the NVTX
// calls return at once.
class ApiRange {
 public:
  explicit ApiRange(const char* name) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(domain(), &a);
  }
  ~ApiRange() { nvtxDomainRangePop(domain()); }
  ApiRange(const ApiRange&) = delete;
  ApiRange& operator=(const ApiRange&) = delete;

 private:
  static nvtxDomainHandle_t domain() {
    static const nvtxDomainHandle_t d = nvtxDomainCreateA("fp8q");
    return d;
  }
};

}  // namespace
}  // namespace fp8q

using namespace fp8q;

namespace {

fp8_status cast_transpose_impl(const void* x, bool f32, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                               const float* scale, float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col,
                               void* s_col, cudaStream_t stream);

// Validation and launch parameters of one cast; no device work.  fp8_cast_transpose and
// every job of fp8_cast_transpose_multi go through the same checks.
struct CastPlan {
  bool empty = false;   // no elements: nothing to launch
  bool tiled = false;   // the TMA path (else the plain per-tensor path)
  bool f32 = false;     // binary32 input (else bf16)
  CastParams p{};
  CUtensorMap tm_x, tm_qr, tm_qc;
};

fp8_status plan_cast(const void* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt, const float* scale,
                     float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col, void* s_col, CastPlan* plan,
                     bool f32 = false) {
  plan->f32 = f32;
  if (rows < 0 || cols < 0 || !valid_fmt(fmt) || !valid_recipe(recipe)) return FP8_ERR_INVALID_ARG;
  if (rows * cols == 0) {
    if (!aligned(amax_out, 4)) return FP8_ERR_ALIGNMENT;
    plan->empty = true;
    return FP8_OK;
  }
  const bool do_row = q_row != nullptr, do_col = q_col != nullptr;
  if (!do_row && !do_col) return FP8_ERR_INVALID_ARG;
  if (x == nullptr) return FP8_ERR_INVALID_ARG;
  const bool mx = is_mx(recipe);
  if (recipe == FP8_TENSOR) {
    if (scale == nullptr) return FP8_ERR_INVALID_ARG;
  } else {
    if ((do_row && s_row == nullptr) || (do_col && s_col == nullptr)) return FP8_ERR_INVALID_ARG;
  }
  // blocked dimensions
  switch (recipe) {
    case FP8_BLOCK_1x128:
      if ((do_row && cols % 128) || (do_col && rows % 128)) return FP8_ERR_SHAPE;
      break;
    case FP8_BLOCK_128x128:
      if (rows % 128 || cols % 128) return FP8_ERR_SHAPE;
      break;
    case FP8_MX_1x32:
    case FP8_MX_1x32_FLOOR:
      if ((do_row && cols % 32) || (do_col && rows % 32)) return FP8_ERR_SHAPE;
      break;
    case FP8_MX_1x32_TILED:
    case FP8_MX_1x32_FLOOR_TILED:
      if (rows % 128 || cols % 128) return FP8_ERR_SHAPE;
      break;
    default:
      break;
  }
  if (rows > kMaxDim || cols > kMaxDim) return FP8_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(q_row, 16) || !aligned(q_col, 16)) return FP8_ERR_ALIGNMENT;
  if (!mx && (!aligned(s_row, 4) || !aligned(s_col, 4))) return FP8_ERR_ALIGNMENT;
  if (is_mx_tiled(recipe) && (!aligned(s_row, 16) || !aligned(s_col, 16))) return FP8_ERR_ALIGNMENT;
  if (!aligned(scale, 4) || !aligned(amax_out, 4)) return FP8_ERR_ALIGNMENT;

  CastParams& p = plan->p;
  p.R = rows;
  p.C = cols;
  p.recipe = mx ? kMx : static_cast<int>(recipe);
  p.e5m2 = fmt == FP8_E5M2;
  p.mx_tiled = is_mx_tiled(recipe);
  p.mx_floor = is_mx_floor(recipe);
  p.do_row = do_row;
  p.do_col = do_col;
  p.scale = scale;
  p.amax_out = amax_out;
  p.q_row = q_row;
  p.q_col = q_col;
  p.s_row = s_row;
  p.s_col = s_col;
  p.tiles_r = static_cast<int>((rows + 127) / 128);
  p.tiles_c = static_cast<int>((cols + 127) / 128);
  plan->tiled = (cols % 16 == 0) && (!do_col || rows % 16 == 0);
  if (plan->tiled) {
    std::memset(&plan->tm_qr, 0, sizeof(plan->tm_qr));
    std::memset(&plan->tm_qc, 0, sizeof(plan->tm_qc));
    const bool ok = f32 ? make_map(&plan->tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, x, cols, rows, 32, 128)
                        : make_map(&plan->tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, cols, rows, 64, 128);
    if (!ok) return FP8_ERR_CUDA;
    if (do_row && !make_map(&plan->tm_qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q_row, cols, rows, 128, 128))
      return FP8_ERR_CUDA;
    if (do_col && !make_map(&plan->tm_qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, q_col, rows, cols, 128, 128))
      return FP8_ERR_CUDA;
  }
  return FP8_OK;
}

// Optional outputs of the fused epilogue (all null for the plain GEMM).
struct GemmExtra {
  float* c_amax = nullptr;
  const float* c_scale = nullptr;
  fp8_format fc = FP8_E4M3;
  uint8_t* cq = nullptr;
  float* c_scale_inv = nullptr;
};

// The GEMM kind of a recipe pairing (the guide's pairings: per-tensor x per-tensor,
// 1x128 x 128x128, 1x128 x 1x128 for the weight gradient, MXFP8 x MXFP8 in the tiled layout).
fp8_status gemm_kind(fp8_recipe ra, fp8_recipe rb, int* kind, int* b_1x128) {
  *b_1x128 = 0;
  if (ra == FP8_TENSOR && rb == FP8_TENSOR) {
    *kind = kTensor;
  } else if (ra == FP8_BLOCK_1x128 && rb == FP8_BLOCK_128x128) {
    *kind = kBlock1x128;
  } else if (ra == FP8_BLOCK_1x128 && rb == FP8_BLOCK_1x128) {
    *kind = kBlock1x128;
    *b_1x128 = 1;
  } else if (is_mx_tiled(ra) && is_mx_tiled(rb)) {
    *kind = kMx;   // either exponent rule: the tensor core reads E8M0 bytes either way
  } else if (valid_recipe(ra) && valid_recipe(rb)) {
    return FP8_ERR_UNSUPPORTED;
  } else {
    return FP8_ERR_INVALID_ARG;
  }
  return FP8_OK;
}

fp8_status scaled_gemm(const uint8_t* A, fp8_format fa, fp8_recipe ra, const void* sA, const uint8_t* B, fp8_format fb,
                       fp8_recipe rb, const void* sB, int64_t M, int64_t N, int64_t K, void* C, fp8_out_dtype out,
                       const GemmExtra& x, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || !valid_fmt(fa) || !valid_fmt(fb) || (out != FP8_OUT_BF16 && out != FP8_OUT_FP32))
    return FP8_ERR_INVALID_ARG;
  int kind;
  int b_1x128 = 0;
  if (fp8_status st = gemm_kind(ra, rb, &kind, &b_1x128)) return st;
  const bool fused = x.c_amax != nullptr || x.cq != nullptr;
  const int64_t outsz = out == FP8_OUT_FP32 ? 4 : 2;
  if (fused) {
    if (!valid_fmt(x.fc)) return FP8_ERR_INVALID_ARG;
    if (x.cq != nullptr && x.c_scale == nullptr) return FP8_ERR_INVALID_ARG;
    if (x.c_scale_inv != nullptr && x.cq == nullptr) return FP8_ERR_INVALID_ARG;
  } else if (C == nullptr && M > 0 && N > 0) {
    return FP8_ERR_INVALID_ARG;
  }
  if (M % 128 || N % 128 || K % 128) return FP8_ERR_SHAPE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8_ERR_SHAPE;
  if ((C != nullptr && !aligned(C, 16)) || (x.cq != nullptr && !aligned(x.cq, 16))) return FP8_ERR_ALIGNMENT;
  if (x.c_amax != nullptr && !aligned(x.c_amax, 4)) return FP8_ERR_ALIGNMENT;
  if (K > 0 && M > 0 && N > 0) {
    if (A == nullptr || B == nullptr || sA == nullptr || sB == nullptr) return FP8_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(B, 16)) return FP8_ERR_ALIGNMENT;
    const uintptr_t sal = kind == kMx ? 16 : 4;
    if (!aligned(sA, sal) || !aligned(sB, sal)) return FP8_ERR_ALIGNMENT;
  }
  if (!fused && (M == 0 || N == 0)) return FP8_OK;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  if (x.c_amax != nullptr) {
    if (launch_zero_f32(x.c_amax, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
  }
  if (M == 0 || N == 0 || K == 0) {
    // C = 0: amax 0 (set above), FP8 copy all +0 codes, scale_inv still written
    const size_t mn = static_cast<size_t>(M * N);
    if (C != nullptr && mn && cudaMemsetAsync(C, 0, mn * outsz, stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (x.cq != nullptr && mn && cudaMemsetAsync(x.cq, 0, mn, stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (x.c_scale_inv != nullptr) return cuda_status(launch_reciprocal(x.c_scale, x.c_scale_inv, stream));
    return FP8_OK;
  }

  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.kind = kind;
  p.b_1x128 = b_1x128;
  p.e5m2_a = fa == FP8_E5M2;
  p.e5m2_b = fb == FP8_E5M2;
  p.out_fp32 = out == FP8_OUT_FP32;
  p.sa = sA;
  p.sb = sB;
  p.c = C;
  p.c_amax = x.c_amax;
  p.c_scale = x.c_scale;
  p.cq = x.cq;
  p.c_scale_inv = x.c_scale_inv;
  p.e5m2_c = x.fc == FP8_E5M2;
  p.err = d->err;
  p.wide160 = gemm_select_wide(p, d->num_sms) ? 1 : 0;
  CUtensorMap tm_a, tm_b;
  if (!make_map(&tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, M, 128, 128)) return FP8_ERR_CUDA;
  if (!make_map(&tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, N, 128, static_cast<uint32_t>(gemm_b_box_rows(p))))
    return FP8_ERR_CUDA;
  // MX: the tiled scale buffers as rows of 256 bytes, two rows (one 512-byte atom) per box
  CUtensorMap tm_sfa, tm_sfb;
  std::memset(&tm_sfa, 0, sizeof(tm_sfa));
  std::memset(&tm_sfb, 0, sizeof(tm_sfb));
  if (kind == kMx) {
    const uint64_t atoms_a = static_cast<uint64_t>(M / 128) * (K / 128), atoms_b = static_cast<uint64_t>(N / 128) * (K / 128);
    if (!make_map(&tm_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sA, 256, 2 * atoms_a, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&tm_sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sB, 256, 2 * atoms_b, 256, 2, CU_TENSOR_MAP_SWIZZLE_NONE))
      return FP8_ERR_CUDA;
  }
  // C leaves through TMA stores of 32-row x 128-byte boxes (all kernels but the blockwise
  // ones with 128-deep stages, which store directly; the 160-wide blockwise tiles use
  // unswizzled 32-row x 16-column boxes)
  CUtensorMap tm_c;
  std::memset(&tm_c, 0, sizeof(tm_c));
  if (C != nullptr) {
    const uint32_t box_cols = static_cast<uint32_t>(gemm_c_box_cols(p));
    const bool ok = out == FP8_OUT_FP32
                        ? make_map(&tm_c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, N, M, 32, 32)
                    : box_cols != 0
                        ? make_map(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, N, M, box_cols, 32, CU_TENSOR_MAP_SWIZZLE_NONE)
                        : make_map(&tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, N, M, 64, 32);
    if (!ok) return FP8_ERR_CUDA;
  }
  return cuda_status(launch_gemm(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, d->num_sms, stream));
}

}  // namespace

extern "C" {

const char* fp8_status_string(fp8_status s) {
  switch (s) {
    case FP8_OK: return "FP8_OK";
    case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
    case FP8_ERR_SHAPE: return "FP8_ERR_SHAPE";
    case FP8_ERR_ALIGNMENT: return "FP8_ERR_ALIGNMENT";
    case FP8_ERR_UNSUPPORTED: return "FP8_ERR_UNSUPPORTED";
    case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    case FP8_ERR_DEVICE_STATE: return "FP8_ERR_DEVICE_STATE";
    case FP8_ERR_INDEX: return "FP8_ERR_INDEX";
  }
  return "FP8_ERR_UNKNOWN";
}

fp8_status fp8_amax(const void* x, int64_t rows, int64_t cols, float* amax, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_amax");
  if (rows < 0 || cols < 0 || amax == nullptr) return FP8_ERR_INVALID_ARG;
  const int64_t n = rows * cols;
  if (n > 0 && x == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(amax, 4)) return FP8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  if (launch_zero_f32(amax, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
  if (n == 0) return FP8_OK;
  return cuda_status(launch_amax(x, n, amax, d->num_sms, stream));
}

fp8_status fp8_compute_scale(const float* amax, fp8_format fmt, float* scale, float* scale_inv,
                             cudaStream_t stream) {
  ApiRange nvtx_range("fp8_compute_scale");
  if (amax == nullptr || scale == nullptr || scale_inv == nullptr || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (!aligned(amax, 4) || !aligned(scale, 4) || !aligned(scale_inv, 4)) return FP8_ERR_ALIGNMENT;
  return cuda_status(launch_compute_scale(amax, fmt == FP8_E5M2, scale, scale_inv, stream));
}

fp8_status amax_history_update(float* hist, int32_t len, int32_t* pos, const float* amax, fp8_format fmt,
                               float* scale, float* scale_inv, cudaStream_t stream) {
  ApiRange nvtx_range("amax_history_update");
  if (hist == nullptr || pos == nullptr || amax == nullptr || scale == nullptr || scale_inv == nullptr || len < 1 ||
      !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (!aligned(hist, 4) || !aligned(pos, 4) || !aligned(amax, 4) || !aligned(scale, 4) || !aligned(scale_inv, 4))
    return FP8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  return cuda_status(launch_history_update(hist, len, pos, amax, fmt == FP8_E5M2, scale, scale_inv, d->err, stream));
}

fp8_status fp8_cast_transpose(const void* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                              const float* scale, float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col,
                              void* s_col, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_cast_transpose");
  return cast_transpose_impl(x, false, rows, cols, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, stream);
}

fp8_status fp8_cast_transpose_f32(const float* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                                  const float* scale, float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col,
                                  void* s_col, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_cast_transpose_f32");
  return cast_transpose_impl(x, true, rows, cols, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, stream);
}

fp8_status fp8_amax_f32(const float* x, int64_t rows, int64_t cols, float* amax, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_amax_f32");
  if (rows < 0 || cols < 0 || amax == nullptr) return FP8_ERR_INVALID_ARG;
  const int64_t n = rows * cols;
  if (n > 0 && x == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(amax, 4)) return FP8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  if (launch_zero_f32(amax, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
  if (n == 0) return FP8_OK;
  return cuda_status(launch_amax_f32(x, n, amax, d->num_sms, stream));
}

}  // extern "C"

namespace {

fp8_status cast_transpose_impl(const void* x, bool f32, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                               const float* scale, float* amax_out, uint8_t* q_row, void* s_row, uint8_t* q_col,
                               void* s_col, cudaStream_t stream) {
  CastPlan plan;
  if (fp8_status st = plan_cast(x, rows, cols, recipe, fmt, scale, amax_out, q_row, s_row, q_col, s_col, &plan, f32))
    return st;
  if (plan.empty) {
    // nothing to cast (outputs of an empty tensor may be NULL); amax of nothing is 0
    if (amax_out != nullptr && launch_zero_f32(amax_out, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
    return FP8_OK;
  }
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  if (amax_out != nullptr && launch_zero_f32(amax_out, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
  plan.p.err = d->err;
  // only the per-tensor recipe can miss the tiled path (block recipes imply its alignment)
  if (f32) {
    if (!plan.tiled) return cuda_status(launch_cast_generic_f32(plan.p, x, stream));
    return cuda_status(launch_cast_transpose_tiled_f32(plan.p, plan.tm_x, plan.tm_qr, plan.tm_qc, d->num_sms, stream));
  }
  if (!plan.tiled) return cuda_status(launch_cast_generic(plan.p, x, stream));
  return cuda_status(launch_cast_transpose_tiled(plan.p, plan.tm_x, plan.tm_qr, plan.tm_qc, d->num_sms, stream));
}

}  // namespace

extern "C" {

fp8_status fp8_cast_transpose_multi(const fp8_cast_job* jobs, int32_t n_jobs, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_cast_transpose_multi");
  if (n_jobs < 0 || n_jobs > kMaxCastJobs || (n_jobs > 0 && jobs == nullptr)) return FP8_ERR_INVALID_ARG;
  CastPlan plans[kMaxCastJobs];
  // every job is checked before any device work
  for (int i = 0; i < n_jobs; ++i) {
    const fp8_cast_job& j = jobs[i];
    if (fp8_status st = plan_cast(j.x, j.rows, j.cols, j.recipe, j.fmt, j.scale, j.amax_out, j.q_row, j.s_row, j.q_col,
                                  j.s_col, &plans[i]))
      return st;
  }
  if (n_jobs == 0) return FP8_OK;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  CastJobs launch{};
  for (int i = 0; i < n_jobs; ++i) {
    CastPlan& pl = plans[i];
    if (jobs[i].amax_out != nullptr && launch_zero_f32(jobs[i].amax_out, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
    if (pl.empty) continue;
    pl.p.err = d->err;
    if (!pl.tiled) {
      if (fp8_status st = cuda_status(launch_cast_generic(pl.p, jobs[i].x, stream))) return st;
      continue;
    }
    launch.p[launch.n] = pl.p;
    launch.m[launch.n].x = pl.tm_x;
    launch.m[launch.n].qrow = pl.tm_qr;
    launch.m[launch.n].qcol = pl.tm_qc;
    launch.tile_start[launch.n + 1] = launch.tile_start[launch.n] + pl.p.tiles_r * pl.p.tiles_c;
    ++launch.n;
  }
  if (launch.n == 0) return FP8_OK;
  return cuda_status(launch_cast_jobs(launch, d->num_sms, stream));
}

fp8_status fp8_quantize(const void* x, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                        const float* scale, float* amax_out, uint8_t* q, void* s, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_quantize");
  if (q == nullptr && rows > 0 && cols > 0) return FP8_ERR_INVALID_ARG;
  return fp8_cast_transpose(x, rows, cols, recipe, fmt, scale, amax_out, q, s, nullptr, nullptr, stream);
}

fp8_status fp8_dequantize(const uint8_t* q, int64_t rows, int64_t cols, fp8_recipe recipe, fp8_format fmt,
                          const void* s, void* y, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_dequantize");
  if (rows < 0 || cols < 0 || !valid_fmt(fmt) || !valid_recipe(recipe)) return FP8_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return FP8_OK;
  if (q == nullptr || s == nullptr || y == nullptr) return FP8_ERR_INVALID_ARG;
  if (rows > kMaxDim || cols > kMaxDim) return FP8_ERR_SHAPE;
  switch (recipe) {
    case FP8_BLOCK_1x128:
      if (cols % 128) return FP8_ERR_SHAPE;
      break;
    case FP8_BLOCK_128x128:
    case FP8_MX_1x32_TILED:
    case FP8_MX_1x32_FLOOR_TILED:
      if (rows % 128 || cols % 128) return FP8_ERR_SHAPE;
      break;
    case FP8_MX_1x32:
    case FP8_MX_1x32_FLOOR:
      if (cols % 32) return FP8_ERR_SHAPE;
      break;
    default:
      break;
  }
  if (!aligned(q, 16) || !aligned(y, 16)) return FP8_ERR_ALIGNMENT;
  const bool mx = is_mx(recipe);
  if (!mx && !aligned(s, 4)) return FP8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  const int kind = recipe == FP8_TENSOR ? kTensor : recipe == FP8_BLOCK_1x128 ? kBlock1x128
                   : recipe == FP8_BLOCK_128x128 ? kBlock128x128 : kMx;
  return cuda_status(launch_dequantize(q, rows, cols, kind, is_mx_tiled(recipe), fmt == FP8_E5M2, s, y,
                                       d->num_sms, stream));
}

fp8_status fp8_allreduce_sum(const void* g, int32_t k, int64_t n, fp8_format fmt, float* amax, uint8_t* q,
                             float* scale_inv, float* out, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_allreduce_sum");
  if (k < 1 || n < 0 || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (n == 0) return FP8_OK;
  if (g == nullptr || amax == nullptr || q == nullptr || scale_inv == nullptr || out == nullptr)
    return FP8_ERR_INVALID_ARG;
  if (n % 8 || n > kMaxDim || static_cast<int64_t>(k) * n / k != n) return FP8_ERR_SHAPE;
  if (!aligned(g, 16) || !aligned(out, 16) || !aligned(q, 8) || !aligned(amax, 4) || !aligned(scale_inv, 4))
    return FP8_ERR_ALIGNMENT;
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  if (launch_zero_f32(amax, 1, stream) != cudaSuccess) return FP8_ERR_CUDA;
  if (fp8_status st = cuda_status(launch_amax(g, static_cast<int64_t>(k) * n, amax, d->num_sms, stream))) return st;
  return cuda_status(launch_allreduce(g, k, n, amax, fmt == FP8_E5M2, q, scale_inv, out, d->num_sms, stream));
}

fp8_status fp8_allreduce_sum_noalloc(const void* g, int32_t k, int64_t n, fp8_format fmt, uint8_t* q, float* scale_inv,
                                     float* out, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_allreduce_sum_noalloc");
  if (k < 1 || n < 0 || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (k > noalloc_max_ranks()) return FP8_ERR_SHAPE;   // more ranks than the scratch has slots
  if (n == 0) return FP8_OK;
  if (g == nullptr || q == nullptr || scale_inv == nullptr || out == nullptr) return FP8_ERR_INVALID_ARG;
  if (n % 8 || n > kMaxDim) return FP8_ERR_SHAPE;
  if (!aligned(g, 16) || !aligned(out, 16) || !aligned(q, 8) || !aligned(scale_inv, 4)) return FP8_ERR_ALIGNMENT;
  const cudaError_t e = launch_allreduce_noalloc(g, k, n, fmt == FP8_E5M2, q, scale_inv, out, stream);
  // the first call on a device was made inside a stream capture: refused before any work
  if (e == cudaErrorStreamCaptureUnsupported) return FP8_ERR_INVALID_ARG;
  return cuda_status(e);
}

fp8_status fp8_scaled_gemm(const uint8_t* A, fp8_format fa, fp8_recipe ra, const void* sA, const uint8_t* B,
                           fp8_format fb, fp8_recipe rb, const void* sB, int64_t M, int64_t N, int64_t K, void* C,
                           fp8_out_dtype out, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_scaled_gemm");
  return scaled_gemm(A, fa, ra, sA, B, fb, rb, sB, M, N, K, C, out, GemmExtra{}, stream);
}

fp8_status fp8_scaled_gemm_amax(const uint8_t* A, fp8_format fa, fp8_recipe ra, const void* sA, const uint8_t* B,
                                fp8_format fb, fp8_recipe rb, const void* sB, int64_t M, int64_t N, int64_t K, void* C,
                                fp8_out_dtype out, float* c_amax, const float* c_scale, fp8_format fc, uint8_t* C_q,
                                float* c_scale_inv, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_scaled_gemm_amax");
  if (c_amax == nullptr && C_q == nullptr) return FP8_ERR_INVALID_ARG;
  GemmExtra x;
  x.c_amax = c_amax;
  x.c_scale = c_scale;
  x.fc = fc;
  x.cq = C_q;
  x.c_scale_inv = c_scale_inv;
  return scaled_gemm(A, fa, ra, sA, B, fb, rb, sB, M, N, K, C, out, x, stream);
}

fp8_status fp8_get_device_status(cudaStream_t stream) {
  ApiRange nvtx_range("fp8_get_device_status");
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FP8_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, d->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(d->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FP8_ERR_CUDA;
  }
  if (word & (kErrTimeoutTmaLoad | kErrTimeoutMma | kErrTimeoutStage)) return FP8_ERR_TIMEOUT;
  if (word & kErrBadState) return FP8_ERR_DEVICE_STATE;
  if (word & kErrIndex) return FP8_ERR_INDEX;
  return FP8_OK;
}

fp8_status fp8_debug_gemm_plan(fp8_recipe ra, fp8_recipe rb, fp8_out_dtype out, int64_t M, int64_t N, int64_t K,
                               int32_t fused, int32_t num_sms, int32_t resident_pairs, int64_t* plan) {
  if (plan == nullptr || M <= 0 || N <= 0 || K <= 0 || num_sms < 2 || (out != FP8_OUT_BF16 && out != FP8_OUT_FP32))
    return FP8_ERR_INVALID_ARG;
  int kind, b_1x128;
  if (fp8_status st = gemm_kind(ra, rb, &kind, &b_1x128)) return st;
  if (M % 128 || N % 128 || K % 128) return FP8_ERR_SHAPE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8_ERR_SHAPE;
  // the parameters the dispatch reads; the pointers only say which outputs exist
  static uint8_t present;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.kind = kind;
  p.b_1x128 = b_1x128;
  p.out_fp32 = out == FP8_OUT_FP32;
  p.c = &present;
  if (fused) p.cq = &present;
  p.wide160 = gemm_select_wide(p, num_sms) ? 1 : 0;
  const GemmPlan g = gemm_plan(p, num_sms, resident_pairs);
  plan[0] = g.pair;
  plan[1] = g.variant;
  plan[2] = g.block_n;
  plan[3] = g.ntiles;
  plan[4] = g.div.streamk;
  plan[5] = g.div.split;
  plan[6] = g.div.tail0;
  plan[7] = g.div.launched;
  return FP8_OK;
}

fp8_status fp8_debug_index_check(int64_t index, int64_t extent, cudaStream_t stream) {
  ApiRange nvtx_range("fp8_debug_index_check");
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  return cuda_status(launch_index_selftest(index, extent, d->err, stream));
}

fp8_status fp8_debug_wait_timeout(cudaStream_t stream) {
  ApiRange nvtx_range("fp8_debug_wait_timeout");
  DeviceInfo* d;
  if (fp8_status st = device_info(&d)) return st;
  return cuda_status(launch_wait_selftest(d->err, stream));
}

}  // extern "C"
