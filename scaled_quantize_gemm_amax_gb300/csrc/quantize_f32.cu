// quantize_f32.cu -- quantize / cast-transpose of a binary32 matrix (e.g. the FP32
// master copy of a weight) into row-wise and column-wise FP8 plus scales, for the
// four recipes of quantize.cu.  The search-result page's mixed-precision dataflow
// paragraph keeps weights in higher precision and quantizes that copy to FP8; reading
// the binary32 values directly means no bf16 copy of the weight is written and read
// again, and the element rule is the same: q = saturating RNE FP8 of (x * scale), one
// binary32 product, block amaxes over the binary32 values (NaN ignored).
//
// Design (tiled path): a persistent grid, one CTA per SM, 512 threads, 128 x 128 tiles.
// A 2-stage ring of 64 KB tiles is filled by TMA (four 32-column boxes, 128-byte
// swizzle).  For each tile:
//   row pass  -- warp w owns rows 8w .. 8w+7, lane l columns 4l .. 4l+3 (16-byte shared
//                loads, conflict-free); the 8 rows' 1x128 (or 1x32 MX block) maxima are
//                reduce-scattered over the warp (or the block's 8 lanes), so each lane
//                computes one scale, and the scales return by shuffles;
//   col pass  -- warp w owns columns 32 (w % 4) + lane over rows 32 (w / 4) .. +31 (one
//                MX block along the rows; scalar shared loads, conflict-free); a column's
//                1x128 amax combines the four row quarters through shared memory;
//   staged FP8 tiles (double-buffered) leave through TMA stores.
#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 2;
constexpr int kTile = 128;
constexpr uint32_t kXBytes = kTile * kTile * 4;      // 64 KB binary32 tile
constexpr uint32_t kQBytes = kTile * kTile;          // 16 KB fp8 tile
constexpr uint32_t kOffOutR = kStages * kXBytes;     // 128 KB
constexpr uint32_t kOffOutT = kOffOutR + 2 * kQBytes;
constexpr uint32_t kOffBar = kOffOutT + 2 * kQBytes;  // 192 KB
constexpr uint32_t kOffRed = kOffBar + 64;            // [2][kWarps] block maxima
constexpr uint32_t kOffCol = kOffRed + 2 * kWarps * 4;   // [4][128] column-quarter maxima
// MX with the tiled layout: [tile parity][row, col][512 B], one tile's exponents of a copy
// (exactly one atom of the GEMM-ready layout), sent out by one bulk copy each
constexpr uint32_t kOffSf = kOffCol + 4 * kTile * 4;
constexpr uint32_t kSmemBytes = kOffSf + 2 * 2 * 512 + 1024;   // + alignment slack

// Element (r, c) of a binary32 tile held as four 32-column boxes, each [128 rows][128 B]
// with the 128-byte swizzle (16-byte chunk k of row r at chunk k ^ (r % 8)).
__device__ __forceinline__ uint32_t xf_addr(uint32_t base, int r, int c) {
  return base + ((c >> 5) << 14) + (r << 7) + ((((c >> 2) & 7) ^ (r & 7)) << 4) + ((c & 3) << 2);
}
// Byte (r, c) of a [128][128 B] swizzled fp8 tile.
__device__ __forceinline__ uint32_t q_addr(uint32_t base, int r, int c) {
  return base + (r << 7) + ((((c >> 4) ^ (r & 7))) << 4) + (c & 15);
}

__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds32f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// max(m, |v|) with NaN ignored (fmaxf returns the other operand of a NaN)
__device__ __forceinline__ float absmax4(float m, float4 v) {
  return fmaxf(fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fabsf(v.y)), fabsf(v.z)), fabsf(v.w));
}
// four binary32 values times s -> four FP8 bytes (first value in the low byte)
__device__ __forceinline__ uint32_t q4(float4 v, float s, bool e5) {
  return cvt_pair(__fmul_rn(v.x, s), __fmul_rn(v.y, s), e5) | (cvt_pair(__fmul_rn(v.z, s), __fmul_rn(v.w, s), e5) << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Block maximum with one barrier; the caller alternates two `red` buffers (a buffer is
// written again only two calls later, after every thread has passed the caller's own
// barrier in between).
__device__ __forceinline__ float block_max_1(float v, float* red, int warp, int lane) {
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, red[w]);
  return r;
}

// The GEMM-ready tiled E8M0 layout: 128-row x 4-block atoms of 512 B, atom (r/128, b/4)
// at ((r/128) * atoms_per_row + b/4) * 512; exponent (local row r, local block b) at
// (r%32)*16 + (r/32)*4 + b inside it.
__device__ __forceinline__ uint32_t mx_atom_offset(int r, int b) {
  return static_cast<uint32_t>((r & 31) * 16 + (r >> 5) * 4 + b);
}
__device__ __forceinline__ void sts8(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

template <int RECIPE>
__device__ __forceinline__ void cast_tile_f32(const CastParams& p, uint32_t xs, uint32_t outR, uint32_t outT, int tr,
                                              int tc, int64_t row0, int64_t col0, float g_scale, float& thr_amax,
                                              float* red, float* colmax, uint32_t sf, int warp, int lane) {
  const bool e5 = p.e5m2 != 0;
  const float fmax = fmax_of(e5);
  const int fexp = fmax_exp_of(e5);
  const int64_t nb128_c = p.C / 128, nb128_r = p.R / 128, nb32_c = p.C / 32, nb32_r = p.R / 32;
  // ---------------- row pass
  float4 v[8];
  float a[8];
  float tmax_local = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = lds128f(xf_addr(xs, 8 * warp + i, 4 * lane));
    a[i] = absmax4(0.0f, v[i]);
    tmax_local = fmaxf(tmax_local, a[i]);
  }
  thr_amax = fmaxf(thr_amax, tmax_local);
  float tile_scale = g_scale;
  if (RECIPE == kBlock128x128) {
    const float tmax = block_max_1(tmax_local, red, warp, lane);
    tile_scale = scale_from_amax(tmax, fmax);
    if (warp == 0 && lane == 0) {
      const float si = recip_rn(tile_scale);
      const int64_t nblk = nb128_r * nb128_c;
      if (p.do_row && p.s_row) FP8Q_GUARD(tr * nb128_c + tc, 1, nblk, p.err) {
        static_cast<float*>(p.s_row)[tr * nb128_c + tc] = si;
      }
      if (p.do_col && p.s_col) FP8Q_GUARD(tc * nb128_r + tr, 1, nblk, p.err) {
        static_cast<float*>(p.s_col)[tc * nb128_r + tr] = si;
      }
    }
  }
  if (p.do_row) {
    // the scale of each of this lane's 8 rows
    float sc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i] = tile_scale;
    if (RECIPE == kBlock1x128 || RECIPE == kMx) {
      // Reduce-scatter the 8 rows' maxima: each exchange halves the rows a lane keeps, so
      // one scale computation per lane serves a whole row (1x128: lanes 4r .. 4r+3 end with
      // row r's maximum over the warp) or a whole 1x32 block (MX: lane 8b + r ends with row
      // r's maximum over block b's 8 lanes); the scales then go back by shuffles.
      constexpr int X0 = RECIPE == kMx ? 4 : 16, X1 = X0 / 2, X2 = X0 / 4;
      const bool k0 = lane & X0, k1 = lane & X1, k2 = lane & X2;
      float b4[4], b2[2];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        b4[k] = fmaxf(k0 ? a[k + 4] : a[k], __shfl_xor_sync(0xFFFFFFFFu, k0 ? a[k] : a[k + 4], X0));
#pragma unroll
      for (int k = 0; k < 2; ++k)
        b2[k] = fmaxf(k1 ? b4[k + 2] : b4[k], __shfl_xor_sync(0xFFFFFFFFu, k1 ? b4[k] : b4[k + 2], X1));
      float m = fmaxf(k2 ? b2[1] : b2[0], __shfl_xor_sync(0xFFFFFFFFu, k2 ? b2[0] : b2[1], X2));
      // the row this lane now holds: 4 k0 + 2 k1 + k2
      const int rr = (k0 ? 4 : 0) + (k1 ? 2 : 0) + (k2 ? 1 : 0);
      const int64_t grow = row0 + 8 * warp + rr;
      float s_mine;
      if (RECIPE == kBlock1x128) {
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        s_mine = scale_from_amax(m, fmax);
        if ((lane & 3) == 0 && grow < p.R) FP8Q_GUARD(grow * nb128_c + tc, 1, p.R * nb128_c, p.err) {
          static_cast<float*>(p.s_row)[grow * nb128_c + tc] = recip_rn(s_mine);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i] = __shfl_sync(0xFFFFFFFFu, s_mine, 4 * i);
      } else {
        const int e = (p.mx_floor ? mx_exponent_floor(m, fexp) : mx_exponent(m, fexp));
        s_mine = pow2_neg(e);
        const int64_t b = static_cast<int64_t>(tc) * 4 + (lane >> 3);
        if (p.mx_tiled)   // the tile's atom (both dims are multiples of 128)
          sts8(sf + mx_atom_offset(8 * warp + rr, lane >> 3), static_cast<uint32_t>(e + 127));
        else if (grow < p.R && b < nb32_c)   // a tile hanging over C has blocks past the last one
          FP8Q_GUARD(grow * nb32_c + b, 1, p.R * nb32_c, p.err) {
            static_cast<uint8_t*>(p.s_row)[grow * nb32_c + b] = static_cast<uint8_t>(e + 127);
          }
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[i] = __shfl_sync(0xFFFFFFFFu, s_mine, (lane & ~7) | i);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sts32(q_addr(outR, 8 * warp + i, 4 * lane), q4(v[i], sc[i], e5));
  }
  // ---------------- col pass
  if (p.do_col) {
    const int cg = warp & 3, rq = warp >> 2;
    const int c = 32 * cg + lane;
    const int64_t gcol = col0 + c;
    float w[32];
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      w[i] = lds32f(xf_addr(xs, 32 * rq + i, c));
      am = fmaxf(am, fabsf(w[i]));
    }
    float s = tile_scale;
    if (RECIPE == kBlock1x128) {
      colmax[rq * kTile + c] = am;
      __syncthreads();
      const float m = fmaxf(fmaxf(colmax[c], colmax[kTile + c]), fmaxf(colmax[2 * kTile + c], colmax[3 * kTile + c]));
      s = scale_from_amax(m, fmax);
      if (rq == 0 && gcol < p.C) FP8Q_GUARD(gcol * nb128_r + tr, 1, p.C * nb128_r, p.err) {
        static_cast<float*>(p.s_col)[gcol * nb128_r + tr] = recip_rn(s);
      }
    } else if (RECIPE == kMx) {
      const int e = (p.mx_floor ? mx_exponent_floor(am, fexp) : mx_exponent(am, fexp));
      s = pow2_neg(e);
      const int64_t b = static_cast<int64_t>(tr) * 4 + rq;
      if (p.mx_tiled)
        sts8(sf + 512 + mx_atom_offset(c, rq), static_cast<uint32_t>(e + 127));
      else if (gcol < p.C && b < nb32_r)
        FP8Q_GUARD(gcol * nb32_r + b, 1, p.C * nb32_r, p.err) {
          static_cast<uint8_t*>(p.s_col)[gcol * nb32_r + b] = static_cast<uint8_t>(e + 127);
        }
    }
    uint32_t qw[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) qw[k] = q4(make_float4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]), s, e5);
    // row c of the column-wise staging tile, bytes 32 rq .. 32 rq + 31 (chunks 2 rq, 2 rq + 1)
    const uint32_t rowb = outT + (static_cast<uint32_t>(c) << 7);
    sts128(rowb + (((2 * rq) ^ (c & 7)) << 4), qw[0], qw[1], qw[2], qw[3]);
    sts128(rowb + (((2 * rq + 1) ^ (c & 7)) << 4), qw[4], qw[5], qw[6], qw[7]);
  }
}

template <int RECIPE>
__global__ void __launch_bounds__(kThreads, 1)
    k_cast_transpose_f32(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_qrow,
                         const __grid_constant__ CUtensorMap tm_qcol, const CastParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  float* const red = reinterpret_cast<float*>(base_ptr + kOffRed);
  float* const colmax = reinterpret_cast<float*>(base_ptr + kOffCol);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = p.tiles_r * p.tiles_c;

  if (tid == 0) {
    prefetch_tmap(&tm_x);
    if (p.do_row) prefetch_tmap(&tm_qrow);
    if (p.do_col) prefetch_tmap(&tm_qcol);
    for (int s = 0; s < kStages; ++s) mbar_init(base + kOffBar + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // with amax_out a zeroing kernel ran just before this one: only the atomic waits (as the
  // BF16-input kernel)
  const bool zeroed = p.amax_out != nullptr;
  if (!zeroed) pdl_wait();   // from here on: global memory
  pdl_launch_dependents();

  float g_scale = 1.0f;
  if (RECIPE == kTensor) {
    g_scale = *p.scale;
    if (blockIdx.x == 0 && tid == 0) {
      const float si = recip_rn(g_scale);
      if (p.do_row && p.s_row) *static_cast<float*>(p.s_row) = si;
      if (p.do_col && p.s_col) *static_cast<float*>(p.s_col) = si;
    }
  }

  auto issue_load = [&](int it, int tile) {
    const int s = it % kStages;
    const uint32_t bar = base + kOffBar + 8 * s;
    const int row0 = (tile / p.tiles_c) * kTile, col0 = (tile % p.tiles_c) * kTile;
    mbar_arrive_expect_tx(bar, kXBytes);
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_load_2d(base + s * kXBytes + b * (kXBytes / 4), &tm_x, col0 + 32 * b, row0, bar);
  };
  if (tid == 0) {
    for (int it = 0; it < kStages; ++it) {
      const int tile = blockIdx.x + it * gridDim.x;
      if (tile < ntiles) issue_load(it, tile);
    }
  }

  float thr_amax = 0.0f;
  int it = 0;
  bool failed = false;
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
    const int s = it % kStages;
    const uint32_t xs = base + s * kXBytes;
    const int ob = it & 1;
    const uint32_t outR = base + kOffOutR + ob * kQBytes;
    const uint32_t outT = base + kOffOutT + ob * kQBytes;
    const int tr = tile / p.tiles_c, tc = tile % p.tiles_c;
    const int64_t row0 = static_cast<int64_t>(tr) * kTile, col0 = static_cast<int64_t>(tc) * kTile;

    // One barrier a tile, plus one inside the body for the 128x128 tile maximum and one
    // for the 1x128 column maxima.  Staging buffer `ob` was last read by the stores of two
    // tiles ago, which thread 0 waited for before the previous tile's barrier.  A wait that
    // timed out still runs the body (its results are dropped) so that every thread reaches
    // the same barriers; the tile barrier then ends the loop on every thread.
    const bool ok = mbar_wait(base + kOffBar + 8 * s, (it / kStages) & 1, p.err, kErrTimeoutTmaLoad, nullptr);
    const uint32_t sf = base + kOffSf + static_cast<uint32_t>(ob) * 1024u;
    cast_tile_f32<RECIPE>(p, xs, outR, outT, tr, tc, row0, col0, g_scale, thr_amax, red + (it & 1) * kWarps, colmax, sf,
                          warp, lane);
    fence_proxy_async_smem();
    if (tid == 0) bulk_wait_read<0>();  // the previous tile's stores have read their staging buffer
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0) {
      if (p.do_row) tma_store_2d(&tm_qrow, outR, static_cast<int>(col0), static_cast<int>(row0));
      if (p.do_col) tma_store_2d(&tm_qcol, outT, static_cast<int>(row0), static_cast<int>(col0));
      if (RECIPE == kMx && p.mx_tiled) {   // the staged atoms: row copy's (tr, tc), column copy's (tc, tr)
        const int64_t atoms = static_cast<int64_t>(p.tiles_r) * p.tiles_c * 512;
        const int64_t orow = (static_cast<int64_t>(tr) * p.tiles_c + tc) * 512;
        const int64_t ocol = (static_cast<int64_t>(tc) * p.tiles_r + tr) * 512;
        if (p.do_row) FP8Q_GUARD(orow, 512, atoms, p.err) { bulk_store(static_cast<uint8_t*>(p.s_row) + orow, sf, 512); }
        if (p.do_col) FP8Q_GUARD(ocol, 512, atoms, p.err) { bulk_store(static_cast<uint8_t*>(p.s_col) + ocol, sf + 512, 512); }
      }
      bulk_commit();
      const int next = tile + kStages * gridDim.x;
      if (next < ntiles) issue_load(it + kStages, next);
    }
  }

  if (failed && tid == 0) {
    // wait (bounded) for loads still in flight into this CTA's ring before leaving
    for (int k = it; k < it + kStages; ++k) {
      const int tile = blockIdx.x + k * gridDim.x;
      if (tile >= ntiles) break;
      mbar_wait(base + kOffBar + 8 * (k % kStages), (k / kStages) & 1, p.err, kErrTimeoutTmaLoad, nullptr);
    }
  }
  if (tid == 0) bulk_wait_all<0>();

  if (zeroed) {
    // the block maximum (the red buffer of the next tile index is free: every thread has
    // passed the last tile barrier)
    float* const r = red + (it & 1) * kWarps;
    const float am = block_max_1(thr_amax, r, warp, lane);
    if (tid == 0) {
      pdl_wait();   // the zeroing of amax_out is done
      if (am > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(am));
    }
  }
}

// ------------------------------------------------------------------ per-tensor, any shape
// 32x32 tiles, 256 threads: row-wise bytes straight from the input, column-wise
// bytes through a transposed shared tile.
__global__ void __launch_bounds__(256) k_cast_generic_f32(const float* __restrict__ x, CastParams p) {
  __shared__ float tile[32][33];
  const bool zeroed = p.amax_out != nullptr;   // as the tiled kernel: only the atomic waits then
  if (!zeroed) pdl_wait();
  pdl_launch_dependents();
  const bool e5 = p.e5m2 != 0;
  const float s = *p.scale;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  float amax = 0.0f;
  for (int k = ty; k < 32; k += 8) {
    const int64_t r = r0 + k, c = c0 + tx;
    float v = 0.0f;
    if (r < p.R && c < p.C) {
      v = x[r * p.C + c];
      amax = fmaxf(amax, fabsf(v));
      if (p.do_row) FP8Q_GUARD(r * p.C + c, 1, p.R * p.C, p.err) {
        p.q_row[r * p.C + c] = static_cast<uint8_t>(cvt_pair(__fmul_rn(v, s), 0.0f, e5) & 0xFF);
      }
    }
    tile[k][tx] = v;
  }
  __syncthreads();
  if (p.do_col) {
    for (int k = ty; k < 32; k += 8) {
      const int64_t c = c0 + k, r = r0 + tx;
      if (r < p.R && c < p.C) FP8Q_GUARD(c * p.R + r, 1, p.R * p.C, p.err) {
        p.q_col[c * p.R + r] = static_cast<uint8_t>(cvt_pair(__fmul_rn(tile[tx][k], s), 0.0f, e5) & 0xFF);
      }
    }
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    const float si = recip_rn(s);
    if (p.do_row && p.s_row) *static_cast<float*>(p.s_row) = si;
    if (p.do_col && p.s_col) *static_cast<float*>(p.s_col) = si;
  }
  if (zeroed) {
    amax = warp_max(amax);
    if (tx == 0) {
      pdl_wait();
      if (amax > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(amax));
    }
  }
}

template <int RECIPE>
cudaError_t launch_tiled_f32(const CastParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_qrow,
                             const CUtensorMap& tm_qcol, int num_sms, cudaStream_t s) {
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_limit(k_cast_transpose_f32<RECIPE>, static_cast<int>(kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  const int ntiles = p.tiles_r * p.tiles_c;
  const int grid = ntiles < num_sms ? ntiles : num_sms;
  return launch_pdl(k_cast_transpose_f32<RECIPE>, dim3(grid), dim3(kThreads), kSmemBytes, s, 1, tm_x, tm_qrow, tm_qcol,
                    p);
}

}  // namespace

cudaError_t launch_cast_transpose_tiled_f32(const CastParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_qrow,
                                            const CUtensorMap& tm_qcol, int num_sms, cudaStream_t s) {
  switch (p.recipe) {
    case kTensor: return launch_tiled_f32<kTensor>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
    case kBlock1x128: return launch_tiled_f32<kBlock1x128>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
    case kBlock128x128: return launch_tiled_f32<kBlock128x128>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
    default: return launch_tiled_f32<kMx>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
  }
}

cudaError_t launch_cast_generic_f32(const CastParams& p, const void* x, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((p.C + 31) / 32), static_cast<unsigned>((p.R + 31) / 32));
  return launch_pdl(k_cast_generic_f32, grid, dim3(256), 0, s, 1, static_cast<const float*>(x), p);
}

}  // namespace fp8q
