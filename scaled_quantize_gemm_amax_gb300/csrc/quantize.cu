// quantize.cu -- quantize / cast-transpose of a BF16 matrix into row-wise and
// column-wise FP8 plus scales, for the four recipes:
//   per-tensor (current or delayed: the scale is an input),
//   blockwise 1x128 (rows of the stored copy) and 128x128,
//   MXFP8 1x32 with E8M0 exponents.
// (FP8 quantized-training guide: "tensor-level scaling", "block-level scaling",
// "MXFP8 scaling"; the column-wise copy feeds the backward GEMMs, which read the
// operands along the other axis -- the mixed-precision dataflow paragraph.)
//
// Design (tiled path): a persistent grid, one CTA per SM, 512 threads.  Each CTA
// walks 128x128 tiles of the input.  A 4-stage ring of 32 KB shared buffers is
// filled by TMA (two 64-column boxes, 128-byte swizzle).  For each tile:
//   row pass  -- 16-byte shared loads, 16 lanes per row; per-row / per-32 amax by
//                a shuffle reduce-scatter, so each lane derives one block scale and
//                the others receive it; quantized bytes go to a swizzled staging tile;
//   col pass  -- ldmatrix.trans gives each lane two consecutive rows of one column;
//                per-column amax by shuffles; bytes go to a second staging tile
//                already transposed;
//   both staging tiles leave through TMA stores (double-buffered), and one barrier
//   per tile separates a tile's shared-memory writes from its stores and the
//   refill of its ring slot.
// The optional per-tensor amax of the input (delayed scaling records it while
// casting with the previous scale) is a block max + one atomicMax per CTA.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 4;
constexpr int kTile = 128;
constexpr uint32_t kXBytes = kTile * kTile * 2;      // 32 KB bf16 tile
constexpr uint32_t kQBytes = kTile * kTile;          // 16 KB fp8 tile
constexpr uint32_t kOffOutR = kStages * kXBytes;     // 128 KB
constexpr uint32_t kOffOutT = kOffOutR + 2 * kQBytes;
constexpr uint32_t kOffBar = kOffOutT + 2 * kQBytes;  // 192 KB
constexpr uint32_t kOffRed = kOffBar + 64;
// MX with the tiled layout: a tile's exponents of one copy are exactly one 512-byte atom of
// the GEMM-ready layout; they are staged here ([tile parity][row, col][512 B]) and leave by
// one bulk copy each instead of 512 scattered byte stores
constexpr uint32_t kOffSf = kOffRed + 128;
constexpr uint32_t kSmemBytes = kOffSf + 2 * 2 * 512 + 1024;  // + alignment slack

// Address of 16-byte chunk `c16` (0..15) of row r in a bf16 tile held as two
// 64-column halves, each [128 rows][128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t x_addr(uint32_t base, int r, int c16) {
  return base + ((c16 >> 3) << 14) + (r << 7) + ((((c16 & 7) ^ (r & 7))) << 4);
}
// Byte (r, c) of a [128][128 B] swizzled fp8 tile, c a multiple of 2.
__device__ __forceinline__ uint32_t q_addr(uint32_t base, int r, int c) {
  return base + (r << 7) + ((((c >> 4) ^ (r & 7))) << 4) + (c & 15);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts8(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(static_cast<uint16_t>(v)) : "memory");
}
// A 1x128 column-scale store with the L2 evict-last policy: a 32-byte sector of the
// column-scale array ([C, R/128] floats) is written by 8 tile-rows, one tile-row at a time,
// and should stay in L2 until it is complete rather than leave partly written (a row-scale
// sector is completed by 8 neighbouring tiles of one tile-row, within one round).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_f32_l2_last(float* a, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t a, uint32_t (&d)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
               : "r"(a));
}

// Running max of |.| over bf16 pairs: the magnitude of max.xorsign.abs is
// max(|a|, |b|) (its sign bit is meaningless and masked at the end); NaN inputs
// are ignored.
__device__ __forceinline__ uint32_t xabs_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float pair_abs_f32(uint32_t m) { return pair_max_f32(m & 0x7FFF7FFFu); }
__device__ __forceinline__ float absmax_chunk(uint4 v) {
  return pair_abs_f32(xabs_max(xabs_max(v.x, v.y), xabs_max(v.z, v.w)));
}

// Quantize one bf16 pair with scale s -> two FP8 bytes (low half -> low byte):
// both binary32 products in one packed multiply, then the saturating cast.
__device__ __forceinline__ uint32_t q_pair(uint32_t w, float s, bool e5) {
  uint64_t x2, s2, p2;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x2) : "r"(w << 16), "r"(w & 0xFFFF0000u));
  asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(s));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p2) : "l"(x2), "l"(s2));
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p2));
  return cvt_pair(lo, hi, e5);
}
// Eight bf16 (one 16-byte chunk) -> eight FP8 bytes.
__device__ __forceinline__ uint2 q_chunk(uint4 w, float s, bool e5) {
  uint2 r;
  r.x = q_pair(w.x, s, e5) | (q_pair(w.y, s, e5) << 16);
  r.y = q_pair(w.z, s, e5) | (q_pair(w.w, s, e5) << 16);
  return r;
}

// Reduce-scatter of four per-lane maxima a[0..3] over the four lanes
// {l, l^hi, l^lo, l^hi^lo}: afterwards lane l holds the maximum of
// a[2*(l has hi) + (l has lo)] over those lanes (two rounds, three shuffles).
__device__ __forceinline__ float reduce_scatter4(const float (&a)[4], int lane, int hi, int lo) {
  const bool h = (lane & hi) != 0;
  float k0 = h ? a[2] : a[0], k1 = h ? a[3] : a[1];
  const float s0 = h ? a[0] : a[2], s1 = h ? a[1] : a[3];
  k0 = fmaxf(k0, __shfl_xor_sync(0xFFFFFFFFu, s0, hi));
  k1 = fmaxf(k1, __shfl_xor_sync(0xFFFFFFFFu, s1, hi));
  const bool l = (lane & lo) != 0;
  const float keep = l ? k1 : k0, send = l ? k0 : k1;
  return fmaxf(keep, __shfl_xor_sync(0xFFFFFFFFu, send, lo));
}

// The same with one barrier, for a caller that alternates between two `red` buffers: a
// buffer is written again only two calls later, after every thread has passed the
// caller's own barrier in between.
__device__ __forceinline__ float block_max_1(float v, float* red, int warp, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float block_max(float v, float* red, int warp, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}


// One 128x128 tile already in shared memory (stage buffer xs): both passes, scales
// written to global memory, quantized bytes staged in outR (row-wise) and outT
// (column-wise) for the TMA stores.  thr_amax accumulates this thread's |x| maximum.
// `red` is this tile's block-maximum buffer (the caller alternates two), and every
// thread of the CTA calls this (the 128x128 recipe synchronises inside).
// The staged atoms of tile (tr, tc) to their places in the tiled scale arrays: the row
// copy's atom (tr, tc) of [R, C], the column copy's atom (tc, tr) of [C, R].
__device__ __forceinline__ void store_mx_atoms(const CastParams& p, uint32_t sf, int tr, int tc) {
  const int64_t atoms = static_cast<int64_t>(p.tiles_r) * p.tiles_c * 512;   // bytes of either tiled array
  const int64_t orow = (static_cast<int64_t>(tr) * p.tiles_c + tc) * 512, ocol = (static_cast<int64_t>(tc) * p.tiles_r + tr) * 512;
  if (p.do_row) FP8Q_GUARD(orow, 512, atoms, p.err) { bulk_store(static_cast<uint8_t*>(p.s_row) + orow, sf, 512); }
  if (p.do_col) FP8Q_GUARD(ocol, 512, atoms, p.err) { bulk_store(static_cast<uint8_t*>(p.s_col) + ocol, sf + 512, 512); }
}

// The GEMM-ready tiled E8M0 layout: 128-row x 4-block atoms of 512 B, atom (r/128, b/4)
// at ((r/128) * atoms_per_row + b/4) * 512; exponent (local row r, local block b) at
// (r%32)*16 + (r/32)*4 + b inside it.
__device__ __forceinline__ uint32_t mx_atom_offset(int r, int b) {
  return static_cast<uint32_t>((r & 31) * 16 + (r >> 5) * 4 + b);
}

// A 1x128 tile with both copies.  The row maxima (each row's 128 columns of the tile) and
// the column maxima (each column's 128 rows) are both found before any scale is formed, so
// that one correctly rounded division and one reciprocal a lane serve both copies: in each
// group of four lanes, lanes 0-1 form their row's scale and lanes 2-3 their column's.  Same
// bytes and scales as the two passes of cast_tile_body.
__device__ __forceinline__ void cast_tile_1x128_both(const CastParams& p, uint32_t xs, uint32_t outR, uint32_t outT,
                                                     int tr, int tc, int64_t row0, int64_t col0, float& thr_amax,
                                                     int warp, int lane) {
  const bool e5 = p.e5m2 != 0;
  const float fmax = fmax_of(e5);
  const int64_t nb128_c = p.C / 128, nb128_r = p.R / 128;
  const int j = lane & 15;
  // rows i*32 + 2w + (lane / 16), 16-byte chunk j
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = lds128(x_addr(xs, i * 32 + warp * 2 + (lane >> 4), j));
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = absmax_chunk(v[i]);
  thr_amax = fmaxf(thr_amax, fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])));
  // row i = j / 4 ends up in lanes j = 4i..4i+3 of each half-warp
  float mr = reduce_scatter4(a, lane, 8, 4);
  mr = fmaxf(mr, __shfl_xor_sync(0xFFFFFFFFu, mr, 2));
  mr = fmaxf(mr, __shfl_xor_sync(0xFFFFFFFFu, mr, 1));
  // column cc = 8w + lane / 4, transposed: lanes 4k..4k+3 hold its 128 rows between them
  uint32_t d[4][4];
#pragma unroll
  for (int t = 0; t < 4; ++t) ldsm_x4_trans(x_addr(xs, 32 * t + 8 * (lane >> 3) + (lane & 7), warp), d[t]);
  uint32_t mb = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) mb = xabs_max(mb, d[t][q]);
  float mc = pair_abs_f32(mb);
  mc = fmaxf(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, 1));
  mc = fmaxf(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, 2));
  const float y = scale_from_amax((lane & 2) ? mc : mr, fmax);
  const float yi = recip_rn(y);
  const int64_t grow = row0 + (j >> 2) * 32 + warp * 2 + (lane >> 4);
  if ((j & 3) == 0 && grow < p.R) FP8Q_GUARD(grow * nb128_c + tc, 1, p.R * nb128_c, p.err) {
    static_cast<float*>(p.s_row)[grow * nb128_c + tc] = yi;
  }
  const int cc = 8 * warp + (lane >> 2);
  const int64_t gcol = col0 + cc;
  if ((lane & 3) == 2 && gcol < p.C) FP8Q_GUARD(gcol * nb128_r + tr, 1, p.C * nb128_r, p.err) {
    float* const dst = static_cast<float*>(p.s_col) + gcol * nb128_r + tr;
    if (p.keep_col_scales) st_f32_l2_last(dst, yi, l2_evict_last_policy());
    else *dst = yi;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float sr = __shfl_sync(0xFFFFFFFFu, y, (lane & 16) | (i << 2));
    const int r = i * 32 + warp * 2 + (lane >> 4);
    const uint2 q = q_chunk(v[i], sr, e5);
    sts64(outR + (r << 7) + ((((j >> 1) ^ (r & 7))) << 4) + ((j & 1) << 3), q.x, q.y);
  }
  const float s1 = __shfl_sync(0xFFFFFFFFu, y, (lane & ~3) | 2);
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) sts16(q_addr(outT, cc, 32 * t + 8 * q + 2 * (lane & 3)), q_pair(d[t][q], s1, e5));
}

template <int RECIPE>
__device__ __forceinline__ void cast_tile_body(const CastParams& p, uint32_t xs, uint32_t outR, uint32_t outT, int tr,
                                               int tc, int64_t row0, int64_t col0, float g_scale, float& thr_amax,
                                               float* red, uint32_t sf, int tid, int warp, int lane) {
  const bool e5 = p.e5m2 != 0;
  const float fmax = fmax_of(e5);
  const int fexp = fmax_exp_of(e5);
  const int64_t nb128_c = p.C / 128, nb128_r = p.R / 128, nb32_c = p.C / 32, nb32_r = p.R / 32;
  const int j = lane & 15;
  if (RECIPE == kBlock1x128 && p.do_row && p.do_col && p.one_division) {
    cast_tile_1x128_both(p, xs, outR, outT, tr, tc, row0, col0, thr_amax, warp, lane);
    return;
  }
  // Recipes whose two copies share one scale per tile (per-tensor, 128x128): the column
  // copy is the byte transpose of the row copy.  When the launcher chose that (col_from_row),
  // each warp quantizes 8 consecutive rows, so that its column pass transposes the bytes it
  // staged itself; otherwise rows i*32 + 2w and +1 (the row scales' reduce-scatter depends
  // on that order).
  constexpr bool kOneScale = RECIPE == kTensor || RECIPE == kBlock128x128;
  const bool contig = kOneScale && p.col_from_row != 0;
  auto row_of = [&](int i) { return contig ? 8 * warp + 2 * i + (lane >> 4) : i * 32 + warp * 2 + (lane >> 4); };
  // ---------------- row pass
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = lds128(x_addr(xs, row_of(i), j));
  float a[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = absmax_chunk(v[i]);

  float tile_scale = g_scale;
  if (RECIPE == kBlock128x128) {
    const float tmax = block_max_1(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), red, warp, lane);
    thr_amax = fmaxf(thr_amax, tmax);
    tile_scale = scale_from_amax(tmax, fmax);
    if (tid == 0) {
      const float si = recip_rn(tile_scale);
      const int64_t nblk = static_cast<int64_t>(nb128_r) * nb128_c;
      if (p.do_row && p.s_row) FP8Q_GUARD(static_cast<int64_t>(tr) * nb128_c + tc, 1, nblk, p.err) {
        static_cast<float*>(p.s_row)[tr * nb128_c + tc] = si;
      }
      if (p.do_col && p.s_col) FP8Q_GUARD(static_cast<int64_t>(tc) * nb128_r + tr, 1, nblk, p.err) {
        static_cast<float*>(p.s_col)[tc * nb128_r + tr] = si;
      }
    }
  } else {
    thr_amax = fmaxf(thr_amax, fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])));
  }

  if (p.do_row) {
    float sc[4] = {tile_scale, tile_scale, tile_scale, tile_scale};
    if (RECIPE == kBlock1x128) {
      // row i = j / 4 ends up in lanes j = 4i..4i+3 of each half-warp
      float m = reduce_scatter4(a, lane, 8, 4);
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      const float mine = scale_from_amax(m, fmax);
      const int64_t grow = row0 + (j >> 2) * 32 + warp * 2 + (lane >> 4);
      if ((j & 3) == 0 && grow < p.R) FP8Q_GUARD(grow * nb128_c + tc, 1, p.R * nb128_c, p.err) {
        static_cast<float*>(p.s_row)[grow * nb128_c + tc] = recip_rn(mine);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[i] = __shfl_sync(0xFFFFFFFFu, mine, (lane & 16) | (i << 2));
    } else if (RECIPE == kMx) {
      // the 32-column block of lane j is lanes 4 (j/4) .. +3; row i = j % 4 ends up in lane 4 (j/4) + i
      const float m = reduce_scatter4(a, lane, 2, 1);
      const int e = (p.mx_floor ? mx_exponent_floor(m, fexp) : mx_exponent(m, fexp));
      const float mine = pow2_neg(e);
      const int lrow = (j & 3) * 32 + warp * 2 + (lane >> 4);
      const int64_t grow = row0 + lrow;
      const int64_t b = tc * 4 + (j >> 2);
      if (p.mx_tiled) {
        sts8(sf + mx_atom_offset(lrow, j >> 2), static_cast<uint32_t>(e + 127));   // the tile's atom (dims % 128 == 0)
      } else if (grow < p.R && b < nb32_c) {   // a tile hanging over C has blocks past the last one
        FP8Q_GUARD(grow * nb32_c + b, 1, p.R * nb32_c, p.err) {
          static_cast<uint8_t*>(p.s_row)[grow * nb32_c + b] = static_cast<uint8_t>(e + 127);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[i] = __shfl_sync(0xFFFFFFFFu, mine, (lane & ~3) | i);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = row_of(i);
      const uint2 q = q_chunk(v[i], sc[i], e5);
      sts64(outR + (r << 7) + ((((j >> 1) ^ (r & 7))) << 4) + ((j & 1) << 3), q.x, q.y);
    }
  }

  // ---------------- col pass
  if (contig && p.do_col && p.do_row) {
    // This warp's rows 8w..8w+7 of the staged row copy, loaded transposed as 2-byte
    // elements: thread T gets, for each 16-byte column chunk m, rows ra = 8w + 2(T%4) and
    // ra + 1 at byte columns c = 16m + 2(T/4) and c + 1; column c's two bytes and column
    // c+1's go to the column copy's rows c and c+1 at byte ra.  The upper half-warp stores
    // column c+1 first, so that each store instruction meets eight different 16-byte
    // chunks of the swizzled tile (no bank conflict).
    __syncwarp();
    uint32_t d[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = 8 * warp + (lane & 7), m = 4 * h + (lane >> 3);
      ldsm_x4_trans(outR + (r << 7) + ((m ^ (r & 7)) << 4), d[h]);
    }
    const int ra = 8 * warp + 2 * (lane & 3), up = lane >> 4;
    const int c_first = 2 * (lane >> 2) + up, c_second = 2 * (lane >> 2) + 1 - up;
    const uint32_t sel_first = up ? 0x31u : 0x20u, sel_second = up ? 0x20u : 0x31u;
    const uint32_t a_first = q_addr(outT, c_first, ra), a_second = q_addr(outT, c_second, ra);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t m = static_cast<uint32_t>(4 * h + q);   // column chunk: rows c + 16m of the column copy
        sts16(a_first + (m << 11), __byte_perm(d[h][q], 0u, sel_first));
        sts16(a_second + (m << 11), __byte_perm(d[h][q], 0u, sel_second));
      }
  } else if (p.do_col) {
    const int g = warp;
    uint32_t d[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) ldsm_x4_trans(x_addr(xs, 32 * t + 8 * (lane >> 3) + (lane & 7), g), d[t]);
    const int cc = 8 * g + (lane >> 2);
    const int64_t gcol = col0 + cc;
    float sc[4] = {tile_scale, tile_scale, tile_scale, tile_scale};
    if (RECIPE == kBlock1x128) {
      uint32_t m = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int q = 0; q < 4; ++q) m = xabs_max(m, d[t][q]);
      float am = pair_abs_f32(m);
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
      const float s1 = scale_from_amax(am, fmax);
      sc[0] = sc[1] = sc[2] = sc[3] = s1;
      if ((lane & 3) == 0 && gcol < p.C) FP8Q_GUARD(gcol * nb128_r + tr, 1, p.C * nb128_r, p.err) {
        float* const dst = static_cast<float*>(p.s_col) + gcol * nb128_r + tr;
        if (p.keep_col_scales) st_f32_l2_last(dst, recip_rn(s1), l2_evict_last_policy());
        else *dst = recip_rn(s1);
      }
    } else if (RECIPE == kMx) {
      float at[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) at[t] = pair_abs_f32(xabs_max(xabs_max(d[t][0], d[t][1]), xabs_max(d[t][2], d[t][3])));
      // block t = lane % 4 of this column ends up in this lane
      const float m = reduce_scatter4(at, lane, 2, 1);
      const int e = (p.mx_floor ? mx_exponent_floor(m, fexp) : mx_exponent(m, fexp));
      const float mine = pow2_neg(e);
      const int64_t b = static_cast<int64_t>(tr) * 4 + (lane & 3);
      if (p.mx_tiled) {
        sts8(sf + 512 + mx_atom_offset(cc, lane & 3), static_cast<uint32_t>(e + 127));
      } else if (gcol < p.C && b < nb32_r) {
        FP8Q_GUARD(gcol * nb32_r + b, 1, p.C * nb32_r, p.err) {
          static_cast<uint8_t*>(p.s_col)[gcol * nb32_r + b] = static_cast<uint8_t>(e + 127);
        }
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) sc[t] = __shfl_sync(0xFFFFFFFFu, mine, (lane & ~3) | t);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r0 = 32 * t + 8 * q + 2 * (lane & 3);
        sts16(q_addr(outT, cc, r0), q_pair(d[t][q], sc[t], e5));
      }
  }

}

template <int RECIPE>
__global__ void __launch_bounds__(kThreads, 1)
    k_cast_transpose(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_qrow,
                     const __grid_constant__ CUtensorMap tm_qcol, const CastParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  float* const red = reinterpret_cast<float*>(base_ptr + kOffRed);
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
  // With amax_out, the host launched the zeroing of amax_out just before this kernel; that
  // kernel waited for every earlier one before letting this one start, so only the atomic
  // on amax_out has to wait (griddepcontrol.wait) for it.  Otherwise wait here.
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
    tma_load_2d(base + s * kXBytes, &tm_x, col0, row0, bar);
    tma_load_2d(base + s * kXBytes + kXBytes / 2, &tm_x, col0 + 64, row0, bar);
  };
  if (tid == 0) {
    for (int it = 0; it < kStages; ++it) {
      const int tile = blockIdx.x + it * gridDim.x;
      if (tile < ntiles) issue_load(it, tile);
    }
  }

  // Row pass: lane j = lane % 16 of a half-warp owns 16-byte chunk j of rows
  // r(i) = 32 i + 2 warp + lane / 16, i = 0..3.  Column pass: warp w owns the
  // 8-column chunk w; lane holds column 8 w + lane / 4, rows 32 t + 8 q + 2 (lane % 4) + {0, 1}.
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

    // One barrier a tile.  Staging buffer `ob` was last read by the stores of two tiles
    // ago, which thread 0 waited for before the previous tile's barrier.  A wait that
    // timed out still runs the body (its results are dropped) so that every thread
    // reaches the same barriers; the barrier then ends the loop on every thread.
    const bool ok = mbar_wait(base + kOffBar + 8 * s, (it / kStages) & 1, p.err, kErrTimeoutTmaLoad, nullptr);

    const uint32_t sf = base + kOffSf + static_cast<uint32_t>(ob) * 1024u;
    cast_tile_body<RECIPE>(p, xs, outR, outT, tr, tc, row0, col0, g_scale, thr_amax, red + (it & 1) * kWarps, sf, tid,
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
      if (RECIPE == kMx && p.mx_tiled) store_mx_atoms(p, sf, tr, tc);
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
    const float am = block_max(thr_amax, red, warp, lane);
    if (tid == 0) {
      pdl_wait();   // the zeroing of amax_out is done
      if (am > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(am));
    }
  }
}

// ------------------------------------------------------------------ per-tensor, any shape
// 32x32 tiles, 256 threads: row-wise bytes straight from the input, column-wise
// bytes through a transposed shared tile.
__global__ void __launch_bounds__(256) k_cast_generic(const uint16_t* __restrict__ x, CastParams p) {
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
      v = __uint_as_float(static_cast<uint32_t>(x[r * p.C + c]) << 16);
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (tx == 0) {
      pdl_wait();
      if (amax > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(amax));
    }
  }
}

// Several casts in one persistent grid: the tiles of job 0, then job 1, ... are dealt
// round-robin to the CTAs as in k_cast_transpose; each tile runs the body of its
// job's recipe and leaves through its job's tensor maps.  A CTA meets the jobs in
// order, so it folds its amax of a job into that job's amax_out when it moves on.
__global__ void __launch_bounds__(kThreads, 1) k_cast_jobs(const __grid_constant__ CastJobs J) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  float* const red = reinterpret_cast<float*>(base_ptr + kOffRed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = J.tile_start[J.n];

  if (tid == 0) {
    for (int j = 0; j < J.n; ++j) prefetch_tmap(&J.m[j].x);
    for (int s = 0; s < kStages; ++s) mbar_init(base + kOffBar + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // a zeroing kernel ran just before this one when any job has amax_out (as the single cast)
  bool zeroed = false;
  for (int j = 0; j < J.n; ++j) zeroed = zeroed || J.p[j].amax_out != nullptr;
  if (!zeroed) pdl_wait();   // from here on: global memory
  pdl_launch_dependents();

  if (blockIdx.x == 0 && tid == 0) {
    for (int j = 0; j < J.n; ++j) {
      const CastParams& p = J.p[j];
      if (p.recipe != kTensor) continue;
      const float si = recip_rn(*p.scale);
      if (p.do_row && p.s_row) *static_cast<float*>(p.s_row) = si;
      if (p.do_col && p.s_col) *static_cast<float*>(p.s_col) = si;
    }
  }
  auto job_of = [&](int gt) {
    int j = 0;
    while (j + 1 < J.n && gt >= J.tile_start[j + 1]) ++j;
    return j;
  };
  auto issue_load = [&](int it, int gt) {
    const int j = job_of(gt);
    const int lt = gt - J.tile_start[j];
    const int s = it % kStages;
    const uint32_t bar = base + kOffBar + 8 * s;
    const int row0 = (lt / J.p[j].tiles_c) * kTile, col0 = (lt % J.p[j].tiles_c) * kTile;
    mbar_arrive_expect_tx(bar, kXBytes);
    tma_load_2d(base + s * kXBytes, &J.m[j].x, col0, row0, bar);
    tma_load_2d(base + s * kXBytes + kXBytes / 2, &J.m[j].x, col0 + 64, row0, bar);
  };
  if (tid == 0) {
    for (int it = 0; it < kStages; ++it) {
      const int gt = blockIdx.x + it * gridDim.x;
      if (gt < ntiles) issue_load(it, gt);
    }
  }
  // fold this CTA's |x| maximum of job j into its amax_out (all threads take part)
  auto flush_amax = [&](int j, float thr_amax) {
    if (J.p[j].amax_out == nullptr) return;
    const float am = block_max(thr_amax, red, warp, lane);
    if (tid == 0) {
      pdl_wait();   // the zeroing of the amaxes is done
      if (am > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(J.p[j].amax_out), __float_as_uint(am));
    }
  };

  float thr_amax = 0.0f, g_scale = 1.0f;
  int cur = -1;
  int it = 0;
  bool failed = false;
  for (int gt = blockIdx.x; gt < ntiles; gt += gridDim.x, ++it) {
    const int j = job_of(gt);
    if (j != cur) {
      if (cur >= 0) flush_amax(cur, thr_amax);
      cur = j;
      thr_amax = 0.0f;
      g_scale = J.p[j].recipe == kTensor ? *J.p[j].scale : 1.0f;
    }
    const CastParams& p = J.p[j];
    const int lt = gt - J.tile_start[j];
    const int s = it % kStages;
    const uint32_t xs = base + s * kXBytes;
    const int ob = it & 1;
    const uint32_t outR = base + kOffOutR + ob * kQBytes;
    const uint32_t outT = base + kOffOutT + ob * kQBytes;
    const int tr = lt / p.tiles_c, tc = lt % p.tiles_c;
    const int64_t row0 = static_cast<int64_t>(tr) * kTile, col0 = static_cast<int64_t>(tc) * kTile;

    // one barrier a tile, as in k_cast_transpose
    const bool ok = mbar_wait(base + kOffBar + 8 * s, (it / kStages) & 1, p.err, kErrTimeoutTmaLoad, nullptr);
    float* const red_t = red + (it & 1) * kWarps;
    const uint32_t sf = base + kOffSf + static_cast<uint32_t>(ob) * 1024u;
    switch (p.recipe) {
      case kTensor:
        cast_tile_body<kTensor>(p, xs, outR, outT, tr, tc, row0, col0, g_scale, thr_amax, red_t, sf, tid, warp, lane);
        break;
      case kBlock1x128:
        cast_tile_body<kBlock1x128>(p, xs, outR, outT, tr, tc, row0, col0, g_scale, thr_amax, red_t, sf, tid, warp,
                                    lane);
        break;
      case kBlock128x128:
        cast_tile_body<kBlock128x128>(p, xs, outR, outT, tr, tc, row0, col0, g_scale, thr_amax, red_t, sf, tid, warp,
                                      lane);
        break;
      default:
        cast_tile_body<kMx>(p, xs, outR, outT, tr, tc, row0, col0, g_scale, thr_amax, red_t, sf, tid, warp, lane);
        break;
    }
    fence_proxy_async_smem();
    if (tid == 0) bulk_wait_read<0>();  // the previous tile's stores have read their staging buffer
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    if (tid == 0) {
      if (p.do_row) tma_store_2d(&J.m[j].qrow, outR, static_cast<int>(col0), static_cast<int>(row0));
      if (p.do_col) tma_store_2d(&J.m[j].qcol, outT, static_cast<int>(row0), static_cast<int>(col0));
      if (p.recipe == kMx && p.mx_tiled) store_mx_atoms(p, sf, tr, tc);
      bulk_commit();
      const int next = gt + kStages * gridDim.x;
      if (next < ntiles) issue_load(it + kStages, next);
    }
  }

  if (failed && tid == 0) {
    // wait (bounded) for loads still in flight into this CTA's ring before leaving
    for (int k = it; k < it + kStages; ++k) {
      const int gt = blockIdx.x + k * gridDim.x;
      if (gt >= ntiles) break;
      mbar_wait(base + kOffBar + 8 * (k % kStages), (k / kStages) & 1, J.p[0].err, kErrTimeoutTmaLoad, nullptr);
    }
  }
  if (tid == 0) bulk_wait_all<0>();
  if (!failed && cur >= 0) flush_amax(cur, thr_amax);
}

// Two casts in one persistent grid with their recipes known at compile time (the common
// pairings: an activation and a weight of one layer).  As k_cast_jobs, but each tile's
// body and stores read job 0's or job 1's parameters at fixed places in the parameter
// block; with the job index a run-time value every parameter read inside the tile body
// is an indexed load.  Measured on the 4096^2 activation / weight pair (1x128, 128x128):
// 32.3 us for this launch against 32.8-33.5 for two single launches and 34.8 for the
// generic jobs kernel.
template <int R0, int R1>
__global__ void __launch_bounds__(kThreads, 1) k_cast_two(const __grid_constant__ CastJobs J) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  float* const red = reinterpret_cast<float*>(base_ptr + kOffRed);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = J.tile_start[1], ntiles = J.tile_start[2];

  if (tid == 0) {
    prefetch_tmap(&J.m[0].x);
    prefetch_tmap(&J.m[1].x);
    for (int s = 0; s < kStages; ++s) mbar_init(base + kOffBar + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // a zeroing kernel ran just before this one when either job has amax_out (as the single cast)
  const bool zeroed = J.p[0].amax_out != nullptr || J.p[1].amax_out != nullptr;
  if (!zeroed) pdl_wait();   // from here on: global memory
  pdl_launch_dependents();

  if (blockIdx.x == 0 && tid == 0) {
    if (R0 == kTensor) {
      const float si = recip_rn(*J.p[0].scale);
      if (J.p[0].do_row && J.p[0].s_row) *static_cast<float*>(J.p[0].s_row) = si;
      if (J.p[0].do_col && J.p[0].s_col) *static_cast<float*>(J.p[0].s_col) = si;
    }
    if (R1 == kTensor) {
      const float si = recip_rn(*J.p[1].scale);
      if (J.p[1].do_row && J.p[1].s_row) *static_cast<float*>(J.p[1].s_row) = si;
      if (J.p[1].do_col && J.p[1].s_col) *static_cast<float*>(J.p[1].s_col) = si;
    }
  }
  auto issue_load = [&](int it, int gt) {
    const bool j1 = gt >= n0;
    const CUtensorMap* tx = j1 ? &J.m[1].x : &J.m[0].x;
    const int lt = j1 ? gt - n0 : gt, tc_n = j1 ? J.p[1].tiles_c : J.p[0].tiles_c;
    const int s = it % kStages;
    const uint32_t bar = base + kOffBar + 8 * s;
    const int row0 = (lt / tc_n) * kTile, col0 = (lt % tc_n) * kTile;
    mbar_arrive_expect_tx(bar, kXBytes);
    tma_load_2d(base + s * kXBytes, tx, col0, row0, bar);
    tma_load_2d(base + s * kXBytes + kXBytes / 2, tx, col0 + 64, row0, bar);
  };
  if (tid == 0) {
    for (int it = 0; it < kStages; ++it) {
      const int gt = blockIdx.x + it * gridDim.x;
      if (gt < ntiles) issue_load(it, gt);
    }
  }
  // fold this CTA's |x| maximum of a job into its amax_out (all threads take part)
  auto flush_amax = [&](float* amax_out, float thr_amax) {
    if (amax_out == nullptr) return;
    const float am = block_max(thr_amax, red, warp, lane);
    if (tid == 0) {
      pdl_wait();   // the zeroing of the amaxes is done
      if (am > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax_out), __float_as_uint(am));
    }
  };
  const float g0 = R0 == kTensor ? *J.p[0].scale : 1.0f, g1 = R1 == kTensor ? *J.p[1].scale : 1.0f;
  float thr_amax = 0.0f;
  bool in_job1 = false;
  int it = 0;
  bool failed = false;
  // one tile of job JJ (its body, then its stores): JJ fixes which parameters are read
  auto tile = [&](auto jc, int lt, int s, int ob, bool ok) -> bool {
    constexpr int JJ = decltype(jc)::value;
    constexpr int RR = JJ == 0 ? R0 : R1;
    const CastParams& p = J.p[JJ];
    const uint32_t xs = base + s * kXBytes;
    const uint32_t outR = base + kOffOutR + ob * kQBytes;
    const uint32_t outT = base + kOffOutT + ob * kQBytes;
    const int tr = lt / p.tiles_c, tc = lt % p.tiles_c;
    const int64_t row0 = static_cast<int64_t>(tr) * kTile, col0 = static_cast<int64_t>(tc) * kTile;
    const uint32_t sf = base + kOffSf + static_cast<uint32_t>(ob) * 1024u;
    cast_tile_body<RR>(p, xs, outR, outT, tr, tc, row0, col0, JJ == 0 ? g0 : g1, thr_amax, red + (it & 1) * kWarps, sf, tid,
                       warp, lane);
    fence_proxy_async_smem();
    if (tid == 0) bulk_wait_read<0>();  // the previous tile's stores have read their staging buffer
    if (__syncthreads_or(!ok)) return false;
    if (tid == 0) {
      if (p.do_row) tma_store_2d(&J.m[JJ].qrow, outR, static_cast<int>(col0), static_cast<int>(row0));
      if (p.do_col) tma_store_2d(&J.m[JJ].qcol, outT, static_cast<int>(row0), static_cast<int>(col0));
      if (RR == kMx && p.mx_tiled) store_mx_atoms(p, sf, tr, tc);
    }
    return true;
  };
  for (int gt = blockIdx.x; gt < ntiles; gt += gridDim.x, ++it) {
    const bool j1 = gt >= n0;
    if (j1 && !in_job1) {   // a CTA meets job 0's tiles first
      flush_amax(J.p[0].amax_out, thr_amax);
      thr_amax = 0.0f;
      in_job1 = true;
    }
    const int s = it % kStages;
    const int ob = it & 1;
    // one barrier a tile, as in k_cast_transpose
    const bool ok = mbar_wait(base + kOffBar + 8 * s, (it / kStages) & 1, J.p[0].err, kErrTimeoutTmaLoad, nullptr);
    const bool done = j1 ? tile(std::integral_constant<int, 1>{}, gt - n0, s, ob, ok)
                         : tile(std::integral_constant<int, 0>{}, gt, s, ob, ok);
    if (!done) {
      failed = true;
      break;
    }
    if (tid == 0) {
      bulk_commit();
      const int next = gt + kStages * gridDim.x;
      if (next < ntiles) issue_load(it + kStages, next);
    }
  }

  if (failed && tid == 0) {
    // wait (bounded) for loads still in flight into this CTA's ring before leaving
    for (int k = it; k < it + kStages; ++k) {
      const int gt = blockIdx.x + k * gridDim.x;
      if (gt >= ntiles) break;
      mbar_wait(base + kOffBar + 8 * (k % kStages), (k / kStages) & 1, J.p[0].err, kErrTimeoutTmaLoad, nullptr);
    }
  }
  if (tid == 0) bulk_wait_all<0>();
  if (!failed) flush_amax(in_job1 ? J.p[1].amax_out : J.p[0].amax_out, thr_amax);
}

// Whether a one-scale cast takes its column copy from the staged row copy: always for
// per-tensor (measured side by side: equal or faster at every size, 0.68 against 0.60 of
// HBM at 4096^2); for 128x128 up to 64 tiles a CTA (0.56 / 0.92 at 4096^2 / 8192^2 against
// 0.53 / 0.84 quantizing the column copy again, but 0.92 / 0.89 at 16384^2 / 32768^2
// against 0.97 / 1.00).
int col_from_row(const CastParams& p, int num_sms) {
  if (p.recipe == kTensor) return 1;
  if (p.recipe != kBlock128x128) return 0;
  return static_cast<int64_t>(p.tiles_r) * p.tiles_c <= 64LL * num_sms ? 1 : 0;
}

// Whether the 1x128 column scales are stored with the L2 evict-last policy: a sector of
// them is written by 8 tile-rows, between which 8 * 128 rows * C * 4 bytes stream through
// L2 (128 MB at C = 32768, about the whole L2).  Measured side by side, both orders: 32768^2
// 0.95 of HBM with the policy against 0.86, 16384^2 (64 MB) 0.914 against 0.924.  So from
// three quarters of L2 (C >= 24576) on.
int keep_col_scales(const CastParams& p) { return p.recipe == kBlock1x128 && p.C >= 24576 ? 1 : 0; }

// Whether a 1x128 tile with both copies forms its row and column scales with one division a
// lane (cast_tile_1x128_both): up to 64 tiles a CTA, where the cast is bound by its
// instructions (measured side by side, both orders: the step's two-job launch 30.8 against
// 31.2 us, 1x128 casts +2 % at 4096^2 and 8192^2; at 16384^2, bound by HBM, 2.5 % slower).
int one_division(const CastParams& p, int num_sms) {
  return p.recipe == kBlock1x128 && static_cast<int64_t>(p.tiles_r) * p.tiles_c <= 64LL * num_sms ? 1 : 0;
}

template <int RECIPE>
cudaError_t launch_tiled(const CastParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_qrow,
                         const CUtensorMap& tm_qcol, int num_sms, cudaStream_t s) {
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_limit(k_cast_transpose<RECIPE>, static_cast<int>(kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  const int ntiles = p.tiles_r * p.tiles_c;
  const int grid = ntiles < num_sms ? ntiles : num_sms;
  CastParams q = p;
  q.col_from_row = col_from_row(p, num_sms);
  q.keep_col_scales = keep_col_scales(p);
  q.one_division = one_division(p, num_sms);
  return launch_pdl(k_cast_transpose<RECIPE>, dim3(grid), dim3(kThreads), kSmemBytes, s, 1, tm_x, tm_qrow, tm_qcol, q);
}

}  // namespace

cudaError_t launch_cast_transpose_tiled(const CastParams& p, const CUtensorMap& tm_x, const CUtensorMap& tm_qrow,
                                        const CUtensorMap& tm_qcol, int num_sms, cudaStream_t s) {
  switch (p.recipe) {
    case kTensor: return launch_tiled<kTensor>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
    case kBlock1x128: return launch_tiled<kBlock1x128>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
    case kBlock128x128: return launch_tiled<kBlock128x128>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
    default: return launch_tiled<kMx>(p, tm_x, tm_qrow, tm_qcol, num_sms, s);
  }
}

namespace {
template <int R0, int R1>
cudaError_t launch_two(const CastJobs& jobs, int grid, cudaStream_t s) {
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_limit(k_cast_two<R0, R1>, static_cast<int>(kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_cast_two<R0, R1>, dim3(grid), dim3(kThreads), kSmemBytes, s, 1, jobs);
}
}  // namespace

cudaError_t launch_cast_jobs(const CastJobs& jobs_in, int num_sms, cudaStream_t s) {
  CastJobs jobs = jobs_in;
  for (int j = 0; j < jobs.n; ++j) {
    jobs.p[j].col_from_row = col_from_row(jobs.p[j], num_sms);
    jobs.p[j].keep_col_scales = keep_col_scales(jobs.p[j]);
    jobs.p[j].one_division = one_division(jobs.p[j], num_sms);
  }
  const int ntiles = jobs.tile_start[jobs.n];
  const int grid = ntiles < num_sms ? ntiles : num_sms;
  if (jobs.n == 2) {
    const int r0 = jobs.p[0].recipe, r1 = jobs.p[1].recipe;
    if (r0 == kBlock1x128 && r1 == kBlock128x128) return launch_two<kBlock1x128, kBlock128x128>(jobs, grid, s);
    if (r0 == kMx && r1 == kMx) return launch_two<kMx, kMx>(jobs, grid, s);
    if (r0 == kTensor && r1 == kTensor) return launch_two<kTensor, kTensor>(jobs, grid, s);
  }
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_limit(k_cast_jobs, static_cast<int>(kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_cast_jobs, dim3(grid), dim3(kThreads), kSmemBytes, s, 1, jobs);
}

cudaError_t launch_cast_generic(const CastParams& p, const void* x, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((p.C + 31) / 32), static_cast<unsigned>((p.R + 31) / 32));
  return launch_pdl(k_cast_generic, grid, dim3(256), 0, s, 1, static_cast<const uint16_t*>(x), p);
}

}  // namespace fp8q
