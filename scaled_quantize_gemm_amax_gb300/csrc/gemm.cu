// gemm.cu -- scaled FP8 GEMM on the 5th-generation tensor cores (tcgen05).
//
//   C[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k],  A [M, K], B [N, K], both K-major FP8,
//   FP32 accumulation, C row-major BF16 (fprop / dgrad) or FP32 (wgrad)
// (mixed-precision dataflow paragraph of the search-result page: quantized inputs,
// FP32 accumulation, BF16 output; wgrad stays FP32).  Dequantization by recipe:
//   per-tensor  C = sA_inv * sB_inv * sum qA qB                (epilogue scale)
//   blockwise   C = sum_kb sA[m, kb] * sB[n/128 | n, kb] * sum_{k in kb} qA qB
//               (guide, "block-level scaling": 1x128 activations, 128x128 weights;
//                each 128-deep partial product is promoted into FP32 registers)
//   MXFP8       the tensor core applies 2^(eA - 127) * 2^(eB - 127) per 32-deep block
//               (guide, "MXFP8 scaling"; kind::mxf8f6f4.block_scale)
//
// Structure: a persistent grid (one CTA per SM).
//   warp 0      TMA producer: A / B tiles (128-byte swizzle) into a ring of stages,
//               plus MX scale atoms by bulk copy
//   warp 1      TMEM allocation; lane 0 issues the tcgen05.mma (and the scale copies)
//   warps 2..9  epilogue: tcgen05.ld from TMEM,
//               scale, convert, store.  Warp w reads TMEM lanes 32*(w%4).. (its quarter)
//               and column slice (w-2)/4 of the tile.
//   blockwise with 256-deep stages: warps 0..3 are the control warpgroup (warp 2's lane
//               0 issues the MMAs of each stage's second partial) and warps 4..11 the
//               epilogue, with registers moved from the former to the latter
// Every wait is time-bounded (ptx.cuh); a timeout sets the device error word, the
// other roles see a shared abort flag, and the CTA drains and frees TMEM.
#include <cuda_bf16.h>

#include <atomic>
#include <mutex>

#include "gemm_util.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "recipes.cuh"

namespace fp8q {

namespace {

using namespace gemm_util;

constexpr int kBM = 128;
constexpr int kBK = 128;               // bytes (= FP8 elements) of K per stage
constexpr int kUmmaK = 32;             // K of one MMA instruction for 8-bit inputs
constexpr uint32_t kTmemCols = 512;

// Blockwise with per-row B scales (1x128 x 1x128, the wgrad pairing): its own
// instantiation so the common 1x128 x 128x128 promotion carries no extra registers.
constexpr int kBlockRowsB = 4;

template <int KIND>
struct Cfg;
template <>
struct Cfg<kTensor> {
  static constexpr int BN = 256, STAGES = 4, ACC = 2, EPI = 8, KSUB = 1, CTRL = 2;
};
template <>
struct Cfg<kBlock1x128> {
  static constexpr int BN = 128, STAGES = 6, ACC = 4, EPI = 8, KSUB = 1, CTRL = 2;   // ACC = TMEM partial buffers
};
template <>
struct Cfg<kBlockRowsB> : Cfg<kBlock1x128> {};
// Blockwise with 256-deep stages: two 128-deep partials per stage, handed to the
// promotion as one group (one commit, one release).  Every barrier operation of
// the MMA-issuing thread stalls its next MMA while the tensor core streams shared
// memory (measured), so halving them per MMA matters most for 128-wide tiles.
constexpr int kBlockK2 = 5;
template <>
struct Cfg<kBlockK2> {
  static constexpr int BN = 128, STAGES = 3, ACC = 4, EPI = 8, KSUB = 2, CTRL = 4;
};
// The same with per-row B scales (1x128 x 1x128): each output column has its own factor
// sB[n, kb].  The epilogue copies the tile's B scales into a shared table (per half of the
// tile's columns, [kb][64] floats, K / 128 <= kMaxTableKb; two buffers, the next tile's
// fetched a tile ahead, when K / 128 <= kMaxTableKb / 2) and reads a k-block's 64 factors
// as broadcast 16-byte loads.
constexpr int kBlockK2RowsB = 6;
constexpr int kMaxTableKb = 64;
template <>
struct Cfg<kBlockK2RowsB> : Cfg<kBlockK2> {};
// MMA-issuing threads.  One thread needs about 74 cycles to issue a 256x128x32 MMA
// (measured by a clock trace), close to the 88 cycles the MMA runs, so with 128-wide
// tiles a single issuer starves the tensor core once it also waits and commits.  With
// 256-deep stages the two 128-deep partials of a stage go to different TMEM buffers
// and need no ordering between them: each gets its own issuing thread (warp 1 and the
// warp after the epilogue warps), and both commit every stage.
template <int KIND>
__host__ __device__ constexpr int issuers_of() { return (KIND == kBlockK2 || KIND == kBlockK2RowsB || KIND == kMx) ? 2 : 1; }
template <>
struct Cfg<kMx> {
  static constexpr int BN = 256, STAGES = 3, ACC = 1, EPI = 8, KSUB = 1, CTRL = 2;
};
// Blockwise 1x128 x 128x128 on 256 x 160 pair tiles with 128-deep stages (BF16 out, no
// fused output cast), for K / 128 odd, where the 256-deep stages above do not fit and the
// alternative is one CTA per 128 x 128 tile (measured: 1.10-1.34x faster than that).
// Three 160-column partial buffers fill 480 of TMEM's 512 columns; a single MMA issuer
// (a 256 x 160 x 32 MMA runs longer than the ~74 cycles one thread needs to issue it);
// the promotion holds a whole partial (80 columns a thread) next to its 80 accumulators,
// with registers from the control warpgroup as below.  (A 256 x N x 32 pair MMA costs
// about 88 + 0.34 N cycles inside these kernels, so 160 columns would do 1.14x the work a
// cycle of 128, but with K / 128 even this kernel ran at 0.55 of the FP8 peak at 8192^3
// against 0.68 for the 256-deep stages, measured.)
constexpr int kBlock160 = 7;
template <>
struct Cfg<kBlock160> {
  static constexpr int BN = 160, STAGES = 6, ACC = 3, EPI = 8, KSUB = 1, CTRL = 4;
};

// CTRL = 4: warps 0..3 (producer, the two MMA issuers, an idle warp) form a warpgroup
// that gives registers to the two epilogue warpgroups (warps 4..11) with setmaxnreg, so
// that the promotion can hold a group's partials (the 1x128 x 128x128 kind: both, its 64
// columns of each) in registers and hand the group back before its FMAs.  The kernel
// must be launched with kSplitLaunchRegs a thread (checked on the host before the first
// launch: an increase beyond the launch pool is never granted).
constexpr int kSplitLaunchRegs = 168, kCtrlRegs = 72, kEpiRegs = 216;
static_assert(128 * kCtrlRegs + 256 * kEpiRegs <= 384 * kSplitLaunchRegs, "register split exceeds the launch pool");
static_assert(kCtrlRegs + 2 * kEpiRegs <= 512, "register split exceeds a sub-partition");
// The 160-wide blockwise kernel: its single MMA issuer's loop needs more than 72 (it
// spilled), its promotion less than 216.
constexpr int kCtrlRegs160 = 80, kEpiRegs160 = 208;
static_assert(128 * kCtrlRegs160 + 256 * kEpiRegs160 <= 384 * kSplitLaunchRegs, "register split exceeds the launch pool");
static_assert(kCtrlRegs160 + 2 * kEpiRegs160 <= 512, "register split exceeds a sub-partition");

// Stages of the 2-CTA (pair) variant: each CTA holds 128 rows of A and half of B
// (blockwise with 256-deep stages: 48 KB a stage; three ran 3 % faster than four at
// 4096^3 and 8192^3, measured).
template <int KIND>
constexpr int pair_stages() {
  return KIND == kBlock160 ? Cfg<kBlock160>::STAGES
                           : (Cfg<KIND>::KSUB == 2 ? 3 : (KIND == kMx ? 5 : (Cfg<KIND>::BN == 256 ? 6 : 8)));
}

template <int KIND, bool PAIR>
struct Layout {
  static constexpr int BN = Cfg<KIND>::BN, S = PAIR ? pair_stages<KIND>() : Cfg<KIND>::STAGES;
  static constexpr int KSUB = Cfg<KIND>::KSUB;
  // per K sub-block: A [128 rows][128 B], B [BN (or BN/2) rows][128 B]; a stage holds KSUB of each
  static constexpr uint32_t A_SUB = kBM * kBK, B_SUB = (PAIR ? BN / 2 : BN) * kBK;
  static constexpr uint32_t A_BYTES = A_SUB * KSUB, B_BYTES = B_SUB * KSUB;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  // MX scale atoms per stage: this CTA's rows of A and all BN rows of B
  static constexpr uint32_t SF_BYTES = (KIND == kMx) ? 512 + 512 * (BN / 128) : 0;
  static constexpr uint32_t OFF_SF = S * STAGE_BYTES;
  // per-tensor / MX / blockwise with 256-deep stages: one 4 KB staging box per epilogue
  // warp for the TMA stores of C
  // (32 rows x 128 B, 128-byte swizzle; the box must start on 1024 bytes).  The 160-wide
  // blockwise tiles: five unswizzled 1 KB boxes a warp (32 rows x 16 BF16 columns each).
  static constexpr bool TSTORE = !(KIND == kBlock1x128 || KIND == kBlockRowsB);
  static constexpr uint32_t STG_WARP = KIND == kBlock160 ? 5 * 1024 : 4096;
  static constexpr uint32_t STG_BYTES = TSTORE ? Cfg<KIND>::EPI * STG_WARP : 0;
  static constexpr uint32_t OFF_STG = (OFF_SF + S * SF_BYTES + 1023) & ~1023u;
  // per-row B scales on CTA pairs: the tile's B-scale table, one part of [kb][COLS] floats
  // per epilogue warpgroup (its COLS columns)
  static constexpr int NPART = Cfg<KIND>::EPI / 4, PCOLS = BN / NPART;
  static constexpr uint32_t TBL_PART = KIND == kBlockK2RowsB ? kMaxTableKb * PCOLS * 4 : 0;
  static constexpr uint32_t OFF_TBL = OFF_STG + STG_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_TBL + NPART * TBL_PART;
  // barriers: full[S], empty[S], tfull[4], tempty[4], final
  static constexpr uint32_t OFF_FULL = OFF_BAR, OFF_EMPTY = OFF_BAR + 8 * S;
  static constexpr uint32_t OFF_TFULL = OFF_EMPTY + 8 * S, OFF_TEMPTY = OFF_TFULL + 32;
  static constexpr uint32_t OFF_FINAL = OFF_TEMPTY + 32;
  static constexpr uint32_t OFF_SFR = OFF_FINAL + 8;   // MX: a stage's scale factors are in TMEM
  static constexpr uint32_t OFF_TMEM = OFF_SFR + 8 * S, OFF_ABORT = OFF_TMEM + 4;
  // B-scale table barriers per (part, buffer): filled, then (at 8 * 2 * NPART) read
  static constexpr uint32_t OFF_TBAR = (OFF_ABORT + 4 + 7) & ~7u;
  static constexpr uint32_t SMEM = OFF_TBAR + 32 * NPART + 1024;   // + alignment slack
  // bytes one stage's full barrier expects (in a pair: the leader's barrier sees both CTAs' loads)
  static constexpr uint32_t TX_BYTES = PAIR ? 2 * (STAGE_BYTES + SF_BYTES) : STAGE_BYTES + SF_BYTES;
};

// Store 32 consecutive FP32 values (already scaled) of one output row.
__device__ __forceinline__ void store_row32(void* c, int64_t off, const float (&v)[32], bool fp32) {
  if (fp32) {
    float* p = static_cast<float*>(c) + off;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      stg128(p + 4 * i, __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
             __float_as_uint(v[4 * i + 3]));
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(c) + off;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      stg128(p + 8 * i, pack_bf16(v[8 * i], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
             pack_bf16(v[8 * i + 4], v[8 * i + 5]), pack_bf16(v[8 * i + 6], v[8 * i + 7]));
  }
}

// control warps (producer, MMA), EPI epilogue warps, then (CTRL = 2) the second MMA issuer if any
template <int KIND>
constexpr int threads_of() {
  return 32 * (Cfg<KIND>::CTRL + Cfg<KIND>::EPI + (Cfg<KIND>::CTRL == 2 ? issuers_of<KIND>() - 1 : 0));
}

// PAIR: a 2-CTA cluster computes a 256-row tile with the 2-SM MMA (cta_group::2).
// CTA rank r of the pair loads A rows [128 r, 128 r + 128) and B rows
// [r BN/2, (r + 1) BN/2) of the tile into its own shared memory; both loads
// signal the leader's (rank 0) stage barrier; the leader issues every MMA and
// multicasts its commits to both CTAs; each CTA's TMEM holds its 128 rows of D,
// and both CTAs' epilogues release an accumulator on the leader's barrier.
// QOUT: the epilogue may also write C's FP8 copy and amax (a separate instantiation, so
// the plain GEMM's epilogue carries none of it).
template <int KIND, bool PAIR, bool QOUT>
__global__ void __launch_bounds__(threads_of<KIND>(), 1)
    k_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
           const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
           const __grid_constant__ CUtensorMap tm_c, const GemmParams p) {
  using L = Layout<KIND, PAIR>;
  constexpr int BN = L::BN, S = L::S, ACC = Cfg<KIND>::ACC, EPI = Cfg<KIND>::EPI;
  constexpr bool BLOCK = (KIND == kBlock1x128 || KIND == kBlockRowsB || KIND == kBlockK2 || KIND == kBlockK2RowsB ||
                          KIND == kBlock160);   // promotion path
  constexpr int KSUB = L::KSUB;
  constexpr int GROUPS = ACC / KSUB;   // partial-buffer groups (blockwise)
  static_assert(KSUB == 1 || BLOCK, "multi-block stages: blockwise only");
  // Blockwise: a stage's full barrier also counts the epilogue's release of the partial
  // group that stage will write (in a pair, both CTAs' epilogues release on the
  // leader's barrier), so the MMA thread waits once per stage.
  constexpr bool GATED = BLOCK;
  constexpr bool B_ROWS = (KIND == kBlockRowsB || KIND == kBlockK2RowsB);   // B scales per row
  constexpr bool TABLE = (KIND == kBlockK2RowsB);                         // ... read from the shared table
  constexpr int COLS = BN / (EPI / 4);   // columns of the tile each epilogue thread owns
  constexpr int NISS = issuers_of<KIND>();
  // MX with two issuers: the second thread copies each stage's scale factors into TMEM
  // (tcgen05.cp) and signals the MMA thread, which then only issues MMAs
  constexpr bool SFCP = KIND == kMx && NISS > 1;
  static_assert(NISS == 1 || NISS == KSUB || SFCP, "MMA issuers");
  constexpr int CTRL = Cfg<KIND>::CTRL;                 // warps before the epilogue warps
  constexpr int ISS1 = CTRL == 4 ? 2 : 2 + EPI;         // warp of the second MMA issuer
  constexpr bool REGSPLIT = CTRL == 4;                  // registers move to the epilogue (see Cfg)
  constexpr bool WIDE = REGSPLIT && KIND != kBlock160;  // 64-column partial loads of 256-deep stages
  static_assert(!WIDE || (BLOCK && KSUB == 2 && COLS == 64 && B_ROWS == TABLE), "wide promotion layout");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - smem_u32(smem_raw));
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(base_ptr + L::OFF_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  constexpr int TM = PAIR ? 2 * kBM : kBM;                  // rows of one tile
  constexpr int kRasterM = BN == 256 ? 16 : 8;              // M-tiles that walk N together
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;      // 0 = the pair's leader
  const bool leader = rank == 0;
  const int tiles_m = static_cast<int>(p.M / TM), tiles_n = static_cast<int>((p.N + BN - 1) / BN);
  const int ntiles = tiles_m * tiles_n;
  const int KB = static_cast<int>(p.K / kBK);
  const int NG = KB / KSUB;   // stages per tile (K / 128 is a multiple of KSUB)
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);   // tile-walker index
  const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // This unit's work.  Whole tiles unit0, unit0 + units, ... below tail0, then (when the
  // last partial wave is split) K range c = unit0 / ntail of tail tile tail0 + unit0 % ntail.
  // Or (stream-K) whole tiles unit0, unit0 + units, ... below tail0, then the share
  // [W unit0 / units, W (unit0 + 1) / units) of the W = (ntiles - tail0) * NG K blocks of the
  // tiles from tail0 on, in tile order: a part of a tile at each end of the share, whole
  // tiles between (a share is at least one tile long, so a tile has at most two parts).
  // Both keep the tiles in flight at one time neighbours, which the raster needs for L2.
  constexpr bool SPLITK = PAIR && (KIND == kTensor || KIND == kMx);
  const bool streamk = SPLITK && p.streamk != 0;
  const int split = SPLITK && !streamk && p.split > 1 ? p.split : 1;
  const int tail0 = split > 1 || streamk ? p.tail0 : ntiles;
  const int ntail = ntiles - tail0;
  const int nfull = split > 1 || streamk ? tail0 / units : 0;
  // The share's first tile and K block and its last tile and end, divided out once here: the
  // 64-bit divisions cost the single MMA-issuing thread 0.5-1.4 us at each work item of the
  // share when done there (measured), with the tensor core idle.
  int sk_t0 = 0, sk_kg0 = 0, sk_t1 = -1, sk_kg1 = 0;
  if (streamk) {
    const int64_t sk_w = static_cast<int64_t>(ntail) * NG;
    if (sk_w * units < (int64_t{1} << 31)) {   // 32-bit divisions suffice (every size in practice)
      const int w32 = static_cast<int>(sk_w);
      const int s32 = w32 * unit0 / units, e32 = w32 * (unit0 + 1) / units;
      if (e32 > s32) {
        sk_t0 = tail0 + s32 / NG;
        sk_kg0 = s32 % NG;
        sk_t1 = tail0 + (e32 - 1) / NG;
        sk_kg1 = (e32 - 1) % NG + 1;
      }
    } else {
      const int64_t sk_s = sk_w * unit0 / units, sk_e = sk_w * (unit0 + 1) / units;
      if (sk_e > sk_s) {
        sk_t0 = tail0 + static_cast<int>(sk_s / NG);
        sk_kg0 = static_cast<int>(sk_s % NG);
        sk_t1 = tail0 + static_cast<int>((sk_e - 1) / NG);
        sk_kg1 = static_cast<int>((sk_e - 1) % NG) + 1;
      }
    }
  }
  const int nwork = streamk    ? nfull + (sk_t1 >= sk_t0 ? sk_t1 - sk_t0 + 1 : 0)
                    : split > 1 ? nfull + (unit0 < ntail * split ? 1 : 0)
                                : (unit0 < ntiles ? (ntiles - unit0 + units - 1) / units : 0);
  struct Work {
    int t, kg0, kg1;
    int part;     // -1: the whole tile; 0: adds the other parts' slots to its own; 1: leaves its part in `slot`
    int slot;     // part 1: its slot; part 0: the first slot it adds
    int nslot;    // part 0: how many slots it adds, `sstride` apart
    int sstride;
  };
  auto work_at = [&](int i) -> Work {
    if (streamk && i >= nfull) {
      i -= nfull;
      const int t = sk_t0 + i;
      const int kg0 = i == 0 ? sk_kg0 : 0;
      const int kg1 = t == sk_t1 ? sk_kg1 : NG;
      if (kg0 > 0) return Work{t, kg0, kg1, 1, unit0, 0, 0};            // the later part of a tile begun by unit0 - 1
      if (kg1 < NG) return Work{t, kg0, kg1, 0, unit0 + 1, 1, 0};       // the earlier part: adds unit0 + 1's slot
      return Work{t, 0, NG, -1, 0, 0, 0};
    }
    if ((split == 1 && !streamk) || i < nfull) return Work{unit0 + i * units, 0, NG, -1, 0, 0, 0};
    const int c = unit0 / ntail, j = unit0 % ntail;
    if (c > 0) return Work{tail0 + j, c * NG / split, (c + 1) * NG / split, 1, (c - 1) * ntail + j, 0, 0};
    return Work{tail0 + j, 0, NG / split, 0, j, split - 1, ntail};
  };
  const int64_t row_off = static_cast<int64_t>(rank) * kBM;   // this CTA's rows within a tile

  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    for (int s = 0; s < S; ++s) {
      mbar_init(base + L::OFF_FULL + 8 * s, GATED ? 1 + (PAIR ? 2 : 1) * EPI : 1);
      mbar_init(base + L::OFF_EMPTY + 8 * s, SFCP ? 1 : NISS);
      mbar_init(base + L::OFF_SFR + 8 * s, 1);
    }
    for (int a = 0; a < 4; ++a) {
      mbar_init(base + L::OFF_TFULL + 8 * a, SFCP ? 1 : NISS);
      mbar_init(base + L::OFF_TEMPTY + 8 * a, PAIR ? 2 * EPI : EPI);
    }
    mbar_init(base + L::OFF_FINAL, NISS);
    if (TABLE) {
      for (int hb = 0; hb < 2 * L::NPART; ++hb) {   // (part, table buffer)
        mbar_init(base + L::OFF_TBAR + 8 * hb, 4 * 32);                  // filled: every lane's copies of the part's four warps
        mbar_init(base + L::OFF_TBAR + 16 * L::NPART + 8 * hb, 4);       // read: one arrive per warp
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(base + L::OFF_TMEM, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(base + L::OFF_TMEM, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // (Arriving on the cluster barrier before the TMEM allocation and waiting here made the
  // pair's allocation itself ~0.5 us slower: no gain, measured.)
  if (PAIR) cluster_sync();   // the peer's barriers are initialised before anyone signals them
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base_ptr + L::OFF_TMEM);

  if (warp < CTRL || (CTRL == 2 && NISS > 1 && warp == ISS1)) {
  if constexpr (REGSPLIT) setmaxnreg_dec<KIND == kBlock160 ? kCtrlRegs160 : kCtrlRegs>();
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ producer
    pdl_wait();   // operands may come from the previous kernel in the stream
    int n_issued = 0;   // loads issued so far; stage s received n_issued / S (+1 if s < n_issued % S)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int wi = 0; wi < nwork && ok; ++wi) {
      const Work w = work_at(wi);
      int tm, tn;
      tile_coords<kRasterM>(w.t, tiles_m, tiles_n, tm, tn);
      for (int kg = w.kg0; kg < w.kg1; ++kg) {
        const int kb = kg * KSUB;   // first 128-deep K block of this stage
        const uint32_t full = base + L::OFF_FULL + 8 * stage;
        const uint32_t full_sig = PAIR ? mapa_shared(full, 0) : full;   // the barrier the loads signal
        if (!mbar_wait(base + L::OFF_EMPTY + 8 * stage, phase ^ 1u, p.err, kErrTimeoutStage, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t sa = base + stage * L::STAGE_BYTES;
        if (PAIR) {
          if (leader) mbar_arrive_expect_tx(full, L::TX_BYTES);
#pragma unroll
          for (int sub = 0; sub < KSUB; ++sub) {
            tma_load_2d_pair(sa + sub * L::A_SUB, &tm_a, (kb + sub) * kBK, tm * TM + static_cast<int>(row_off), full_sig);
            tma_load_2d_pair(sa + L::A_BYTES + sub * L::B_SUB, &tm_b, (kb + sub) * kBK,
                             tn * BN + static_cast<int>(rank) * (BN / 2), full_sig);
          }
        } else {
          mbar_arrive_expect_tx(full, L::TX_BYTES);
#pragma unroll
          for (int sub = 0; sub < KSUB; ++sub) {
            tma_load_2d(sa + sub * L::A_SUB, &tm_a, (kb + sub) * kBK, tm * kBM, full);
            tma_load_2d(sa + L::A_BYTES + sub * L::B_SUB, &tm_b, (kb + sub) * kBK, tn * BN, full);
          }
        }
        if (KIND == kMx && PAIR) {
          // this CTA's A-scale atom and the B-scale atoms of the whole tile width, each a
          // 2 x 256-byte box of the tiled scale buffer, signalled on the leader's barrier
          const uint32_t sf = base + L::OFF_SF + stage * L::SF_BYTES;
          const int atom_a = (tm * 2 + static_cast<int>(rank)) * KB + kb;
          tma_load_2d_pair(sf, &tm_sfa, 0, 2 * atom_a, full_sig);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            const int brow = min(tn * (BN / 128) + h, static_cast<int>((p.N - 1) / 128));
            tma_load_2d_pair(sf + 512 + 512 * h, &tm_sfb, 0, 2 * (brow * KB + kb), full_sig);
          }
        } else if (KIND == kMx) {
          const uint32_t sf = base + L::OFF_SF + stage * L::SF_BYTES;
          const uint8_t* ga = static_cast<const uint8_t*>(p.sa) + (static_cast<int64_t>(tm) * KB + kb) * 512;
          bulk_load(sf, ga, 512, full);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            // a tile hanging over N reuses the last real atom (its B rows are zero-filled)
            const int64_t atom_row = min(static_cast<int64_t>(tn * (BN / 128) + h), (p.N - 1) / 128);
            const uint8_t* gb = static_cast<const uint8_t*>(p.sb) + (atom_row * KB + kb) * 512;
            bulk_load(sf + 512 + 512 * h, gb, 512, full);
          }
        }
        ++n_issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // loads this CTA issued must land before it exits (they have, unless a consumer aborted).
    // A pair's loads complete on the leader's barrier, so there the stage's release by the
    // MMA (which follows the loads) is awaited instead.
    for (int s = 0; s < S; ++s) {
      const int issued_s = n_issued / S + (s < n_issued % S ? 1 : 0);
      if (issued_s > 0) {
        if (PAIR)
          mbar_wait(base + L::OFF_EMPTY + 8 * s, static_cast<uint32_t>(issued_s - 1) & 1u, p.err, kErrTimeoutStage,
                    abort_flag);
        else
          mbar_wait(base + L::OFF_FULL + 8 * s, static_cast<uint32_t>(issued_s - 1) & 1u, p.err, kErrTimeoutTmaLoad,
                    nullptr);
      }
    }
  } else if ((warp == 1 || (NISS > 1 && warp == ISS1)) && lane == 0 && !leader) {
    // ------------------------------------------------ pair peer: no MMAs; wait for the leader's last ones
    mbar_wait(base + L::OFF_FINAL, 0, p.err, kErrTimeoutMma, abort_flag);
  } else if (SFCP && warp == ISS1 && lane == 0) {
    // ------------------------------------------------ MX scale-factor copies (leader)
    auto commit_sfr = [&](uint32_t bar) {
      if (PAIR) tc_commit_pair_mc(bar, 1);   // the leader's MMA thread waits on it
      else tc_commit(bar);
    };
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int wi = 0; wi < nwork && ok; ++wi) {
      const Work w = work_at(wi);
      for (int kg = w.kg0; kg < w.kg1; ++kg) {
        if (!mbar_wait(base + L::OFF_FULL + 8 * stage, phase, p.err, kErrTimeoutTmaLoad, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the slot of this stage was last read by the MMAs of the stage's previous use,
        // which finished before the producer could refill the stage (and so before the
        // wait above returned)
        const uint32_t sf = base + L::OFF_SF + stage * L::SF_BYTES;
        const uint32_t sf_col = 256u + static_cast<uint32_t>(stage) * (4u + 4u * (BN / 128));
        if (PAIR) {
          tc_cp_32x128b_warpx4_pair(tmem + sf_col, sdesc_rows16(sf));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tc_cp_32x128b_warpx4_pair(tmem + sf_col + 4 + 4 * h, sdesc_rows16(sf + 512 + 512 * h));
        } else {
          tc_cp_32x128b_warpx4(tmem + sf_col, sdesc_rows16(sf));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) tc_cp_32x128b_warpx4(tmem + sf_col + 4 + 4 * h, sdesc_rows16(sf + 512 + 512 * h));
        }
        commit_sfr(base + L::OFF_SFR + 8 * stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (PAIR) tc_commit_pair_mc(base + L::OFF_FINAL, 3);
    else tc_commit(base + L::OFF_FINAL);
    mbar_wait(base + L::OFF_FINAL, 0, p.err, kErrTimeoutMma, nullptr);
  } else if ((warp == 1 || (NISS > 1 && warp == ISS1)) && lane == 0) {
    // ------------------------------------------------ MMA issuer(s)
    const int my_sub = warp == 1 ? 0 : 1;   // with two issuers: the partial of the stage this thread issues
    uint32_t idesc;
    if (KIND == kMx) {
      idesc = (static_cast<uint32_t>(p.e5m2_a) << 7) | (static_cast<uint32_t>(p.e5m2_b) << 10) |
              (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(TM >> 4) << 24);
    } else {
      idesc = (1u << 4) | (static_cast<uint32_t>(p.e5m2_a) << 7) | (static_cast<uint32_t>(p.e5m2_b) << 10) |
              (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(TM >> 4) << 24);
    }
    // a stage / accumulator barrier wait on the leader: the peer CTA arrives on it too
    auto wait_free = [&](uint32_t bar, uint32_t parity) -> bool {
      return PAIR ? mbar_wait_cluster(bar, parity, p.err, kErrTimeoutMma, abort_flag)
                  : mbar_wait(bar, parity, p.err, kErrTimeoutMma, abort_flag);
    };
    auto commit = [&](uint32_t bar) {
      if (PAIR) tc_commit_pair_mc(bar, 3);
      else tc_commit(bar);
    };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_it = 0, part_it = 0;
    bool ok = true;
    for (int wi = 0; wi < nwork && ok; ++wi) {
      const Work w = work_at(wi);
      const int kb_first = w.kg0 * KSUB;   // the accumulator starts over here
      uint32_t d = tmem;
      if (!BLOCK) {
        const uint32_t a = acc_it % ACC;
        if (!wait_free(base + L::OFF_TEMPTY + 8 * a, ((acc_it / ACC) & 1u) ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        d = tmem + a * BN;
      }
      for (int kg = w.kg0; kg < w.kg1; ++kg) {
        const int kb = kg * KSUB;
        if (BLOCK) {
          const uint32_t pb = part_it % GROUPS;   // partial group: buffers pb*KSUB .. +KSUB-1
          if (!GATED) {
            if (!wait_free(base + L::OFF_TEMPTY + 8 * pb, ((part_it / GROUPS) & 1u) ^ 1u)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }   // gated: the full-barrier wait below also covers the group's release
          d = tmem + pb * KSUB * BN;
        }
        // MX with a copying thread: its signal implies the stage's data and scale factors
        if (!mbar_wait(base + (SFCP ? L::OFF_SFR : L::OFF_FULL) + 8 * stage, phase, p.err, kErrTimeoutTmaLoad,
                       abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = base + stage * L::STAGE_BYTES;
        const uint32_t sb = sa + L::A_BYTES;
        if (KIND == kMx && PAIR) {
          // each CTA's atoms go to the same TMEM columns of its own TMEM
          const uint32_t sf = base + L::OFF_SF + stage * L::SF_BYTES;
          const uint32_t sf_col = 256u + static_cast<uint32_t>(stage) * (4u + 4u * (BN / 128));
          if (!SFCP) {
            tc_cp_32x128b_warpx4_pair(tmem + sf_col, sdesc_rows16(sf));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tc_cp_32x128b_warpx4_pair(tmem + sf_col + 4 + 4 * h, sdesc_rows16(sf + 512 + 512 * h));
          }
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint32_t id = idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
            tc_mma_mxf8f6f4_pair(d, sdesc_k_sw128(sa + k * kUmmaK), sdesc_k_sw128(sb + k * kUmmaK), id, tmem + sf_col,
                                 tmem + sf_col + 4, ((kb - kb_first) | k) != 0 ? 1u : 0u);
          }
        } else if (KIND == kMx) {
          const uint32_t sf = base + L::OFF_SF + stage * L::SF_BYTES;
          const uint32_t sf_col = 256u + static_cast<uint32_t>(stage) * (4u + 4u * (BN / 128));
          if (!SFCP) {
            tc_cp_32x128b_warpx4(tmem + sf_col, sdesc_rows16(sf));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tc_cp_32x128b_warpx4(tmem + sf_col + 4 + 4 * h, sdesc_rows16(sf + 512 + 512 * h));
          }
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint32_t id = idesc | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
            tc_mma_mxf8f6f4(d, sdesc_k_sw128(sa + k * kUmmaK), sdesc_k_sw128(sb + k * kUmmaK), id, tmem + sf_col,
                            tmem + sf_col + 4, ((kb - kb_first) | k) != 0 ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int sub = 0; sub < KSUB; ++sub) {
            if (NISS > 1 && sub != my_sub) continue;
            const uint32_t dsub = d + (BLOCK ? sub * BN : 0);   // blockwise: one partial per sub-block
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              const uint32_t accumulate = (BLOCK) ? (k != 0) : (((kb - kb_first) | k) != 0);
              const uint32_t a_k = sa + sub * L::A_SUB + k * kUmmaK, b_k = sb + sub * L::B_SUB + k * kUmmaK;
              if (PAIR)
                tc_mma_f8f6f4_pair(dsub, sdesc_k_sw128(a_k), sdesc_k_sw128(b_k), idesc, accumulate);
              else
                tc_mma_f8f6f4(dsub, sdesc_k_sw128(a_k), sdesc_k_sw128(b_k), idesc, accumulate);
            }
          }
        }
        commit(base + L::OFF_EMPTY + 8 * stage);
        if (BLOCK) {
          commit(base + L::OFF_TFULL + 8 * (part_it % GROUPS));
          ++part_it;
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (!BLOCK) {
        commit(base + L::OFF_TFULL + 8 * (acc_it % ACC));
        ++acc_it;
      }
    }
    // every MMA this thread issued has finished before TMEM is released (in both CTAs of a
    // pair); with two issuers the barrier completes once both have committed
    commit(base + L::OFF_FINAL);
    mbar_wait(base + L::OFF_FINAL, 0, p.err, kErrTimeoutMma, nullptr);
  }
  } else if (warp >= CTRL && warp < CTRL + EPI) {
    // ------------------------------------------------ epilogue
    if constexpr (REGSPLIT) setmaxnreg_inc<KIND == kBlock160 ? kEpiRegs160 : kEpiRegs>();
    pdl_wait();   // scales and C: ordered after the previous kernel in the stream
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int h = (warp - CTRL) >> 2;       // which COLS-wide slice of the tile's columns
    const int row = 32 * q + lane;          // row within the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    const bool fp32 = p.out_fp32 != 0;
    float tensor_scale = 1.0f;
    if (KIND == kTensor) tensor_scale = __fmul_rn(*static_cast<const float*>(p.sa), *static_cast<const float*>(p.sb));
    // Fused output quantization: the next layer's per-tensor cast of y (the value stored
    // in C, bf16-rounded for bf16 output) with a scale known before the GEMM (delayed
    // scaling), and the amax of y that feeds that scale's history.
    const bool want_q = QOUT && p.cq != nullptr, want_amax = QOUT && p.c_amax != nullptr;
    const float c_scale = want_q ? *p.c_scale : 1.0f;
    const bool e5_c = p.e5m2_c != 0;
    float y_amax = 0.0f;
    if (want_q && p.c_scale_inv != nullptr && blockIdx.x == 0 && warp == CTRL && lane == 0)
      *p.c_scale_inv = recip_rn(c_scale);
    // 32 consecutive output values of one row, starting at column gcol
    const int64_t mn = p.M * p.N;   // elements of C (and of its FP8 copy)
    auto emit = [&](const float (&v)[32], int64_t grow_, int64_t gcol, bool store_c = true) {
      const int64_t off = grow_ * p.N + gcol;
      if (store_c && p.c != nullptr) FP8Q_GUARD(off, 32, mn, p.err) { store_row32(p.c, off, v, fp32); }
      if (QOUT && (want_q || want_amax)) {
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          y[j] = fp32 ? v[j] : __bfloat162float(__float2bfloat16_rn(v[j]));
          y_amax = fmaxf(y_amax, fabsf(y[j]));   // NaN ignored
        }
        if (want_q) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = cvt_pair(__fmul_rn(y[4 * i], c_scale), __fmul_rn(y[4 * i + 1], c_scale), e5_c) |
                   (cvt_pair(__fmul_rn(y[4 * i + 2], c_scale), __fmul_rn(y[4 * i + 3], c_scale), e5_c) << 16);
          FP8Q_GUARD(off, 32, mn, p.err) {
            stg128(p.cq + off, w[0], w[1], w[2], w[3]);
            stg128(p.cq + off + 16, w[4], w[5], w[6], w[7]);
          }
        }
      }
    };
    // release of an accumulator / partial buffer: on the leader's barrier (remote for the peer)
    auto release = [&](uint32_t bar) {
      if (PAIR && !leader) mbar_arrive_remote(mapa_shared(bar, 0));
      else mbar_arrive(bar);
    };
    // C leaves through TMA stores: this warp's 32 rows x 128 bytes (32 fp32 or 64 bf16
    // columns) at a time are staged in its swizzled box, so that every store writes whole
    // lines (a thread per row storing its own 16 bytes would not).  Chunk c holds columns
    // [gcol + 32 c, gcol + 32 c + 32) of this thread's row; bf16 chunks go out in pairs.
    auto store_chunk = [&](const float (&v)[32], int c, int64_t gcol, int box_row) {
      const uint32_t stg = base + L::OFF_STG + static_cast<uint32_t>(warp - CTRL) * L::STG_WARP;
      if (fp32 || (c & 1) == 0) {
        // the box is free once the previous store from it has read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
      }
      // 16-byte chunk k of this thread's row of the box sits at chunk k ^ (row % 8)
      const uint32_t rowb = stg + static_cast<uint32_t>(lane) * 128u;
      if (fp32) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          sts128(rowb + ((static_cast<uint32_t>(k) ^ (lane & 7u)) << 4), __float_as_uint(v[4 * k]),
                 __float_as_uint(v[4 * k + 1]), __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
      } else {
        const uint32_t k0 = (c & 1) * 4;   // 32 bf16 = chunks 0..3 (even c) or 4..7 (odd c) of the row
#pragma unroll
        for (int k = 0; k < 4; ++k)
          sts128(rowb + (((k0 + k) ^ (lane & 7u)) << 4), pack_bf16(v[8 * k], v[8 * k + 1]),
                 pack_bf16(v[8 * k + 2], v[8 * k + 3]), pack_bf16(v[8 * k + 4], v[8 * k + 5]),
                 pack_bf16(v[8 * k + 6], v[8 * k + 7]));
      }
      if (fp32 || (c & 1) == 1) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_c, stg, static_cast<int>(fp32 ? gcol + 32 * c : gcol + 32 * (c - 1)), box_row);
          bulk_commit();
        }
      }
    };
    uint32_t acc_it = 0, part_it = 0;
    uint32_t tile_it = 0;   // tiles this CTA has finished (B-scale table phases)
    // blockwise scale arrays: sA [M, K/128]; sB [N/128, K/128], or [N, K/128] per row
    const int64_t sa_len = p.M * KB, sb_len = (B_ROWS ? p.N : (p.N + 127) / 128) * KB;
    // stages (partial groups) this CTA runs in all; gated: the first GROUPS stages find
    // their partial groups free
    const uint32_t total_groups = static_cast<uint32_t>(nwork) * static_cast<uint32_t>(NG);   // blockwise: never split
    if (GATED && lane == 0) {
      for (uint32_t g = 0; g < static_cast<uint32_t>(GROUPS) && g < total_groups; ++g) release(base + L::OFF_FULL + 8 * (g % S));
    }
    for (int wi = 0; wi < nwork; ++wi) {
      const Work w = work_at(wi);
      int tm, tn;
      tile_coords<kRasterM>(w.t, tiles_m, tiles_n, tm, tn);
      const int64_t grow = static_cast<int64_t>(tm) * TM + row_off + row;
      const int64_t gcol0 = static_cast<int64_t>(tn) * BN + h * COLS;
      if constexpr (KIND == kBlock160) {
        // Promotion, one 128-deep partial per TMEM wait: this thread's 80 columns as five
        // 16-column loads, issued together; the buffer goes back to the MMA issuer once they
        // land and the FMAs follow while the MMAs refill it.  Tiles and their column halves
        // start on multiples of 16 and B's scale blocks on multiples of 128, so a chunk lies
        // in one block: its factor is sA[m, kb] * sB[nb, kb] (rounded once, then the FMA, as
        // the other blockwise kernels), and this thread's columns span at most two blocks.
        constexpr int NCH = COLS / 16;
        const float* sa_row = static_cast<const float*>(p.sa) + grow * KB;
        const int64_t nlast = (p.N - 1) / 128;   // columns past N (a ragged last tile) are never stored
        const int64_t nb_lo = min(gcol0 / 128, nlast), nb_hi = min((gcol0 + COLS - 1) / 128, nlast);
        const float* sb_lo = static_cast<const float*>(p.sb) + nb_lo * KB;
        const float* sb_hi = static_cast<const float*>(p.sb) + nb_hi * KB;
        const int64_t lo_cols = (nb_lo + 1) * 128 - gcol0;   // chunks [0, nlo) take the low block
        const int nlo = lo_cols <= 0 ? 0 : (lo_cols >= COLS ? NCH : static_cast<int>(lo_cols / 16));
        uint64_t acc[COLS / 2];
#pragma unroll
        for (int j = 0; j < COLS / 2; ++j) acc[j] = 0;
        uint32_t r[NCH][16];
        float sa_n = 0.0f, sl_n = 0.0f, sh_n = 0.0f;
        FP8Q_GUARD(grow * KB, 1, sa_len, p.err) { sa_n = sa_row[0]; }
        FP8Q_GUARD(nb_lo * KB, 1, sb_len, p.err) { sl_n = __ldg(sb_lo); }
        FP8Q_GUARD(nb_hi * KB, 1, sb_len, p.err) { sh_n = __ldg(sb_hi); }
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          const float sa_v = sa_n, sl_v = sl_n, sh_v = sh_n;
          if (kb + 1 < KB) {
            FP8Q_GUARD(grow * KB + kb + 1, 1, sa_len, p.err) { sa_n = sa_row[kb + 1]; }
            FP8Q_GUARD(nb_lo * KB + kb + 1, 1, sb_len, p.err) { sl_n = __ldg(sb_lo + kb + 1); }
            FP8Q_GUARD(nb_hi * KB + kb + 1, 1, sb_len, p.err) { sh_n = __ldg(sb_hi + kb + 1); }
          }
          const uint32_t b = part_it % GROUPS;
          // warp-uniform decision: the TMEM loads that follow are .sync.aligned
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(base + L::OFF_TFULL + 8 * b, (part_it / GROUPS) & 1u, p.err, kErrTimeoutMma, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t col = lane_base + b * BN + h * COLS;
#pragma unroll
          for (int c = 0; c < NCH; ++c) tc_ld_32x32b_x16(col + 16 * c, r[c]);
          tc_wait_ld(r[0]);
#pragma unroll
          for (int c = 1; c < NCH; ++c) tc_tie(r[c]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            // the stage that writes this buffer next is GROUPS stages later
            const uint32_t next = part_it + GROUPS;
            if (next < total_groups) release(base + L::OFF_FULL + 8 * (next % S));
          }
          ++part_it;
          const float fl = sa_v * sl_v, fh = sa_v * sh_v;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const float f1 = c < nlo ? fl : fh;
            const uint64_t f = pack_f32x2(f1, f1);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[8 * c + j] = fma_f32x2(f, pack_f32x2(r[c][2 * j], r[c][2 * j + 1]), acc[8 * c + j]);
          }
        }
        if (!ok) break;
        // C: this warp's 32 rows x 80 columns staged as five 32-row x 16-column boxes
        // (32-byte rows), each leaving by one TMA store unless it lies past N
        const int box_row = static_cast<int>(static_cast<int64_t>(tm) * TM + row_off) + 32 * q;
        const uint32_t stg = base + L::OFF_STG + static_cast<uint32_t>(warp - CTRL) * L::STG_WARP;
        if (lane == 0) bulk_wait_read<0>();   // the previous tile's stores have read the boxes
        __syncwarp();
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 8; ++j) unpack_f32x2(acc[8 * c + j], v[2 * j], v[2 * j + 1]);
          const uint32_t rowb = stg + static_cast<uint32_t>(c) * 1024u + static_cast<uint32_t>(lane) * 32u;
          sts128(rowb, pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
          sts128(rowb + 16u, pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                 pack_bf16(v[14], v[15]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            if (gcol0 + 16 * c < p.N) tma_store_2d(&tm_c, stg + static_cast<uint32_t>(c) * 1024u, static_cast<int>(gcol0 + 16 * c), box_row);
          bulk_commit();
        }
      } else if constexpr (WIDE) {
        // Promotion, one partial group (two 128-deep partials; this thread's 64 columns
        // of each: four 32-column loads) per TMEM wait.  All four loads are issued
        // together and the group goes back to the MMA issuers as soon as they land;
        // the FMAs follow, overlapping the MMAs that refill the group.  Releasing only
        // after the FMAs (of this group's first partial and the previous group's
        // second) left the tensor pipe idle for part of every hand-off.  Buffers
        // pa / pb hold the group's two partials.
        const float* sa_row = static_cast<const float*>(p.sa) + grow * KB;
        const float* sb_tile = static_cast<const float*>(p.sb) + (gcol0 / 128) * KB;
        uint64_t acc[COLS / 2];
#pragma unroll
        for (int j = 0; j < COLS / 2; ++j) acc[j] = 0;
        uint32_t pa[2][32], pb[2][32];
        auto wait_full = [&]() -> bool {
          const uint32_t g = part_it % GROUPS;
          // warp-uniform decision: the TMEM loads that follow are .sync.aligned
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(base + L::OFF_TFULL + 8 * g, (part_it / GROUPS) & 1u, p.err, kErrTimeoutMma, abort_flag)))
            return false;
          tc_fence_after();
          return true;
        };
        auto load64 = [&](int sub, uint32_t (&r)[2][32]) {
          const uint32_t col = lane_base + ((part_it % GROUPS) * KSUB + sub) * BN + h * COLS;
          tc_ld_32x32b_x32(col, r[0]);
          tc_ld_32x32b_x32(col + 32, r[1]);
        };
        auto promote64 = [&](const uint32_t (&r)[2][32], float f) {
          const uint64_t f2 = pack_f32x2(f, f);
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[16 * c + j] = fma_f32x2(f2, pack_f32x2(r[c][2 * j], r[c][2 * j + 1]), acc[16 * c + j]);
        };
        // per-row B scales: this warpgroup's part of the table ([kb][COLS] floats), and the
        // factor of column j at k-block kb: sA[m, kb] * sB[n0 + j, kb] rounded once, then
        // the FMA (as the single-CTA kernel)
        const uint32_t tbl = base + L::OFF_TBL + static_cast<uint32_t>(h) * L::TBL_PART;
        uint32_t tbl_cur = tbl;   // the table buffer of this tile
        // One chunk q of the group: partial q / 2, columns CW (q % 2) .. +CW-1 of this
        // thread's COLS; its factors fk[j] = sA * (sB[c0 + 2 j], sB[c0 + 2 j + 1]) (each
        // product rounded once) from broadcast table loads, and its FMAs into
        // acc[CW / 2 (q % 2) + j].
        constexpr int CW = COLS / 2;
        uint32_t ra[CW], rb[CW];
        uint64_t fk[CW / 2];
        auto ldc = [&](int q4, uint32_t (&r)[CW]) {
          tc_ld_32x32b(lane_base + ((part_it % GROUPS) * KSUB + (q4 >> 1)) * BN + h * COLS + CW * (q4 & 1), r);
        };
        auto factors = [&](uint64_t (&f)[CW / 2], float sa, int kb, int half) {
          const uint64_t sa2 = pack_f32x2(sa, sa);
          const uint32_t trow = tbl_cur + static_cast<uint32_t>(kb * COLS + half * CW) * 4u;
#pragma unroll
          for (int jj = 0; jj < CW / 4; ++jj) {
            const float4 fb = lds128f(trow + static_cast<uint32_t>(jj) * 16u);
            f[2 * jj] = mul_f32x2(sa2, pack_f32x2(fb.x, fb.y));
            f[2 * jj + 1] = mul_f32x2(sa2, pack_f32x2(fb.z, fb.w));
          }
        };
        auto fmac = [&](const uint32_t (&r)[CW], const uint64_t (&f)[CW / 2], int half) {
#pragma unroll
          for (int j = 0; j < CW / 2; ++j)
            acc[CW / 2 * half + j] = fma_f32x2(f[j], pack_f32x2(r[2 * j], r[2 * j + 1]), acc[CW / 2 * half + j]);
        };
        if constexpr (TABLE) {
          // The part's four warps fill its table with a tile's B scales (warp q: its COLS / 4
          // columns, every k-block) by asynchronous copies that arrive on the buffer's
          // "filled" barrier when they land.  With K / 128 <= 32 the table has two buffers and
          // the next tile's scales are fetched at the start of this one, a whole tile ahead;
          // otherwise this tile's fill is awaited at its start.  A buffer is refilled once the
          // part's four warps have finished reading it (its "read" barrier).
          const int nbuf = KB <= kMaxTableKb / 2 ? 2 : 1;
          auto tbar_full = [&](uint32_t b) { return base + L::OFF_TBAR + 8 * (2 * h + b); };
          auto tbar_free = [&](uint32_t b) { return base + L::OFF_TBAR + 16 * L::NPART + 8 * (2 * h + b); };
          auto fill = [&](int tile, uint32_t b) {
            constexpr int CPW = COLS / 4;   // columns a warp fills
            int ftm, ftn;
            tile_coords<kRasterM>(tile, tiles_m, tiles_n, ftm, ftn);
            const int cq = CPW * q + (lane % CPW);
            const float* src = static_cast<const float*>(p.sb) + (static_cast<int64_t>(ftn) * BN + h * COLS + cq) * KB;
            const uint32_t dst = tbl + b * (L::TBL_PART / 2);
            const int64_t src_i = (static_cast<int64_t>(ftn) * BN + h * COLS + cq) * KB;
            for (int kb = lane / CPW; kb < KB; kb += 32 / CPW)
              FP8Q_GUARD(src_i + kb, 1, sb_len, p.err) { cp_async_4(dst + static_cast<uint32_t>(kb * COLS + cq) * 4u, src + kb); }
            cp_async_arrive_noinc(tbar_full(b));
          };
          bool tok = true;
          if (nbuf == 2) {
            if (tile_it == 0) fill(w.t, 0);
            const int tnext = w.t + units;   // blockwise work is whole tiles, units apart
            if (tnext < ntiles) {
              const uint32_t bn = (tile_it + 1) & 1u;
              if (tile_it >= 1)   // the tile before this one read buffer bn
                tok = __all_sync(0xFFFFFFFFu, mbar_wait(tbar_free(bn), ((tile_it - 1) >> 1) & 1u, p.err,
                                                        kErrTimeoutMma, abort_flag));
              if (tok) fill(tnext, bn);
            }
          } else {
            if (tile_it > 0)
              tok = __all_sync(0xFFFFFFFFu, mbar_wait(tbar_free(0), (tile_it - 1) & 1u, p.err, kErrTimeoutMma, abort_flag));
            if (tok) fill(w.t, 0);
          }
          tbl_cur = tbl + (nbuf == 2 ? (tile_it & 1u) * (L::TBL_PART / 2) : 0u);
          if (!tok || !__all_sync(0xFFFFFFFFu, mbar_wait(tbar_full(nbuf == 2 ? (tile_it & 1u) : 0u),
                                                         (nbuf == 2 ? (tile_it >> 1) : tile_it) & 1u, p.err,
                                                         kErrTimeoutMma, abort_flag)))
            break;
        }
        // scale factors of the group to promote next (loads in flight)
        float sa0 = 0.0f, sa1 = 0.0f;
        FP8Q_GUARD(grow * KB, 2, sa_len, p.err) {
          sa0 = sa_row[0];
          sa1 = sa_row[1];
        }
        float sb0 = 0.0f, sb1 = 0.0f;
        if constexpr (!TABLE) {
          FP8Q_GUARD((gcol0 / 128) * KB, 2, sb_len, p.err) {
            sb0 = __ldg(sb_tile);
            sb1 = __ldg(sb_tile + 1);
          }
        }
        bool ok = true;
        if constexpr (TABLE) {
          // Per-row B scales: every column n has its own factor sA[m, kb] * sB[n, kb], so
          // the promotion does twice the FP32 work of the common pairing and, with the MMAs
          // far ahead, its own instruction stream sets the pace.  The group is taken in four
          // 32-column chunks (partial 0 columns 0-31, 32-63, then partial 1), software-
          // pipelined over two register buffers: each chunk's TMEM load is in flight while
          // the previous chunk's FMAs and the next chunk's factors (table loads, packed
          // multiplies) run; the group goes back to the MMA issuers once the last chunk has
          // landed.  The next group's barrier is tested right after that and its answer used
          // after the last FMAs.  (Two loads in flight per warp over three buffers ran
          // slower: the TMEM read rate, not the load latency, bounds the loop.)
          bool ready_next = false;   // the next group's partials were seen complete early
          for (int kg = 0; kg < NG; ++kg) {
            const float a0 = sa0, a1 = sa1;
            if (kg + 1 < NG) {
              FP8Q_GUARD(grow * KB + 2 * kg + 2, 2, sa_len, p.err) {
                sa0 = sa_row[2 * kg + 2];
                sa1 = sa_row[2 * kg + 3];
              }
            }
            if (!__all_sync(0xFFFFFFFFu, ready_next)) {
              ok = wait_full();
              if (!ok) break;
            } else {
              tc_fence_after();
            }
            ldc(0, ra);
            factors(fk, a0, 2 * kg, 0);
            tc_wait_ld(ra);
            ldc(1, rb);
            fmac(ra, fk, 0);
            factors(fk, a0, 2 * kg, 1);
            tc_wait_ld(rb);
            ldc(2, ra);
            fmac(rb, fk, 1);
            factors(fk, a1, 2 * kg + 1, 0);
            tc_wait_ld(ra);
            ldc(3, rb);
            fmac(ra, fk, 0);
            factors(fk, a1, 2 * kg + 1, 1);
            tc_wait_ld(rb);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              const uint32_t next = part_it + GROUPS;
              if (next < total_groups) release(base + L::OFF_FULL + 8 * (next % S));
            }
            ++part_it;
            ready_next = kg + 1 < NG &&
                         mbar_test_wait(base + L::OFF_TFULL + 8 * (part_it % GROUPS), (part_it / GROUPS) & 1u);
            fmac(rb, fk, 1);
          }
        }
        if constexpr (!TABLE)
        for (int kg = 0; kg < NG; ++kg) {
          ok = wait_full();
          if (!ok) break;
          load64(0, pa);
          load64(1, pb);
          tc_wait_ld(pa[0]);          // both partials of the group have landed
          tc_tie(pa[1]);
          tc_tie(pb[0]);
          tc_tie(pb[1]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            // the stage that reuses this group is GROUPS stages later
            const uint32_t next = part_it + GROUPS;
            if (next < total_groups) release(base + L::OFF_FULL + 8 * (next % S));
          }
          ++part_it;
          // the scale factors are used only after the release (a tile's first ones were
          // loaded at its start and may still be in flight)
          {
            const float f0 = sa0 * sb0, f1 = sa1 * sb1;
            if (kg + 1 < NG) {
              FP8Q_GUARD(grow * KB + 2 * kg + 2, 2, sa_len, p.err) {
                sa0 = sa_row[2 * kg + 2];
                sa1 = sa_row[2 * kg + 3];
              }
              FP8Q_GUARD((gcol0 / 128) * KB + 2 * kg + 2, 2, sb_len, p.err) {
                sb0 = __ldg(sb_tile + 2 * kg + 2);
                sb1 = __ldg(sb_tile + 2 * kg + 3);
              }
            }
            promote64(pa, f0);          // the FMAs run while the MMAs refill the group
            promote64(pb, f1);
          }
        }
        if (!ok) break;
        if constexpr (TABLE) {
          __syncwarp();   // every lane's table reads of this tile are done
          const uint32_t b = KB <= kMaxTableKb / 2 ? (tile_it & 1u) : 0u;
          if (lane == 0) mbar_arrive(base + L::OFF_TBAR + 16 * L::NPART + 8 * (2 * h + b));
          ++tile_it;
        }
        // C through TMA stores of this warp's staged box (as the other kinds)
        const int box_row = static_cast<int>(static_cast<int64_t>(tm) * TM + row_off) + 32 * q;
#pragma unroll
        for (int c32 = 0; c32 < COLS / 32; ++c32) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) unpack_f32x2(acc[16 * c32 + j], v[2 * j], v[2 * j + 1]);
          if (QOUT && (want_q || want_amax) && gcol0 + 32 * c32 < p.N) emit(v, grow, gcol0 + 32 * c32, false);
          if (p.c != nullptr) store_chunk(v, c32, gcol0, box_row);
        }
      } else if (BLOCK) {
        const float* sa_row = static_cast<const float*>(p.sa) + grow * KB;
        const float* sb_blk = static_cast<const float*>(p.sb);
        // Promotion: TMEM loads of CW columns (32, or 16 when a thread owns 128 columns or
        // loads a B scale per column, to fit the registers), software-pipelined: while the FMAs of one chunk run, the
        // load of the next chunk (of this partial, or the first of the next partial) is in
        // flight.  A partial buffer is released once all its chunks are in registers.
        constexpr int CW = (COLS >= 128 || B_ROWS) ? 16 : 32;
        constexpr int NC = COLS / CW;
        static_assert(!BLOCK || (NC % 2 == 0 && COLS % 32 == 0), "blockwise promotion chunking");
        const float* sb_tile = sb_blk + (gcol0 / 128) * KB;   // 128x128 B: one factor per k-block
        uint64_t acc[COLS / 2];              // column pairs (2j, 2j+1) of this thread's columns
#pragma unroll
        for (int j = 0; j < COLS / 2; ++j) acc[j] = 0;
        // scale factors are fetched two k-blocks ahead, off the promotion's critical path
        float sa0 = 0.0f, sa1 = 0.0f, sb0 = 0.0f, sb1 = 0.0f;
        FP8Q_GUARD(grow * KB, KB > 1 ? 2 : 1, sa_len, p.err) {
          sa0 = sa_row[0];
          sa1 = KB > 1 ? sa_row[1] : 0.0f;
        }
        if (!B_ROWS) FP8Q_GUARD((gcol0 / 128) * KB, KB > 1 ? 2 : 1, sb_len, p.err) {
          sb0 = __ldg(sb_tile);
          sb1 = KB > 1 ? __ldg(sb_tile + 1) : 0.0f;
        }
        auto wait_full = [&]() -> bool {
          const uint32_t pb = part_it % GROUPS;
          // warp-uniform decision: the TMEM loads that follow are .sync.aligned
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(base + L::OFF_TFULL + 8 * pb, (part_it / GROUPS) & 1u, p.err, kErrTimeoutMma, abort_flag)))
            return false;
          tc_fence_after();
          return true;
        };
        auto promote = [&](const uint32_t (&r)[CW], int c, float sa_v, float sb_v, int kb) {
          if (B_ROWS) {
            // per-column B scales: sB[n, kb]
            const float* sbc = sb_blk + (gcol0 + CW * c) * KB + kb;
            if constexpr (kDebugIndex) {   // every column's scale of this k-block
              for (int j = 0; j < CW; ++j) in_range((gcol0 + CW * c + j) * KB + kb, sb_len, p.err);
            }
#pragma unroll
            for (int j = 0; j < CW / 2; ++j) {
              const uint64_t f = pack_f32x2(sa_v * __ldg(sbc + (2 * j) * KB), sa_v * __ldg(sbc + (2 * j + 1) * KB));
              acc[(CW / 2) * c + j] = fma_f32x2(f, pack_f32x2(r[2 * j], r[2 * j + 1]), acc[(CW / 2) * c + j]);
            }
          } else {
            const float f1 = sa_v * sb_v;
            const uint64_t f = pack_f32x2(f1, f1);
#pragma unroll
            for (int j = 0; j < CW / 2; ++j)
              acc[(CW / 2) * c + j] = fma_f32x2(f, pack_f32x2(r[2 * j], r[2 * j + 1]), acc[(CW / 2) * c + j]);
          }
        };
        uint32_t rbuf[2][CW];
        // column offset in TMEM of chunk c of sub-block `sub` of partial group `pb`
        auto chunk_col = [&](uint32_t pb, int sub, int c) -> uint32_t {
          return lane_base + (pb * KSUB + sub) * BN + h * COLS + CW * c;
        };
        bool ok = wait_full();
        if (ok) tc_ld_32x32b(chunk_col(part_it % GROUPS, 0, 0), rbuf[0]);
        for (int kg = 0; ok && kg < NG; ++kg) {
          const uint32_t group_seq = part_it;   // stages (= partial groups) this CTA has used before
          const uint32_t pb = part_it % GROUPS;
#pragma unroll
          for (int sub = 0; sub < KSUB; ++sub) {
            const int kb = kg * KSUB + sub;
            const float sa_v = sa0, sb_v = sb0;
            sa0 = sa1;
            sb0 = sb1;
            if (kb + 2 < KB) {
              FP8Q_GUARD(grow * KB + kb + 2, 1, sa_len, p.err) { sa1 = sa_row[kb + 2]; }
              if (!B_ROWS) FP8Q_GUARD((gcol0 / 128) * KB + kb + 2, 1, sb_len, p.err) { sb1 = __ldg(sb_tile + kb + 2); }
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              const int i = sub * NC + c;   // chunk index within the group (NC is even)
              tc_wait_ld(rbuf[i & 1]);
              if (c + 1 < NC) {
                tc_ld_32x32b(chunk_col(pb, sub, c + 1), rbuf[(i + 1) & 1]);
              } else if (sub + 1 < KSUB) {
                tc_ld_32x32b(chunk_col(pb, sub + 1, 0), rbuf[(i + 1) & 1]);
              } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                  if (GATED) {
                    // the stage that reuses this group is GROUPS stages later
                    const uint32_t next = group_seq + GROUPS;
                    if (next < total_groups) release(base + L::OFF_FULL + 8 * (next % S));
                  } else {
                    release(base + L::OFF_TEMPTY + 8 * pb);   // the group's partials fully read
                  }
                }
                ++part_it;
                if (kg + 1 < NG) {
                  ok = wait_full();
                  if (ok) tc_ld_32x32b(chunk_col(part_it % GROUPS, 0, 0), rbuf[(i + 1) & 1]);
                }
              }
              promote(rbuf[i & 1], c, sa_v, sb_v, kb);
            }
          }
        }
        if (!ok) break;
#pragma unroll
        for (int c32 = 0; c32 < COLS / 32; ++c32) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) unpack_f32x2(acc[16 * c32 + j], v[2 * j], v[2 * j + 1]);
          if (gcol0 + 32 * c32 < p.N) emit(v, grow, gcol0 + 32 * c32);
        }
      } else {
        const uint32_t a = acc_it % ACC;
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(base + L::OFF_TFULL + 8 * a, (acc_it / ACC) & 1u, p.err, kErrTimeoutMma, abort_flag)))
          break;
        tc_fence_after();
        const uint32_t col_base = lane_base + a * BN + h * COLS;
        constexpr int CH = COLS / 32;
        if (SPLITK && w.part >= 0) {
          const int box_row = static_cast<int>(static_cast<int64_t>(tm) * TM + row_off) + 32 * q;
          // A part of a tile cut along K: 32 columns at a time straight from TMEM, the
          // accumulator released at the end.  A part 1 leaves its raw FP32 values in its slot
          // and counts its warps there; a part 0 (the tile's first K blocks) waits for each of
          // its slots' counts, adds their values in order, then scales and stores as a whole
          // tile would.  Both CTAs' epilogue warps of a pair count on (and, for part 0, read)
          // a slot.  A slot holds 16-byte pieces [column slice][chunk][piece][row of the tile],
          // so a warp's 16-byte stores and loads cover 512 consecutive bytes.
          constexpr int kSlotWarps = 2 * EPI;
          if (w.part == 0) {
            bool got = true;
            if (lane == 0)
              for (int k = 0; k < w.nslot && got; ++k)
                FP8Q_GUARD(w.slot + k * w.sstride, 1, p.ws_nflags, p.err) {
                  got = wait_count(p.ws_flags + w.slot + k * w.sstride, kSlotWarps, p.err, kErrTimeoutMma);
                }
            if (!__shfl_sync(0xFFFFFFFFu, got, 0)) break;   // timed out: the error word says so
          }
          // float offset of 16-byte piece i of chunk c of this thread's row in slot `sl`
          auto piece = [&](int sl, int c, int i) -> int64_t {
            return ((static_cast<int64_t>(sl) * (BN / 4) + (h * CH + c) * 8 + i) * TM + row_off + row) * 4;
          };
          if (w.part > 0) {
            // the thread's whole row slice from TMEM at once; the accumulator goes back to the
            // MMA issuer before the pieces are stored (with one accumulator, MX, its next work
            // item waited ~2.6 us for these stores, measured)
            uint32_t r[CH][32];
#pragma unroll
            for (int c = 0; c < CH; ++c) tc_ld_32x32b_x32(col_base + 32 * c, r[c]);
#pragma unroll
            for (int c = 0; c < CH; ++c) tc_wait_ld(r[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(base + L::OFF_TEMPTY + 8 * a);
#pragma unroll
            for (int c = 0; c < CH; ++c)
#pragma unroll
              for (int i = 0; i < 8; ++i)
                FP8Q_GUARD(piece(w.slot, c, i), 4, p.ws_len, p.err) {
                  stg128(p.ws + piece(w.slot, c, i), r[c][4 * i], r[c][4 * i + 1], r[c][4 * i + 2], r[c][4 * i + 3]);
                }
          } else {
            // the first slot's pieces of the next chunk are in flight while this chunk is
            // summed (further slots are loaded as they are added)
            float4 o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              o[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              FP8Q_GUARD(piece(w.slot, 0, i), 4, p.ws_len, p.err) {
                o[i] = __ldcg(reinterpret_cast<const float4*>(p.ws + piece(w.slot, 0, i)));
              }
            }
            for (int c = 0; c < CH; ++c) {
              uint32_t rc[32];
              tc_ld_32x32b_x32(col_base + 32 * c, rc);
              tc_wait_ld(rc);
              float v[32];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                v[4 * i] = __uint_as_float(rc[4 * i]) + o[i].x;
                v[4 * i + 1] = __uint_as_float(rc[4 * i + 1]) + o[i].y;
                v[4 * i + 2] = __uint_as_float(rc[4 * i + 2]) + o[i].z;
                v[4 * i + 3] = __uint_as_float(rc[4 * i + 3]) + o[i].w;
              }
              if (c + 1 < CH) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  FP8Q_GUARD(piece(w.slot, c + 1, i), 4, p.ws_len, p.err) {
                    o[i] = __ldcg(reinterpret_cast<const float4*>(p.ws + piece(w.slot, c + 1, i)));
                  }
              }
              for (int k = 1; k < w.nslot; ++k) {
                const int sl = w.slot + k * w.sstride;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  float4 e = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                  FP8Q_GUARD(piece(sl, c, i), 4, p.ws_len, p.err) {
                    e = __ldcg(reinterpret_cast<const float4*>(p.ws + piece(sl, c, i)));
                  }
                  v[4 * i] += e.x;
                  v[4 * i + 1] += e.y;
                  v[4 * i + 2] += e.z;
                  v[4 * i + 3] += e.w;
                }
              }
              if (KIND == kTensor) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], tensor_scale);
              }
              if (QOUT && (want_q || want_amax) && gcol0 + 32 * c < p.N) emit(v, grow, gcol0 + 32 * c, false);
              if (p.c != nullptr) store_chunk(v, c, gcol0, box_row);
            }
          }
          if (w.part == 0) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(base + L::OFF_TEMPTY + 8 * a);
          }
          if (w.part > 0) {
            __threadfence();   // this thread's slot values, before the warp is counted
            __syncwarp();
            if (lane == 0) FP8Q_GUARD(w.slot, 1, p.ws_nflags, p.err) { atomicAdd(p.ws_flags + w.slot, 1); }
          } else if (lane == 0) {
            // the last of the two pairs' warps to count on a slot (all have read it) resets it
            for (int k = 0; k < w.nslot; ++k) {
              int* f = p.ws_flags + w.slot + k * w.sstride;
              FP8Q_GUARD(w.slot + k * w.sstride, 1, p.ws_nflags, p.err) {
                if (atomicAdd(f, 1) == 2 * kSlotWarps - 1) atomicExch(f, 0);
              }
            }
          }
          ++acc_it;
          continue;
        }
        {
          // pull the whole half-row into registers, free the accumulator, then scale and store
          uint32_t r[CH][32];
#pragma unroll
          for (int c = 0; c < CH; ++c) tc_ld_32x32b_x32(col_base + 32 * c, r[c]);
#pragma unroll
          for (int c = 0; c < CH; ++c) tc_wait_ld(r[c]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release(base + L::OFF_TEMPTY + 8 * a);
          const int box_row = static_cast<int>(static_cast<int64_t>(tm) * TM + row_off) + 32 * q;
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = (KIND == kTensor) ? __fmul_rn(__uint_as_float(r[c][j]), tensor_scale) : __uint_as_float(r[c][j]);
            if (QOUT && (want_q || want_amax) && gcol0 + 32 * c < p.N) emit(v, grow, gcol0 + 32 * c, false);
            if (p.c != nullptr) store_chunk(v, c, gcol0, box_row);
          }
        }
        ++acc_it;
      }
    }
    if (L::TSTORE && lane == 0) bulk_wait_all<0>();   // this warp's TMA stores have finished
    if (TABLE) cp_async_wait_all();                  // no table copy of this thread still in flight
    if (QOUT && want_amax) {
      // one atomic per warp, on the (non-negative) float bits, which order like the values
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) y_amax = fmaxf(y_amax, __shfl_xor_sync(0xFFFFFFFFu, y_amax, o));
      if (lane == 0 && y_amax > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(p.c_amax), __float_as_uint(y_amax));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
}

// Workspaces of the K-split last wave: one per (device, stream), slots of 256 x 256 FP32
// partial tiles (one per pair at most) and their warp counters, allocated on a stream's
// first split launch and kept for the process's lifetime.  A stream in capture that has
// none yet (or a full table, or a failed allocation) runs the GEMM unsplit.  Launches on
// one stream are ordered, so they never share a workspace concurrently.
constexpr int kMaxSplit = 8;
constexpr bool kStreamK = true;
constexpr int kMaxSplitStreams = 16;
constexpr size_t kSplitSlotBytes = size_t(2 * kBM) * 256 * sizeof(float);
struct SplitWorkspace {
  cudaStream_t stream;
  float* ws;
  int* flags;
};
std::mutex g_split_mu;
SplitWorkspace g_split_ws[kMaxDevices][kMaxSplitStreams];
int g_split_n[kMaxDevices];

bool split_workspace(cudaStream_t s, int slots, float** ws, int** flags) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_split_mu);
  for (int i = 0; i < g_split_n[dev]; ++i) {
    if (g_split_ws[dev][i].stream == s) {
      *ws = g_split_ws[dev][i].ws;
      *flags = g_split_ws[dev][i].flags;
      return true;
    }
  }
  if (g_split_n[dev] == kMaxSplitStreams) return false;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return false;
  }
  // relaxed capture mode: allocating here must not invalidate another thread's capture
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  cudaThreadExchangeStreamCaptureMode(&mode);
  float* w = nullptr;
  int* f = nullptr;
  bool ok = cudaMalloc(&w, static_cast<size_t>(slots) * kSplitSlotBytes) == cudaSuccess &&
            cudaMalloc(&f, static_cast<size_t>(slots) * sizeof(int)) == cudaSuccess &&
            cudaMemsetAsync(f, 0, static_cast<size_t>(slots) * sizeof(int), s) == cudaSuccess;
  cudaThreadExchangeStreamCaptureMode(&mode);
  if (!ok) {
    if (w != nullptr) cudaFree(w);
    if (f != nullptr) cudaFree(f);
    cudaGetLastError();
    return false;
  }
  g_split_ws[dev][g_split_n[dev]++] = SplitWorkspace{s, w, f};
  *ws = w;
  *flags = f;
  return true;
}

// A kernel that moves registers between warpgroups must have been given exactly the
// launch registers the split was sized for (with fewer, an increase would never be
// granted and the epilogue warps would not start).  Checked once per device.
template <class K>
cudaError_t check_split_regs(K kern, bool split, std::atomic<bool> (&checked)[kMaxDevices]) {
  if (!split) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (checked[dev].load(std::memory_order_acquire)) return cudaSuccess;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kSplitLaunchRegs) return cudaErrorInvalidConfiguration;
  checked[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

}  // namespace

PairDivision pair_division(int kind, int64_t ntiles, int64_t pairs, int64_t k) {
  PairDivision d{0, 1, static_cast<int>(ntiles), ntiles < pairs ? ntiles : pairs};
  if (kind != kTensor && kind != kMx) return d;
  const int64_t full = ntiles / pairs, rest = ntiles % pairs, ng = k / kBK;
  // Two or three full waves and a partial one: all but the last full wave as whole tiles,
  // then every pair an equal share of the remaining tiles' K blocks (each share over one
  // tile long).  With more waves the partial one costs less than the hand-overs (measured:
  // MX 8192 x 12288 x 4096, 20 waves, 4 % slower).  With one full wave every tile is
  // shared: worth it for K >= 8192 (2560 x 2304 x 8192: 0.54 -> 0.61 against the K-range
  // cut), not at K = 4096 (MX 2048 x 4096 x 4096: 0.55 -> 0.50 against whole tiles).
  if (kStreamK && full >= 1 && rest > 0 && full <= 3 && (full >= 2 || ng >= 64)) {
    d.streamk = 1;
    d.tail0 = static_cast<int>((full - 1) * pairs);
    d.launched = pairs;
    return d;
  }
  // A last wave that would leave at least half of the pairs idle is cut along K: its R
  // tiles into S ranges on R * S pairs (every pair resident, so the waits end).  The
  // hand-over of the ranges costs a few microseconds whatever K is, the time saved grows
  // with K: measured side by side, +1-2 % at 8192^3, +3 % at 2048 x 36864 x 12288, +9 % at
  // 2048 x 12288 x 49152, but nothing at 4096^3 and -6 % at 49152 x 12288 x 2048.  So the
  // cut is made for K >= 8192, or when there is only the one partial wave.
  if (rest > 0 && 2 * rest <= pairs && ng >= 2 && (full == 0 || ng >= 64)) {
    int64_t split = pairs / rest;
    if (split > ng) split = ng;
    if (split > kMaxSplit) split = kMaxSplit;
    d.split = static_cast<int>(split);
    d.tail0 = static_cast<int>(full * pairs);
    d.launched = full > 0 ? pairs : rest * split;
  }
  return d;
}

namespace {

template <int KIND, bool QOUT>
cudaError_t launch_kind(const GemmParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_sfa,
                        const CUtensorMap& tm_sfb, const CUtensorMap& tm_c, int num_sms, cudaStream_t s) {
  using L = Layout<KIND, false>;
  static_assert(L::SMEM <= 232448, "shared memory budget");
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_limit(k_gemm<KIND, false, QOUT>, static_cast<int>(L::SMEM), attr_done);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> regs_checked[kMaxDevices] = {};
  e = check_split_regs(k_gemm<KIND, false, QOUT>, Cfg<KIND>::CTRL == 4, regs_checked);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (p.M / kBM) * ((p.N + L::BN - 1) / L::BN);
  const int grid = static_cast<int>(ntiles < num_sms ? ntiles : num_sms);
  return launch_pdl(k_gemm<KIND, false, QOUT>, dim3(grid), dim3(threads_of<KIND>()), L::SMEM, s, 1, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, p);
}

// 2-CTA clusters; the grid is as many pairs as can be resident at once (at most
// one per two SMs), each walking the 256-row tiles with a stride of the pair count.
template <int KIND, bool QOUT>
cudaError_t launch_pair(const GemmParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_sfa,
                        const CUtensorMap& tm_sfb, const CUtensorMap& tm_c, int num_sms, cudaStream_t s) {
  using L = Layout<KIND, true>;
  static_assert(L::SMEM <= 232448, "shared memory budget");
  auto kern = k_gemm<KIND, true, QOUT>;
  static std::atomic<bool> attr_done[kMaxDevices] = {};
  cudaError_t e = ensure_smem_limit(kern, static_cast<int>(L::SMEM), attr_done);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> regs_checked[kMaxDevices] = {};
  e = check_split_regs(kern, Cfg<KIND>::CTRL == 4, regs_checked);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(threads_of<KIND>());
  cfg.dynamicSmemBytes = L::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int64_t ntiles = (p.M / (2 * kBM)) * ((p.N + L::BN - 1) / L::BN);
  int64_t pairs = num_sms / 2;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  // resident pairs: queried once per device
  static std::atomic<int> max_clusters[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (max_clusters[dev].load(std::memory_order_relaxed) == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = static_cast<int>(pairs);
    max_clusters[dev].store(n, std::memory_order_relaxed);
  }
  const int resident = max_clusters[dev].load(std::memory_order_relaxed);
  if (resident < pairs) pairs = resident;
  GemmParams q = p;
  q.split = 1;
  q.tail0 = static_cast<int>(ntiles);
  q.streamk = 0;
  q.ws = nullptr;
  q.ws_flags = nullptr;
  const PairDivision d = pair_division(KIND, ntiles, pairs, p.K);
  int64_t launched = ntiles < pairs ? ntiles : pairs;
  if (d.streamk || d.split > 1) {
    // both need the stream's workspace; without one (a capture that has none yet, a full
    // table, a failed allocation) the tiles run whole
    float* ws = nullptr;
    int* flags = nullptr;
    if (split_workspace(s, static_cast<int>(num_sms / 2), &ws, &flags)) {
      q.streamk = d.streamk;
      q.split = d.split;
      q.tail0 = d.tail0;
      q.ws = ws;
      q.ws_flags = flags;
      q.ws_len = static_cast<int64_t>(num_sms / 2) * static_cast<int64_t>(kSplitSlotBytes / sizeof(float));
      q.ws_nflags = num_sms / 2;
      launched = d.launched;
    }
  }
  cfg.gridDim = dim3(static_cast<unsigned>(2 * launched));
  return launch_pdl(kern, cfg.gridDim, cfg.blockDim, L::SMEM, s, 2, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, q);
}

}  // namespace

bool gemm_select_wide(const GemmParams& p, int num_sms) {
  if (p.kind != kBlock1x128 || p.b_1x128 || p.out_fp32 || p.c == nullptr || p.cq != nullptr || p.c_amax != nullptr)
    return false;
  if (p.M % (2 * kBM) != 0 || num_sms < 2) return false;
  // The other pair kernel needs K / 128 even (else one CTA per 128 x 128 tile, slower).
  return (p.K / kBK) % 2 != 0;
}

int gemm_block_n(const GemmParams& p) {
  if (p.wide160) return Cfg<kBlock160>::BN;
  return p.kind == kBlock1x128 ? Cfg<kBlock1x128>::BN : (p.kind == kMx ? Cfg<kMx>::BN : Cfg<kTensor>::BN);
}

int gemm_c_box_cols(const GemmParams& p) { return p.wide160 ? 16 : 0; }

// CTA pairs need M a multiple of 256.  Blockwise runs on pairs only with 256-deep
// stages (K / 128 even) and 128x128 B scales: there each stage's two partials go to
// the promotion as one group, so the cross-SM release is paid once per 8 MMAs.  The
// release is a CTA-scope arrive on the leader's barrier: with cluster-scope release
// semantics each arrive also waited for the epilogue's earlier global stores, which
// made the blockwise pair 40 % slower (measured).
bool gemm_uses_pair(const GemmParams& p) {
  if (p.M % (2 * kBM) != 0) return false;
  if (p.wide160) return true;
  if (p.kind == kBlock1x128) return (p.K / kBK) % 2 == 0 && (!p.b_1x128 || p.K / kBK <= kMaxTableKb);
  return true;
}

int gemm_b_box_rows(const GemmParams& p) { return gemm_uses_pair(p) ? gemm_block_n(p) / 2 : gemm_block_n(p); }

GemmPlan gemm_plan(const GemmParams& p, int num_sms, int resident_pairs) {
  GemmPlan g{};
  g.pair = gemm_uses_pair(p) ? 1 : 0;
  g.block_n = gemm_block_n(p);
  if (p.kind == kBlock1x128) {
    if (p.b_1x128) g.variant = g.pair ? kBlockK2RowsB : kBlockRowsB;
    else if (p.wide160) g.variant = kBlock160;
    else g.variant = (g.pair || (p.K / kBK) % 2 == 0) ? kBlockK2 : kBlock1x128;
  } else {
    g.variant = p.kind;
  }
  const int64_t rows = g.pair ? 2 * kBM : kBM;
  g.ntiles = (p.M / rows) * ((p.N + g.block_n - 1) / g.block_n);
  if (g.pair) {
    int64_t pairs = num_sms / 2;
    if (resident_pairs > 0 && resident_pairs < pairs) pairs = resident_pairs;
    g.div = pair_division(g.variant, g.ntiles, pairs, p.K);
  } else {
    g.div = PairDivision{0, 1, static_cast<int>(g.ntiles), g.ntiles < num_sms ? g.ntiles : num_sms};
  }
  return g;
}

template <bool QOUT>
cudaError_t launch_gemm_q(const GemmParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_sfa,
                          const CUtensorMap& tm_sfb, const CUtensorMap& tm_c, int num_sms, cudaStream_t s) {
  switch (p.kind) {
    case kTensor:
      return gemm_uses_pair(p) ? launch_pair<kTensor, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s)
                               : launch_kind<kTensor, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
    case kBlock1x128:
      if (p.b_1x128)
        return gemm_uses_pair(p) ? launch_pair<kBlockK2RowsB, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s)
                                 : launch_kind<kBlockRowsB, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
      if constexpr (!QOUT)
        if (p.wide160) return launch_pair<kBlock160, false>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
      if (gemm_uses_pair(p)) return launch_pair<kBlockK2, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
      return (p.K / kBK) % 2 == 0 ? launch_kind<kBlockK2, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s)
                                  : launch_kind<kBlock1x128, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
    default:
      return gemm_uses_pair(p) ? launch_pair<kMx, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s)
                               : launch_kind<kMx, QOUT>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
  }
}

cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_sfa,
                        const CUtensorMap& tm_sfb, const CUtensorMap& tm_c, int num_sms, cudaStream_t s) {
  if (p.cq != nullptr || p.c_amax != nullptr) return launch_gemm_q<true>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
  return launch_gemm_q<false>(p, tm_a, tm_b, tm_sfa, tm_sfb, tm_c, num_sms, s);
}

}  // namespace fp8q
