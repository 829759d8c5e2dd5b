// Persistent grouped GEMM on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, over the tile schedule that mgemm_fill_args wrote:
//   kRows mode (forward, dgrad):   out[r, n] = sum_k A[r, k] B_e(r)[n, k]
//       one tile = 128 token rows of one non-empty group x BN output columns;
//       tiles of empty groups do not exist ("F8I4 Grouped Gemm Optimization
//       for Sparse M", Summary).
//   kExperts mode (wgrad):         out_e[k, n] = sum_{r in group e} A[r, k] G[r, n]
//       one tile = 128 rows of K x BN columns of N of expert e, contracting
//       over the rows of group e ("dynamic k"); experts are visited in the
//       order sorted by group size, largest first, and empty experts get a
//       zero tile with no main loop ("Support GPU-resident batch sizes",
//       review of csrc/fill_arguments.cuh and ZeroOutK0Outputs).
// BN (64, 128, 192 or 256) is chosen per launch on the host to balance the tile
// count against the number of SMs.
//
// CTA layout (64 + 32 x EPI threads, one CTA per SM, grid = number of SMs,
// tiles strided by the grid; with CTA pairs, tiles strided by the clusters):
//   warp 0      TMA producer: one thread fills a ring (4, 6 or 8 stages) of
//               (A 128 rows x 128 B, B BN rows x 128 B) shared-memory tiles,
//               128-byte swizzled, each stage guarded by a full/empty mbarrier.
//   warp 1      TMEM owner and MMA issuer: allocates two 128 x BN_MAX fp32
//               accumulators in TMEM, one thread issues
//               tcgen05.mma (M=128, N=BN, K=16 bf16 / 32 e4m3) per 32-byte
//               K step and commits stage-release / accumulator-ready events.
//               On the partial last block of a group in bf16 wgrad the warp
//               issues only the k-steps that hold group rows and first zeroes
//               the few out-of-group positions inside the partial step (FP8
//               wgrad reads the padded layout, whose blocks are whole).
//   warps 2..   epilogue, EPI = 4 warps (one per TMEM lane quarter, 32 output
//               rows each) or 8 (two per quarter, each taking every other
//               64-column chunk): tcgen05.ld, optional FP8 scale division
//               (packed fp32x2 multiplies by power-of-two reciprocals fetched
//               one tile ahead), bf16 rounding, then 128-byte-swizzled
//               shared-memory staging buffers and a TMA store of each 32-row x
//               64-column block.  A warp whose 32 rows are not all valid (group
//               edge) stores those rows directly instead, so nothing outside
//               the tile's rows is ever written.  The accumulator is released
//               right after its last tcgen05.ld, so the next tile's main loop
//               overlaps the stores.
// CTA pairs (FP8 wgrad): a cluster of two CTAs computes one 256-row tile with
// cta_group::2 MMAs issued by the even CTA.  Each CTA copies its 128 rows of A
// and half of B's columns; the odd CTA's copies complete on the even CTA's
// full barrier (which expects both CTAs' bytes), MMA commits free the stage
// and publish the accumulator in both CTAs (multicast), and both CTAs'
// epilogue warps hand the accumulator back on the even CTA's barrier.  Per SM
// that is 32 KB of operands per contraction block instead of 48 KB, and six
// ring stages instead of four.
// Every mbarrier wait is bounded (about 1 s); on expiry the kernel records
// MGEMM_STATUS_TIMEOUT in the args block, lets the other roles leave their
// loops, drains its own outstanding copies and MMAs, frees TMEM and returns.
#pragma once

#include "common.cuh"

namespace mgemm {

enum { kModeRows = 0, kModeExperts = 1 };

// kBnMax / kStages: the widest output tile this instantiation serves and its
// ring depth.  Wide (256, 4 stages), 192-wide (5), mid (128, 6) and narrow
// (64, 8) forms fill the same shared memory; the narrower forms serve
// weight-streaming launches, where a deeper ring keeps more HBM reads in
// flight per SM, and the 192-wide one gives the weight tile the largest share
// of the ring (the A tile, re-read from L2, is the same 16 KB in every form).
// kPair: a cluster of two CTAs computes one 256-row tile with cta_group::2
// MMAs (each CTA loads its 128 rows of A and half of B's columns), so every SM
// reads half of the B tile it would otherwise read.
// kEpiWarps: epilogue warps, 4 (one per TMEM lane quarter) or 8 (two per
// quarter, splitting the tile's 64-column chunks between them).
// kDynRing: the ring's stages are [A slot of a_rows x 128 B][B slot of BN x
// 128 B] and their number is chosen per launch (kStages is then the most
// there can be): with few token rows (sparse routing) the A slot shrinks to
// those rows and the weight stream gets the rest of shared memory.
// kKc: contraction blocks per ring stage (run-time rings only).  With kKc > 1
// each operand comes in one box of kKc consecutive 128-byte k-chunks (a 3-d /
// 4-d view of the K-major tensor, chunk stride 128 B), landing as kKc
// consecutive MMA tiles: fewer, larger copies, which is what latency-bound
// launches with few rows need.
template <bool kFp8, bool kAMn, bool kBMn, int kMode, int kBnMax = 256, int kStages = 4, int kOutBufs = 2,
          bool kPair = false, int kEpiWarps = 4, bool kDynRing = false, int kKc = 1, bool kMx = false>
struct GemmCfg {
  static constexpr bool Fp8 = kFp8;
  // kMx: MXFP8 -- e4m3 operands with one e8m0 scale per 32 contraction
  // elements of every row, applied by block-scaled MMAs (no epilogue scales)
  static constexpr bool Mx = kMx;
  static constexpr bool Scaled = kFp8 && !kMx;  // FP8 with row / column scales in the epilogue
  static_assert(!kMx || (kFp8 && !kAMn && !kBMn && !kPair && !kDynRing &&
                          (kBnMax == 128 || kBnMax == 192 || kBnMax == 256)),
                "MXFP8: K-major operands, 128-, 192- or 256-wide tiles");
  // MXFP8 scale rows per contraction block: the rows schedule's scale rows
  // are [rows][ld_sf] (16 bytes = four blocks per row); the experts schedule's
  // (wgrad) are k-block-major [blocks][rows][4 B] (one block per load)
  static constexpr int KPS = kMode == kModeRows ? 4 : 1;
  static constexpr bool AMn = kAMn;  // A stored MN-major (contraction is the strided dim)
  static constexpr bool BMn = kBMn;
  static constexpr int Mode = kMode;
  static constexpr int BM = 128, BN_MAX = kBnMax;
  static constexpr int ESIZE = kFp8 ? 1 : 2;
  static constexpr int BK = 128 / ESIZE;  // contraction elements per stage (one 128-byte row)
  static constexpr int UK = 32 / ESIZE;   // contraction elements per MMA
  static constexpr int KSTEPS = BK / UK;  // 4
  static constexpr bool Pair = kPair;
  static constexpr bool DynRing = kDynRing;
  static constexpr int KC = kKc;
  static_assert(kKc == 1 || (kDynRing && !kAMn && !kBMn), "multi-block stages: run-time rings of K-major operands");
  static_assert(!kDynRing || (kMode == kModeRows && !kPair), "run-time rings serve the rows schedule");
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = (kPair ? BN_MAX / 2 : BN_MAX) * 128;
  static constexpr int STAGES = kStages;
  static constexpr int CHUNK = 64 * 128;  // MN-major: one 64-element x BK-row block (8 KB)
  // two accumulators of BN_MAX columns, allocated as a power of two >= 32
  static constexpr int TMEM_COLS = kMx                ? 512  // + the scale factors of every stage
                                   : 2 * BN_MAX <= 32  ? 32
                                   : 2 * BN_MAX <= 64  ? 64
                                   : 2 * BN_MAX <= 128 ? 128
                                   : 2 * BN_MAX <= 256 ? 256
                                                       : 512;
  static_assert(2 * BN_MAX <= 512, "two accumulators fit in TMEM");
  // TMEM accumulators: two (the next tile's MMAs run while the epilogue
  // drains the last), or one for 256-wide MXFP8 tiles, whose scale factors
  // need the columns a second accumulator would take (the MMAs of the next
  // tile then wait until the epilogue has read the accumulator)
  static constexpr int NACC = (kMx && kBnMax == 256) ? 1 : 2;
  static constexpr int EPI = kEpiWarps;
  static_assert(EPI == 4 || EPI == 8, "one or two epilogue warps per TMEM lane quarter");
  static constexpr int HN = EPI / 4;         // epilogue warps per lane quarter
  static constexpr int THREADS = 64 + 32 * EPI + (kMx ? 32 : 0);  // MXFP8: + the scale warp
  static constexpr int OUT_BUF = 32 * 128;  // 32 rows x 64 bf16 columns
  static constexpr int NBUF = kOutBufs;      // staging buffers per epilogue warp
  static constexpr size_t TAIL_BYTES = 16 * STAGES + 256;  // barriers, flags
  // MXFP8: per stage, the two 512-byte scale tiles rearranged for the
  // tensor-memory copy; and a ring of SF_SLOTS slots holding the scale rows
  // of A (128 x 16 B) and B (BN x 16 B) as loaded, one slot per four
  // contraction blocks
  static constexpr int SF_TILES_B = BN_MAX > 128 ? 2 : 1;  // B scale tiles per stage (128 columns each)
  static constexpr int SF_STAGE = kMx ? (1 + SF_TILES_B) * 512 : 0;
  static constexpr int SF_COLS = 4 + 4 * SF_TILES_B;        // tensor-memory columns of a stage's scales
  static constexpr int SF_SLOTS = 2;
  static constexpr int SF_SLOT = kMx ? 128 * 16 + BN_MAX * 16 : 0;
  static constexpr size_t SF_BYTES = (size_t)STAGES * SF_STAGE + (size_t)SF_SLOTS * SF_SLOT;
  static constexpr size_t SF_BARS = kMx ? 8 * (STAGES + 1 + 2 * SF_SLOTS) : 0;
  static constexpr size_t FIXED_BYTES = 1024 /*align slack*/ + (size_t)EPI * NBUF * OUT_BUF /*epilogue staging*/ +
                                        SF_BYTES + SF_BARS + TAIL_BYTES;
  // a run-time ring takes what the launch needs, up to the per-CTA limit
  static constexpr size_t SMEM_BYTES =
      kDynRing ? (size_t)227 * 1024 : FIXED_BYTES + (size_t)STAGES * (A_BYTES + B_BYTES);
  static_assert(SMEM_BYTES <= (size_t)227 * 1024, "one CTA's shared memory");
  static_assert(!kMx || NACC * BN_MAX + STAGES * SF_COLS <= TMEM_COLS, "MXFP8: accumulators and scales fit in TMEM");
};

struct GemmParams {
  const uint8_t *args;
  int E;
  int bn;           // output tile width: 64, 128 or 256
  int b_one_box;    // rows mode, MN-major B: the whole BN-column tile is one 4-d box (N % 64 == 0)
  int stages;       // run-time ring: stages, and bytes per stage ((a_rows + bn) x 128)
  int stage_bytes;
  int a_rows;       // rows mode: rows of each A box (128, or fewer when M itself is smaller)
  uint32_t idesc;   // tcgen05 instruction descriptor for M=128, N=bn
  int n_tiles;      // ceil(Nout / bn)
  int mt_k;         // kExperts: ceil(Kout / BM)
  int Kc;           // kRows: contraction length
  int Nout;         // output columns
  int Kout;         // kExperts: output rows per expert
  __nv_bfloat16 *out;
  const float *rscale;  // FP8: per output row (indexed by out_row0 + r)
  const float *cscale;  // FP8: per (expert, column): cscale[e * Nout + col]
  // bf16 rows mode, scattered output (routed layers): row i of the row-sorted
  // result goes to output row row_map[i] when 0 <= row_map[i] < map_limit and
  // nowhere otherwise; with row_weight, the fp32 accumulator row is first
  // multiplied by row_weight[row_map[i]] (one rounding to bf16 after it)
  const int32_t *row_map;
  int64_t map_limit;
  const float *row_weight;
  // bf16 rows mode, K-major B: gated output (the first GEMM of a SiLU-gated
  // MLP).  A tile's B stage holds bn / 2 rows of the gate half of w
  // (rows n0 ..) then the bn / 2 matching rows of the up half (rows
  // gate_rows + n0 ..); the epilogue writes silu(gate) * up for output
  // columns n0 .. n0 + bn / 2 - 1.
  int gated;
  int gate_rows;
  // bf16 rows mode, run-time ring with k-chunk boxes: with a_ids, row i of
  // the sorted rows is row a_ids[i] / a_top_k of x (a_src, a_ld bytes per
  // row; a_ids[i] >= a_numel: padding, a row of zeros)
  const int32_t *a_ids;
  int64_t a_numel;
  int a_top_k;
  const uint8_t *a_src;
  int64_t a_ld;
  int a_kbytes;  // 2 K: bytes of a row inside the contraction
};

struct TileInfo {
  int e, kb_count, a_row, b_row, n0, x0, lo, hi, out_row0, out_rows;
};

// FP8 with fewer than 128 token rows in all (the run-time-ring kernels with an
// A box of a_rows < 128 rows): every group has fewer than 128 rows, so every
// active group owns exactly one row tile (mtile_start[a] = a) and a tile's
// group is found without the prefix search.
template <class C>
__device__ __forceinline__ bool one_tile_per_group(const GemmParams &p) {
  return C::Mode == kModeRows && C::DynRing && C::Fp8 && p.a_rows < C::BM;
}

template <class C>
__device__ __forceinline__ int total_tiles(const GemmParams &p, const ArgsView &av, int na) {
  if (C::Mode == kModeRows) {
    if (one_tile_per_group<C>(p)) return na * p.n_tiles;
    return (C::Pair ? av.ptile_start[na] : av.mtile_start[na]) * p.n_tiles;
  }
  return p.E * p.mt_k * p.n_tiles;
}

// The j-th tile of the CTA (or pair) c of P: round j covers tiles j P ..
// j P + P - 1.  For wgrad (tiles of an expert cost in proportion to its rows,
// experts in decreasing size) odd rounds run backwards, so the CTA that took
// the costliest tile of one round takes the cheapest of the next (static
// round-robin left the DeepSeek wgrad ~10% longer than balanced; this order
// ~2%).  Row tiles all cost the same and keep the plain order.
template <class C>
__device__ __forceinline__ int tile_of(int j, int c, int P) {
  if (C::Mode == kModeExperts && (j & 1)) return j * P + (P - 1 - c);
  return j * P + c;
}

template <class C>
__device__ __forceinline__ TileInfo decode_tile(int t, const GemmParams &p, const ArgsView &av, uint32_t rank) {
  TileInfo ti;
  if (C::Mode == kModeRows) {
    // Group a owns tiles [start[a] * n_tiles, start[a+1] * n_tiles), start being
    // the 128-row tile prefix (or, for CTA pairs, the 256-row pair prefix).
    // Inside a group the row tile varies fastest, so CTAs running together
    // share one weight tile through L2 instead of each streaming its own.
    const int *start = C::Pair ? av.ptile_start : av.mtile_start;
    const int gm = t / p.n_tiles;
    int lo = gm, m_first = gm, mt_g = 1;
    if (!one_tile_per_group<C>(p)) {
      lo = 0;
      int hi = *av.n_active - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(start + mid) <= gm) lo = mid; else hi = mid - 1;
      }
      m_first = __ldg(start + lo);
      mt_g = __ldg(start + lo + 1) - m_first;
    }
    ti.e = __ldg(av.active + lo);
    const int local = t - m_first * p.n_tiles;
    const int mt = local % mt_g;
    ti.n0 = (local / mt_g) * (p.gated ? p.bn / 2 : p.bn);
    const int64_t rs = __ldg(av.offsets + ti.e), re = __ldg(av.offsets + ti.e + 1);
    // a CTA pair's tile is 256 rows: rank r takes rows 128 r .. 128 r + 127 (the
    // odd CTA's half may lie past the group: loaded, never stored) and columns
    // n0 + r bn / 2 .. of B
    const int row0 = (int)rs + (C::Pair ? mt * 2 * C::BM + (int)rank * C::BM : mt * C::BM);
    ti.kb_count = (p.Kc + C::BK * C::KC - 1) / (C::BK * C::KC);
    ti.a_row = row0;
    ti.out_row0 = row0;
    ti.out_rows = (int)max((int64_t)0, min((int64_t)C::BM, re - row0));
    // a run-time ring's A slot holds a_rows rows: the MMA rows past them read
    // stale shared memory and are not stored (they are padding rows there)
    if (C::DynRing && ti.out_rows > p.a_rows) ti.out_rows = p.a_rows;
    ti.b_row = C::Pair ? ti.n0 + (int)rank * (p.bn / 2) : ti.n0;
    ti.x0 = 0; ti.lo = 0; ti.hi = 0;
  } else {
    ti.n0 = (t % p.n_tiles) * p.bn;
    const int per_e = p.mt_k * p.n_tiles;
    const int i = t / per_e;
    const int mk = (t % per_e) / p.n_tiles;
    ti.e = __ldg(av.wgrad_order + i);
    if (C::Fp8) {
      // padded column-major operands: the group's rows start 128-aligned at
      // poffsets[e] and are followed by zeros up to a multiple of 128, so
      // every block is whole and nothing is masked
      const int64_t ps = __ldg(av.poffsets + ti.e), pe = __ldg(av.poffsets + ti.e + 1);
      ti.x0 = (int)ps;
      ti.lo = 0;
      ti.hi = (int)(pe - ps);
      ti.kb_count = ti.hi / C::BK;
    } else {
      // row-major operands: the group's rows are the TMA outer coordinate
      const int64_t rs = __ldg(av.offsets + ti.e), re = __ldg(av.offsets + ti.e + 1);
      ti.x0 = (int)rs;
      ti.lo = 0;
      ti.hi = (int)(re - rs);
      ti.kb_count = re > rs ? (ti.hi + C::BK - 1) / C::BK : 0;
    }
    // a CTA pair's tile is 256 rows of K: rank r takes rows 128 r .. 128 r + 127
    // and columns n0 + r bn / 2 .. of B
    ti.a_row = C::Pair ? mk * 2 * C::BM + (int)rank * C::BM : mk * C::BM;
    ti.b_row = C::Pair ? ti.n0 + (int)rank * (p.bn / 2) : ti.n0;
    ti.out_row0 = ti.e * p.Kout + ti.a_row;
    ti.out_rows = max(0, min(C::BM, p.Kout - ti.a_row));
  }
  return ti;
}

// Zero contraction positions [zlo, zhi) of one stage (positions relative to
// the block start, all inside one MMA k-step).  Executed by all 32 lanes of
// the MMA warp.  Only bf16 wgrad has partial blocks (the tail of a group's
// rows; its operands are the row-major activations, MN-major in shared
// memory): the rows of those positions are cleared in A and B, so a
// non-finite value in the next group cannot leak in.  FP8 wgrad reads the
// padded column-major layout, whose blocks are always whole.
template <class C>
__device__ __forceinline__ void mask_positions(uint8_t *sa, uint8_t *sb, int bn, int zlo, int zhi, int lane) {
  static_assert(!C::Fp8 && C::AMn && C::BMn, "only MN-major bf16 operands have partial blocks");
  const int nA = C::BM / 64, nch = nA + bn / 64;
  const int nrows = zhi - zlo;
  for (int idx = lane; idx < nch * nrows * 8; idx += 32) {  // 16-byte granules
    const int g = idx & 7, rr = idx >> 3;
    const int ch = rr / nrows, pos = zlo + rr % nrows;
    uint8_t *base = ch < nA ? sa + ch * C::CHUNK : sb + (ch - nA) * C::CHUNK;
    *reinterpret_cast<uint4 *>(base + pos * 128 + g * 16) = make_uint4(0, 0, 0, 0);
  }
}

// 1 / s for a power of two s in [2^-126, 2^126] (exact: the exponent is negated)
__device__ __forceinline__ float pow2_recip(float s) { return __uint_as_float(0x7F000000u - __float_as_uint(s)); }

// (a0, a1) * (b0, b1) elementwise, round to nearest (one packed fp32 multiply)
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; }
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  return f32x2(__float_as_uint(lo), __float_as_uint(hi));
}
// two packed fp32 values -> bf16x2 (round to nearest even), low element in the low half
__device__ __forceinline__ uint32_t pack_bf16x2_u64(uint64_t v) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float((uint32_t)v), __uint_as_float((uint32_t)(v >> 32)));
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// One CTA's share of a launch: CTA cta of ncta (CTA pairs: the cluster's
// place among the clusters) takes tiles cta, cta + ncta, ...
template <class C>
__device__ __forceinline__ void gemm_cta(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmOut,
                                         const CUtensorMap &tmSFA, const CUtensorMap &tmSFB, const GemmParams &p,
                                         int cta, int ncta) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // ring stages, then the epilogue staging [EPI warps][NBUF buffers][32 x 128 B], then barriers
  const int nst = C::DynRing ? p.stages : C::STAGES;
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::STAGES * C::A_BYTES;
  uint8_t *sOut = C::DynRing ? smem + (size_t)nst * p.stage_bytes : sB + C::STAGES * C::B_BYTES;
  auto stage_a = [&](int st) -> uint8_t * { return C::DynRing ? smem + (size_t)st * p.stage_bytes : sA + st * C::A_BYTES; };
  auto stage_b = [&](int st) -> uint8_t * {
    return C::DynRing ? smem + (size_t)st * p.stage_bytes + C::KC * p.a_rows * 128 : sB + st * C::B_BYTES;
  };
  // MXFP8 scales: per stage the A and B tiles for the copy, then the slots of loaded scale rows
  uint8_t *sSF = sOut + C::EPI * C::NBUF * C::OUT_BUF;
  auto sf_tile = [&](int st, int op) -> uint8_t * { return sSF + st * C::SF_STAGE + op * 512; };
  auto sfa_slot = [&](int q) -> uint8_t * { return sSF + C::STAGES * C::SF_STAGE + q * C::SF_SLOT; };
  auto sfb_slot = [&](int q) -> uint8_t * { return sSF + C::STAGES * C::SF_STAGE + q * C::SF_SLOT + 128 * 16; };
  // MXFP8 barriers: a stage's scales are in tensor memory; the scale warp's
  // copies have drained; a slot of scale rows has landed / is free again
  uint64_t *sfready = reinterpret_cast<uint64_t *>(sSF + C::SF_BYTES);
  uint64_t *sfdrain = sfready + C::STAGES;
  uint64_t *sf_full = sfdrain + 1;
  uint64_t *sf_empty = sf_full + C::SF_SLOTS;
  uint64_t *full = reinterpret_cast<uint64_t *>(sSF + C::SF_BYTES + C::SF_BARS);
  uint64_t *empty = full + C::STAGES;
  uint64_t *tfull = empty + C::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pairs walk the tiles per cluster: both CTAs of a pair see the same
  // sequence and leave (or stay) together
  const uint32_t rank = C::Pair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int t_first = C::Pair ? (int)cluster_id_x() : cta;
  const int t_step = C::Pair ? (int)ncluster_x() : ncta;

  // Set-up (barriers, tensor memory, descriptor prefetch) reads nothing an
  // earlier kernel writes, so it runs before the wait for the previous grid of
  // the stream and overlaps that grid's tail.  A CTA with no tile (or a
  // non-zero status) runs no role loop and goes straight to the teardown.
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], p.a_ids ? 1 + 32 : 1);  // gathered rows: + each producer lane's copies
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      // one arrival per thread of the four epilogue warps, or per warp with
      // eight of them (pair: per warp of each CTA, on the leader's barrier)
      mbar_init(&tempty[a], C::Pair ? 2 * C::EPI : (C::EPI == 4 ? 128 : C::EPI));
    }
    mbar_init(drain, 1);
    if constexpr (C::Mx) {
      for (int s = 0; s < nst; ++s) mbar_init(&sfready[s], 1);
      mbar_init(sfdrain, 1);
      for (int q = 0; q < C::SF_SLOTS; ++q) {
        mbar_init(&sf_full[q], 1);
        mbar_init(&sf_empty[q], 1);
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
    if constexpr (C::Mx) {
      tma_prefetch_desc(&tmSFA);
      tma_prefetch_desc(&tmSFB);
    }
  }
  if (warp == 1) {
    if constexpr (C::Pair) {
      tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (C::Pair)
    cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  const ArgsView av(p.args, p.E);
  const int status0 = *av.status, n_active0 = *av.n_active;  // two independent loads
  const int total = status0 != 0 ? 0 : total_tiles<C>(p, av, n_active0);
  volatile int *vabort = abort_flag;
  const int bn = p.bn;
  // an abort in one CTA of a pair is raised in the other as well
  auto raise_abort = [&]() {
    *vabort = 1;
    if constexpr (C::Pair) st_cluster_u32(cluster_addr(abort_flag, rank ^ 1u), 1u);
  };

  // Producer bookkeeping kept for the drain after an abort.
  uint32_t issued = 0, sf_issued = 0;

  if (warp == 0) {
    if (C::Mode == kModeRows && C::KC > 1 && !C::Pair && !C::Mx && p.a_ids) {
      // Gathered A rows (few rows per group, a_rows <= 32): the whole warp
      // produces.  Lane r copies sorted row r of the tile (x row a_ids[a_row +
      // r] / a_top_k) in 16-byte asynchronous copies into the stage's
      // [KC chunks][a_rows][128 B] layout with its 128-byte swizzle (unit u of
      // row r at u ^ (r & 7)); padding rows and chunks past K are zeros (nothing
      // read), as in the gathered copy.  Lane 0 also arms the full barrier with
      // the weight bytes and loads the weight box; every lane's copies then
      // count one arrival when they land.
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t tx = C::KC * bn * 128;
      const uint32_t a_off = (uint32_t)lane * 128u;
      for (int j = 0; j * t_step < total && !*vabort; ++j) {
        const int t = tile_of<C>(j, t_first, t_step);
        if (t >= total) continue;
        const TileInfo ti = decode_tile<C>(t, p, av, rank);
        int xrow = -1;
        if (lane < p.a_rows) {
          const int32_t id = __ldg(p.a_ids + ti.a_row + lane);
          if (id >= 0 && id < p.a_numel) xrow = id / p.a_top_k;
        }
        bool ok = true;
        for (int kb = 0; kb < ti.kb_count; ++kb) {
          if (!mbar_wait_warp(&empty[stage], phase ^ 1, vabort)) {
            ok = false;
            break;
          }
          uint8_t *b = stage_b(stage);
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[stage], tx);
            ++issued;
            if (p.gated)
              tma_load_5d(b, &tmB, &full[stage], 0, ti.b_row, 0, kb * C::KC, ti.e);
            else
              tma_load_4d(b, &tmB, &full[stage], 0, ti.b_row, kb * C::KC, ti.e);
          }
          if (lane < p.a_rows) {
            const uint32_t a_s = smem_u32(stage_a(stage)) + a_off;
#pragma unroll
            for (int c = 0; c < C::KC; ++c) {
              const int kx = (kb * C::KC + c) * 128;
              const bool live = xrow >= 0 && kx < p.a_kbytes;
              const uint8_t *src = p.a_src + (live ? (int64_t)xrow * p.a_ld + kx : 0);
              const uint32_t dst = a_s + (uint32_t)(c * p.a_rows * 128), nb = live ? 16u : 0u;
#pragma unroll
              for (int u = 0; u < 8; ++u) cp_async16(dst + ((u ^ (lane & 7)) << 4), src + (live ? u * 16 : 0), nb);
            }
          }
          cp_async_mbar_arrive(&full[stage]);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) {
          if (lane == 0) {
            set_status(av.status, MGEMM_STATUS_TIMEOUT);
            raise_abort();
          }
          break;
        }
      }
    } else if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      // with fewer than 128 token rows the A box is cut to them (rounded up to 8);
      // the MMA's remaining A rows hold stale data and only feed output rows
      // that are never stored
      // pair: the leader's full barrier counts the bytes of both CTAs
      const uint32_t tx = C::Pair ? 2u * (uint32_t)(C::A_BYTES + (bn / 2) * 128)
                                  : C::KC * ((C::Mode == kModeRows ? p.a_rows * 128 : C::A_BYTES) + bn * 128);
      int qslot = 0;
      uint32_t qphase = 0;
      for (int j = 0; j * t_step < total && !*vabort; ++j) {
        const int t = tile_of<C>(j, t_first, t_step);
        if (t >= total) continue;
        const TileInfo ti = decode_tile<C>(t, p, av, rank);
        for (int kb = 0; kb < ti.kb_count; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, vabort)) {
            set_status(av.status, MGEMM_STATUS_TIMEOUT);
            raise_abort();
            break;
          }
          uint8_t *a = stage_a(stage);
          uint8_t *b = stage_b(stage);
          if constexpr (C::Mx) {
            if (kb % C::KPS == 0) {
              if (!mbar_wait(&sf_empty[qslot], qphase ^ 1, vabort)) {
                set_status(av.status, MGEMM_STATUS_TIMEOUT);
                raise_abort();
                break;
              }
              if constexpr (C::Mode == kModeRows) {
                // the scale rows of this and the next three contraction blocks
                // (16 bytes per row; x is a multiple of 16 bytes): A rows of the
                // tile, and rows e N + n0 .. of B's [E N, ld_sf] scales
                mbar_arrive_expect_tx(&sf_full[qslot], (uint32_t)(128 * 16 + bn * 16));
                tma_load_2d(sfa_slot(qslot), &tmSFA, &sf_full[qslot], (kb >> 2) * 16, ti.a_row);
                tma_load_2d(sfb_slot(qslot), &tmSFB, &sf_full[qslot], (kb >> 2) * 16, ti.e * p.Nout + ti.n0);
              } else {
                // one contraction block of the padded layout (its block index is
                // x0 / 128 + kb): 4 bytes per row, rows viewed in fours (16 bytes)
                mbar_arrive_expect_tx(&sf_full[qslot], (uint32_t)(128 * 4 + bn * 4));
                tma_load_3d(sfa_slot(qslot), &tmSFA, &sf_full[qslot], 0, ti.a_row / 4, ti.x0 / C::BK + kb);
                tma_load_3d(sfb_slot(qslot), &tmSFB, &sf_full[qslot], 0, ti.n0 / 4, ti.x0 / C::BK + kb);
              }
              ++sf_issued;
              if (++qslot == C::SF_SLOTS) {
                qslot = 0;
                qphase ^= 1;
              }
            }
          }
          if constexpr (C::Pair) {
            static_assert(C::Pair ? (C::Fp8 && !C::AMn && !C::BMn) : true, "CTA pairs serve K-major FP8 operands");
            // each CTA copies its own halves; the peer's copies complete on the leader's barrier
            // (wgrad: column-major operands, contraction inner; rows: x [M, K], w [E, N, K])
            const int xr = C::Mode == kModeExperts ? ti.x0 + kb * C::BK : kb * C::BK;
            if (leader) {
              mbar_arrive_expect_tx(&full[stage], tx);
              ++issued;
              tma_load_2d(a, &tmA, &full[stage], xr, ti.a_row);
              if (C::Mode == kModeExperts)
                tma_load_2d(b, &tmB, &full[stage], xr, ti.b_row);
              else
                tma_load_3d(b, &tmB, &full[stage], xr, ti.b_row, ti.e);
            } else {
              const uint32_t lbar = cluster_addr(&full[stage], 0);
              tma_load_2d_pair(a, &tmA, lbar, xr, ti.a_row);
              if (C::Mode == kModeExperts)
                tma_load_2d_pair(b, &tmB, lbar, xr, ti.b_row);
              else
                tma_load_3d_pair(b, &tmB, lbar, xr, ti.b_row, ti.e);
            }
            if (++stage == nst) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          mbar_arrive_expect_tx(&full[stage], tx);
          ++issued;
          if (C::Mode == kModeRows && C::KC > 1) {
            // [KC chunks][a_rows][128 B] and [KC chunks][bn][128 B] in one copy each; the gated
            // form's B view adds a gate / up dimension, so a chunk lands as its bn / 2 gate rows
            // followed by the matching up rows
            tma_load_3d(a, &tmA, &full[stage], 0, ti.a_row, kb * C::KC);
            if (p.gated)
              tma_load_5d(b, &tmB, &full[stage], 0, ti.b_row, 0, kb * C::KC, ti.e);
            else
              tma_load_4d(b, &tmB, &full[stage], 0, ti.b_row, kb * C::KC, ti.e);
          } else if (C::Mode == kModeRows) {
            tma_load_2d(a, &tmA, &full[stage], kb * C::BK, ti.a_row);
            if (C::BMn) {
              if (p.b_one_box) {  // [chunk][row][64 columns] in one copy: the layout the MMA reads
                tma_load_4d(b, &tmB, &full[stage], 0, kb * C::BK, ti.n0 / 64, ti.e);
              } else {
                for (int j = 0; j < bn / 64; ++j)
                  tma_load_3d(b + j * C::CHUNK, &tmB, &full[stage], ti.n0 + 64 * j, kb * C::BK, ti.e);
              }
            } else {
              if (p.gated) {  // gate rows, then the matching up rows (boxes of bn / 2 rows)
                tma_load_3d(b, &tmB, &full[stage], kb * C::BK, ti.n0, ti.e);
                tma_load_3d(b + (bn / 2) * 128, &tmB, &full[stage], kb * C::BK, p.gate_rows + ti.n0, ti.e);
              } else {
                tma_load_3d(b, &tmB, &full[stage], kb * C::BK, ti.n0, ti.e);
              }
            }
          } else {
            const int xr = ti.x0 + kb * C::BK;
            if (C::AMn) {
#pragma unroll
              for (int j = 0; j < C::BM / 64; ++j)
                tma_load_2d(a + j * C::CHUNK, &tmA, &full[stage], ti.a_row + 64 * j, xr);
              for (int j = 0; j < bn / 64; ++j)
                tma_load_2d(b + j * C::CHUNK, &tmB, &full[stage], ti.n0 + 64 * j, xr);
            } else {
              tma_load_2d(a, &tmA, &full[stage], xr, ti.a_row);
              tma_load_2d(b, &tmB, &full[stage], xr, ti.n0);
            }
          }
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    // pair: only the leader issues MMAs (for both CTAs); the peer's warp 1 only owns its TMEM
    const bool issues = !C::Pair || leader;
    for (int j = 0; issues && j * t_step < total && ok; ++j) {
      const int t = tile_of<C>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<C>(t, p, av, rank);
      if (ti.kb_count == 0) continue;
      if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1, vabort)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::BN_MAX;
      for (int kb = 0; kb < ti.kb_count; ++kb) {
        if (!mbar_wait_warp(&full[stage], phase, vabort)) { ok = false; break; }
        if (C::Mode == kModeRows && C::KC > 1 && p.a_ids) fence_proxy_async_smem();  // rows written by cp.async
        // MXFP8: and the stage's scales are in tensor memory
        if (C::Mx && !mbar_wait_warp(&sfready[stage], phase, vabort)) { ok = false; break; }
        tc_fence_after();
        uint8_t *a = stage_a(stage);
        uint8_t *b = stage_b(stage);
        // bf16 wgrad: at the partial last block of a group only the MMA
        // k-steps [k_first, k_last] hold group rows; the others are skipped,
        // and the out-of-group positions inside the partial step are cleared
        constexpr bool kPartial = C::Mode == kModeExperts && !C::Fp8;
        const bool edge = kPartial && (ti.lo - kb * C::BK > 0 || ti.hi - kb * C::BK < C::BK);
        int k_first = 0, k_last = C::KSTEPS - 1;
        if (edge) {
          const int lo = max(ti.lo - kb * C::BK, 0), hi = min(ti.hi - kb * C::BK, C::BK);
          k_first = lo / C::UK;
          k_last = (hi - 1) / C::UK;
          const bool head = lo > k_first * C::UK, tail = hi < (k_last + 1) * C::UK;
          if constexpr (kPartial) {
            if (head) mask_positions<C>(a, b, bn, k_first * C::UK, lo, lane);
            if (tail) mask_positions<C>(a, b, bn, hi, (k_last + 1) * C::UK, lane);
          }
          if (head || tail) {
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if constexpr (C::Mx) {
          // MXFP8: sub-block k of the stage reads byte k of the scale words
          // (the scale-factor ids of the instruction descriptor)
          if (lane == 0) {
            const uint32_t sfa_t = tmem_base + C::NACC * C::BN_MAX + stage * C::SF_COLS, sfb_t = sfa_t + 4;
            const uint32_t abase = smem_u32(a), bbase = smem_u32(b);
#pragma unroll
            for (int k = 0; k < C::KSTEPS; ++k) {
              const uint64_t ad = smem_desc_sw128(abase + k * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(bbase + k * 32, 16, 1024);
              const uint32_t idk = p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29);
              mma_mx(d_tmem, ad, bd, idk, sfa_t, sfb_t, (kb | k) != 0);
            }
            mma_commit(&empty[stage]);
          }
        } else if (lane == 0) {
          const uint32_t abase = smem_u32(a), bbase = smem_u32(b);
          if (!edge) {
#pragma unroll
            for (int j = 0; j < C::KC; ++j) {  // the stage's contraction blocks (one unless KC > 1)
              const uint32_t aj = abase + j * p.a_rows * 128, bj = bbase + j * bn * 128;
#pragma unroll
              for (int k = 0; k < C::KSTEPS; ++k) {
                const uint64_t ad = C::AMn ? smem_desc_sw128(aj + k * C::UK * 128, C::CHUNK, 1024)
                                           : smem_desc_sw128(aj + k * 32, 16, 1024);
                const uint64_t bd = C::BMn ? smem_desc_sw128(bj + k * C::UK * 128, C::CHUNK, 1024)
                                           : smem_desc_sw128(bj + k * 32, 16, 1024);
                // the tile's first MMA overwrites the accumulator
                const bool acc_on = (kb | j | k) != 0;
                if constexpr (C::Pair)
                  mma_f8_pair(d_tmem, ad, bd, p.idesc, acc_on);
                else if (C::Fp8)
                  mma_f8(d_tmem, ad, bd, p.idesc, acc_on);
                else
                  mma_f16(d_tmem, ad, bd, p.idesc, acc_on);
              }
            }
          } else {
            for (int k = k_first; k <= k_last; ++k) {
              const uint64_t ad = C::AMn ? smem_desc_sw128(abase + k * C::UK * 128, C::CHUNK, 1024)
                                         : smem_desc_sw128(abase + k * 32, 16, 1024);
              const uint64_t bd = C::BMn ? smem_desc_sw128(bbase + k * C::UK * 128, C::CHUNK, 1024)
                                         : smem_desc_sw128(bbase + k * 32, 16, 1024);
              const bool acc_on = kb > 0 || k > k_first;
              if (C::Fp8)
                mma_f8(d_tmem, ad, bd, p.idesc, acc_on);
              else
                mma_f16(d_tmem, ad, bd, p.idesc, acc_on);
            }
          }
          if constexpr (C::Pair)
            mma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
          else
            mma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == nst) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        if constexpr (C::Pair)
          mma_commit_pair(&tfull[acc], 0x3);  // both CTAs' accumulators are ready
        else
          mma_commit(&tfull[acc]);
      }
      __syncwarp();
      if (++acc == C::NACC) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (!ok) {
      if (lane == 0) set_status(av.status, MGEMM_STATUS_TIMEOUT);
      raise_abort();
    }
    // all MMAs this thread issued have completed before TMEM is released
    if (lane == 0 && (!C::Pair || leader)) {
      if constexpr (C::Pair)
        mma_commit_pair(drain, 0x1);
      else
        mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (C::Mx && warp == 2 + C::EPI) {
    // MXFP8 scale warp.  A slot holds the scale rows of KPS contraction
    // blocks of 128 (rows schedule: 16 bytes per row, four blocks; experts
    // schedule: 4 bytes per row, one block); word w = kb % KPS of each row
    // holds block kb's four 32-element scales.  Tensor memory takes them as a
    // 512-byte tile per operand, row l holding rows l, l + 32, l + 64, l + 96
    // of the tile (byte 4 m + s: sub-block s of row l + 32 m), copied into
    // each lane quarter at columns NACC BN_MAX + SF_COLS stage (A) and + 4 (B).  Lane
    // l builds row l of both tiles.  A stage's tiles and columns are reused
    // once its previous MMAs are done (its empty barrier, which the producer
    // waits for too); the copies' commit arms the stage's sfready barrier,
    // which the MMA warp waits for; a slot is released after its fourth block
    // (or the tile's last).
    int stage = 0, qslot = 0;
    uint32_t phase = 0, qphase = 0;
    bool ok = true;
    for (int j = 0; j * t_step < total && ok; ++j) {
      const int t = tile_of<C>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<C>(t, p, av, rank);
      if (ti.kb_count == 0) continue;
      for (int kb = 0; kb < ti.kb_count; ++kb) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1, vabort)) { ok = false; break; }
        if (kb % C::KPS == 0 && !mbar_wait_warp(&sf_full[qslot], qphase, vabort)) { ok = false; break; }
        const int w = kb % C::KPS;
        const uint32_t *la = reinterpret_cast<const uint32_t *>(sfa_slot(qslot));
        const uint32_t *lb = reinterpret_cast<const uint32_t *>(sfb_slot(qslot));
        constexpr int S = C::KPS;  // words per row of a slot
        const uint4 va = make_uint4(la[lane * S + w], la[(lane + 32) * S + w], la[(lane + 64) * S + w],
                                    la[(lane + 96) * S + w]);
        const uint4 vb = make_uint4(lb[lane * S + w], lb[(lane + 32) * S + w], lb[(lane + 64) * S + w],
                                    lb[(lane + 96) * S + w]);
        reinterpret_cast<uint4 *>(sf_tile(stage, 0))[lane] = va;
        reinterpret_cast<uint4 *>(sf_tile(stage, 1))[lane] = vb;
        if constexpr (C::SF_TILES_B > 1) {
          // B columns 128 .. BN_MAX - 1 (the slot has BN_MAX rows; the rest are zero)
          const uint4 vc = make_uint4(lb[(lane + 128) * S + w], lb[(lane + 160) * S + w],
                                      C::BN_MAX > 192 ? lb[(lane + 192) * S + w] : 0u,
                                      C::BN_MAX > 224 ? lb[(lane + 224) * S + w] : 0u);
          reinterpret_cast<uint4 *>(sf_tile(stage, 2))[lane] = vc;
        }
        fence_proxy_async_smem();  // the tiles are read by tcgen05.cp
        __syncwarp();
        if (lane == 0) {
          // column n of B reads the word at column sfb_t + n / 32: the second
          // B tile (columns 128 ..) sits 4 columns after the first
          const uint32_t sfa_t = tmem_base + C::NACC * C::BN_MAX + stage * C::SF_COLS, sfb_t = sfa_t + 4;
          tmem_cp_32x128b_warpx4(sfa_t, smem_desc_rows16(smem_u32(sf_tile(stage, 0))));
          tmem_cp_32x128b_warpx4(sfb_t, smem_desc_rows16(smem_u32(sf_tile(stage, 1))));
          if constexpr (C::SF_TILES_B > 1)
            tmem_cp_32x128b_warpx4(sfb_t + 4, smem_desc_rows16(smem_u32(sf_tile(stage, 2))));
          mma_commit(&sfready[stage]);
          if (w == C::KPS - 1 || kb == ti.kb_count - 1) mbar_arrive(&sf_empty[qslot]);  // the slot's rows are read
        }
        __syncwarp();
        if (w == C::KPS - 1 || kb == ti.kb_count - 1) {
          if (++qslot == C::SF_SLOTS) {
            qslot = 0;
            qphase ^= 1;
          }
        }
        if (++stage == nst) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (!ok) {
      if (lane == 0) set_status(av.status, MGEMM_STATUS_TIMEOUT);
      raise_abort();
    }
    // every copy this warp issued has landed before tensor memory is freed
    if (lane == 0) {
      mma_commit(sfdrain);
      mbar_wait_drain(sfdrain, 0);
    }
    __syncwarp();
  } else {
    // epilogue warps 2 .. EPI + 1: warp w reads TMEM lane quarter q = w % 4 (tile
    // rows 32q .. 32q + 31) and, with two warps per quarter, every other
    // 64-column chunk of the tile (h = its place among the quarter's warps)
    const int ew = warp - 2;
    const int q = warp & 3;
    const int h = ew / 4;
    const int r = q * 32 + lane;
    constexpr int kCpw = (C::BN_MAX / 64 + C::HN - 1) / C::HN;  // chunks per warp, at most
    uint8_t *my_buf = sOut + (size_t)ew * C::NBUF * C::OUT_BUF;
    uint32_t nstored = 0;  // TMA-stored chunks so far; buffers rotate with it
    int acc = 0;
    uint32_t acc_phase = 0;
    // FP8: the row-scale reciprocal of this thread's row and the column-scale
    // reciprocals of the warp's chunks of one tile (lane l: columns col0 + l
    // and col0 + 32 + l of each chunk), loaded one tile ahead so their latency
    // never sits between an accumulator and its stores (scales are powers of
    // two: the reciprocals are exact)
    float rinv_next = 1.f, csr_next[2 * kCpw] = {};
    auto load_scales = [&](int tn) {
      if (!C::Scaled || tn >= total) return;
      const TileInfo tj = decode_tile<C>(tn, p, av, rank);
      const bool live = tj.kb_count > 0;
      rinv_next = live && r < tj.out_rows ? pow2_recip(__ldg(p.rscale + tj.out_row0 + r)) : 1.f;
#pragma unroll
      for (int i = 0; i < 2 * kCpw; ++i) {
        const int c = h + C::HN * (i >> 1);
        const int col = tj.n0 + c * 64 + 32 * (i & 1) + lane;
        csr_next[i] = live && c * 64 < bn && col < p.Nout ? pow2_recip(__ldg(p.cscale + (int64_t)tj.e * p.Nout + col))
                                                           : 0.f;
      }
    };
    // hand the accumulator back to the MMA warp (one arrival per warp)
    auto release = [&](int a) {
      tc_fence_before();
      if constexpr (!C::Pair && C::EPI == 4) {
        mbar_arrive(&tempty[a]);  // every thread arrives
      } else {
        __syncwarp();
        if (lane == 0) {
          if (!C::Pair || leader)
            mbar_arrive(&tempty[a]);
          else
            mbar_arrive_cluster(cluster_addr(&tempty[a], 0));
        }
      }
    };
    load_scales(t_first);
    for (int j = 0; j * t_step < total; ++j) {
      const int t = tile_of<C>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<C>(t, p, av, rank);
      const bool has_acc = ti.kb_count > 0;
      bool row_ok = r < ti.out_rows;
      bool warp_full = q * 32 + 32 <= ti.out_rows;
      int64_t out_row = (int64_t)ti.out_row0 + r;
      float wgt = 1.f;
      if constexpr (C::Mode == kModeRows && !C::Fp8) {
        if (p.row_map) {  // scattered rows: plain per-row stores
          const int32_t d = row_ok ? __ldg(p.row_map + ti.out_row0 + r) : -1;
          row_ok = d >= 0 && d < p.map_limit;
          out_row = row_ok ? d : 0;
          warp_full = false;
          if (row_ok && p.row_weight) wgt = __ldg(p.row_weight + d);
        }
      }
      __nv_bfloat16 *orow = p.out + out_row * p.Nout;
      float rinv = 1.f, csr[2 * kCpw];
      if constexpr (C::Scaled) {
        rinv = rinv_next;
#pragma unroll
        for (int i = 0; i < 2 * kCpw; ++i) csr[i] = csr_next[i];
        load_scales(tile_of<C>(j + 1, t_first, t_step));
      }
      if (has_acc) {
        if (!mbar_wait_warp(&tfull[acc], acc_phase, vabort)) {
          set_status(av.status, MGEMM_STATUS_TIMEOUT);
          raise_abort();
          break;
        }
        tc_fence_after();
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::BN_MAX;
      // with one warp per quarter, TMEM -> registers runs one chunk ahead (chunk
      // c + 1 loads while chunk c is converted and stored; the loop is unrolled
      // so both register sets keep fixed names); with two, the other warp of the
      // quarter hides the load latency and registers stay within the budget
      constexpr int kNb = C::HN == 1 ? 2 : 1;
      uint32_t va[kNb][32], vb[kNb][32];
      if constexpr (C::Mode == kModeRows && !C::Fp8 && !C::BMn && C::HN == 1) {
        if (p.gated) {
          // accumulator columns [0, bn / 2) hold the gate, [bn / 2, bn) the up
          // projection of the same output columns: h = silu(g) * u in fp32,
          // silu(g) = g / (1 + exp(-g)), one rounding to bf16
          const int half = bn / 2, nout = half / 64;
          uint32_t(&g)[32] = va[0];  // gate columns c*64 .. +31, then +32 .. +63 in vb[0]
          uint32_t(&u)[32] = va[1];  // up columns, likewise in vb[1]
          for (int c = 0; c < nout; ++c) {
            const int col0 = ti.n0 + c * 64;
            uint32_t pk[32];
            if (has_acc) {
              tmem_ld_32x32b_x32(taddr + c * 64, g);
              tmem_ld_32x32b_x32(taddr + c * 64 + 32, vb[0]);
              tmem_ld_32x32b_x32(taddr + half + c * 64, u);
              tmem_ld_32x32b_x32(taddr + half + c * 64 + 32, vb[1]);
              tmem_ld_wait();
              if (c == nout - 1) release(acc);  // the accumulator is read
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
                pk[j] = pack_bf16x2(g0 / (1.f + expf(-g0)) * u0, g1 / (1.f + expf(-g1)) * u1);
                const float g2 = __uint_as_float(vb[0][2 * j]), g3 = __uint_as_float(vb[0][2 * j + 1]);
                const float u2 = __uint_as_float(vb[1][2 * j]), u3 = __uint_as_float(vb[1][2 * j + 1]);
                pk[16 + j] = pack_bf16x2(g2 / (1.f + expf(-g2)) * u2, g3 / (1.f + expf(-g3)) * u3);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) pk[j] = 0u;
            }
            if (col0 >= p.Nout) continue;
            if (warp_full) {
              uint8_t *buf = my_buf + (nstored % C::NBUF) * C::OUT_BUF;
              if (lane == 0) bulk_wait_read<C::NBUF - 1>();
              __syncwarp();
              uint8_t *rowp = buf + lane * 128;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4 *>(rowp + ((j ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmOut, buf, col0, ti.out_row0 + q * 32);
                bulk_commit();
              }
              ++nstored;
            } else if (row_ok) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + col0);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (col0 + 8 * j < p.Nout) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
          }
          if (has_acc) {
            if (nout == 0) release(acc);
            if (++acc == C::NACC) {
              acc = 0;
              acc_phase ^= 1;
            }
          }
          continue;
        }
      }
      const int nchunks = bn / 64;
      bool released = false;
      if (kNb == 2 && has_acc && h < nchunks) {
        tmem_ld_32x32b_x32(taddr + h * 64, va[0]);
        tmem_ld_32x32b_x32(taddr + h * 64 + 32, vb[0]);
      }
#pragma unroll
      for (int ci = 0; ci < kCpw; ++ci) {
        const int c = h + C::HN * ci;
        if (c >= nchunks) break;
        const int cur = kNb == 2 ? (ci & 1) : 0;
        const int col0 = ti.n0 + c * 64;
        // the staging buffer of this chunk; the store group that last read it is
        // NBUF groups back (FP8 parks the chunk's column scales in it first, so
        // it waits for the buffer before the math; bf16 only before its stores)
        uint8_t *buf = my_buf + (nstored % C::NBUF) * C::OUT_BUF;
        if constexpr (C::Scaled) {
          if (lane == 0) bulk_wait_read<C::NBUF - 1>();
          __syncwarp();
        }
        uint32_t pk[32];
        if (has_acc) {
          if (kNb == 1) {
            tmem_ld_32x32b_x32(taddr + c * 64, va[0]);
            tmem_ld_32x32b_x32(taddr + c * 64 + 32, vb[0]);
          }
          tmem_ld_wait();
          if (c + C::HN >= nchunks) {  // the warp's last chunk: the accumulator is read
            release(acc);
            released = true;
          } else if (kNb == 2) {
            tmem_ld_32x32b_x32(taddr + (c + C::HN) * 64, va[cur ^ (kNb - 1)]);
            tmem_ld_32x32b_x32(taddr + (c + C::HN) * 64 + 32, vb[cur ^ (kNb - 1)]);
          }
          if (C::Scaled) {
            // the chunk's column-scale reciprocals, staged in the (free) staging
            // buffer and read as broadcasts before the codes overwrite them
            float *cs = reinterpret_cast<float *>(buf);
            cs[lane] = csr[2 * ci];
            cs[lane + 32] = csr[2 * ci + 1];
            __syncwarp();
            // two packed multiplies per pair of elements: by the row's, then the columns' reciprocals
            const uint64_t r2 = f32x2(rinv, rinv);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 c0 = *reinterpret_cast<const float4 *>(cs + 4 * j);
              const float4 c1 = *reinterpret_cast<const float4 *>(cs + 32 + 4 * j);
              pk[2 * j] = pack_bf16x2_u64(mul_f32x2(mul_f32x2(f32x2(va[cur][4 * j], va[cur][4 * j + 1]), r2), f32x2(c0.x, c0.y)));
              pk[2 * j + 1] =
                  pack_bf16x2_u64(mul_f32x2(mul_f32x2(f32x2(va[cur][4 * j + 2], va[cur][4 * j + 3]), r2), f32x2(c0.z, c0.w)));
              pk[16 + 2 * j] =
                  pack_bf16x2_u64(mul_f32x2(mul_f32x2(f32x2(vb[cur][4 * j], vb[cur][4 * j + 1]), r2), f32x2(c1.x, c1.y)));
              pk[16 + 2 * j + 1] =
                  pack_bf16x2_u64(mul_f32x2(mul_f32x2(f32x2(vb[cur][4 * j + 2], vb[cur][4 * j + 3]), r2), f32x2(c1.z, c1.w)));
            }
            __syncwarp();
          } else if (C::Mode == kModeRows && p.row_weight) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              pk[j] = pack_bf16x2(__uint_as_float(va[cur][2 * j]) * wgt, __uint_as_float(va[cur][2 * j + 1]) * wgt);
              pk[16 + j] =
                  pack_bf16x2(__uint_as_float(vb[cur][2 * j]) * wgt, __uint_as_float(vb[cur][2 * j + 1]) * wgt);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              pk[j] = pack_bf16x2(__uint_as_float(va[cur][2 * j]), __uint_as_float(va[cur][2 * j + 1]));
              pk[16 + j] = pack_bf16x2(__uint_as_float(vb[cur][2 * j]), __uint_as_float(vb[cur][2 * j + 1]));
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) pk[j] = 0u;
        }
        if (col0 >= p.Nout) continue;
        if (warp_full) {
          if constexpr (!C::Scaled) {
            if (lane == 0) bulk_wait_read<C::NBUF - 1>();
            __syncwarp();
          }
          uint8_t *rowp = buf + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4 *>(rowp + ((j ^ (lane & 7)) << 4)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmOut, buf, col0, ti.out_row0 + q * 32);
            bulk_commit();
          }
          ++nstored;
        } else if (row_ok) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + col0);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (col0 + 8 * j < p.Nout) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
      if (has_acc) {
        if (!released) release(acc);  // a warp with no chunk of this tile (narrow tiles)
        if (++acc == C::NACC) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // teardown: every role has left its loop
  tc_fence_before();
  __syncthreads();
  if (*vabort && warp == 0 && lane == 0) {
    // wait for the TMA copies this CTA armed, bounded
    for (int s = 0; s < nst; ++s) {
      const uint32_t armed = issued / nst + ((uint32_t)s < issued % nst ? 1u : 0u);
      if (armed) mbar_wait_drain(&full[s], (armed - 1) & 1);
    }
    if constexpr (C::Mx) {  // and the scale-row copies
      for (int q = 0; q < C::SF_SLOTS; ++q) {
        const uint32_t armed = sf_issued / C::SF_SLOTS + ((uint32_t)q < sf_issued % C::SF_SLOTS ? 1u : 0u);
        if (armed) mbar_wait_drain(&sf_full[q], (armed - 1) & 1);
      }
    }
    // pair: copies a peer issued for stages its leader never armed are not
    // counted anywhere; give them far longer than a copy takes to land
    if constexpr (C::Pair) {
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 100000ull) __nanosleep(1000);
    }
  }
  if constexpr (C::Pair)
    cluster_sync();  // every MMA into either CTA's TMEM and every remote arrival is done
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (C::Pair)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if constexpr (C::Pair) cluster_sync();  // neither CTA leaves while the other may still address it
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    mgemm_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmSFA,
                      const __grid_constant__ CUtensorMap tmSFB, const __grid_constant__ GemmParams p) {
  gemm_cta<C>(tmA, tmB, tmOut, tmSFA, tmSFB, p, (int)blockIdx.x, (int)gridDim.x);
}

// Two GEMMs of one backward pass in one launch: split of the grid's CTAs run
// the first (C0, maps a0 b0 o0, params p0), the others the second.  Neither
// reads what the other writes; a memory-bound weight stream (dgrad) and an
// epilogue-bound one (wgrad's grad_w stores) then share the SMs and HBM
// instead of taking turns.  The first GEMM's CTAs are spread evenly over the
// block indices (CTA b is one of them when floor((b + 1) split / grid) >
// floor(b split / grid); its index among them is floor(b split / grid)), so
// neither half is packed onto a few GPCs whatever order the CTAs are placed
// in.
template <class C0, class C1>
__global__ void __launch_bounds__(C0::THREADS, 1)
    mgemm_dual_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap b0,
                      const __grid_constant__ CUtensorMap o0, const __grid_constant__ CUtensorMap a1,
                      const __grid_constant__ CUtensorMap b1, const __grid_constant__ CUtensorMap o1,
                      const __grid_constant__ GemmParams p0, const __grid_constant__ GemmParams p1, int split) {
  static_assert(C0::THREADS == C1::THREADS && !C0::Pair && !C1::Pair && !C0::Mx && !C1::Mx,
                "both forms run the same warps, one CTA each");
  const int b = (int)blockIdx.x, g = (int)gridDim.x;
  const int lo = (int)((int64_t)b * split / g), hi = (int)((int64_t)(b + 1) * split / g);
  if (hi > lo)
    gemm_cta<C0>(a0, b0, o0, a0, a0, p0, lo, split);
  else
    gemm_cta<C1>(a1, b1, o1, a1, a1, p1, b - lo, g - split);
}

}  // namespace mgemm
