// mgemm_fwd_f8i4: the FP8 x INT4 grouped forward GEMM ("F8I4 Grouped Gemm
// Optimization for Sparse M", FBGEMM PR #3854: FP8 activations, INT4 weights,
// problems only for the non-empty groups).
//
//   out[r, n] = sum_k (e4m3(x[r, k]) / sx[r]) * q[e, n, k] * 2^(b[e, n, k / 32] - 127)
//
// over the rows tile schedule of mgemm_fill_args.  The weights stream from
// HBM as packed nibbles (half the bytes of FP8), which is what bounds the
// latency at sparse M; the tensor cores take them as e4m3 (every integer in
// [-8, 7] is an e4m3 value) in the block-scaled kind::mxf8f6f4 MMA, with the
// weight blocks' e8m0 bytes as one operand's scale factors and each token
// row's power-of-two FP8 scale written as the e8m0 byte 127 - log2(sx[r]) on
// all of the other operand's blocks of row r, so both scales are applied
// inside the MMA and the epilogue only rounds.
//
// The operands are swapped with respect to mgemm_fwd: a tile is 128 weight
// rows (output columns n0 .. n0 + 127, the MMA's M side) by the TB token rows
// of one group (the N side, TB = the token rows rounded up to 16, at most
// 128), D[n][t] = sum_k w[n, k] x[t, k].  With few token rows per group the
// MMA then does TB / 128 of the work a 128-token-row tile would, per weight
// byte, which keeps the tensor cores well below the rate at which the packed
// weights arrive.
//
// CTA (persistent, one per SM, 448 threads):
//   warp 0      TMA producer: a deep "raw" ring whose slot holds KC
//               contraction blocks of 128: token rows [KC][TB][128 B]
//               (swizzled), packed weights [KC][128][64 B] and their scale
//               words [KC][128][4 B]; the number of slots is set per launch by
//               the shared memory left.
//   warp 1      TMEM owner and MMA issuer (one thread, which also does the
//               waits): per raw slot, the
//               4 KC block-scaled MMAs (K = 32 each; the scale-factor ids
//               select byte k of the scale words); commits free the expanded
//               slot and the raw slot (its token rows are read by the MMAs),
//               and at a tile's end publish the accumulator and free the
//               tile's token-scale columns.
//   warps 2-9   converters, one handoff per raw slot: the packed nibbles of
//               its KC blocks expanded to e4m3 bytes in the 128-byte swizzled
//               K-major layout the MMA reads (a shallow "expanded" ring of
//               whole slots); the scale factors go straight into tensor memory
//               with tcgen05.st by one warp per lane quarter (lane l of every
//               quarter holds the words of rows l, l + 32, l + 64, l + 96 in
//               four columns), for the weights per block and for the tokens
//               once per tile (token row t's byte replicated into a word).
//   warps 10-13 epilogue: warp w reads the accumulator lanes of quarter w % 4
//               (weight rows, i.e. output columns), tcgen05.ld of the token
//               columns, bf16 rounding, stores out[token][column] (a warp's 32
//               lanes write 64 contiguous bytes of one token row).
// PAIR form (at most 16 token rows, and tiles for at most half of the SMs):
// clusters of two CTAs take the tiles, each CTA one half of the contraction
// blocks, so that every SM streams nibbles; the second CTA writes its fp32
// partial sums into the first's shared memory (st.shared::cluster, each lane
// arriving on the first's barrier with release at cluster scope) and the first
// adds them before rounding.
// Every wait is bounded; on expiry the kernel records MGEMM_STATUS_TIMEOUT,
// drains the copies and MMAs it issued, frees TMEM and returns.
#include "gemm_launch.cuh"

namespace mgemm {
namespace {

constexpr int kConvWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kI4Threads = 64 + 32 * (kConvWarps + kEpiWarps);

template <int kKc, int kXs, bool kPair = false>
struct I4Cfg {
  static constexpr bool PAIR = kPair;  // CTA pairs split each tile's contraction (16 token rows)
  static constexpr int BW = 128;   // weight rows (output columns) per tile: the MMA's M
  static constexpr int TB_MAX = 128;  // token rows per tile at most: the MMA's N
  static constexpr int KC = kKc;   // contraction blocks of 128 per raw slot
  static constexpr int XS = kXs;   // expanded slots (each holds a raw slot's KC blocks)
  static constexpr int RS_MAX = 16;
  static constexpr int XB_SLOT = KC * BW * 128;                            // expanded weights of KC blocks
  static constexpr int SFT_COL = 2 * TB_MAX;   // token scale columns (4 per accumulator)
  static constexpr int SFW_COL = 2 * TB_MAX + 8;  // weight scale columns (4 per block of each expanded slot)
  static constexpr int COLS = 2 * TB_MAX + 8 + 4 * KC * XS;
  static constexpr int TMEM_COLS = COLS <= 256 ? 256 : 512;
  static_assert(COLS <= 512, "tensor memory");
  static_assert(XB_SLOT % 1024 == 0, "swizzle atoms");
  static constexpr int RECV_BYTES = 128 * 16 * 4;  // PAIR: the partner's partial sums, 128 rows x 16 fp32
  static constexpr size_t TAIL = 8 * (2 * RS_MAX + 2 * XS + 8 + 1 + 2) + 64 + (PAIR ? 16 + RECV_BYTES : 0);
  // a raw slot: [tokens KC x TB x 128][weights packed KC x 128 x 64][weight scales KC x 128 x 4]
  static size_t raw_slot_bytes(int tb) {
    return ((size_t)KC * ((size_t)tb * 128 + BW * 64 + BW * 4) + 1023) / 1024 * 1024;
  }
  static size_t fixed_bytes() { return 1024 /*align*/ + (size_t)XS * XB_SLOT + TAIL; }
};

// ---- the decode of a tile: the rows schedule of the grouped GEMM, a "row
// tile" being up to 128 token rows of one group and a "column tile" 128 weight
// rows; out_rows is clipped to the TB token rows the tile's box holds
template <int kKc>
using I4Decode = GemmCfg<true, false, false, kModeRows, 128, 24, 1, false, 8, true, kKc, false>;

// 8 packed nibbles (element 0 in bits 0-3) -> 8 e4m3 bytes.  The low three
// bits of each nibble select a byte of one of two 8-entry tables (prmt): the
// codes of 0 .. 7 and of -8 .. -1; bit 3 (the sign) picks the table through a
// byte mask made by prmt's sign-replicating mode.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint2 int4x8_to_e4m3(uint32_t w) {
  // e4m3 codes: 0, 1, 2, 3 -> 00 38 40 44; 4 .. 7 -> 48 4A 4C 4E;
  // -8, -7, -6, -5 -> D0 CE CC CA; -4 .. -1 -> C8 C4 C0 B8
  constexpr uint32_t P0 = 0x44403800u, P1 = 0x4E4C4A48u, N0 = 0xCACCCED0u, N1 = 0xB8C0C4C8u;
  const uint32_t sl = w & 0x7777u, sh = (w >> 16) & 0x7777u;
  const uint32_t s4 = w << 4;
  // byte i of the mask = 0xFF when nibble i has bit 3 set: nibble 2j's bit 3 is
  // the top bit of byte j of (w << 4), nibble 2j + 1's that of byte j of w
  const uint32_t mlo = prmt(s4, w, 0xD9C8u), mhi = prmt(s4, w, 0xFBEAu);
  const uint32_t plo = prmt(P0, P1, sl), nlo = prmt(N0, N1, sl);
  const uint32_t phi = prmt(P0, P1, sh), nhi = prmt(N0, N1, sh);
  return make_uint2((plo & ~mlo) | (nlo & mlo), (phi & ~mhi) | (nhi & mhi));
}

struct I4Params {
  GemmParams g;      // args, E, bn, a_rows, idesc, n_tiles, Kc, Nout, out, rscale (sx)
  int raw_slots;
  int raw_slot_bytes;
};

template <class C>
__global__ void __launch_bounds__(kI4Threads, 1)
    f8i4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmS, const I4Params P) {
  using D = I4Decode<C::KC>;
  const GemmParams &p = P.g;
  const int TB = p.a_rows;  // token rows per tile (a multiple of 16)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int RS = P.raw_slots;
  uint8_t *sX = smem;                                     // expanded ring
  uint8_t *sR = sX + C::XS * C::XB_SLOT;                  // raw ring
  auto raw_t = [&](int r, int j) { return sR + (size_t)r * P.raw_slot_bytes + (size_t)j * TB * 128; };
  auto raw_w = [&](int r) { return sR + (size_t)r * P.raw_slot_bytes + (size_t)C::KC * TB * 128; };
  auto raw_s = [&](int r, int j) {
    return sR + (size_t)r * P.raw_slot_bytes + (size_t)C::KC * (TB * 128 + C::BW * 64) + (size_t)j * C::BW * 4;
  };
  auto xb = [&](int x, int j) { return sX + x * C::XB_SLOT + j * C::BW * 128; };
  uint64_t *bars = reinterpret_cast<uint64_t *>(sR + (size_t)RS * P.raw_slot_bytes);
  uint64_t *raw_full = bars, *raw_empty = bars + C::RS_MAX;
  uint64_t *xb_full = raw_empty + C::RS_MAX, *xb_empty = xb_full + C::XS;
  uint64_t *ts_full = xb_empty + C::XS, *ts_empty = ts_full + 2;
  uint64_t *tfull = ts_empty + 2, *tempty = tfull + 2, *drain = tempty + 2;
  uint64_t *part_full = drain + 1, *part_empty = part_full + 1;  // PAIR: recv holds a partial / may be rewritten
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(part_empty + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  float *recv = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(abort_flag + 1) + 15) & ~uintptr_t(15));
  const uint32_t rank = C::PAIR ? cluster_ctarank() : 0u;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t_first = C::PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int t_step = C::PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // a tile's contraction blocks (raw slots) [g_lo, g_hi) of its kb_count for this CTA
  auto g_range = [&](int kb_count, int &g_lo, int &g_hi) {
    const int half = (kb_count + 1) / 2;
    g_lo = C::PAIR && rank == 1 ? half : 0;
    g_hi = C::PAIR && rank == 0 ? half : kb_count;
  };
  // set-up before the wait for the previous grid (it reads nothing that grid
  // writes); a CTA without tiles runs no role loop
  if (threadIdx.x == 0) {
    for (int r = 0; r < RS; ++r) {
      mbar_init(&raw_full[r], 1);
      mbar_init(&raw_empty[r], 1);
    }
    for (int x = 0; x < C::XS; ++x) {
      mbar_init(&xb_full[x], kConvWarps);
      mbar_init(&xb_empty[x], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ts_full[a], kConvWarps);
      mbar_init(&ts_empty[a], 1);
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(part_full, 128);
    mbar_init(part_empty, 128);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmS);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (C::PAIR) cluster_sync();  // the partner's barriers are initialised before any arrival on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  const ArgsView av(p.args, p.E);
  const int status0 = *av.status, n_active0 = *av.n_active;
  const int total = status0 != 0 ? 0 : total_tiles<D>(p, av, n_active0);
  volatile int *vabort = abort_flag;
  uint32_t issued = 0;  // raw slots armed (for the drain after an abort)

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t tx = (uint32_t)C::KC * (uint32_t)(TB * 128 + C::BW * 64 + C::BW * 4);
      int r = 0;
      uint32_t ph = 0;
      for (int j = 0; j * t_step < total && !*vabort; ++j) {
        const int t = tile_of<D>(j, t_first, t_step);
        if (t >= total) continue;
        const TileInfo ti = decode_tile<D>(t, p, av, 0u);
        int g_lo, g_hi;
        g_range(ti.kb_count, g_lo, g_hi);
        for (int g = g_lo; g < g_hi; ++g) {
          if (!mbar_wait(&raw_empty[r], ph ^ 1, vabort)) {
            set_status(av.status, MGEMM_STATUS_TIMEOUT);
            *vabort = 1;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[r], tx);
          ++issued;
          // weights first (the long pole), then their scales and the token rows
          tma_load_4d(raw_w(r), &tmB, &raw_full[r], 0, ti.n0, g * C::KC, ti.e);
          tma_load_4d(raw_s(r, 0), &tmS, &raw_full[r], 0, ti.n0 / 4, g * C::KC, ti.e);
          tma_load_3d(raw_t(r, 0), &tmA, &raw_full[r], 0, ti.a_row, g * C::KC);
          if (++r == RS) {
            r = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // one thread waits and issues (no warp-wide vote per slot)
    if (lane == 0) {
      int r = 0, x = 0, acc = 0;
      uint32_t rph = 0, xph = 0, aph = 0;
      bool ok = true;
      for (int j = 0; j * t_step < total && ok; ++j) {
        const int t = tile_of<D>(j, t_first, t_step);
        if (t >= total) continue;
        const TileInfo ti = decode_tile<D>(t, p, av, 0u);
        if (!mbar_wait(&tempty[acc], aph ^ 1, vabort) || !mbar_wait(&ts_full[acc], aph, vabort)) {
          ok = false;
          break;
        }
        const uint32_t d_tmem = tmem_base + acc * C::TB_MAX;
        const uint32_t sft = tmem_base + C::SFT_COL + 4 * acc;
        int g_lo, g_hi;
        g_range(ti.kb_count, g_lo, g_hi);
        for (int g = g_lo; g < g_hi; ++g) {
          if (!mbar_wait(&raw_full[r], rph, vabort) || !mbar_wait(&xb_full[x], xph, vabort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < C::KC; ++jj) {
            const uint32_t sfw = tmem_base + C::SFW_COL + 4 * (x * C::KC + jj);
            // descriptors advance by (byte offset >> 4) in their start-address field
            const uint64_t ad = smem_desc_sw128(smem_u32(xb(x, jj)), 16, 1024);    // weights: M side
            const uint64_t bd = smem_desc_sw128(smem_u32(raw_t(r, jj)), 16, 1024);  // tokens: N side
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t idk = p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29);
              mma_mx(d_tmem, ad + 2 * k, bd + 2 * k, idk, sfw, sft, (g != g_lo) | jj | k);
            }
          }
          mma_commit(&xb_empty[x]);
          mma_commit(&raw_empty[r]);  // the slot's token rows are read
          if (++x == C::XS) {
            x = 0;
            xph ^= 1;
          }
          if (++r == RS) {
            r = 0;
            rph ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        mma_commit(&ts_empty[acc]);  // the tile's token-scale columns are read
        if (++acc == 2) {
          acc = 0;
          aph ^= 1;
        }
      }
      if (!ok) {
        set_status(av.status, MGEMM_STATUS_TIMEOUT);
        *vabort = 1;
      }
      // every MMA this thread issued has completed before TMEM is freed
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp < 2 + kConvWarps) {
    constexpr int NT = 32 * kConvWarps;
    const int c = threadIdx.x - 64;                 // 0 .. NT - 1
    const bool sf_writer = warp < 2 + 4;            // one warp per TMEM lane quarter writes the scales
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int r = 0, x = 0, acc = 0;
    uint32_t rph = 0, xph = 0, aph = 0;
    bool ok = true;
    for (int j = 0; j * t_step < total && ok; ++j) {
      const int t = tile_of<D>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<D>(t, p, av, 0u);
      // token scales of this tile: token row i's word is its byte 127 - log2(sx)
      // (254 minus the biased exponent of the power of two sx) in all four
      // sub-blocks; rows past the tile's rows get the unit byte
      if (!mbar_wait_warp(&ts_empty[acc], aph ^ 1, vabort)) { ok = false; break; }
      if (sf_writer) {
        uint32_t wv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int i = lane + 32 * m;
          wv[m] = 0x7F7F7F7Fu;
          if (i < ti.out_rows)
            wv[m] = (254u - (__float_as_uint(__ldg(p.rscale + ti.out_row0 + i)) >> 23)) * 0x01010101u;
        }
        tmem_st_32x32b_x4(tmem_base + lane_base + C::SFT_COL + 4 * acc, wv);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ts_full[acc]);
      int g_lo, g_hi;
      g_range(ti.kb_count, g_lo, g_hi);
      for (int g = g_lo; g < g_hi; ++g) {
        if (!mbar_wait_warp(&raw_full[r], rph, vabort) || !mbar_wait_warp(&xb_empty[x], xph ^ 1, vabort)) {
          ok = false;
          break;
        }
        // expand: output chunk ch (16 elements) of weight row n of block jj.  All of a
        // thread's packed chunks are read first (the raw and expanded slots are distinct,
        // but the compiler cannot tell), so the reads overlap instead of each waiting
        // behind the previous chunk's conversion and store.
        const uint8_t *src = raw_w(r);
        uint8_t *dst = xb(x, 0);
        constexpr int kChunks = C::KC * C::BW * 8;
        static_assert(kChunks % NT == 0, "whole rounds");
        constexpr int kIt = kChunks / NT;
        uint2 v[kIt];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
          const int idx = c + it * NT;
          v[it] = *reinterpret_cast<const uint2 *>(src + (size_t)idx * 8);  // = (jj * BW + n) * 64 + ch * 8
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
          const int idx = c + it * NT;
          const int jj = idx / (C::BW * 8), rem = idx % (C::BW * 8);
          const int n = rem >> 3, ch = rem & 7;
          const uint2 lo = int4x8_to_e4m3(v[it].x), hi = int4x8_to_e4m3(v[it].y);
          *reinterpret_cast<uint4 *>(dst + (jj * C::BW + n) * 128 + ((ch ^ (n & 7)) << 4)) =
              make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
        if (sf_writer) {  // weight scales of the slot's blocks: lane l holds rows l, l + 32, l + 64, l + 96
#pragma unroll
          for (int jj = 0; jj < C::KC; ++jj) {
            const uint32_t *sw = reinterpret_cast<const uint32_t *>(raw_s(r, jj));
            const uint32_t wv[4] = {sw[lane], sw[lane + 32], sw[lane + 64], sw[lane + 96]};
            tmem_st_32x32b_x4(tmem_base + lane_base + C::SFW_COL + 4 * (x * C::KC + jj), wv);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();  // generic writes -> tensor-core reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&xb_full[x]);
        if (++x == C::XS) {
          x = 0;
          xph ^= 1;
        }
        if (++r == RS) {
          r = 0;
          rph ^= 1;
        }
      }
      if (!ok) break;
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
    if (!ok) {
      if (lane == 0) set_status(av.status, MGEMM_STATUS_TIMEOUT);
      *vabort = 1;
    }
  } else {
    // epilogue: warp w reads accumulator lanes of quarter q = w % 4, i.e. output
    // columns n0 + 32 q + lane, and the token columns 0 .. TB - 1
    const int q = warp & 3;
    int acc = 0;
    uint32_t aph = 0, part_phase = 0;
    for (int j = 0; j * t_step < total; ++j) {
      const int t = tile_of<D>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<D>(t, p, av, 0u);
      if (!mbar_wait_warp(&tfull[acc], aph, vabort)) {
        set_status(av.status, MGEMM_STATUS_TIMEOUT);
        *vabort = 1;
        break;
      }
      tc_fence_after();
      const int col = ti.n0 + q * 32 + lane;
      const bool col_ok = col < p.Nout;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::TB_MAX;
      bool pair_ok = true;
      for (int c0 = 0; c0 < TB; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(taddr + c0, v);
        tmem_ld_wait();
        if (c0 + 16 >= TB) {  // the accumulator is read: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        if (C::PAIR) {  // TB == 16: one chunk
          const int row = q * 32 + lane;
          if (rank == 1) {
            // the second half's partial sums into the first CTA's recv, once it has read the last ones
            if (!mbar_wait_cluster_warp(part_empty, part_phase ^ 1, vabort)) {
              pair_ok = false;
              break;
            }
            part_phase ^= 1;
            const uint32_t dst = cluster_addr(recv + row * 16, 0);
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + i * 4), "r"(v[i]),
                           "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3])
                           : "memory");
            mbar_arrive_cluster(cluster_addr(part_full, 0));
            continue;
          }
          if (!mbar_wait_cluster_warp(part_full, part_phase, vabort)) {
            pair_ok = false;
            break;
          }
          part_phase ^= 1;
          const float4 *src = reinterpret_cast<const float4 *>(recv + row * 16);
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 f4 = src[i / 4];
            v[i] = __float_as_uint(__uint_as_float(v[i]) + f4.x);
            v[i + 1] = __float_as_uint(__uint_as_float(v[i + 1]) + f4.y);
            v[i + 2] = __float_as_uint(__uint_as_float(v[i + 2]) + f4.z);
            v[i + 3] = __float_as_uint(__uint_as_float(v[i + 3]) + f4.w);
          }
          mbar_arrive_cluster(cluster_addr(part_empty, 1));
        }
        if (col_ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c0 + i < ti.out_rows)
              p.out[((int64_t)ti.out_row0 + c0 + i) * p.Nout + col] = __float2bfloat16_rn(__uint_as_float(v[i]));
        }
      }
      if (!pair_ok) {
        set_status(av.status, MGEMM_STATUS_TIMEOUT);
        *vabort = 1;
        break;
      }
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*vabort && warp == 0 && lane == 0) {
    // wait for the TMA copies this CTA armed, bounded
    for (int r = 0; r < RS; ++r) {
      const uint32_t armed = issued / RS + ((uint32_t)r < issued % RS ? 1u : 0u);
      if (armed) mbar_wait_drain(&raw_full[r], (armed - 1) & 1);
    }
  }
  __syncthreads();
  if (C::PAIR) cluster_sync();  // neither CTA of a pair leaves while the other may still reach its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <class C>
int launch_f8i4(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &s, I4Params P, int grid,
                cudaStream_t st) {
  const size_t slot = C::raw_slot_bytes(P.g.a_rows);
  const size_t room = (size_t)227 * 1024 - C::fixed_bytes();
  int rs = (int)(room / slot);
  if (rs > C::RS_MAX) rs = C::RS_MAX;
  if (rs < 2 || P.g.a_rows % 16) return MGEMM_EINVAL;
  P.raw_slots = rs;
  P.raw_slot_bytes = (int)slot;
  const size_t smem = C::fixed_bytes() + (size_t)rs * slot;
  static bool attr_done[64] = {};
  int dev = 0;
  int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return MGEMM_EINVAL;
  if (!attr_done[dev]) {
    rc = cuda_rc(cudaFuncSetAttribute(f8i4_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024),
                 "cudaFuncSetAttribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  return launch_pdl(f8i4_gemm_kernel<C>, dim3((unsigned)grid), dim3(kI4Threads), smem, st, C::PAIR ? 2u : 1u,
                    C::PAIR ? "F8I4 GEMM launch (CTA pairs)" : "F8I4 GEMM launch", a, b, s, P);
}

}  // namespace
}  // namespace mgemm

using namespace mgemm;

extern "C" int mgemm_fwd_f8i4(const void *args, const uint8_t *x, const float *sx, const uint8_t *w_packed,
                              const uint8_t *w_scales, void *out, int64_t M, int K, int N, int E,
                              mgemm_stream_t stream) {
  if (!args || !x || !sx || !w_packed || !w_scales || !out) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || K <= 0 || N <= 0) return MGEMM_EINVAL;
  if ((int64_t)E * N >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (K % 128 || N % 8) return MGEMM_EALIGN;
  if (((uintptr_t)args & 15) || ((uintptr_t)x & 15) || ((uintptr_t)sx & 3) || ((uintptr_t)w_packed & 15) ||
      ((uintptr_t)w_scales & 15) || ((uintptr_t)out & 15))
    return MGEMM_EALIGN;
  if (M == 0) return MGEMM_OK;
  int rc = ensure_context();
  if (rc) return rc;
  const int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  // tiles of 128 weight rows (output columns) by TB token rows of one group:
  // TB = the token rows rounded up to 16 (the MMA's N), at most 128
  const int64_t groups = M < E ? M : E;
  const uint32_t tb = M < 128 ? (uint32_t)((M + 15) / 16 * 16) : 128u;
  const int kc = 2;
  CUtensorMap ta, tb_map, ts;
  {  // x [M, K] e4m3 as 128-byte k-chunks: {128, M, K / 128}, boxes of kc chunks of tb rows
    const uint64_t d[3] = {128, (uint64_t)M, (uint64_t)K / 128};
    const uint64_t st[2] = {(uint64_t)K, 128};
    const uint32_t box[3] = {128, tb, (uint32_t)kc};
    if (!make_tensor_map(&ta, true, 3, x, d, st, box)) return MGEMM_ECUDA;
  }
  {  // packed w [E, N, K / 2] as 64-byte k-chunks: {64, N, K / 128, E}, unswizzled
    const uint64_t d[4] = {64, (uint64_t)N, (uint64_t)K / 128, (uint64_t)E};
    const uint64_t st[3] = {(uint64_t)K / 2, 64, (uint64_t)N * K / 2};
    const uint32_t box[4] = {64, 128, (uint32_t)kc, 1};
    if (!make_tensor_map(&tb_map, true, 4, w_packed, d, st, box, false)) return MGEMM_ECUDA;
  }
  {  // scales [E][K / 128][N][4 B] as 16-byte rows of four: {16, N / 4, K / 128, E}
    const uint64_t d[4] = {16, (uint64_t)N / 4, (uint64_t)K / 128, (uint64_t)E};
    const uint64_t st[3] = {16, (uint64_t)N * 4, (uint64_t)K / 128 * N * 4};
    const uint32_t box[4] = {16, 32, (uint32_t)kc, 1};
    if (!make_tensor_map(&ts, true, 4, w_scales, d, st, box, false)) return MGEMM_ECUDA;
  }
  I4Params P{};
  GemmParams &p = P.g;
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = 128;
  p.a_rows = (int)tb;
  p.idesc = make_idesc_mx(128, (int)tb, 1);  // M = 128 weight rows, N = tb token rows, ue8m0 scale factors
  p.n_tiles = (N + 127) / 128;
  p.Kc = K;
  p.Nout = N;
  p.out = (__nv_bfloat16 *)out;
  p.rscale = sx;
  const int64_t upper = ((M + 127) / 128 + groups) * p.n_tiles;
  cudaStream_t s = (cudaStream_t)stream;
  // pairs: 16 token rows (every group in one row tile: at most groups x n_tiles tiles), two
  // contraction slots per tile at least, and tiles for at most half of the SMs
  const int64_t tiles16 = groups * p.n_tiles;
  if (tb == 16 && K >= 2 * 128 * kc && 2 * tiles16 <= sms)
    return launch_f8i4<I4Cfg<2, 2, true>>(ta, tb_map, ts, P, (int)(2 * tiles16), s);
  const int grid = (int)(upper < sms ? upper : sms);
  return launch_f8i4<I4Cfg<2, 2>>(ta, tb_map, ts, P, grid, s);
}
