// mgemm_fwd_f8i4: the FP8 x INT4 grouped forward GEMM ("F8I4 Grouped Gemm
// Optimization for Sparse M", FBGEMM PR #3854: FP8 activations, INT4 weights,
// problems only for the non-empty groups).
//
//   out[r, n] = sum_k (e4m3(x[r, k]) / sx[r]) * q[e, n, k] * 2^(b[e, n, k / 32] - 127)
//
// over the rows tile schedule of mgemm_fill_args (tiles of 128 token rows of
// one non-empty group x BN output columns).  The weights stream from HBM as
// packed nibbles (half the bytes of FP8), which is what bounds the latency at
// sparse M; the tensor cores take them as e4m3 (every integer in [-8, 7] is an
// e4m3 value) in the block-scaled kind::mxf8f6f4 MMA, with the weight blocks'
// e8m0 bytes as B's scale factors and each token row's power-of-two FP8 scale
// written as the e8m0 byte 127 - log2(sx[r]) on all of A's blocks of row r,
// so both scales are applied inside the MMA and the epilogue only rounds.
//
// CTA (persistent, one per SM, 320 threads):
//   warp 0      TMA producer: a deep "raw" ring whose slot holds KC
//               contraction blocks of 128: A rows [KC][a_rows][128 B]
//               (swizzled), packed B [KC][BN][64 B] and B's scale words
//               [KC][BN][4 B]; the number of slots is set per launch by the
//               shared memory left.
//   warp 1      TMEM owner and MMA issuer (one thread): per tile, copies the A
//               scale tile into tensor memory; per contraction block, copies
//               the block's B scale tile and issues four block-scaled MMAs
//               (K = 32 each, the scale-factor ids selecting byte k of the
//               scale words); commits free the expanded slot, then the raw
//               slot (its A rows are read by the MMAs), then publish the
//               accumulator.
//   warps 2-5   converters: per tile, the A scale tile (row r's byte
//               replicated into a word); per contraction block, the packed
//               nibbles of BN rows expanded to e4m3 bytes in the 128-byte
//               swizzled K-major layout the MMA reads (a shallow "expanded"
//               ring), and the B scale tile (row l of the 512-byte tile holds
//               the words of rows l, l + 32, l + 64, l + 96).
//   warps 6-9   epilogue: tcgen05.ld of the accumulator (two in TMEM, so the
//               next tile's main loop overlaps), bf16 rounding, direct stores
//               of the tile's valid rows.
// Every wait is bounded; on expiry the kernel records MGEMM_STATUS_TIMEOUT,
// drains the copies and MMAs it issued, frees TMEM and returns.
#include "gemm_launch.cuh"

namespace mgemm {
namespace {

constexpr int kConvWarps = 4;
constexpr int kEpiWarps = 4;
constexpr int kI4Threads = 64 + 32 * (kConvWarps + kEpiWarps);

template <int kBn, int kKc, int kXs>
struct I4Cfg {
  static constexpr int BN = kBn;   // output columns per tile (64 or 128)
  static constexpr int KC = kKc;   // contraction blocks of 128 per raw slot
  static constexpr int XS = kXs;   // expanded slots
  static constexpr int RS_MAX = 16;
  static constexpr int XB_BYTES = BN * 128;                                // expanded B, one block
  static constexpr int XB_SLOT = (XB_BYTES + 512 + 1023) / 1024 * 1024;    // + its scale tile
  static constexpr int TMEM_COLS = 2 * BN + 8 + 4 * XS <= 256 ? 256 : 512;
  static constexpr int SFA_COL = 2 * BN;       // A scale tiles (one per accumulator), 4 columns each
  static constexpr int SFB_COL = 2 * BN + 8;   // B scale tiles (one per expanded slot)
  static_assert(2 * BN + 8 + 4 * XS <= 512, "tensor memory");
  static constexpr size_t TAIL = 8 * (2 * RS_MAX + 2 * XS + 8 + 1) + 64;
  // a raw slot: [A KC x a_rows x 128][B packed KC x BN x 64][B scales KC x BN x 4]
  static size_t raw_slot_bytes(int a_rows) {
    return ((size_t)KC * ((size_t)a_rows * 128 + BN * 64 + BN * 4) + 1023) / 1024 * 1024;
  }
  static size_t fixed_bytes() { return 1024 /*align*/ + (size_t)XS * XB_SLOT + 1024 /*A scale tiles*/ + TAIL; }
};

// ---- the decode of a tile: the rows schedule of the grouped GEMM (one group
// per tile; out_rows clipped to the A box's rows)
template <int kBn, int kKc>
using I4Decode = GemmCfg<true, false, false, kModeRows, kBn, 24, 1, false, 8, true, kKc, false>;

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
  using D = I4Decode<C::BN, C::KC>;
  const GemmParams &p = P.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int RS = P.raw_slots;
  uint8_t *sX = smem;                                     // expanded ring
  uint8_t *sAT = sX + C::XS * C::XB_SLOT;                 // two A scale tiles
  uint8_t *sR = sAT + 1024;                               // raw ring
  auto raw_a = [&](int r, int j) { return sR + (size_t)r * P.raw_slot_bytes + (size_t)j * p.a_rows * 128; };
  auto raw_b = [&](int r, int j) {
    return sR + (size_t)r * P.raw_slot_bytes + (size_t)C::KC * p.a_rows * 128 + (size_t)j * C::BN * 64;
  };
  auto raw_s = [&](int r, int j) {
    return sR + (size_t)r * P.raw_slot_bytes + (size_t)C::KC * (p.a_rows * 128 + C::BN * 64) + (size_t)j * C::BN * 4;
  };
  auto xb = [&](int x) { return sX + x * C::XB_SLOT; };
  auto xb_tile = [&](int x) { return sX + x * C::XB_SLOT + C::XB_BYTES; };
  uint64_t *bars = reinterpret_cast<uint64_t *>(sR + (size_t)RS * P.raw_slot_bytes);
  uint64_t *raw_full = bars, *raw_empty = bars + C::RS_MAX;
  uint64_t *xb_full = raw_empty + C::RS_MAX, *xb_empty = xb_full + C::XS;
  uint64_t *as_full = xb_empty + C::XS, *as_empty = as_full + 2;
  uint64_t *tfull = as_empty + 2, *tempty = tfull + 2, *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const ArgsView av(p.args, p.E);
  if (*av.status != 0) return;
  const int total = total_tiles<D>(p, av);
  const int t_first = (int)blockIdx.x, t_step = (int)gridDim.x;
  if (t_first >= total) return;
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
      mbar_init(&as_full[a], kConvWarps);
      mbar_init(&as_empty[a], 1);
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
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
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int *vabort = abort_flag;
  uint32_t issued = 0;  // raw slots armed (for the drain after an abort)

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t tx = (uint32_t)C::KC * (uint32_t)(p.a_rows * 128 + C::BN * 64 + C::BN * 4);
      int r = 0;
      uint32_t ph = 0;
      for (int j = 0; j * t_step < total && !*vabort; ++j) {
        const int t = tile_of<D>(j, t_first, t_step);
        if (t >= total) continue;
        const TileInfo ti = decode_tile<D>(t, p, av, 0u);
        for (int g = 0; g < ti.kb_count; ++g) {
          if (!mbar_wait(&raw_empty[r], ph ^ 1, vabort)) {
            set_status(av.status, MGEMM_STATUS_TIMEOUT);
            *vabort = 1;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[r], tx);
          ++issued;
          // weights first (the long pole), then the scales and the token rows
          tma_load_4d(raw_b(r, 0), &tmB, &raw_full[r], 0, ti.b_row, g * C::KC, ti.e);
          tma_load_4d(raw_s(r, 0), &tmS, &raw_full[r], 0, ti.b_row / 4, g * C::KC, ti.e);
          tma_load_3d(raw_a(r, 0), &tmA, &raw_full[r], 0, ti.a_row, g * C::KC);
          if (++r == RS) {
            r = 0;
            ph ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    int r = 0, x = 0, acc = 0;
    uint32_t rph = 0, xph = 0, aph = 0;
    bool ok = true;
    for (int j = 0; j * t_step < total && ok; ++j) {
      const int t = tile_of<D>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<D>(t, p, av, 0u);
      if (!mbar_wait_warp(&tempty[acc], aph ^ 1, vabort) || !mbar_wait_warp(&as_full[acc], aph, vabort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::BN;
      const uint32_t sfa = tmem_base + C::SFA_COL + 4 * acc;
      if (lane == 0) {
        tmem_cp_32x128b_warpx4(sfa, smem_desc_rows16(smem_u32(sAT + acc * 512)));
        mma_commit(&as_empty[acc]);
      }
      __syncwarp();
      for (int g = 0; g < ti.kb_count && ok; ++g) {
        if (!mbar_wait_warp(&raw_full[r], rph, vabort)) { ok = false; break; }
        for (int jj = 0; jj < C::KC; ++jj) {
          if (!mbar_wait_warp(&xb_full[x], xph, vabort)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sfb = tmem_base + C::SFB_COL + 4 * x;
            tmem_cp_32x128b_warpx4(sfb, smem_desc_rows16(smem_u32(xb_tile(x))));
            const uint32_t abase = smem_u32(raw_a(r, jj)), bbase = smem_u32(xb(x));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = smem_desc_sw128(abase + k * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(bbase + k * 32, 16, 1024);
              const uint32_t idk = p.idesc | ((uint32_t)k << 4) | ((uint32_t)k << 29);
              mma_mx(d_tmem, ad, bd, idk, sfa, sfb, (g | jj | k) != 0);
            }
            mma_commit(&xb_empty[x]);
          }
          __syncwarp();
          if (++x == C::XS) {
            x = 0;
            xph ^= 1;
          }
        }
        if (!ok) break;
        if (lane == 0) mma_commit(&raw_empty[r]);  // the slot's A rows are read
        __syncwarp();
        if (++r == RS) {
          r = 0;
          rph ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&tfull[acc]);
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        aph ^= 1;
      }
    }
    if (!ok) {
      if (lane == 0) set_status(av.status, MGEMM_STATUS_TIMEOUT);
      *vabort = 1;
    }
    if (lane == 0) {  // every MMA and copy this thread issued has completed before TMEM is freed
      mma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp < 2 + kConvWarps) {
    const int c = threadIdx.x - 64;  // 0 .. 127
    int r = 0, x = 0, acc = 0;
    uint32_t rph = 0, xph = 0, aph = 0;
    bool ok = true;
    for (int j = 0; j * t_step < total && ok; ++j) {
      const int t = tile_of<D>(j, t_first, t_step);
      if (t >= total) continue;
      const TileInfo ti = decode_tile<D>(t, p, av, 0u);
      // A scale tile of this tile: word of token row i = its byte 127 - log2(sx)
      // (254 minus the biased exponent of the power of two sx) in all four
      // sub-blocks; rows past the tile's rows get the unit byte
      if (!mbar_wait_warp(&as_empty[acc], aph ^ 1, vabort)) { ok = false; break; }
      {
        const int i = c;  // token row i of the tile: row l = i % 32, word i / 32 of the tile row
        uint32_t wv = 0x7F7F7F7Fu;
        if (i < ti.out_rows) {
          const uint32_t b = 254u - (__float_as_uint(__ldg(p.rscale + ti.out_row0 + i)) >> 23);
          wv = b * 0x01010101u;
        }
        reinterpret_cast<uint32_t *>(sAT + acc * 512)[(i & 31) * 4 + (i >> 5)] = wv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&as_full[acc]);
      for (int g = 0; g < ti.kb_count && ok; ++g) {
        if (!mbar_wait_warp(&raw_full[r], rph, vabort)) { ok = false; break; }
        for (int jj = 0; jj < C::KC; ++jj) {
          if (!mbar_wait_warp(&xb_empty[x], xph ^ 1, vabort)) { ok = false; break; }
          const uint8_t *src = raw_b(r, jj);
          uint8_t *dst = xb(x);
#pragma unroll 2
          for (int idx = c; idx < C::BN * 8; idx += 32 * kConvWarps) {
            const int n = idx >> 3, ch = idx & 7;  // output chunk ch (16 elements) of row n
            const uint2 v = *reinterpret_cast<const uint2 *>(src + n * 64 + ch * 8);
            const uint2 lo = int4x8_to_e4m3(v.x), hi = int4x8_to_e4m3(v.y);
            *reinterpret_cast<uint4 *>(dst + n * 128 + ((ch ^ (n & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
          }
          if (c < 32) {  // B scale tile: row l holds the words of rows l, l + 32, l + 64, l + 96
            const uint32_t *sw = reinterpret_cast<const uint32_t *>(raw_s(r, jj));
            const uint4 tv = make_uint4(sw[c], C::BN > 32 ? sw[c + 32] : 0u, C::BN > 64 ? sw[c + 64] : 0u,
                                        C::BN > 96 ? sw[c + 96] : 0u);
            reinterpret_cast<uint4 *>(xb_tile(x))[c] = tv;
          }
          fence_proxy_async_smem();  // generic writes -> tensor-core reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&xb_full[x]);
          if (++x == C::XS) {
            x = 0;
            xph ^= 1;
          }
        }
        if (++r == RS) {
          r = 0;
          rph ^= 1;
        }
      }
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
    // epilogue: warp w reads TMEM lane quarter w % 4 (tile rows 32 q ..)
    const int q = warp & 3;
    const int rr = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
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
      const bool row_ok = rr < ti.out_rows;
      __nv_bfloat16 *orow = p.out + ((int64_t)ti.out_row0 + (row_ok ? rr : 0)) * p.Nout;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::BN;
#pragma unroll
      for (int cc = 0; cc < C::BN / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + cc * 32, v);
        tmem_ld_wait();
        if (cc == C::BN / 32 - 1) {  // the accumulator is read: hand it back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        const int col0 = ti.n0 + cc * 32;
        if (row_ok && col0 < p.Nout) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint4 *dst = reinterpret_cast<uint4 *>(orow + col0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (col0 + 8 * i < p.Nout) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
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
  if (rs < 2 || P.g.a_rows % 8) return MGEMM_EINVAL;
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
  return launch_pdl(f8i4_gemm_kernel<C>, dim3((unsigned)grid), dim3(kI4Threads), smem, st, 1u, "F8I4 GEMM launch", a,
                    b, s, P);
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
  // 64-column tiles while the weights stream (few rows per group), 128 beyond
  const int64_t groups = M < E ? M : E;
  const bool narrow = M / groups < 128;
  const int bn = narrow ? 64 : 128, kc = narrow ? 4 : 2;
  const uint32_t a_rows = M < 128 ? (uint32_t)((M + 7) / 8 * 8) : 128u;
  CUtensorMap ta, tb, ts;
  {  // x [M, K] e4m3 as 128-byte k-chunks: {128, M, K / 128}, boxes of kc chunks of a_rows rows
    const uint64_t d[3] = {128, (uint64_t)M, (uint64_t)K / 128};
    const uint64_t st[2] = {(uint64_t)K, 128};
    const uint32_t box[3] = {128, a_rows, (uint32_t)kc};
    if (!make_tensor_map(&ta, true, 3, x, d, st, box)) return MGEMM_ECUDA;
  }
  {  // packed w [E, N, K / 2] as 64-byte k-chunks: {64, N, K / 128, E}, unswizzled
    const uint64_t d[4] = {64, (uint64_t)N, (uint64_t)K / 128, (uint64_t)E};
    const uint64_t st[3] = {(uint64_t)K / 2, 64, (uint64_t)N * K / 2};
    const uint32_t box[4] = {64, (uint32_t)bn, (uint32_t)kc, 1};
    if (!make_tensor_map(&tb, true, 4, w_packed, d, st, box, false)) return MGEMM_ECUDA;
  }
  {  // scales [E][K / 128][N][4 B] as 16-byte rows of four: {16, N / 4, K / 128, E}
    const uint64_t d[4] = {16, (uint64_t)N / 4, (uint64_t)K / 128, (uint64_t)E};
    const uint64_t st[3] = {16, (uint64_t)N * 4, (uint64_t)K / 128 * N * 4};
    const uint32_t box[4] = {16, (uint32_t)bn / 4, (uint32_t)kc, 1};
    if (!make_tensor_map(&ts, true, 4, w_scales, d, st, box, false)) return MGEMM_ECUDA;
  }
  I4Params P{};
  GemmParams &p = P.g;
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = bn;
  p.a_rows = (int)a_rows;
  p.idesc = make_idesc_mx(128, bn, 1);  // ue8m0 scale factors
  p.n_tiles = (N + bn - 1) / bn;
  p.Kc = K;
  p.Nout = N;
  p.out = (__nv_bfloat16 *)out;
  p.rscale = sx;
  const int64_t upper = ((M + 127) / 128 + groups) * p.n_tiles;
  const int grid = (int)(upper < sms ? upper : sms);
  cudaStream_t s = (cudaStream_t)stream;
  if (narrow) return launch_f8i4<I4Cfg<64, 4, 4>>(ta, tb, ts, P, grid, s);
  return launch_f8i4<I4Cfg<128, 2, 3>>(ta, tb, ts, P, grid, s);
}
