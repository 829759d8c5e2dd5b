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
// BN (64, 128 or 256) is chosen per launch on the host to balance the tile
// count against the number of SMs.
//
// CTA layout (192 threads, one CTA per SM, grid = number of SMs, tiles
// strided by gridDim.x):
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
//   warps 2-5   epilogue, one TMEM lane quarter (32 output rows) each:
//               tcgen05.ld, optional FP8 scale division, bf16 rounding, then
//               128-byte-swizzled shared-memory staging buffers (2 per warp,
//               4 for wgrad, whose short main loops leave the stores as the
//               critical path) and a TMA store of each 32-row x 64-column block.  A
//               warp whose 32 rows are not all valid (group edge) stores
//               those rows directly instead, so nothing outside the tile's
//               rows is ever written.  The accumulator is released right
//               after its last tcgen05.ld, so the next tile's main loop
//               overlaps the stores.
// Every mbarrier wait is bounded (about 1 s); on expiry the kernel records
// MGEMM_STATUS_TIMEOUT in the args block, lets the other roles leave their
// loops, drains its own outstanding copies and MMAs, frees TMEM and returns.
#pragma once

#include "common.cuh"

namespace mgemm {

enum { kModeRows = 0, kModeExperts = 1 };

// kBnMax / kStages: the widest output tile this instantiation serves and its
// ring depth.  Wide (256, 4 stages), mid (128, 6) and narrow (64, 8) forms
// fill the same shared memory; the narrower forms serve weight-streaming
// launches, where a deeper ring keeps more HBM reads in flight per SM.
template <bool kFp8, bool kAMn, bool kBMn, int kMode, int kBnMax = 256, int kStages = 4, int kOutBufs = 2>
struct GemmCfg {
  static constexpr bool Fp8 = kFp8;
  static constexpr bool AMn = kAMn;  // A stored MN-major (contraction is the strided dim)
  static constexpr bool BMn = kBMn;
  static constexpr int Mode = kMode;
  static constexpr int BM = 128, BN_MAX = kBnMax;
  static constexpr int ESIZE = kFp8 ? 1 : 2;
  static constexpr int BK = 128 / ESIZE;  // contraction elements per stage (one 128-byte row)
  static constexpr int UK = 32 / ESIZE;   // contraction elements per MMA
  static constexpr int KSTEPS = BK / UK;  // 4
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN_MAX * 128;
  static constexpr int STAGES = kStages;
  static constexpr int CHUNK = 64 * 128;  // MN-major: one 64-element x BK-row block (8 KB)
  static constexpr int TMEM_COLS = 2 * BN_MAX;  // a power of two >= 32
  static constexpr int THREADS = 192;
  static constexpr int OUT_BUF = 32 * 128;  // 32 rows x 64 bf16 columns
  static constexpr int NBUF = kOutBufs;      // staging buffers per epilogue warp
  static constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)STAGES * (A_BYTES + B_BYTES) +
                                       4 * NBUF * OUT_BUF /*epilogue staging*/ + 4 * 64 * 4 /*column scales*/ +
                                       256 /*barriers, flags*/;
};

struct GemmParams {
  const uint8_t *args;
  int E;
  int bn;           // output tile width: 64, 128 or 256
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
};

struct TileInfo {
  int e, kb_count, a_row, n0, x0, lo, hi, out_row0, out_rows;
};

template <class C>
__device__ __forceinline__ int total_tiles(const GemmParams &p, const ArgsView &av) {
  if (C::Mode == kModeRows) {
    const int na = *av.n_active;
    return av.mtile_start[na] * p.n_tiles;
  }
  return p.E * p.mt_k * p.n_tiles;
}

template <class C>
__device__ __forceinline__ TileInfo decode_tile(int t, const GemmParams &p, const ArgsView &av) {
  TileInfo ti;
  if (C::Mode == kModeRows) {
    // Group a owns tiles [mtile_start[a] * n_tiles, mtile_start[a+1] * n_tiles).
    // Inside a group the row tile varies fastest, so CTAs running together
    // share one weight tile through L2 instead of each streaming its own.
    const int gm = t / p.n_tiles;
    int lo = 0, hi = *av.n_active - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(av.mtile_start + mid) <= gm) lo = mid; else hi = mid - 1;
    }
    ti.e = __ldg(av.active + lo);
    const int m_first = __ldg(av.mtile_start + lo);
    const int mt_g = __ldg(av.mtile_start + lo + 1) - m_first;
    const int local = t - m_first * p.n_tiles;
    const int mt = local % mt_g;
    ti.n0 = (local / mt_g) * p.bn;
    const int64_t rs = __ldg(av.offsets + ti.e), re = __ldg(av.offsets + ti.e + 1);
    const int row0 = (int)rs + mt * C::BM;
    ti.kb_count = (p.Kc + C::BK - 1) / C::BK;
    ti.a_row = row0;
    ti.out_row0 = row0;
    ti.out_rows = (int)min((int64_t)C::BM, re - row0);
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
    ti.a_row = mk * C::BM;
    ti.out_row0 = ti.e * p.Kout + mk * C::BM;
    ti.out_rows = min(C::BM, p.Kout - mk * C::BM);
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

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    mgemm_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmOut, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::STAGES * C::A_BYTES;
  uint8_t *sOut = sB + C::STAGES * C::B_BYTES;  // [4 warps][NBUF buffers][32 x 128 B]
  float *s_csc = reinterpret_cast<float *>(sOut + 4 * C::NBUF * C::OUT_BUF);  // [4 warps][64]
  uint64_t *full = reinterpret_cast<uint64_t *>(s_csc + 4 * 64);
  uint64_t *empty = full + C::STAGES;
  uint64_t *tfull = empty + C::STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ArgsView av(p.args, p.E);
  if (*av.status != 0) return;
  const int total = total_tiles<C>(p, av);
  if ((int)blockIdx.x >= total) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmOut);
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
  const int bn = p.bn;

  // Producer bookkeeping kept for the drain after an abort.
  uint32_t issued = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      // with fewer than 128 token rows the A box is cut to them (rounded up to 8);
      // the MMA's remaining A rows hold stale data and only feed output rows
      // that are never stored
      const uint32_t tx = (C::Mode == kModeRows ? p.a_rows * 128 : C::A_BYTES) + bn * 128;
      for (int t = blockIdx.x; t < total && !*vabort; t += gridDim.x) {
        const TileInfo ti = decode_tile<C>(t, p, av);
        for (int kb = 0; kb < ti.kb_count; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, vabort)) {
            set_status(av.status, MGEMM_STATUS_TIMEOUT);
            *vabort = 1;
            break;
          }
          uint8_t *a = sA + stage * C::A_BYTES;
          uint8_t *b = sB + stage * C::B_BYTES;
          mbar_arrive_expect_tx(&full[stage], tx);
          ++issued;
          if (C::Mode == kModeRows) {
            tma_load_2d(a, &tmA, &full[stage], kb * C::BK, ti.a_row);
            if (C::BMn) {
              for (int j = 0; j < bn / 64; ++j)
                tma_load_3d(b + j * C::CHUNK, &tmB, &full[stage], ti.n0 + 64 * j, kb * C::BK, ti.e);
            } else {
              tma_load_3d(b, &tmB, &full[stage], kb * C::BK, ti.n0, ti.e);
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
          if (++stage == C::STAGES) {
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
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<C>(t, p, av);
      if (ti.kb_count == 0) continue;
      if (!mbar_wait_warp(&tempty[acc], acc_phase ^ 1, vabort)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * C::BN_MAX;
      for (int kb = 0; kb < ti.kb_count; ++kb) {
        if (!mbar_wait_warp(&full[stage], phase, vabort)) { ok = false; break; }
        tc_fence_after();
        uint8_t *a = sA + stage * C::A_BYTES;
        uint8_t *b = sB + stage * C::B_BYTES;
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
        if (lane == 0) {
          const uint32_t abase = smem_u32(a), bbase = smem_u32(b);
          if (!edge) {
#pragma unroll
            for (int k = 0; k < C::KSTEPS; ++k) {
              const uint64_t ad = C::AMn ? smem_desc_sw128(abase + k * C::UK * 128, C::CHUNK, 1024)
                                         : smem_desc_sw128(abase + k * 32, 16, 1024);
              const uint64_t bd = C::BMn ? smem_desc_sw128(bbase + k * C::UK * 128, C::CHUNK, 1024)
                                         : smem_desc_sw128(bbase + k * 32, 16, 1024);
              // the tile's first MMA overwrites the accumulator
              if (C::Fp8)
                mma_f8(d_tmem, ad, bd, p.idesc, (kb | k) != 0);
              else
                mma_f16(d_tmem, ad, bd, p.idesc, (kb | k) != 0);
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
          mma_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&tfull[acc]);
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (!ok) {
      if (lane == 0) set_status(av.status, MGEMM_STATUS_TIMEOUT);
      *vabort = 1;
    }
    // all MMAs this thread issued have completed before TMEM is released
    if (lane == 0) {
      mma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
    __syncwarp();
  } else {
    // epilogue warps 2..5 -> TMEM lane quarter q = warp % 4 -> tile rows 32q..32q+31
    const int q = warp & 3;
    const int r = q * 32 + lane;
    uint8_t *my_buf = sOut + (size_t)q * C::NBUF * C::OUT_BUF;
    uint32_t nstored = 0;  // TMA-stored chunks so far; buffers rotate with it
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile<C>(t, p, av);
      const bool has_acc = ti.kb_count > 0;
      const bool row_ok = r < ti.out_rows;
      const bool warp_full = q * 32 + 32 <= ti.out_rows;
      __nv_bfloat16 *orow = p.out + (int64_t)(ti.out_row0 + r) * p.Nout;
      float rinv = 1.f;
      if (C::Fp8 && row_ok && has_acc) rinv = pow2_recip(__ldg(p.rscale + ti.out_row0 + r));
      // FP8: this tile's column-scale reciprocals, fetched before the accumulator
      // wait so no global load sits between a TMEM read and its stores; lane l
      // holds columns n0 + 32 i + l (scales are powers of two: exact reciprocals)
      float csr[C::BN_MAX / 32];
      if (C::Fp8) {
#pragma unroll
        for (int i = 0; i < C::BN_MAX / 32; ++i) {
          const int col = ti.n0 + 32 * i + lane;
          csr[i] = has_acc && 32 * i < bn && col < p.Nout ? pow2_recip(__ldg(p.cscale + (int64_t)ti.e * p.Nout + col))
                                                          : 0.f;
        }
      }
      if (has_acc) {
        if (!mbar_wait_warp(&tfull[acc], acc_phase, vabort)) {
          set_status(av.status, MGEMM_STATUS_TIMEOUT);
          *vabort = 1;
          break;
        }
        tc_fence_after();
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * C::BN_MAX;
      const int nchunks = bn / 64;
      // TMEM -> registers runs one chunk ahead: chunk c + 1 is loading while
      // chunk c is converted and stored (the loop is unrolled so both register
      // sets keep fixed names)
      uint32_t va[2][32], vb[2][32];
      if (has_acc) {
        tmem_ld_32x32b_x32(taddr, va[0]);
        tmem_ld_32x32b_x32(taddr + 32, vb[0]);
      }
#pragma unroll
      for (int c = 0; c < C::BN_MAX / 64; ++c) {
        if (c >= nchunks) break;
        const int cur = c & 1;
        const int col0 = ti.n0 + c * 64;
        uint32_t pk[32];
        if (has_acc) {
          tmem_ld_wait();
          if (c + 1 < nchunks) {
            tmem_ld_32x32b_x32(taddr + (c + 1) * 64, va[cur ^ 1]);
            tmem_ld_32x32b_x32(taddr + (c + 1) * 64 + 32, vb[cur ^ 1]);
          } else {  // accumulator fully read: hand it back to the MMA warp
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
          }
          if (C::Fp8) {
            // this chunk's column-scale reciprocals, staged per warp and read as broadcasts
            float *cs = s_csc + q * 64;
            cs[lane] = csr[2 * c];
            cs[lane + 32] = csr[2 * c + 1];
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 c0 = *reinterpret_cast<const float4 *>(cs + 4 * j);
              const float4 c1 = *reinterpret_cast<const float4 *>(cs + 32 + 4 * j);
              pk[2 * j] = pack_bf16x2(__uint_as_float(va[cur][4 * j]) * rinv * c0.x,
                                      __uint_as_float(va[cur][4 * j + 1]) * rinv * c0.y);
              pk[2 * j + 1] = pack_bf16x2(__uint_as_float(va[cur][4 * j + 2]) * rinv * c0.z,
                                          __uint_as_float(va[cur][4 * j + 3]) * rinv * c0.w);
              pk[16 + 2 * j] = pack_bf16x2(__uint_as_float(vb[cur][4 * j]) * rinv * c1.x,
                                           __uint_as_float(vb[cur][4 * j + 1]) * rinv * c1.y);
              pk[16 + 2 * j + 1] = pack_bf16x2(__uint_as_float(vb[cur][4 * j + 2]) * rinv * c1.z,
                                               __uint_as_float(vb[cur][4 * j + 3]) * rinv * c1.w);
            }
            __syncwarp();
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
          // one store group per chunk, committed in rotation order: the group
          // that last read this buffer is NBUF groups back
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
      if (has_acc && ++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // teardown: every role has left its loop
  tc_fence_before();
  __syncthreads();
  if (*vabort && warp == 0 && lane == 0) {
    // wait for the TMA copies this CTA issued, bounded
    for (int s = 0; s < C::STAGES; ++s) {
      const uint32_t armed = issued / C::STAGES + ((uint32_t)s < issued % C::STAGES ? 1u : 0u);
      if (armed) mbar_wait(&full[s], (armed - 1) & 1, nullptr);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace mgemm
