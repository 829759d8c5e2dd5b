// mgemm_fwd_fp8_sparse: the sparse-M FP8 forward in one launch -- the group
// sizes scanned, the token rows cast rowwise to e4m3 and the grouped GEMM
// ("F8I4 Grouped Gemm Optimization for Sparse M", FBGEMM PR #3854, Summary:
// problems only for the min(total_M, groups) non-empty groups; "[moe
// training] Optimize FP8 MoE backward pass", commit message: the fused rowwise
// scale + cast).  It computes what mgemm_fill_args + mgemm_quant_rowwise +
// mgemm_fwd (dtype MGEMM_FP8_E4M3, w [E, N, K]) compute, for at most 16 token
// rows, where those three launches cost more than the weights' stream.
//
// Orientation: a tcgen05.mma costs about the same time for every shape up to
// M = 128, N = 128 (K = 32 for e4m3), so the weights take the MMA's 128-row
// side (4 KB of weights per instruction) and the few token rows its N side
// (N = 16).  With the tokens on the 128-row side, as in mgemm_fwd, an
// instruction consumes only N x 32 bytes of weights and the tensor pipe, not
// HBM, bounds the stream.
//
// Work split: a tile is one non-empty group x tw weight rows (output
// columns) x all of K, cut into stages of KC contraction blocks.  The CTAs
// (persistent, one per SM) take equal contiguous ranges of tiles, and
// consecutive tiles mostly share their group, so a CTA writes a group's token
// codes once for the whole run of them.  The host picks tw (96 to 128) so
// that the tiles divide evenly over the SMs.  When 128-row tiles number at
// most half the SMs (one token: one expert's 64 tiles), CTA pairs (clusters
// of two) take them instead, each CTA one half of the contraction, so that
// every SM streams weights: the second CTA hands its fp32 partial sums to the
// first through the first's shared memory, and the first adds them to its
// own before the epilogue.  Without pairs every output equals mgemm_fwd's bit
// for bit; with them it differs by the rounding of that one addition.
//
// CTA roles (320 threads):
//   all         at launch, the token rows are read and their magnitude maxima
//               reduced (all rows when they fit one register batch, else the
//               first group's) while every CTA scans the E group sizes in
//               shared memory (the active groups, their first rows and sizes;
//               validation)
//   warp 0      TMA producer: the weights only, KC contraction blocks of
//               128 rows x 128 B per stage, as many stages as fit; its first
//               copy waits until the first group's token loads are out
//   warp 1      TMEM owner; one thread issues the MMAs: kind::f8f6f4, M = 128
//               (weight rows), N = 16 (token rows), K = 32; two accumulators
//   warps 2-9   at a change of group, the group's token rows cast to e4m3 with
//               their power-of-two scale into a resident B region laid out as
//               the MMA reads it (K / 128 chunks of a_rows x 128 B, 128-byte
//               swizzle), once the MMAs before are done; the next group's row
//               maxima are read while the current tile's MMAs run
//   warps 4-7   the previous tile's epilogue, one TMEM lane quarter each:
//               lane = output column, TMEM column = token row; in a pair's
//               second CTA, the partial sums into the first's shared memory;
//               else (the partner's partial added first) times 1 / sx[row] and
//               1 / sw[e, column] in mgemm_fwd's order, bf16, direct stores.
// Every wait is bounded; on expiry the kernel raises *status to
// MGEMM_STATUS_TIMEOUT, drains the copies and MMAs it issued, frees TMEM and
// returns.
#include "gemm_launch.cuh"

namespace mgemm {
namespace {

constexpr int kSpBw = 128;       // the MMA's M: weight rows (output columns) per tile at most
constexpr int kSpTn = 16;        // the MMA's N: token rows (a group has at most 16)
constexpr int kSpMaxRows = 16;   // token rows of the whole call at most
constexpr int kSpThreads = 320;
constexpr int kSpMaxStages = 12;
constexpr int kSpKeep = 8;       // 16-byte units per cast thread held in registers
constexpr int kSpRecvBytes = kSpBw * kSpTn * 4;  // a pair's partial sums: 128 rows x 16 fp32

struct SpParams {
  const int64_t *sizes;
  int E;
  int M;
  int K, N;
  int a_rows;     // token rows rounded up to 8 (the B region's rows per chunk)
  int tw;         // weight rows per tile (a multiple of 8, at most 128), chosen to balance the SMs
  int stages;
  int n_tiles;    // ceil(N / tw)
  const __nv_bfloat16 *x;
  int64_t ld_x;
  const float *sw;
  __nv_bfloat16 *out;
  int *status;
  uint32_t idesc;
};

struct SpShared {
  int act_e[kSpMaxRows], act_row[kSpMaxRows], act_m[kSpMaxRows];
  int n_active, bad;
  long long warp_tot[kSpThreads / 32];
  int warp_cnt[kSpThreads / 32];
  unsigned amax_bits[kSpMaxRows];  // magnitude maximum of every token row (bits of a float >= 0)
  float rinv[kSpMaxRows];          // row-scale reciprocal of every token row
  uint64_t full[kSpMaxStages], empty[kSpMaxStages], a_full, a_empty, tfull[2], tempty[2], drain, x_go;
  uint64_t part_full, part_empty;  // pairs: the partner's partial is in recv / recv may be rewritten
  uint32_t tmem_slot;
  int abort_flag;
};

// Named barrier 1 over the 256 threads of warps 2-9; returns the OR of v over
// them, so every participant takes the same branch after it.
__device__ __forceinline__ bool bar1_256_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, o;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred o, 1, 256, q;\n\tselp.u32 %0, 1, 0, o;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bar1_256() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// KC: contraction blocks of 128 per stage (a stage is KC x 16 KB of weights);
// PAIR: clusters of two CTAs, each one half of the contraction of every tile.
template <int KC, bool PAIR>
__global__ void __launch_bounds__(kSpThreads, 1)
    sparse_fp8_kernel(const __grid_constant__ CUtensorMap tmW, const SpParams p) {
  const int chunk_bytes = p.tw * 128;  // one contraction block of the tile's weight rows
  const int stage_bytes = KC * chunk_bytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kchunks = p.K / 128;
  uint8_t *sT = smem;                                                  // token codes [kchunks][a_rows][128 B]
  uint8_t *sW = sT + (size_t)kchunks * p.a_rows * 128;                 // ring of weight stages
  // (the MMA reads 128 rows from a block's start; past a tile of tw rows, the next block's or the
  // following bytes, inside the allocation, feed accumulator lanes that are never read)
  SpShared &S = *reinterpret_cast<SpShared *>(sW + (size_t)p.stages * stage_bytes);
  // pairs: the partner's partial sums, [128 rows][16] fp32 (after SpShared, 16-byte aligned)
  float *recv = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(&S + 1) + 15) & ~uintptr_t(15));
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nst = p.stages;
  const int ct = (int)threadIdx.x - 64;  // cast thread 0 .. 255
  const int upr = p.K >> 3;              // 16-byte units (8 elements) per token row
  const int U_all = p.M * upr;           // unit u: row u / upr, elements 8 (u % upr) .. + 7
  // all rows' units fit one register batch: they are read before the scan, all rows' scales at once
  const bool all_rows = U_all <= 256 * kSpKeep;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.a_full, 8);
    mbar_init(&S.a_empty, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&S.tfull[a], 1);
      mbar_init(&S.tempty[a], 4);
    }
    mbar_init(&S.drain, 1);
    mbar_init(&S.x_go, 8);
    mbar_init(&S.part_full, 128);
    mbar_init(&S.part_empty, 128);
    S.abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
  }
  if (threadIdx.x < kSpMaxRows) S.amax_bits[threadIdx.x] = 0u;
  if (warp == 1) {
    tmem_alloc(&S.tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the partner's barriers are initialised before any arrival on them
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_slot;
  pdl_wait();
  pdl_trigger();

  // A cast thread's units: u = base + 256 j + ct (j < kSpKeep), loaded where lo <= u < hi.
  auto load_units = [&](int base, uint4(&v)[kSpKeep], int lo, int hi) {
#pragma unroll
    for (int j = 0; j < kSpKeep; ++j) {
      const int u = base + j * 256 + ct;
      if (u >= lo && u < hi) {
        const int r = u / upr;
        v[j] = ldg_nc_v4(p.x + (int64_t)r * p.ld_x + (int64_t)(u - r * upr) * 8);
      } else {
        v[j] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  uint4 keep[kSpKeep];  // the current batch of units, kept between the maxima and the codes
  int keep_base = 0;
  if (warp >= 2 && all_rows) load_units(0, keep, 0, U_all);  // in flight during the scan

  // ---- scan of the group sizes: thread t holds experts 4t .. 4t + 3
  {
    int64_t m[4];
    int cnt = 0, neg = 0;
    long long sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * threadIdx.x + i;
      m[i] = e < p.E ? p.sizes[e] : 0;
      cnt += m[i] != 0;
      neg |= m[i] < 0;
      sum += m[i];
    }
    // inclusive scans of the counts and sums over the block (warp shuffles, then warp totals)
    int ci = cnt;
    long long si = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int cn = __shfl_up_sync(0xffffffffu, ci, o);
      const long long sn = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) {
        ci += cn;
        si += sn;
      }
    }
    if (lane == 31) {
      S.warp_cnt[warp] = ci;
      S.warp_tot[warp] = si;
    }
    const int any_neg = __syncthreads_or(neg);
    int cbase = 0;
    long long sbase = 0;
    for (int w = 0; w < warp; ++w) {
      cbase += S.warp_cnt[w];
      sbase += S.warp_tot[w];
    }
    int c_ex = cbase + ci - cnt;        // active groups before this thread's experts
    long long s_ex = sbase + si - sum;  // rows before them
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (m[i] > 0) {
        if (c_ex < kSpMaxRows) {
          S.act_e[c_ex] = 4 * threadIdx.x + i;
          S.act_row[c_ex] = (int)s_ex;
          S.act_m[c_ex] = (int)m[i];
        }
        ++c_ex;
      }
      s_ex += m[i];
    }
    if (threadIdx.x == kSpThreads - 1) {
      long long total = 0;
      int n = 0;
      for (int w = 0; w < kSpThreads / 32; ++w) {
        total += S.warp_tot[w];
        n += S.warp_cnt[w];
      }
      S.n_active = n;
      S.bad = any_neg ? MGEMM_STATUS_NEGATIVE_SIZE : (total != p.M ? MGEMM_STATUS_SUM_MISMATCH : 0);
    }
    __syncthreads();
    // the status only rises (0 < validation codes < timeout), so this write and a timeout
    // recorded by another CTA give the same result in either order
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicMax(p.status, S.bad);
  }
  const int kbc = (kchunks + KC - 1) / KC;  // stages per tile
  const int total = S.bad ? 0 : S.n_active * p.n_tiles;
  // this CTA's (or pair's) tiles: [t_lo, t_hi), an even split in order; its stages [kb_lo, kb_hi)
  const int slot = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int nslot = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  // (32-bit arithmetic while total x grid stays below 2^31: a 64-bit division costs ~0.2 us here)
  auto split = [&](int b) {
    return total < (1 << 20) ? (int)((unsigned)total * (unsigned)b / (unsigned)nslot)
                             : (int)((long long)total * b / nslot);
  };
  const int t_lo = split(slot), t_hi = split(slot + 1);
  const int kb_half = (kbc + 1) / 2;
  const int kb_lo = PAIR && rank == 1 ? kb_half : 0, kb_hi = PAIR && rank == 0 ? kb_half : kbc;
  // the group (active index) of a tile; the codes are (re)written when it changes
  auto group_of = [&](int t) { return t / p.n_tiles; };
  auto fresh_at = [&](int t) { return t == t_lo || group_of(t) != group_of(t - 1); };
  volatile int *vabort = &S.abort_flag;
  uint32_t issued = 0;
  auto timeout = [&]() {
    atomicMax(p.status, MGEMM_STATUS_TIMEOUT);
    *vabort = 1;
  };

  if (warp == 0) {
    if (lane == 0 && t_lo < t_hi) {
      // the first token loads go out ahead of the weight stream (with all rows in one batch they
      // were issued before the scan)
      bool ok = all_rows || mbar_wait(&S.x_go, 0, vabort);
      if (!ok) timeout();
      int stage = 0;
      uint32_t phase = 0;
      for (int t = t_lo; t < t_hi && ok && !*vabort; ++t) {
        const int a = group_of(t), n0 = (t % p.n_tiles) * p.tw, e = S.act_e[a];
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(&S.empty[stage], phase ^ 1, vabort)) {
            timeout();
            break;
          }
          mbar_arrive_expect_tx(&S.full[stage], (uint32_t)stage_bytes);
          ++issued;
          tma_load_4d(sW + (size_t)stage * stage_bytes, &tmW, &S.full[stage], 0, n0, kb * KC, e);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // one thread issues every MMA (no warp-wide vote per stage)
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0, a_phase = 0;
      bool ok = true;
      const uint32_t idesc = p.idesc;
      for (int t = t_lo; t < t_hi && ok; ++t) {
        // the token codes change only with the group (they are complete when a_full flips)
        const bool fresh = fresh_at(t);
        if (!mbar_wait(&S.tempty[acc], acc_phase ^ 1, vabort) || (fresh && !mbar_wait(&S.a_full, a_phase, vabort))) {
          ok = false;
          break;
        }
        if (fresh) a_phase ^= 1;
        const uint32_t d_tmem = tmem_base + acc * kSpTn;
        const uint64_t t_desc = smem_desc_sw128(smem_u32(sT), 16, 1024);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(&S.full[stage], phase, vabort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t w_desc = smem_desc_sw128(smem_u32(sW + (size_t)stage * stage_bytes), 16, 1024);
#pragma unroll
          for (int j = 0; j < KC; ++j) {
            const int chunk = kb * KC + j;
            if (chunk >= kchunks) break;  // past K: no token codes there (the weight box holds zeros)
            // descriptors advance by (byte offset >> 4) in their start-address field
            const uint64_t wj = w_desc + (uint64_t)((j * chunk_bytes) >> 4);
            const uint64_t tj = t_desc + (uint64_t)(((uint32_t)chunk * p.a_rows * 128) >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_f8(d_tmem, wj + 2 * k, tj + 2 * k, idesc, (kb != kb_lo) | j | k);
          }
          mma_commit(&S.empty[stage]);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&S.tfull[acc]);
        if (t + 1 < t_hi && fresh_at(t + 1)) mma_commit(&S.a_empty);  // the codes are read and will be rewritten
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      if (!ok) timeout();
      mma_commit(&S.drain);
      mbar_wait_drain(&S.drain, 0);
    }
    __syncwarp();
  } else {
    // ---- warps 2 .. 9: token scales and codes; warps 4 .. 7 also the epilogue
    // magnitude maxima of the units base + 256 j + ct below hi, into S.amax_bits of their rows
    auto reduce_units = [&](int base, const uint4(&v)[kSpKeep], int hi) {
#pragma unroll
      for (int j = 0; j < kSpKeep; ++j) {
        if (base + j * 256 >= hi) break;  // uniform over the block
        const int u = base + j * 256 + ct;
        const int r = u < hi ? u / upr : (hi - 1) / upr;
        const unsigned bits = u < hi ? __float_as_uint(amax8(v[j], 0.f)) : 0u;
        const int r_first = __shfl_sync(0xffffffffu, r, 0);
        if (__all_sync(0xffffffffu, r == r_first)) {
          const unsigned mx = __reduce_max_sync(0xffffffffu, bits);
          if (lane == 0) atomicMax(&S.amax_bits[r_first], mx);
        } else if (bits) {
          atomicMax(&S.amax_bits[r], bits);
        }
      }
    };
    // rows [r_lo, r_hi): maxima of all their units (keep holds the first batch), then their scales.
    // Every one of the eight warps calls it at the same point (it holds a barrier).
    auto scales = [&](int r_lo, int r_hi, bool loaded) {
      const int lo = r_lo * upr, hi = r_hi * upr;
      if (!loaded) load_units(lo, keep, lo, hi);
      keep_base = lo;
      reduce_units(lo, keep, hi);
      for (int b = lo + 256 * kSpKeep; b < hi; b += 256 * kSpKeep) {
        uint4 v[kSpKeep];
        load_units(b, v, lo, hi);
        reduce_units(b, v, hi);
      }
      bar1_256();  // the rows' maxima are complete
      // S.rinv is read by the epilogue warps only after a later barrier of these warps
      if (ct < r_hi - r_lo) S.rinv[r_lo + ct] = pow2_recip(pow2_scale_from_amax(__uint_as_float(S.amax_bits[r_lo + ct])));
    };
    // codes of the units base + 256 j + ct in [lo, hi) (rows r0 ..) into the B region, rows relative to r0
    auto store_units = [&](int base, const uint4(&v)[kSpKeep], int r0, int lo, int hi) {
#pragma unroll
      for (int j = 0; j < kSpKeep; ++j) {
        const int u = base + j * 256 + ct;
        if (u >= lo && u < hi) {
          const int r = u / upr, c = (u - r * upr) * 8, i = r - r0;  // 8 code bytes at column c of row i
          const float sc = pow2_scale_from_amax(__uint_as_float(S.amax_bits[r]));
          const int chunk = c >> 7, b = c & 127;
          uint8_t *dst = sT + ((size_t)chunk * p.a_rows + i) * 128 + ((((b >> 4) ^ (i & 7)) << 4) | (b & 15));
          *reinterpret_cast<uint2 *>(dst) = cast8(v[j], sc);
        }
      }
    };
    if (t_lo < t_hi) {
      if (all_rows) {
        if (lane == 0) mbar_arrive(&S.x_go);
        scales(0, p.M, true);
      } else {
        const int a = group_of(t_lo);
        const int lo = S.act_row[a] * upr;
        load_units(lo, keep, lo, lo + S.act_m[a] * upr);
        if (lane == 0) mbar_arrive(&S.x_go);
        scales(S.act_row[a], S.act_row[a] + S.act_m[a], true);
      }
    }
    const bool epi = warp >= 4 && warp <= 7;
    const int q = warp & 3;  // TMEM lane quarter of an epilogue warp
    uint32_t e_phase = 0, acc_phase = 0, part_phase = 0;
    int acc = 0;
    int prev_t = -1, prev_acc = 0;
    uint32_t prev_phase = 0;
    float sw_prev = 0.f;
    auto epilogue = [&](int t, int ac, uint32_t ph, float swv) -> bool {
      if (!mbar_wait_warp(&S.tfull[ac], ph, vabort)) return false;
      tc_fence_after();
      const int a = group_of(t), row = q * 32 + lane, n = (t % p.n_tiles) * p.tw + row;
      const int r0 = S.act_row[a], m = S.act_m[a];
      uint32_t v[kSpTn];
      tmem_ld_32x32b_x16(tmem_base + ((uint32_t)(q * 32) << 16) + ac * kSpTn, v);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tempty[ac]);
      if (PAIR && rank == 1) {
        // the second half's partial sums into the first CTA's recv, once it has read the last ones
        if (!mbar_wait_cluster_warp(&S.part_empty, part_phase ^ 1, vabort)) return false;
        part_phase ^= 1;
        const uint32_t dst = cluster_addr(recv + row * kSpTn, 0);
#pragma unroll
        for (int j = 0; j < kSpTn; j += 4)
          asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + j * 4), "r"(v[j]), "r"(v[j + 1]),
                       "r"(v[j + 2]), "r"(v[j + 3])
                       : "memory");
        mbar_arrive_cluster(cluster_addr(&S.part_full, 0));
        return true;
      }
      float accv[kSpTn];
#pragma unroll
      for (int j = 0; j < kSpTn; ++j) accv[j] = __uint_as_float(v[j]);
      if (PAIR) {
        // add the second half's partial sums, then hand recv back
        if (!mbar_wait_cluster_warp(&S.part_full, part_phase, vabort)) return false;
        part_phase ^= 1;
        const float4 *src = reinterpret_cast<const float4 *>(recv + row * kSpTn);
#pragma unroll
        for (int j = 0; j < kSpTn; j += 4) {
          const float4 f4 = src[j / 4];
          accv[j] += f4.x;
          accv[j + 1] += f4.y;
          accv[j + 2] += f4.z;
          accv[j + 3] += f4.w;
        }
        mbar_arrive_cluster(cluster_addr(&S.part_empty, 1));
      }
      if (row < p.tw && n < p.N) {
        const float cs = pow2_recip(swv);
        __nv_bfloat16 *o = p.out + (int64_t)r0 * p.N + n;
#pragma unroll
        for (int j = 0; j < kSpTn; ++j)
          if (j < m) o[(int64_t)j * p.N] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(accv[j], S.rinv[r0 + j]), cs));
      }
      return true;
    };
    for (int t = t_lo; t < t_hi; ++t) {
      const int a = group_of(t);
      if (fresh_at(t)) {
        const int r0 = S.act_row[a], m = S.act_m[a];
        const int lo = r0 * upr, hi = (r0 + m) * upr;
        // the codes are rewritten once the MMAs before have read them
        if (!mbar_wait_warp(&S.a_empty, e_phase ^ 1, vabort)) {
          if (lane == 0) timeout();
        } else {
          // keep holds the batch at keep_base (all rows, or this group's first batch)
          store_units(keep_base, keep, r0, lo, hi);
          for (int b = keep_base + 256 * kSpKeep; b < hi; b += 256 * kSpKeep) {
            if (b + 256 * kSpKeep <= lo) continue;  // no unit of the group in this batch
            uint4 v[kSpKeep];
            load_units(b, v, lo, hi);
            store_units(b, v, r0, lo, hi);
          }
        }
        e_phase ^= 1;
        fence_proxy_async_smem();  // the codes are read by the tensor cores
        __syncwarp();
        // the codes (and the group's row scales) are visible; leave together on an abort
        if (bar1_256_or(*vabort != 0)) break;
        if (lane == 0) mbar_arrive(&S.a_full);
      }
      // an epilogue thread's column scale for this tile, loaded ahead of its use
      float swv = 0.f;
      if (epi && !(PAIR && rank == 1)) {
        const int row = q * 32 + lane, n = (t % p.n_tiles) * p.tw + row;
        if (row < p.tw && n < p.N) swv = __ldg(p.sw + (int64_t)S.act_e[a] * p.N + n);
      }
      if (epi && prev_t >= 0 && !epilogue(prev_t, prev_acc, prev_phase, sw_prev) && lane == 0) timeout();
      // the next group's scales while this tile's MMAs run
      if (!all_rows && t + 1 < t_hi && fresh_at(t + 1)) {
        const int an = group_of(t + 1);
        scales(S.act_row[an], S.act_row[an] + S.act_m[an], false);
      }
      prev_t = t;
      prev_acc = acc;
      prev_phase = acc_phase;
      sw_prev = swv;
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (epi && !*vabort && prev_t >= 0 && !epilogue(prev_t, prev_acc, prev_phase, sw_prev) && lane == 0) timeout();
  }

  tc_fence_before();
  __syncthreads();
  if (*vabort && warp == 0 && lane == 0) {
    for (int s = 0; s < nst; ++s) {
      const uint32_t armed = issued / nst + ((uint32_t)s < issued % nst ? 1u : 0u);
      if (armed) mbar_wait_drain(&S.full[s], (armed - 1) & 1);
    }
  }
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA of a pair leaves while the other may still reach its shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace
}  // namespace mgemm

using namespace mgemm;

extern "C" int mgemm_fwd_fp8_sparse(const int64_t *group_sizes, int E, const void *x, int64_t ld_x, const void *w,
                                    const float *sw, void *out, int *status, int64_t M, int K, int N,
                                    mgemm_stream_t stream) {
  if (!group_sizes || !x || !w || !sw || !out || !status) return MGEMM_EINVAL;
  if (E < 1 || E > kSpThreads * 4) return E < 1 ? MGEMM_EINVAL : MGEMM_ETOOMANY;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 1 || M > kSpMaxRows || K <= 0 || N <= 0 || ld_x < K) return MGEMM_EINVAL;
  if ((int64_t)E * N >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (K % 128 || N % 8 || ld_x % 8) return MGEMM_EALIGN;
  if (((uintptr_t)group_sizes & 7) || ((uintptr_t)x & 15) || ((uintptr_t)w & 15) || ((uintptr_t)sw & 3) ||
      ((uintptr_t)out & 15) || ((uintptr_t)status & 3))
    return MGEMM_EALIGN;
  int rc = ensure_context();
  if (rc) return rc;
  const int a_rows = (int)((M + 7) / 8 * 8);
  const size_t a_bytes = (size_t)K * a_rows;
  const int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  const int64_t groups_max = M < E ? M : E;  // non-empty groups at most
  const size_t limit = (size_t)227 * 1024;
  // Weight rows per tile: CTA pairs take 128-row tiles when 128-row tiles cover at most half of
  // the SMs (one token); else the tile height (a multiple of 8 from 96 to 128) that minimizes the
  // weight rows of the busiest CTA when the tiles of groups_max groups are split evenly over the
  // SMs.  (Below 96 rows the MMA, which takes 128 rows per instruction whatever the tile holds,
  // would consume the weights slower than an SM's share of HBM.)
  const int64_t tiles128 = groups_max * ((N + kSpBw - 1) / kSpBw);
  bool pair = 2 * tiles128 <= sms;
  int tw = kSpBw;
  if (!pair) {
    int64_t best = -1;
    for (int h = kSpBw; h >= 96; h -= 8) {
      const int64_t nt = (N + h - 1) / h, per_cta = (groups_max * nt + sms - 1) / sms * h;
      if (best < 0 || per_cta < best) {
        best = per_cta;
        tw = h;
      }
    }
  }
  const int n_tiles = (N + tw - 1) / tw;
  const int64_t tiles_max = groups_max * (int64_t)n_tiles;
  const size_t chunk_bytes = (size_t)tw * 128;
  // past the ring: SpShared, the pair's partial sums, and the MMA's read of 128 rows from a
  // block's start beyond a tile of fewer rows
  auto fixed_bytes = [&](bool pr) {
    return 1024 + a_bytes + sizeof(SpShared) + 16 + (pr ? kSpRecvBytes : 0) + (size_t)(kSpBw - tw) * 128 + 64;
  };
  // stages of 4 blocks (16 MMAs between waits) while three of them fit, else of 2
  auto stage_chunks = [&](size_t fx) { return fx + 3 * 4 * chunk_bytes <= limit ? 4 : 2; };
  // pairs need the partial-sum buffer to fit and two stages per tile
  if (pair) pair = fixed_bytes(true) + 4 * chunk_bytes <= limit;
  if (pair) {
    const int kc_pair = stage_chunks(fixed_bytes(true));
    pair = (K / 128 + kc_pair - 1) / kc_pair >= 2;
  }
  const size_t fixed = fixed_bytes(pair);
  if (fixed + 4 * chunk_bytes > limit) return MGEMM_EINVAL;  // the token rows do not fit on chip
  const int kc = stage_chunks(fixed);
  const size_t stage_bytes = (size_t)kc * chunk_bytes;
  int stages = (int)((limit - fixed) / stage_bytes);
  if (stages > kSpMaxStages) stages = kSpMaxStages;
  CUtensorMap tmap;
  {  // w [E, N, K] e4m3 as 128-byte k-chunks: {128, N, K / 128, E}, boxes of kc chunks of 128 rows
    const uint64_t d[4] = {128, (uint64_t)N, (uint64_t)K / 128, (uint64_t)E};
    const uint64_t st[3] = {(uint64_t)K, 128, (uint64_t)N * K};
    const uint32_t box[4] = {128, (uint32_t)tw, (uint32_t)kc, 1};
    if (!make_tensor_map(&tmap, true, 4, w, d, st, box)) return MGEMM_ECUDA;
  }
  SpParams p{};
  p.sizes = group_sizes;
  p.E = E;
  p.M = (int)M;
  p.K = K;
  p.N = N;
  p.a_rows = a_rows;
  p.stages = stages;
  p.n_tiles = n_tiles;
  p.tw = tw;
  p.x = (const __nv_bfloat16 *)x;
  p.ld_x = ld_x;
  p.sw = sw;
  p.out = (__nv_bfloat16 *)out;
  p.status = status;
  p.idesc = make_idesc(0u, false, false, kSpBw, kSpTn);
  const int grid = pair ? (int)(2 * tiles_max) : (int)(tiles_max < sms ? tiles_max : sms);
  const size_t smem = fixed + (size_t)stages * stage_bytes;
  static bool attr_done[64] = {};
  int dev = 0;
  rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return MGEMM_EINVAL;
  if (!attr_done[dev]) {
    const void *fns[4] = {(const void *)sparse_fp8_kernel<2, false>, (const void *)sparse_fp8_kernel<4, false>,
                          (const void *)sparse_fp8_kernel<2, true>, (const void *)sparse_fp8_kernel<4, true>};
    for (const void *f : fns) {
      rc = cuda_rc(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit),
                   "cudaFuncSetAttribute");
      if (rc) return rc;
    }
    attr_done[dev] = true;
  }
  const cudaStream_t st = (cudaStream_t)stream;
  const char *what = pair ? "sparse FP8 forward launch (CTA pairs)" : "sparse FP8 forward launch";
  if (pair)
    return kc == 4 ? launch_pdl(sparse_fp8_kernel<4, true>, dim3((unsigned)grid), dim3(kSpThreads), smem, st, 2u, what, tmap, p)
                   : launch_pdl(sparse_fp8_kernel<2, true>, dim3((unsigned)grid), dim3(kSpThreads), smem, st, 2u, what, tmap, p);
  return kc == 4 ? launch_pdl(sparse_fp8_kernel<4, false>, dim3((unsigned)grid), dim3(kSpThreads), smem, st, 1u, what, tmap, p)
                 : launch_pdl(sparse_fp8_kernel<2, false>, dim3((unsigned)grid), dim3(kSpThreads), smem, st, 1u, what, tmap, p);
}
