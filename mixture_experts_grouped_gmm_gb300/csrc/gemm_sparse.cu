// mgemm_fwd_fp8_sparse: the sparse-M FP8 forward in one launch -- the group
// sizes scanned, the token rows cast rowwise to e4m3 and the grouped GEMM
// ("F8I4 Grouped Gemm Optimization for Sparse M", FBGEMM PR #3854, Summary:
// problems only for the min(total_M, groups) non-empty groups; "[moe
// training] Optimize FP8 MoE backward pass", commit message: the fused rowwise
// scale + cast).  It computes what mgemm_fill_args + mgemm_quant_rowwise +
// mgemm_fwd (dtype MGEMM_FP8_E4M3, w [E, N, K]) compute, for at most 16 token
// rows, where those three launches cost more than the weights' stream.
//
// CTA (persistent, one per SM, 320 threads), each on a contiguous range of
// tiles; a tile is one non-empty group (every group has fewer than 128 rows,
// so one row tile) x 64 weight rows, and consecutive tiles share their group,
// so a CTA casts a group's rows once for the whole run of its tiles:
//   all         scan of the E group sizes in shared memory (every CTA: the
//               active groups, their first rows and sizes; validation)
//   warp 0      TMA producer: the weights only, KC = 4 contraction blocks of
//               64 rows x 128 B per stage, as many stages as fit; it starts as
//               soon as the scan is done (the weights do not depend on x)
//   warp 1      TMEM owner and MMA issuer: kind::f8f6f4, M = 128 (the token
//               rows of the group, the rest unused), N = 64, K = 32
//   warps 2-9   per tile: on a change of group, the group's token rows cast
//               to e4m3 with their power-of-two scale by all 256 threads: the
//               rows' 16-byte units are loaded and their magnitude maxima
//               reduced while the MMAs of the tile before still run, and the
//               codes are written once those MMAs are done, straight into a
//               resident A region laid out as the MMA reads it (K / 128 chunks
//               of a_rows x 128 B, 128-byte swizzle); then the previous tile's
//               epilogue: TMEM -> registers, times
//               1 / sx[row] and 1 / sw[e, column] (the same packed-multiply
//               order as mgemm_fwd's FP8 epilogue), bf16, direct stores.
// Every wait is bounded; on expiry the kernel records MGEMM_STATUS_TIMEOUT in
// *status, drains the copies and MMAs it issued, frees TMEM and returns.
#include "gemm_launch.cuh"

namespace mgemm {
namespace {

constexpr int kSpBn = 64;        // weight rows (output columns) per tile
constexpr int kSpKc = 4;         // contraction blocks of 128 per stage
constexpr int kSpMaxRows = 16;   // token rows of the whole call at most
constexpr int kSpThreads = 320;
constexpr int kSpStageBytes = kSpKc * kSpBn * 128;
constexpr int kSpMaxStages = 12;
constexpr int kSpKeep = 8;       // 16-byte units per cast thread held in registers between the two passes

struct SpParams {
  const int64_t *sizes;
  int E;
  int M;
  int K, N;
  int a_rows;     // token rows rounded up to 8 (the A region's rows)
  int stages;
  int n_tiles;    // ceil(N / 64)
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
  float rinv[kSpMaxRows];          // row-scale reciprocal of every token row (a row's value never changes)
  float cinv[3][kSpBn];   // column-scale reciprocals of the last three tiles (a tile's epilogue runs
                          // while the next tile's are written, and before the one after it starts)
  uint64_t full[kSpMaxStages], empty[kSpMaxStages], a_full, a_empty, tfull[2], tempty[2], drain;
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

__global__ void __launch_bounds__(kSpThreads, 1)
    sparse_fp8_kernel(const __grid_constant__ CUtensorMap tmB, const SpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kchunks = p.K / 128;
  uint8_t *sA = smem;                                                  // [kchunks][a_rows][128 B]
  uint8_t *sB = sA + (size_t)kchunks * p.a_rows * 128;                 // ring of weight stages
  SpShared &S = *reinterpret_cast<SpShared *>(sB + (size_t)p.stages * kSpStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nst = p.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.a_full, 8);
    mbar_init(&S.a_empty, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&S.tfull[a], 1);
      mbar_init(&S.tempty[a], 8);
    }
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_slot;
  pdl_wait();
  pdl_trigger();

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
    if (threadIdx.x < kSpMaxRows) S.amax_bits[threadIdx.x] = 0u;
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
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.status = S.bad;
  }
  const int total = S.bad ? 0 : S.n_active * p.n_tiles;
  // this CTA's tiles: [t_lo, t_hi), an even split of the tiles in order
  const int t_lo = (int)((long long)total * blockIdx.x / gridDim.x);
  const int t_hi = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  // the A region is (re)written at a tile whose group differs from the previous tile's
  auto recast = [&](int t) { return t == t_lo || t / p.n_tiles != (t - 1) / p.n_tiles; };
  volatile int *vabort = &S.abort_flag;
  uint32_t issued = 0;
  auto timeout = [&]() {
    atomicCAS(p.status, 0, MGEMM_STATUS_TIMEOUT);
    *vabort = 1;
  };
  const int kb_count = (kchunks + kSpKc - 1) / kSpKc;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = t_lo; t < t_hi && !*vabort; ++t) {
        const int a = t / p.n_tiles, n0 = (t % p.n_tiles) * kSpBn, e = S.act_e[a];
        for (int kb = 0; kb < kb_count; ++kb) {
          if (!mbar_wait(&S.empty[stage], phase ^ 1, vabort)) {
            timeout();
            break;
          }
          mbar_arrive_expect_tx(&S.full[stage], (uint32_t)kSpStageBytes);
          ++issued;
          tma_load_4d(sB + (size_t)stage * kSpStageBytes, &tmB, &S.full[stage], 0, n0, kb * kSpKc, e);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0, a_phase = 0;
    bool ok = true;
    for (int t = t_lo; t < t_hi && ok; ++t) {
      // the A region changes only at a recast tile (its codes are complete when a_full flips)
      const bool fresh = recast(t);
      if (!mbar_wait_warp(&S.tempty[acc], acc_phase ^ 1, vabort) ||
          (fresh && !mbar_wait_warp(&S.a_full, a_phase, vabort))) {
        ok = false;
        break;
      }
      if (fresh) a_phase ^= 1;
      const uint32_t d_tmem = tmem_base + acc * kSpBn;
      for (int kb = 0; kb < kb_count; ++kb) {
        if (!mbar_wait_warp(&S.full[stage], phase, vabort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t bbase = smem_u32(sB + (size_t)stage * kSpStageBytes);
#pragma unroll
          for (int j = 0; j < kSpKc; ++j) {
            const int chunk = kb * kSpKc + j;
            if (chunk >= kchunks) break;  // past K: no A rows there (the weight box holds zeros)
            const uint32_t aj = smem_u32(sA) + (uint32_t)chunk * p.a_rows * 128, bj = bbase + j * kSpBn * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8(d_tmem, smem_desc_sw128(aj + k * 32, 16, 1024), smem_desc_sw128(bj + k * 32, 16, 1024), p.idesc,
                     (kb | j | k) != 0);
          }
          mma_commit(&S.empty[stage]);
        }
        __syncwarp();
        if (++stage == nst) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(&S.tfull[acc]);
        if (t + 1 < t_hi && recast(t + 1)) mma_commit(&S.a_empty);  // the A region is read and will be rewritten
      }
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (!ok) {
      if (lane == 0) timeout();
    }
    if (lane == 0) {
      mma_commit(&S.drain);
      mbar_wait_drain(&S.drain, 0);
    }
    __syncwarp();
  } else {
    // warps 2 .. 9: cast the tile's token rows, then the previous tile's epilogue
    const int cw = warp - 2;  // 0 .. 7
    const int q = warp & 3;   // TMEM lane quarter this warp may read
    uint32_t e_phase = 0, acc_phase = 0;
    int acc = 0, cb = 0;
    int prev_t = -1, prev_acc = 0, prev_cb = 0;
    uint32_t prev_phase = 0;
    auto epilogue = [&](int t, int ac, uint32_t ph, int cbuf) -> bool {
      // rows 0 .. 31 live in TMEM lane quarter 0: warps 4 and 8 read it, 32 columns each
      if (!mbar_wait_warp(&S.tfull[ac], ph, vabort)) return false;
      tc_fence_after();
      const int a = t / p.n_tiles, n0 = (t % p.n_tiles) * kSpBn;
      const int r0 = S.act_row[a], m = S.act_m[a];
      if (q == 0) {
        const int h = cw >> 2;  // warp 4 -> columns 0 .. 31, warp 8 -> 32 .. 63
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ac * kSpBn + h * 32, v);
        tmem_ld_wait();
        if (lane < m) {
          const float ri = S.rinv[r0 + lane];
          __nv_bfloat16 *orow = p.out + (int64_t)(r0 + lane) * p.N;
          const uint64_t r2 = f32x2(ri, ri);
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const int col = n0 + h * 32 + c8 * 8;
            uint32_t pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int c = h * 32 + c8 * 8 + 2 * i;
              pk[i] = pack_bf16x2_u64(mul_f32x2(mul_f32x2(f32x2(v[c8 * 8 + 2 * i], v[c8 * 8 + 2 * i + 1]), r2),
                                                f32x2(S.cinv[cbuf][c], S.cinv[cbuf][c + 1])));
            }
            if (col < p.N) *reinterpret_cast<uint4 *>(orow + col) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.tempty[ac]);
      return true;
    };
    // Every one of these eight warps reaches the named barrier once per tile,
    // and the loop is left only right after it (on the abort flag, read by all
    // of them there): a warp whose wait gave up never strands the others at it.
    const int ct = (int)threadIdx.x - 64;  // 0 .. 255
    const int upr = p.K >> 3;                // 16-byte units (8 elements) per row
    for (int t = t_lo; t < t_hi; ++t) {
      const int a = t / p.n_tiles, n0 = (t % p.n_tiles) * kSpBn;
      const int r0 = S.act_row[a], m = S.act_m[a], e = S.act_e[a];
      const bool fresh = recast(t);
      bool ok = true;
      if (fresh) {
        // unit u of the group: row u / upr, elements 8 (u % upr) .. + 7; thread ct holds u = ct + 256 j
        const int U = m * upr;
        auto load = [&](int j0, uint4(&v)[kSpKeep]) {
#pragma unroll
          for (int j = 0; j < kSpKeep; ++j) {
            const int u = j0 + j * 256 + ct;
            if (u < U) {
              const int i = u / upr;
              v[j] = ldg_nc_v4(p.x + (int64_t)(r0 + i) * p.ld_x + (int64_t)(u - i * upr) * 8);
            } else {
              v[j] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        };
        auto reduce = [&](int j0, const uint4(&v)[kSpKeep]) {
#pragma unroll
          for (int j = 0; j < kSpKeep; ++j) {
            if (j0 + j * 256 >= U) break;  // uniform over the warp
            const int u = j0 + j * 256 + ct;
            const int i = u < U ? u / upr : m - 1;
            const unsigned bits = u < U ? __float_as_uint(amax8(v[j], 0.f)) : 0u;
            const int i0 = __shfl_sync(0xffffffffu, i, 0);
            if (__all_sync(0xffffffffu, i == i0)) {
              const unsigned r = __reduce_max_sync(0xffffffffu, bits);
              if (lane == 0) atomicMax(&S.amax_bits[r0 + i0], r);
            } else if (bits) {
              atomicMax(&S.amax_bits[r0 + i], bits);
            }
          }
        };
        auto store = [&](int j0, const uint4(&v)[kSpKeep]) {
#pragma unroll
          for (int j = 0; j < kSpKeep; ++j) {
            const int u = j0 + j * 256 + ct;
            if (u < U) {
              const int i = u / upr, c = (u - i * upr) * 8;  // 8 code bytes at column c of row i
              const float sc = pow2_scale_from_amax(__uint_as_float(S.amax_bits[r0 + i]));
              const int chunk = c >> 7, b = c & 127;
              uint8_t *dst = sA + ((size_t)chunk * p.a_rows + i) * 128 + ((((b >> 4) ^ (i & 7)) << 4) | (b & 15));
              *reinterpret_cast<uint2 *>(dst) = cast8(v[j], sc);
            }
          }
        };
        // pass 1: the row maxima (the first kSpKeep units of every thread stay in registers)
        uint4 keep[kSpKeep];
        load(0, keep);
        reduce(0, keep);
        for (int j0 = 256 * kSpKeep; j0 < U; j0 += 256 * kSpKeep) {
          uint4 v[kSpKeep];
          load(j0, v);
          reduce(j0, v);
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // every row maximum is complete
        if (ct < m) S.rinv[r0 + ct] = pow2_recip(pow2_scale_from_amax(__uint_as_float(S.amax_bits[r0 + ct])));
        // pass 2, once the MMAs of the tile before have read the A region: the codes
        if (!mbar_wait_warp(&S.a_empty, e_phase ^ 1, vabort)) {
          if (lane == 0) timeout();
          ok = false;
        } else {
          store(0, keep);
          for (int j0 = 256 * kSpKeep; j0 < U; j0 += 256 * kSpKeep) {
            uint4 v[kSpKeep];
            load(j0, v);
            store(j0, v);
          }
        }
      }
      if (ok && cw == 0)  // the tile's column-scale reciprocals
        for (int c = lane; c < kSpBn; c += 32)
          S.cinv[cb][c] = n0 + c < p.N ? pow2_recip(__ldg(p.sw + (int64_t)e * p.N + n0 + c)) : 0.f;
      if (fresh) e_phase ^= 1;
      fence_proxy_async_smem();  // the codes are read by the tensor cores
      __syncwarp();
      // the tile's scales are visible to all eight warps; leave together on an abort
      if (bar1_256_or(*vabort != 0)) break;
      if (fresh && lane == 0) mbar_arrive(&S.a_full);
      if (prev_t >= 0 && !epilogue(prev_t, prev_acc, prev_phase, prev_cb) && lane == 0) timeout();
      prev_t = t;
      prev_acc = acc;
      prev_cb = cb;
      prev_phase = acc_phase;
      if (++cb == 3) cb = 0;
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (!*vabort && prev_t >= 0 && !epilogue(prev_t, prev_acc, prev_phase, prev_cb) && lane == 0) timeout();
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 128);
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
  const int a_rows = (int)((M + 7) / 8 * 8);
  const size_t a_bytes = (size_t)K * a_rows;
  const size_t fixed = 1024 + a_bytes + sizeof(SpShared) + 64;
  const size_t limit = (size_t)227 * 1024;
  if (fixed + 2 * (size_t)kSpStageBytes > limit) return MGEMM_EINVAL;  // the token rows do not fit on chip
  int stages = (int)((limit - fixed) / kSpStageBytes);
  if (stages > kSpMaxStages) stages = kSpMaxStages;
  int rc = ensure_context();
  if (rc) return rc;
  const int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  CUtensorMap tb;
  {  // w [E, N, K] e4m3 as 128-byte k-chunks: {128, N, K / 128, E}, boxes of 4 chunks of 64 rows
    const uint64_t d[4] = {128, (uint64_t)N, (uint64_t)K / 128, (uint64_t)E};
    const uint64_t st[3] = {(uint64_t)K, 128, (uint64_t)N * K};
    const uint32_t box[4] = {128, (uint32_t)kSpBn, (uint32_t)kSpKc, 1};
    if (!make_tensor_map(&tb, true, 4, w, d, st, box)) return MGEMM_ECUDA;
  }
  SpParams p{};
  p.sizes = group_sizes;
  p.E = E;
  p.M = (int)M;
  p.K = K;
  p.N = N;
  p.a_rows = a_rows;
  p.stages = stages;
  p.n_tiles = (N + kSpBn - 1) / kSpBn;
  p.x = (const __nv_bfloat16 *)x;
  p.ld_x = ld_x;
  p.sw = sw;
  p.out = (__nv_bfloat16 *)out;
  p.status = status;
  p.idesc = make_idesc(0u, false, false, 128, kSpBn);
  const int64_t upper = (M < E ? M : E) * (int64_t)p.n_tiles;
  const int grid = (int)(upper < sms ? upper : sms);
  const size_t smem = fixed + (size_t)stages * kSpStageBytes;
  static bool attr_done[64] = {};
  int dev = 0;
  rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return MGEMM_EINVAL;
  if (!attr_done[dev]) {
    rc = cuda_rc(cudaFuncSetAttribute(sparse_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit),
                 "cudaFuncSetAttribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  return launch_pdl(sparse_fp8_kernel, dim3((unsigned)grid), dim3(kSpThreads), smem, (cudaStream_t)stream, 1u,
                    "sparse FP8 forward launch", tb, p);
}
