// Entry points mgemm_fwd / mgemm_dgrad / mgemm_wgrad: argument checks,
// tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry
// point, so the library needs no link-time libcuda), grid sizing and dispatch.
#include "gemm_launch.cuh"

using namespace mgemm;

namespace {

bool make_map(CUtensorMap *m, bool fp8, int rank, const void *base, const uint64_t *dims,
              const uint64_t *strides, const uint32_t *box) {
  return make_tensor_map(m, fp8, rank, base, dims, strides, box);
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

int sm_count() { return sm_count_cached(); }

// dtype, expert count and sizes (the checks that need no pointer)
int size_checks(int dtype, int64_t M, int K, int N, int E) {
  if (dtype != MGEMM_BF16 && dtype != MGEMM_FP8_E4M3) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || K <= 0 || N <= 0) return MGEMM_EINVAL;
  return MGEMM_OK;
}

int common_checks(const void *args, int dtype, int64_t M, int K, int N, int E) {
  if (!args) return MGEMM_EINVAL;
  int rc = size_checks(dtype, M, K, N, E);
  if (rc) return rc;
  if (!aligned16(args)) return MGEMM_EALIGN;
  const int kmul = dtype == MGEMM_FP8_E4M3 ? 16 : 8;
  if (K % kmul || N % kmul) return MGEMM_EALIGN;
  return MGEMM_OK;
}

int grid_for(int64_t tiles_upper) {
  const int sms = sm_count();
  if (sms <= 0) return -1;
  return (int)(tiles_upper < sms ? tiles_upper : sms);
}

// Output tile width: the candidate with the fewest waves x (width + per-tile
// overhead), where waves = ceil(estimated tiles / SMs); ties go to the wider
// tile (better operand reuse in shared memory).  m_tiles_est is the host's
// estimate of 128-row tiles (the exact count lives on the device).
int choose_bn_units(int64_t m_tiles_est, int64_t n_cols, int units, bool allow192 = false) {
  const int sms = units > 0 ? units : 1;
  int best = 256;
  int64_t best_cost = -1;
  for (int bn : {256, 192, 128, 64}) {
    if (bn == 192 && !allow192) continue;
    const int64_t tiles = m_tiles_est * ((n_cols + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const int64_t cost = waves * (bn + 64);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

int choose_bn(int64_t m_tiles_est, int64_t n_cols, bool allow192 = false) {
  return choose_bn_units(m_tiles_est, n_cols, sm_count() > 0 ? sm_count() : 148, allow192);
}

// Rows-mode estimate of 128-row tiles: dense groups give about M/128, sparse
// routing about one tile per touched group (at most min(M, E)).
int64_t rows_tiles_estimate(int64_t M, int E) {
  const int64_t dense = (M + 127) / 128;
  const int64_t sparse = M < E ? M : E;
  return dense > sparse ? dense : sparse;
}

// FP8 with few token rows: the operands viewed as 128-byte k-chunks so that one
// box brings kc consecutive contraction blocks (the run-time-ring kernels with
// kc blocks per stage).  A [M, Kc] as {128, M, Kc / 128}; B [E, Nrows, Kc] as
// {128, Nrows, Kc / 128, E} (chunk stride 128 B; Kc % 128 == 0 keeps every box
// row inside its row).
bool few_maps(CUtensorMap *ta, CUtensorMap *tb, const void *a, int64_t M, int Kc, uint32_t a_rows, const void *b,
              int Nrows, int E, int bn, uint32_t kc, uint64_t ld_row = 0, uint64_t ld_exp = 0) {
  const uint64_t da[3] = {128, (uint64_t)M, (uint64_t)Kc / 128};
  const uint64_t sa[2] = {(uint64_t)Kc, 128};
  const uint32_t ba[3] = {128, a_rows, kc};
  const uint64_t db[4] = {128, (uint64_t)Nrows, (uint64_t)Kc / 128, (uint64_t)E};
  // B rows (e, n) at e ld_exp + n ld_row (bytes; by default [E, Nrows, Kc] contiguous)
  const uint64_t sb[3] = {ld_row ? ld_row : (uint64_t)Kc, 128, ld_exp ? ld_exp : (uint64_t)Nrows * Kc};
  const uint32_t bb[4] = {128, (uint32_t)bn, kc, 1};
  CUtensorMap ma, mb;  // the caller's maps stay intact unless both views encode
  if (!make_map(&ma, true, 3, a, da, sa, ba) || !make_map(&mb, true, 4, b, db, sb, bb)) return false;
  *ta = ma;
  *tb = mb;
  return true;
}

// CTA pairs pay where a pair's 256-row tile is mostly real rows: groups that
// average at least 256 rows.  With fewer rows per group (sparse routing) the
// odd CTA's half of most tiles would be empty and the pair only couples two
// epilogues.
bool pairs_pay(int64_t M, int E) {
  const int64_t groups = M < E ? M : E;
  return groups > 0 && M / groups >= 256;
}

// Rows-mode estimate of 256-row pair tiles (CTA pairs).
int64_t pair_tiles_estimate(int64_t M, int E) {
  const int64_t dense = (M + 255) / 256;
  const int64_t sparse = M < E ? M : E;
  return dense > sparse ? dense : sparse;
}

// Map for the epilogue's TMA stores: the output viewed [rows, cols] bf16,
// boxes of 32 rows x 64 columns, 128-byte swizzle.
bool make_out_map(CUtensorMap *m, void *out, int64_t rows, int64_t cols) {
  const uint64_t d[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t st[1] = {(uint64_t)cols * 2};
  const uint32_t box[2] = {64, 32};
  return make_map(m, false, 2, out, d, st, box);
}

}  // namespace

// Every host-side check of mgemm_fwd (the args block aside): the same codes,
// returned before any CUDA call.
int mgemm::fwd_checks(int dtype, int trans_b, const void *x, const float *sx, const void *w, const float *sw,
                      const void *out, int64_t M, int K, int N, int E) {
  int rc = size_checks(dtype, M, K, N, E);
  if (rc) return rc;
  const int kmul = dtype == MGEMM_FP8_E4M3 ? 16 : 8;
  if (K % kmul || N % kmul) return MGEMM_EALIGN;
  if (!x || !w || !out) return MGEMM_EINVAL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out)) return MGEMM_EALIGN;
  const bool fp8 = dtype == MGEMM_FP8_E4M3;
  if (fp8 && !trans_b) return MGEMM_ENOTSUP;
  if (fp8 && (!sx || !sw)) return MGEMM_EINVAL;
  return MGEMM_OK;
}

// mgemm_fwd; mgemm_fwd_scatter when row_map is given; mgemm_fwd_gated when
// gate_rows > 0 (w [E, 2 gate_rows, K], N = 2 gate_rows, output gate_rows wide)
// ld_wn, ld_we (FP8 only; 0 = contiguous [E, N, K]): w[e, n, k] at e ld_we + n ld_wn + k bytes
static int fwd_impl(const void *args, int dtype, int trans_b, const void *x, const float *sx, const void *w,
                    const float *sw, void *out, int64_t M, int K, int N, int E, mgemm_stream_t stream,
                    const int32_t *row_map, int64_t map_limit, const float *row_weight, int gate_rows = 0,
                    int64_t group_rows_max = 0, int64_t ld_wn = 0, int64_t ld_we = 0,
                    const int32_t *a_ids = nullptr, int64_t a_numel = 0, int a_top_k = 1, int64_t a_src_rows = 0) {
  int rc = common_checks(args, dtype, M, K, N, E);
  if (rc) return rc;
  if ((rc = fwd_checks(dtype, trans_b, x, sx, w, sw, out, M, K, N, E))) return rc;
  const bool fp8 = dtype == MGEMM_FP8_E4M3;
  if (M == 0) return MGEMM_OK;
  if ((rc = ensure_context())) return rc;
  const uint64_t es = fp8 ? 1 : 2;
  const uint32_t bk = fp8 ? 128 : 64;
  CUtensorMap ta, tb;
  uint32_t a_rows = M < 128 ? (uint32_t)((M + 7) / 8 * 8) : 128u;
  // Routed rows (gated and scattered forms, bf16, w [E, N, K]): each group's
  // rows sit at the start of its 128-row blocks, followed by padding.  With at
  // most rb < 128 rows in a group (decode-size batches), the A box holds only
  // those rows (rounded up to 8) and the run-time ring gives the weight stream
  // the rest of shared memory; the padding rows' outputs are not stored.
  int64_t rb = 128;
  if (row_map && map_limit < rb) rb = map_limit;  // a group holds at most map_limit entries
  if (gate_rows > 0 && group_rows_max > 0 && group_rows_max < rb) rb = group_rows_max;
  const bool routed_few = !fp8 && trans_b && (row_map || gate_rows > 0) && rb < 128 && M >= 128;
  if (routed_few) a_rows = (uint32_t)((rb > 0 ? rb : 1) + 7) / 8 * 8;
  // gathered rows: the gated form with few rows per group and k-chunk boxes only
  if (a_ids && !(routed_few && gate_rows > 0 && K % 64 == 0)) return MGEMM_ENOTSUP;
  {
    const uint64_t d[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)K * es};
    const uint32_t box[2] = {bk, a_rows};
    if (!make_map(&ta, fp8, 2, x, d, st, box)) return MGEMM_ECUDA;
  }
  // FP8 with at least 128 token rows runs on CTA pairs: 256-row tiles, each CTA
  // copying bn / 2 rows of the weight tile
  const int sms = sm_count();
  if (sms <= 1) return MGEMM_ECUDA;
  const bool pair = fp8 && a_rows == 128 && pairs_pay(M, E);
  // 192-wide tiles (a 5-stage ring whose weight tiles are 24 KB of each 40 KB
  // stage), bf16 with w [E, K, N] in one box per stage (N % 64 == 0) or
  // w [E, N, K], when the weights stream (at most 256 rows per expert on
  // average, so HBM bounds the launch).  With more rows the wider tile's
  // operand reuse wins.
  // (the gated form needs whole 64-column halves: 128 or 256)
  const bool allow192 = !fp8 && gate_rows == 0 && !routed_few && (trans_b || N % 64 == 0) && M <= 256 * (int64_t)E;
  const bool gated = gate_rows > 0;
  // routed rows (the gated and scattered forms) come in groups padded to 128,
  // so M / 128 bounds their row tiles; plain groups may add one partial tile each
  const int64_t row_tiles = gated || row_map ? (M + 127) / 128 : rows_tiles_estimate(M, E);
  int bn = pair ? choose_bn_units(pair_tiles_estimate(M, E), N, sms / 2) : choose_bn(row_tiles, N, allow192);
  if (gated) bn = bn > 128 ? 256 : 128;  // gate and up halves of whole 64-column chunks
  const int out_cols = gated ? gate_rows : N;
  const int tile_cols = gated ? bn / 2 : bn;
  bool b_one_box = false;
  if (trans_b) {  // w [E, N, K] (FP8: rows at the given strides)
    const uint64_t d[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)E};
    const uint64_t st[2] = {ld_wn ? (uint64_t)ld_wn : (uint64_t)K * es, ld_we ? (uint64_t)ld_we : (uint64_t)N * K * es};
    const uint32_t box[3] = {bk, (uint32_t)(pair || gated ? bn / 2 : bn), 1};
    if (!make_map(&tb, fp8, 3, w, d, st, box)) return MGEMM_ECUDA;
  } else {  // w [E, K, N], loaded as 64-column MN-major chunks
    // with N % 64 == 0, w is viewed as [E][N / 64 chunks][K rows][64 columns] (chunk stride 128 B)
    // so one box brings the tile's bn / 64 chunks at once; every box row stays inside w
    bool one = N % 64 == 0;
    if (one) {
      const uint64_t d[4] = {64, (uint64_t)K, (uint64_t)N / 64, (uint64_t)E};
      const uint64_t st[3] = {(uint64_t)N * es, 64 * es, (uint64_t)K * N * es};
      const uint32_t box[4] = {64, bk, (uint32_t)bn / 64, 1};
      one = make_map(&tb, fp8, 4, w, d, st, box);
    }
    if (!one) {
      const uint64_t d[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
      const uint64_t st[2] = {(uint64_t)N * es, (uint64_t)K * N * es};
      const uint32_t box[3] = {64, bk, 1};
      if (!make_map(&tb, fp8, 3, w, d, st, box)) return MGEMM_ECUDA;
    }
    b_one_box = one;
  }
  CUtensorMap to;  // (scattered rows are stored row by row; the map then goes unused)
  if (!make_out_map(&to, out, row_map ? (map_limit > 0 ? map_limit : 1) : M, out_cols)) return MGEMM_ECUDA;
  GemmParams p{};
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = bn;
  p.b_one_box = b_one_box ? 1 : 0;
  p.row_map = row_map;
  p.map_limit = map_limit;
  p.row_weight = row_weight;
  p.gated = gated ? 1 : 0;
  p.gate_rows = gate_rows;
  p.idesc = make_idesc(fp8 ? 0u : 1u, false, !trans_b, pair ? 256 : 128, bn);
  p.a_rows = (int)a_rows;
  p.n_tiles = (out_cols + tile_cols - 1) / tile_cols;
  p.Kc = K;
  p.Nout = out_cols;
  p.out = (__nv_bfloat16 *)out;
  p.rscale = sx;
  p.cscale = sw;
  p.a_ids = a_ids;
  p.a_numel = a_numel;
  p.a_top_k = a_top_k;
  p.a_src = (const uint8_t *)x;
  p.a_ld = (int64_t)K * 2;
  p.a_kbytes = K * 2;
  cudaStream_t s = (cudaStream_t)stream;
  if (pair) {
    const int64_t pupper = pair_tiles_estimate(M, E) * p.n_tiles + (M < E ? M : E) * p.n_tiles;
    const int pairs = (int)(pupper < sms / 2 ? pupper : sms / 2);
    return gemm_fp8_rows_pair(ta, tb, to, p, 2 * pairs, s);
  }
  const int64_t upper = ((M + 127) / 128 + (M < E ? M : E)) * p.n_tiles;
  const int grid = grid_for(upper);
  if (grid < 0) return MGEMM_ECUDA;
  if (routed_few) {  // bf16 routed rows, few per group: run-time rings
    if (K % 64 == 0) {
      // k-chunk views of the bf16 rows as bytes (2K per row): one box per operand and stage
      // (four blocks at 64 columns, and at 128 with at most 8 rows per group; else two)
      const uint32_t kc = bn <= 64 || (bn <= 128 && a_rows <= 8) ? 4 : 2;
      bool maps = false;
      if (gated) {
        const uint64_t da[3] = {128, (uint64_t)M, (uint64_t)K * 2 / 128};
        const uint64_t sa[2] = {(uint64_t)K * 2, 128};
        const uint32_t ba[3] = {128, a_rows, kc};
        // w [E, 2F, K]: {128 B, F rows of a half, gate / up, K / 64 chunks, E}
        const uint64_t db[5] = {128, (uint64_t)gate_rows, 2, (uint64_t)K * 2 / 128, (uint64_t)E};
        const uint64_t sb[4] = {(uint64_t)K * 2, (uint64_t)gate_rows * K * 2, 128, (uint64_t)N * K * 2};
        const uint32_t bb[5] = {128, (uint32_t)bn / 2, 2, kc, 1};
        // (gathered rows are copied by the producer; the A map then describes x's own rows)
        const uint64_t dg[3] = {128, (uint64_t)(a_ids ? a_src_rows : M), (uint64_t)K * 2 / 128};
        CUtensorMap ma, mb;
        maps = make_map(&ma, true, 3, x, a_ids ? dg : da, sa, ba) && make_map(&mb, true, 5, w, db, sb, bb);
        if (maps) {
          ta = ma;
          tb = mb;
        }
      } else {
        maps = few_maps(&ta, &tb, x, M, K * 2, a_rows, w, N, E, bn, kc);
      }
      if (!maps && a_ids) return MGEMM_ECUDA;
      if (maps) {
        if (bn <= 64) return gemm_bf16_rows_few_narrow_kc(ta, tb, to, p, grid, s);
        if (bn <= 128)
          return kc == 4 ? gemm_bf16_rows_few_mid_kc4(ta, tb, to, p, grid, s)
                         : gemm_bf16_rows_few_mid_kc(ta, tb, to, p, grid, s);
        return gemm_bf16_rows_few_wide_kc(ta, tb, to, p, grid, s);
      }
    }
    if (bn <= 64) return gemm_bf16_rows_few_narrow(ta, tb, to, p, grid, s);
    if (bn <= 128) return gemm_bf16_rows_few_mid(ta, tb, to, p, grid, s);
    return gemm_bf16_rows_few_wide(ta, tb, to, p, grid, s);
  }
  if (fp8 && a_rows < 128 && K % 128 == 0) {
    // few token rows: the weight stream gets the shared memory the A slots leave
    // (4 / 2 / 1 contraction blocks per stage for BN 64 / 128 / 256)
    if (bn <= 64 && few_maps(&ta, &tb, x, M, K, a_rows, w, N, E, bn, 4, ld_wn, ld_we))
      return gemm_fp8_rows_few_narrow(ta, tb, to, p, grid, s);
    if (bn > 64 && bn <= 128 && few_maps(&ta, &tb, x, M, K, a_rows, w, N, E, bn, 2, ld_wn, ld_we))
      return gemm_fp8_rows_few_mid(ta, tb, to, p, grid, s);
    if (bn > 128) return gemm_fp8_rows_few(ta, tb, to, p, grid, s);
  }
  if (bn <= 64) {
    if (fp8) return gemm_fp8_rows_narrow(ta, tb, to, p, grid, s);
    return trans_b ? gemm_bf16_rows_bk_narrow(ta, tb, to, p, grid, s)
                   : gemm_bf16_rows_bmn_narrow(ta, tb, to, p, grid, s);
  }
  if (bn <= 128) {
    if (fp8) return gemm_fp8_rows_mid(ta, tb, to, p, grid, s);
    return trans_b ? gemm_bf16_rows_bk_mid(ta, tb, to, p, grid, s) : gemm_bf16_rows_bmn_mid(ta, tb, to, p, grid, s);
  }
  if (gated)  // bf16, w [E, 2F, K]: the wide or mid K-major form
    return bn == 256 ? gemm_bf16_rows_bk(ta, tb, to, p, grid, s) : gemm_bf16_rows_bk_mid(ta, tb, to, p, grid, s);
  if (bn == 192 && trans_b) return gemm_bf16_rows_bk_w192(ta, tb, to, p, grid, s);
  if (bn == 192 && b_one_box) return gemm_bf16_rows_bmn_w192(ta, tb, to, p, grid, s);
  if (fp8) return gemm_fp8_rows(ta, tb, to, p, grid, s);
  return trans_b ? gemm_bf16_rows_bk(ta, tb, to, p, grid, s) : gemm_bf16_rows_bmn(ta, tb, to, p, grid, s);
}

extern "C" int mgemm_fwd(const void *args, int dtype, int trans_b, const void *x, const float *sx, const void *w,
                         const float *sw, void *out, int64_t M, int K, int N, int E, mgemm_stream_t stream) {
  return fwd_impl(args, dtype, trans_b, x, sx, w, sw, out, M, K, N, E, stream, nullptr, 0, nullptr);
}

extern "C" int mgemm_fwd_fp8_strided(const void *args, const void *x, const float *sx, const void *w, int64_t ld_wn,
                                     int64_t ld_we, const float *sw, void *out, int64_t M, int K, int N, int E,
                                     mgemm_stream_t stream) {
  if (ld_wn < K || (E > 1 && ld_we < K) || ld_we < 0) return MGEMM_EINVAL;
  if (ld_wn % 16 || ld_we % 16) return MGEMM_EALIGN;
  // (with one expert the expert stride is never stepped; any multiple of 16 describes it)
  return fwd_impl(args, MGEMM_FP8_E4M3, 1, x, sx, w, sw, out, M, K, N, E, stream, nullptr, 0, nullptr, 0, 0, ld_wn,
                  ld_we > 0 ? ld_we : (int64_t)K);
}

extern "C" int mgemm_fwd_scatter(const void *args, int dtype, int trans_b, const void *x, const void *w, void *out,
                                 const int32_t *row_map, int64_t map_limit, const float *row_weight, int64_t M,
                                 int K, int N, int E, mgemm_stream_t stream) {
  if (dtype != MGEMM_BF16 && dtype != MGEMM_FP8_E4M3) return MGEMM_EINVAL;
  if (dtype != MGEMM_BF16) return MGEMM_ENOTSUP;
  if (!row_map || map_limit < 0 || map_limit >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (((uintptr_t)row_map & 3) || ((uintptr_t)row_weight & 3)) return MGEMM_EALIGN;
  return fwd_impl(args, dtype, trans_b, x, nullptr, w, nullptr, out, M, K, N, E, stream, row_map, map_limit,
                  row_weight);
}

extern "C" int mgemm_fwd_gated(const void *args, const void *x, const void *w, void *out, int64_t M, int K, int F,
                               int E, int64_t group_rows_max, mgemm_stream_t stream) {
  if (F < 1 || F % 8 || F > (1 << 29)) return F % 8 ? MGEMM_EALIGN : MGEMM_EINVAL;
  if (group_rows_max < 0) return MGEMM_EINVAL;
  return fwd_impl(args, MGEMM_BF16, 1, x, nullptr, w, nullptr, out, M, K, 2 * F, E, stream, nullptr, 0, nullptr, F,
                  group_rows_max);
}

extern "C" int mgemm_fwd_gated_gather(const void *args, const void *x, int64_t x_rows, const int32_t *sorted_ids,
                                      int64_t numel, int top_k, const void *w, void *out, int64_t M, int K, int F,
                                      int E, int64_t group_rows_max, mgemm_stream_t stream) {
  if (F < 1 || F % 8 || F > (1 << 29)) return F % 8 ? MGEMM_EALIGN : MGEMM_EINVAL;
  if (!sorted_ids || x_rows < 1 || numel < 0 || top_k < 1) return MGEMM_EINVAL;
  if ((uintptr_t)sorted_ids & 3) return MGEMM_EALIGN;
  if (group_rows_max < 1 || group_rows_max > 32) return MGEMM_ENOTSUP;
  return fwd_impl(args, MGEMM_BF16, 1, x, nullptr, w, nullptr, out, M, K, 2 * F, E, stream, nullptr, 0, nullptr, F,
                  group_rows_max, 0, 0, sorted_ids, numel, top_k, x_rows);
}

extern "C" int mgemm_fwd_mx(const void *args, const uint8_t *x, const uint8_t *sx, const uint8_t *w, const uint8_t *sw,
                            int64_t ld_sf, void *out, int64_t M, int K, int N, int E, mgemm_stream_t stream) {
  if (!args || !x || !sx || !w || !sw || !out) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || K <= 0 || N <= 0 || ld_sf < K / 32) return MGEMM_EINVAL;
  if ((int64_t)E * N >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (K % 128 || N % 8) return MGEMM_EINVAL;
  if (!aligned16(args) || !aligned16(x) || !aligned16(sx) || !aligned16(w) || !aligned16(sw) || !aligned16(out) ||
      ld_sf % 16)
    return MGEMM_EALIGN;
  if (M == 0) return MGEMM_OK;
  int rc = ensure_context();
  if (rc) return rc;
  const int sms = sm_count();
  if (sms <= 0) return MGEMM_ECUDA;
  // the widest tile N needs (less operand traffic per FLOP): 256 columns (one
  // TMEM accumulator: the scale factors take the second one's columns), else
  // 192 or one 128-wide tile
  const int bn = N > 192 ? 256 : N > 128 ? 192 : 128;
  CUtensorMap ta, tb, to, tsa, tsb;
  {
    const uint64_t d[2] = {(uint64_t)K, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)K};
    const uint32_t box[2] = {128, 128};
    if (!make_map(&ta, true, 2, x, d, st, box)) return MGEMM_ECUDA;
  }
  {
    const uint64_t d[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)K, (uint64_t)N * K};
    const uint32_t box[3] = {128, (uint32_t)bn, 1};
    if (!make_map(&tb, true, 3, w, d, st, box)) return MGEMM_ECUDA;
  }
  // scale rows: 16-byte boxes (four contraction blocks of 128) of 128 / bn rows, unswizzled
  {
    const uint64_t d[2] = {(uint64_t)ld_sf, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)ld_sf};
    const uint32_t box[2] = {16, 128};
    if (!make_tensor_map(&tsa, true, 2, sx, d, st, box, false)) return MGEMM_ECUDA;
  }
  {
    const uint64_t d[2] = {(uint64_t)ld_sf, (uint64_t)E * N};
    const uint64_t st[1] = {(uint64_t)ld_sf};
    const uint32_t box[2] = {16, (uint32_t)bn};
    if (!make_tensor_map(&tsb, true, 2, sw, d, st, box, false)) return MGEMM_ECUDA;
  }
  if (!make_out_map(&to, out, M, N)) return MGEMM_ECUDA;
  GemmParams p{};
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = bn;
  p.a_rows = 128;
  p.idesc = make_idesc_mx(128, bn, 1);  // ue8m0 scales
  p.n_tiles = (N + bn - 1) / bn;
  p.Kc = K;
  p.Nout = N;
  p.out = (__nv_bfloat16 *)out;
  const int64_t upper = ((M + 127) / 128 + (M < E ? M : E)) * p.n_tiles;
  const int grid = grid_for(upper);
  if (grid < 0) return MGEMM_ECUDA;
  if (bn == 256) return gemm_fp8_rows_mx256(ta, tb, to, tsa, tsb, p, grid, (cudaStream_t)stream);
  return bn == 192 ? gemm_fp8_rows_mx192(ta, tb, to, tsa, tsb, p, grid, (cudaStream_t)stream)
                   : gemm_fp8_rows_mx(ta, tb, to, tsa, tsb, p, grid, (cudaStream_t)stream);
}

extern "C" int mgemm_wgrad_mx(const void *args, const uint8_t *x, const uint8_t *sx, const uint8_t *grad_out,
                              const uint8_t *sgo, void *grad_w, int64_t M, int K, int N, int E, int64_t ld,
                              mgemm_stream_t stream) {
  if (!args || !grad_w) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || K <= 0 || N <= 0 || K % 16 || N % 16) return MGEMM_EINVAL;
  if (M > 0 && (!x || !sx || !grad_out || !sgo)) return MGEMM_EINVAL;
  if (ld < mgemm_colwise_ld(M, E) || ld >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (!aligned16(args) || !aligned16(grad_w) || ld % 128) return MGEMM_EALIGN;
  if (M > 0 && (!aligned16(x) || !aligned16(sx) || !aligned16(grad_out) || !aligned16(sgo))) return MGEMM_EALIGN;
  int rc = ensure_context();
  if (rc) return rc;
  const int sms = sm_count();
  if (sms <= 0) return MGEMM_ECUDA;
  // with M == 0 every expert is empty: nothing is loaded, the maps only need valid memory
  const void *xa = M > 0 ? (const void *)x : grad_w, *ga = M > 0 ? (const void *)grad_out : grad_w;
  const void *sxa = M > 0 ? (const void *)sx : grad_w, *sga = M > 0 ? (const void *)sgo : grad_w;
  const uint64_t L = M > 0 ? (uint64_t)ld : 128;
  // 256-wide tiles (one TMEM accumulator) when N needs more than 192 columns
  const int bn = N > 192 ? 256 : 192;
  CUtensorMap ta, tb, to, tsa, tsb;
  {
    const uint64_t da[2] = {L, (uint64_t)K}, db[2] = {L, (uint64_t)N};
    const uint64_t st[1] = {L};
    const uint32_t boxa[2] = {128, 128}, boxb[2] = {128, (uint32_t)bn};
    if (!make_map(&ta, true, 2, xa, da, st, boxa)) return MGEMM_ECUDA;
    if (!make_map(&tb, true, 2, ga, db, st, boxb)) return MGEMM_ECUDA;
  }
  // scale rows [ld / 128][rows][4 B], rows viewed in fours: boxes of one block
  {
    const uint64_t d[3] = {16, (uint64_t)K / 4, L / 128};
    const uint64_t st[2] = {16, (uint64_t)K * 4};
    const uint32_t box[3] = {16, 32, 1};
    if (!make_tensor_map(&tsa, true, 3, sxa, d, st, box, false)) return MGEMM_ECUDA;
  }
  {
    const uint64_t d[3] = {16, (uint64_t)N / 4, L / 128};
    const uint64_t st[2] = {16, (uint64_t)N * 4};
    const uint32_t box[3] = {16, (uint32_t)bn / 4, 1};
    if (!make_tensor_map(&tsb, true, 3, sga, d, st, box, false)) return MGEMM_ECUDA;
  }
  if (!make_out_map(&to, grad_w, (int64_t)E * K, N)) return MGEMM_ECUDA;
  GemmParams p{};
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = bn;
  p.idesc = make_idesc_mx(128, bn, 1);  // ue8m0 scales
  p.n_tiles = (N + bn - 1) / bn;
  p.mt_k = (K + 127) / 128;
  p.Nout = N;
  p.Kout = K;
  p.out = (__nv_bfloat16 *)grad_w;
  const int64_t upper = (int64_t)E * p.mt_k * p.n_tiles;
  if (upper >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  const int grid = grid_for(upper);
  if (grid < 0) return MGEMM_ECUDA;
  if (bn == 256) return gemm_fp8_experts_mx256(ta, tb, to, tsa, tsb, p, grid, (cudaStream_t)stream);
  return gemm_fp8_experts_mx(ta, tb, to, tsa, tsb, p, grid, (cudaStream_t)stream);
}

extern "C" int mgemm_dgrad(const void *args, int dtype, const void *grad_out, const float *sgo, const void *w,
                           const float *sw, void *grad_x, int64_t M, int K, int N, int E, mgemm_stream_t stream) {
  int rc = common_checks(args, dtype, M, K, N, E);
  if (rc) return rc;
  if (!grad_out || !w || !grad_x) return MGEMM_EINVAL;
  if (!aligned16(grad_out) || !aligned16(w) || !aligned16(grad_x)) return MGEMM_EALIGN;
  const bool fp8 = dtype == MGEMM_FP8_E4M3;
  if (fp8 && (!sgo || !sw)) return MGEMM_EINVAL;
  if (M == 0) return MGEMM_OK;
  if ((rc = ensure_context())) return rc;
  const uint64_t es = fp8 ? 1 : 2;
  const uint32_t bk = fp8 ? 128 : 64;
  CUtensorMap ta, tb;
  const uint32_t a_rows = M < 128 ? (uint32_t)((M + 7) / 8 * 8) : 128u;
  {  // grad_out [M, N], contraction over N
    const uint64_t d[2] = {(uint64_t)N, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)N * es};
    const uint32_t box[2] = {bk, a_rows};
    if (!make_map(&ta, fp8, 2, grad_out, d, st, box)) return MGEMM_ECUDA;
  }
  const int sms = sm_count();
  if (sms <= 1) return MGEMM_ECUDA;
  const bool pair = fp8 && a_rows == 128 && pairs_pay(M, E);  // CTA pairs, as in mgemm_fwd
  const int bn = pair ? choose_bn_units(pair_tiles_estimate(M, E), K, sms / 2) : choose_bn(rows_tiles_estimate(M, E), K);
  {  // w [E, K, N]: output column k, contraction n contiguous
    const uint64_t d[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N * es, (uint64_t)K * N * es};
    const uint32_t box[3] = {bk, (uint32_t)(pair ? bn / 2 : bn), 1};
    if (!make_map(&tb, fp8, 3, w, d, st, box)) return MGEMM_ECUDA;
  }
  CUtensorMap to;
  if (!make_out_map(&to, grad_x, M, K)) return MGEMM_ECUDA;
  GemmParams p{};
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = bn;
  p.idesc = make_idesc(fp8 ? 0u : 1u, false, false, pair ? 256 : 128, bn);
  p.a_rows = (int)a_rows;
  p.n_tiles = (K + bn - 1) / bn;
  p.Kc = N;
  p.Nout = K;
  p.out = (__nv_bfloat16 *)grad_x;
  p.rscale = sgo;
  p.cscale = sw;
  cudaStream_t s = (cudaStream_t)stream;
  if (pair) {
    const int64_t pupper = pair_tiles_estimate(M, E) * p.n_tiles + (M < E ? M : E) * p.n_tiles;
    const int pairs = (int)(pupper < sms / 2 ? pupper : sms / 2);
    return gemm_fp8_rows_pair(ta, tb, to, p, 2 * pairs, s);
  }
  const int64_t upper = ((M + 127) / 128 + (M < E ? M : E)) * p.n_tiles;
  const int grid = grid_for(upper);
  if (grid < 0) return MGEMM_ECUDA;
  if (fp8 && a_rows < 128 && N % 128 == 0) {
    if (bn <= 64 && few_maps(&ta, &tb, grad_out, M, N, a_rows, w, K, E, bn, 4))
      return gemm_fp8_rows_few_narrow(ta, tb, to, p, grid, s);
    if (bn > 64 && bn <= 128 && few_maps(&ta, &tb, grad_out, M, N, a_rows, w, K, E, bn, 2))
      return gemm_fp8_rows_few_mid(ta, tb, to, p, grid, s);
    if (bn > 128) return gemm_fp8_rows_few(ta, tb, to, p, grid, s);
  }
  if (bn <= 64) return fp8 ? gemm_fp8_rows_narrow(ta, tb, to, p, grid, s) : gemm_bf16_rows_bk_narrow(ta, tb, to, p, grid, s);
  if (bn <= 128) return fp8 ? gemm_fp8_rows_mid(ta, tb, to, p, grid, s) : gemm_bf16_rows_bk_mid(ta, tb, to, p, grid, s);
  return fp8 ? gemm_fp8_rows(ta, tb, to, p, grid, s) : gemm_bf16_rows_bk(ta, tb, to, p, grid, s);
}

extern "C" int mgemm_wgrad(const void *args, int dtype, const void *x, const float *sx, const void *grad_out,
                           const float *sgo, void *grad_w, int64_t M, int K, int N, int E, int64_t ld,
                           mgemm_stream_t stream) {
  int rc = common_checks(args, dtype, M, K, N, E);
  if (rc) return rc;
  if (!grad_w) return MGEMM_EINVAL;
  if (M > 0 && (!x || !grad_out)) return MGEMM_EINVAL;
  if (!aligned16(grad_w) || (M > 0 && (!aligned16(x) || !aligned16(grad_out)))) return MGEMM_EALIGN;
  const bool fp8 = dtype == MGEMM_FP8_E4M3;
  if (fp8 && (!sx || !sgo)) return MGEMM_EINVAL;
  if (fp8 && (ld < mgemm_colwise_ld(M, E) || ld >= (int64_t(1) << 31))) return MGEMM_EINVAL;
  if (fp8 && ld % 16) return MGEMM_EALIGN;
  // With M == 0 every expert is empty: the kernel only writes zeros and never
  // loads, so the maps just need a valid description of some memory.
  const void *xa = M > 0 ? x : grad_w;
  const void *ga = M > 0 ? grad_out : grad_w;
  const uint64_t Mm = M > 0 ? (uint64_t)M : 16;
  const uint64_t Lm = fp8 && ld > 0 ? (uint64_t)ld : 16;
  if ((rc = ensure_context())) return rc;
  // FP8 runs on CTA pairs: one tile is 256 rows of K (each CTA 128) by bn columns
  const int mt_k = fp8 ? (K + 255) / 256 : (K + 127) / 128;
  const int sms = sm_count();
  if (sms <= 1) return MGEMM_ECUDA;
  const int bn = fp8 ? choose_bn_units((int64_t)E * mt_k, N, sms / 2) : choose_bn((int64_t)E * mt_k, N);
  CUtensorMap ta, tb;
  if (fp8) {
    // padded column-major operands: x^T [K, ld] and grad_out^T [N, ld], contraction
    // contiguous; each CTA of a pair loads 128 rows of x^T and bn / 2 rows of grad_out^T
    const uint64_t da[2] = {Lm, (uint64_t)K}, db[2] = {Lm, (uint64_t)N};
    const uint64_t st[1] = {Lm};
    const uint32_t boxa[2] = {128, 128}, boxb[2] = {128, (uint32_t)bn / 2};
    if (!make_map(&ta, true, 2, xa, da, st, boxa)) return MGEMM_ECUDA;
    if (!make_map(&tb, true, 2, ga, db, st, boxb)) return MGEMM_ECUDA;
  } else {
    // row-major x [M, K] and grad_out [M, N], loaded as 64-column MN-major chunks of 64 rows
    const uint64_t da[2] = {(uint64_t)K, Mm}, db[2] = {(uint64_t)N, Mm};
    const uint64_t sta[1] = {(uint64_t)K * 2}, stb[1] = {(uint64_t)N * 2};
    const uint32_t box[2] = {64, 64};
    if (!make_map(&ta, false, 2, xa, da, sta, box)) return MGEMM_ECUDA;
    if (!make_map(&tb, false, 2, ga, db, stb, box)) return MGEMM_ECUDA;
  }
  CUtensorMap to;
  if (!make_out_map(&to, grad_w, (int64_t)E * K, N)) return MGEMM_ECUDA;
  GemmParams p{};
  p.args = (const uint8_t *)args;
  p.E = E;
  p.bn = bn;
  p.idesc = make_idesc(fp8 ? 0u : 1u, !fp8, !fp8, fp8 ? 256 : 128, bn);
  p.n_tiles = (N + bn - 1) / bn;
  p.mt_k = mt_k;
  p.Nout = N;
  p.Kout = K;
  p.out = (__nv_bfloat16 *)grad_w;
  p.rscale = sx;
  p.cscale = sgo;
  const int64_t upper = (int64_t)E * p.mt_k * p.n_tiles;
  if (upper >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  if (fp8) {
    const int pairs = (int)(upper < sms / 2 ? upper : sms / 2);
    return gemm_fp8_experts_pair(ta, tb, to, p, 2 * pairs, s);
  }
  const int grid = grid_for(upper);
  if (grid < 0) return MGEMM_ECUDA;
  return gemm_bf16_experts(ta, tb, to, p, grid, s);
}

// CTAs given to dgrad when it shares one launch with wgrad, or 0 when two
// launches are expected to do about as well.  A makespan model with rates measured
// on GB300 for the bf16 forms: a wgrad tile's epilogue stores ~34 GB/s of
// grad_w per SM; a dgrad CTA streams weights at up to ~60 GB/s; HBM serves
// ~6 TB/s to both; the tensor cores give ~12 TFLOP/s per SM.  Only the
// memory-bound regime is considered (groups of at most 256 rows on average),
// where dgrad streams the weights from HBM and wgrad is bound by its stores:
// two different limits, so sharing the SMs beats taking turns.
static int dual_split(int64_t M, int K, int N, int E, int bn_d, int bn_w, int sms) {
  if (M <= 0 || M > 256 * (int64_t)E || sms < 4) return 0;
  const double rw = 34e9, rd = 60e9, hbm = 6e12, tc = 12e12;
  const double tiles_d = (double)rows_tiles_estimate(M, E) * ((K + bn_d - 1) / bn_d);
  const double tiles_w = (double)E * ((K + 127) / 128) * ((N + bn_w - 1) / bn_w);
  const double rows_e = (double)M / E;
  const double tile_d = fmax((double)bn_d * N * 2 / rd, 2.0 * 128 * bn_d * N / tc);
  const double tile_w = fmax(128.0 * bn_w * 2 / rw, 2.0 * 128 * bn_w * rows_e / tc);
  const double bytes_d = (double)(M < E ? M : E) * K * N * 2;
  auto t_d = [&](int g, int gw) {
    const double share = fmax(hbm - gw * rw, 0.1 * hbm);
    return fmax(ceil(tiles_d / g) * tile_d, bytes_d / share);
  };
  auto t_w = [&](int g) { return ceil(tiles_w / g) * tile_w; };
  const double seq = t_d(sms, 0) + t_w(sms);
  int best = 0;
  double best_t = seq;
  for (int g = 1; g < sms; ++g) {
    const double t = fmax(t_d(g, sms - g), t_w(sms - g));
    if (t < best_t) {
      best_t = t;
      best = g;
    }
  }
  // the model's ratio of the two forms was off by up to ~6% on a sweep of
  // shapes: take the one-launch form only for a larger predicted gain
  return best_t < 0.94 * seq ? best : 0;
}

extern "C" int mgemm_dgrad_wgrad_split(int64_t M, int K, int N, int E) {
  int rc = size_checks(MGEMM_BF16, M, K, N, E);
  if (rc) return rc;
  const int sms = sm_count();
  if (sms <= 1) return MGEMM_ECUDA;
  const int bn_d = choose_bn(rows_tiles_estimate(M, E), K);
  const int bn_w = choose_bn((int64_t)E * ((K + 127) / 128), N);
  return dual_split(M, K, N, E, bn_d, bn_w, sms);
}

extern "C" int mgemm_dgrad_wgrad(const void *args, const void *grad_out, const void *w, const void *x, void *grad_x,
                                 void *grad_w, int64_t M, int K, int N, int E, mgemm_stream_t stream) {
  int rc = common_checks(args, MGEMM_BF16, M, K, N, E);
  if (rc) return rc;
  if (M == 0) return mgemm_wgrad(args, MGEMM_BF16, x, nullptr, grad_out, nullptr, grad_w, M, K, N, E, 0, stream);
  if (!grad_out || !w || !x || !grad_x || !grad_w) return MGEMM_EINVAL;
  if (!aligned16(grad_out) || !aligned16(w) || !aligned16(x) || !aligned16(grad_x) || !aligned16(grad_w))
    return MGEMM_EALIGN;
  if ((rc = ensure_context())) return rc;
  const int sms = sm_count();
  if (sms <= 1) return MGEMM_ECUDA;
  const int bn_d = choose_bn(rows_tiles_estimate(M, E), K);
  const int mt_w = (K + 127) / 128;
  const int bn_w = choose_bn((int64_t)E * mt_w, N);
  const int split = dual_split(M, K, N, E, bn_d, bn_w, sms);
  if (split == 0) {
    rc = mgemm_dgrad(args, MGEMM_BF16, grad_out, nullptr, w, nullptr, grad_x, M, K, N, E, stream);
    if (rc) return rc;
    return mgemm_wgrad(args, MGEMM_BF16, x, nullptr, grad_out, nullptr, grad_w, M, K, N, E, 0, stream);
  }
  // dgrad: grad_out [M, N] (A, contraction over N) and w [E, K, N] (B, K-major), as in mgemm_dgrad
  CUtensorMap da, db, dout;
  const uint32_t a_rows = M < 128 ? (uint32_t)((M + 7) / 8 * 8) : 128u;
  {
    const uint64_t d[2] = {(uint64_t)N, (uint64_t)M};
    const uint64_t st[1] = {(uint64_t)N * 2};
    const uint32_t box[2] = {64, a_rows};
    if (!make_map(&da, false, 2, grad_out, d, st, box)) return MGEMM_ECUDA;
  }
  {
    const uint64_t d[3] = {(uint64_t)N, (uint64_t)K, (uint64_t)E};
    const uint64_t st[2] = {(uint64_t)N * 2, (uint64_t)K * N * 2};
    const uint32_t box[3] = {64, (uint32_t)bn_d, 1};
    if (!make_map(&db, false, 3, w, d, st, box)) return MGEMM_ECUDA;
  }
  if (!make_out_map(&dout, grad_x, M, K)) return MGEMM_ECUDA;
  GemmParams pd{};
  pd.args = (const uint8_t *)args;
  pd.E = E;
  pd.bn = bn_d;
  pd.idesc = make_idesc(1u, false, false, 128, bn_d);
  pd.a_rows = (int)a_rows;
  pd.n_tiles = (K + bn_d - 1) / bn_d;
  pd.Kc = N;
  pd.Nout = K;
  pd.out = (__nv_bfloat16 *)grad_x;
  // wgrad: x [M, K] (A) and grad_out [M, N] (B), both MN-major, as in mgemm_wgrad
  CUtensorMap wa, wb, wout;
  {
    const uint64_t dx[2] = {(uint64_t)K, (uint64_t)M}, dg[2] = {(uint64_t)N, (uint64_t)M};
    const uint64_t sx[1] = {(uint64_t)K * 2}, sg[1] = {(uint64_t)N * 2};
    const uint32_t box[2] = {64, 64};
    if (!make_map(&wa, false, 2, x, dx, sx, box)) return MGEMM_ECUDA;
    if (!make_map(&wb, false, 2, grad_out, dg, sg, box)) return MGEMM_ECUDA;
  }
  if (!make_out_map(&wout, grad_w, (int64_t)E * K, N)) return MGEMM_ECUDA;
  GemmParams pw{};
  pw.args = (const uint8_t *)args;
  pw.E = E;
  pw.bn = bn_w;
  pw.idesc = make_idesc(1u, true, true, 128, bn_w);
  pw.n_tiles = (N + bn_w - 1) / bn_w;
  pw.mt_k = mt_w;
  pw.Nout = N;
  pw.Kout = K;
  pw.out = (__nv_bfloat16 *)grad_w;
  if ((int64_t)E * mt_w * pw.n_tiles >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  return gemm_bf16_dgrad_wgrad(da, db, dout, pd, wa, wb, wout, pw, split, sms, (cudaStream_t)stream);
}
