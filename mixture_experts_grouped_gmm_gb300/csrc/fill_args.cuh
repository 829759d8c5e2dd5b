// The args block fill (mgemm_fill_args) as a CTA-wide device function, shared by
// the fill kernels and the one-CTA routing and alignment kernel.
#pragma once

#include "common.cuh"

namespace mgemm {

template <typename T, int NT>
__device__ __forceinline__ T block_inclusive_scan(T v, T *warp_tot) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (NW == 1) return v;
  if (lane == 31) warp_tot[w] = v;
  __syncthreads();
  if (w == 0) {
    T s = lane < NW ? warp_tot[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < NW) warp_tot[lane] = s;
  }
  __syncthreads();
  if (w > 0) v += warp_tot[w - 1];
  __syncthreads();
  return v;
}

// The fill of one args block by the NT threads of one CTA (NT >= E); m is the
// size of group threadIdx.x (0 for threads past E).
template <int NT>
__device__ __forceinline__ void fill_args_body(int64_t m, int E, int64_t M, uint8_t *__restrict__ args) {
  __shared__ int64_t s_size[NT];
  __shared__ int64_t tot64[NT / 32 > 0 ? NT / 32 : 1];
  __shared__ int tot32[NT / 32 > 0 ? NT / 32 : 1];
  const ArgsLayout L = args_layout(E);
  const int t = threadIdx.x;
  s_size[t] = m;
  const int any_neg = __syncthreads_or(m < 0);

  // exclusive offsets: offsets[t + 1] = inclusive prefix
  const int64_t incl = block_inclusive_scan<int64_t, NT>(m, tot64);
  int64_t *offsets = (int64_t *)(args + L.offsets);
  if (t == 0) offsets[0] = 0;
  if (t < E) offsets[t + 1] = incl;
  __shared__ int64_t total_sh;
  if (t == E - 1) total_sh = incl;

  // padded offsets: every group rounded up to kColPad rows
  const int64_t padded = (m > 0 ? (m + kColPad - 1) / kColPad : 0) * kColPad;
  const int64_t pincl = block_inclusive_scan<int64_t, NT>(padded, tot64);
  int64_t *poffsets = (int64_t *)(args + L.poffsets);
  if (t == 0) poffsets[0] = 0;
  if (t < E) poffsets[t + 1] = pincl;

  // compaction of non-empty groups and their row-tile prefix
  const int flag = (t < E && m > 0) ? 1 : 0;
  const int pos = block_inclusive_scan<int, NT>(flag, tot32);
  const int tiles = flag ? (int)((m + MGEMM_TILE_M - 1) / MGEMM_TILE_M) : 0;
  const int tile_incl = block_inclusive_scan<int, NT>(tiles, tot32);
  const int pairs = (tiles + 1) / 2;  // 256-row tiles of a CTA pair
  const int pair_incl = block_inclusive_scan<int, NT>(pairs, tot32);
  int *active = (int *)(args + L.active);
  int *mtile_start = (int *)(args + L.mtile_start);
  int *ptile_start = (int *)(args + L.ptile_start);
  if (t == 0) {
    mtile_start[0] = 0;
    ptile_start[0] = 0;
  }
  if (flag) {
    active[pos - 1] = t;
    mtile_start[pos] = tile_incl;
    ptile_start[pos] = pair_incl;
  }
  __shared__ int n_active_sh;
  if (t == E - 1) n_active_sh = pos;
  __syncthreads();

  // wgrad order: rank = #{j : m_j > m_t} + #{j < t : m_j == m_t}
  if (t < E) {
    int rank = 0;
    for (int j = 0; j < E; ++j) {
      const int64_t mj = s_size[j];
      rank += (mj > m) || (mj == m && j < t);
    }
    ((int *)(args + L.wgrad_order))[rank] = t;
  }
  if (t == 0) {
    int st = MGEMM_STATUS_OK;
    // M = -1: the rows are whatever the sizes add up to (below 2^31)
    const bool check = M >= 0;
    if (any_neg)
      st = MGEMM_STATUS_NEGATIVE_SIZE;
    else if (check ? total_sh != M : total_sh >= (int64_t(1) << 31))
      st = MGEMM_STATUS_SUM_MISMATCH;
    int *hdr = (int *)args;
    hdr[0] = st;
    hdr[1] = n_active_sh;
    hdr[2] = E;
    hdr[3] = 0;  // work counter of the colwise quantizer
    *(int64_t *)(args + 16) = check ? M : total_sh;
  }
}

}  // namespace mgemm
