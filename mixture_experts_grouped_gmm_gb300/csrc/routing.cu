// moe_align_block_size on the device.
//
// Source: pytorch-labs/applied-ai issue 24 (the column-major fused MoE script,
// built on vLLM's fused_moe.py), docstring of moe_align_block_size: the flat
// (token, slot) entries are grouped by expert and each expert's list is padded
// with the id numel to a multiple of block_size; expert_ids names the expert of
// each block.  The worked example there fixes the order inside an expert
// (ascending flat index).
//
// Three kernels, all integer work:
//   count  one CTA per chunk of kChunk entries: a shared-memory histogram of
//          the chunk's experts, written to the workspace as counts[chunk][e].
//   scan   one CTA (one thread per expert): each expert's total and padded
//          count, an exclusive scan over experts for its first position, and
//          counts[chunk][e] rewritten as the chunk's first position for e; it
//          also writes the padding ids, the block experts, the padded total,
//          the group sizes and the tail past the total.
//   place  one CTA per chunk: the chunk is read in rounds of 256 entries; in a
//          round, an entry's place among equal experts is its rank in its warp
//          (__match_any_sync) plus the counts of earlier warps of the round,
//          plus what earlier rounds placed -- the order the docstring shows,
//          with no sort.
#include "common.cuh"

namespace mgemm {

constexpr int kAlignChunk = 2048;   // entries per CTA of the count and place kernels
constexpr int kAlignThreads = 256;  // threads of those CTAs: 8 warps
constexpr int kAlignRounds = kAlignChunk / kAlignThreads;
static_assert(kAlignRounds < 0xFFFF, "round tags fit 16 bits");

__global__ void __launch_bounds__(kAlignThreads) moe_align_count_kernel(const int32_t *__restrict__ ids, int64_t n,
                                                                          int E, int32_t *__restrict__ counts) {
  extern __shared__ int hist[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kAlignChunk;
  for (int j = threadIdx.x; j < kAlignChunk; j += blockDim.x) {
    const int64_t i = base + j;
    if (i < n) {
      const int e = ids[i];
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// One CTA of 1024 threads; thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024) moe_align_scan_kernel(int32_t *__restrict__ counts, int nch, int E,
                                                                int block, int64_t n, int64_t cap, int max_blocks,
                                                                int32_t *__restrict__ sorted_ids,
                                                                int32_t *__restrict__ expert_ids,
                                                                int32_t *__restrict__ num_post,
                                                                int64_t *__restrict__ group_sizes) {
  __shared__ int warp_sum[32];
  __shared__ int total_sh;
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int c = 0;
  if (e < E)
    for (int k = 0; k < nch; ++k) c += counts[(int64_t)k * E + e];
  const int p = e < E ? (c + block - 1) / block * block : 0;  // padded count
  // exclusive scan of p over the block: warp scans, then a scan of the warp sums
  int incl = p;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += v;
    }
    warp_sum[lane] = s;  // inclusive over warps
    if (lane == 31) total_sh = s;
  }
  __syncthreads();
  const int start = incl - p + (warp > 0 ? warp_sum[warp - 1] : 0);
  const int total = total_sh;
  if (e < E) {
    int run = start;
    for (int k = 0; k < nch; ++k) {  // counts -> first position of each chunk's entries of e
      const int64_t idx = (int64_t)k * E + e;
      const int v = counts[idx];
      counts[idx] = run;
      run += v;
    }
    for (int q = start + c; q < start + p; ++q) sorted_ids[q] = (int32_t)n;  // the expert's padding
    for (int b = start / block; b < (start + p) / block; ++b) expert_ids[b] = e;
    if (group_sizes) group_sizes[e] = p;
  }
  if (e == 0) *num_post = total;
  for (int64_t q = total + e; q < cap; q += blockDim.x) sorted_ids[q] = (int32_t)n;
  for (int b = total / block + e; b < max_blocks; b += blockDim.x) expert_ids[b] = -1;
}

__global__ void __launch_bounds__(kAlignThreads) moe_align_place_kernel(const int32_t *__restrict__ ids, int64_t n,
                                                                          int E, const int32_t *__restrict__ first,
                                                                          int32_t *__restrict__ sorted_ids) {
  extern __shared__ int sm[];
  int *run = sm;                                          // [E]: entries of e placed by earlier rounds
  uint32_t *wcnt = reinterpret_cast<uint32_t *>(sm + E);  // [8 warps][E]: (round << 16) | count
  for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = 0;
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0xFFFFFFFFu;  // no round matches
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;
  const int64_t base = (int64_t)blockIdx.x * kAlignChunk;
  const int32_t *fst = first + (int64_t)blockIdx.x * E;
  for (int r = 0; r < kAlignRounds; ++r) {
    const int64_t i = base + (int64_t)r * kAlignThreads + threadIdx.x;
    int e = -1;
    if (i < n) {
      e = ids[i];
      if (e < 0 || e >= E) e = -1;  // not placed
    }
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & below);
    const bool leader = rank == 0;
    if (e >= 0 && leader) wcnt[warp * E + e] = ((uint32_t)r << 16) | (uint32_t)__popc(same);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) {
        const uint32_t v = wcnt[w * E + e];
        if ((v >> 16) == (uint32_t)r) before += (int)(v & 0xFFFFu);
      }
      sorted_ids[fst[e] + run[e] + before + rank] = (int32_t)i;
    }
    __syncthreads();
    if (e >= 0 && leader) atomicAdd(&run[e], __popc(same));
    __syncthreads();
  }
}

}  // namespace mgemm

using namespace mgemm;

extern "C" int64_t mgemm_moe_align_workspace_bytes(int64_t numel, int E) {
  if (numel < 0 || E < 1 || E > MGEMM_MAX_EXPERTS) return -1;
  const int64_t nch = (numel + kAlignChunk - 1) / kAlignChunk;
  const int64_t b = nch * E * 4;
  return b < 16 ? 16 : (b + 15) / 16 * 16;
}

extern "C" int mgemm_moe_align(const int32_t *topk_ids, int64_t numel, int E, int block_size, int32_t *sorted_ids,
                               int32_t *expert_ids, int32_t *num_post_padded, int64_t *group_sizes, void *workspace,
                               mgemm_stream_t stream) {
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (numel < 0 || block_size < 1 || block_size > 4096) return MGEMM_EINVAL;
  const int64_t cap = numel + (int64_t)E * (block_size - 1);
  if (cap >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (!sorted_ids || !expert_ids || !num_post_padded || !workspace || (numel > 0 && !topk_ids)) return MGEMM_EINVAL;
  if (((uintptr_t)topk_ids & 3) || ((uintptr_t)sorted_ids & 3) || ((uintptr_t)expert_ids & 3) ||
      ((uintptr_t)num_post_padded & 3) || ((uintptr_t)group_sizes & 7) || ((uintptr_t)workspace & 15))
    return MGEMM_EALIGN;
  const int max_blocks = (int)(cap / block_size);
  const int nch = (int)((numel + kAlignChunk - 1) / kAlignChunk);
  int32_t *counts = static_cast<int32_t *>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  if (nch > 0) {
    moe_align_count_kernel<<<nch, kAlignThreads, (size_t)E * 4, s>>>(topk_ids, numel, E, counts);
    int rc = cuda_rc(cudaGetLastError(), "moe_align count launch");
    if (rc) return rc;
  }
  moe_align_scan_kernel<<<1, 1024, 0, s>>>(counts, nch, E, block_size, numel, cap, max_blocks, sorted_ids,
                                           expert_ids, num_post_padded, group_sizes);
  int rc = cuda_rc(cudaGetLastError(), "moe_align scan launch");
  if (rc) return rc;
  if (nch > 0) {
    const size_t smem = (size_t)E * 4 * 9;  // run[E] + 8 warps x E counts: at most 36 KB
    moe_align_place_kernel<<<nch, kAlignThreads, smem, s>>>(topk_ids, numel, E, counts, sorted_ids);
    rc = cuda_rc(cudaGetLastError(), "moe_align place launch");
  }
  return rc;
}
