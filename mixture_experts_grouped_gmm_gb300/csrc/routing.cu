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
#include "fill_args.cuh"

namespace mgemm {

constexpr int kAlignChunk = 2048;   // entries per CTA of the count and place kernels
constexpr int kAlignThreads = 256;  // threads of those CTAs: 8 warps
constexpr int kAlignRounds = kAlignChunk / kAlignThreads;
static_assert(kAlignRounds < 0xFFFF, "round tags fit 16 bits");

__global__ void __launch_bounds__(kAlignThreads) moe_align_count_kernel(const int32_t *__restrict__ ids, int64_t n,
                                                                          int E, int32_t *__restrict__ counts) {
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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

// Row s of dst (s below the padded total and dst_rows) is row ids[s] / top_k of
// src, or zeros for a padding entry (ids[s] >= numel) -- the rows the masked
// loads of fused_moe_kernel see.  One warp per row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ src, int64_t src_rows,
                                                            int64_t row_chunks, int64_t src_ld, int64_t dst_ld,
                                                            const int32_t *__restrict__ ids,
                                                            const int32_t *__restrict__ num_post, int64_t numel,
                                                            int top_k, uint4 *__restrict__ dst, int64_t dst_rows) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = *num_post;
  const int64_t rows = total < dst_rows ? total : dst_rows;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t s = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); s < rows; s += nwarps) {
    const int32_t id = __ldg(ids + s);
    const int64_t r = id >= 0 && id < numel ? id / top_k : -1;
    const bool ok = r >= 0 && r < src_rows;
    const uint4 *sp = src + (ok ? r : 0) * src_ld;
    uint4 *dp = dst + s * dst_ld;
#pragma unroll 4
    for (int64_t c = lane; c < row_chunks; c += 32) dp[c] = ok ? __ldg(sp + c) : make_uint4(0, 0, 0, 0);
  }
}

// out[r, j] = silu(in[r, j]) * in[r, F + j], silu(v) = v / (1 + exp(-v)),
// in fp32 from the bf16 inputs, rounded to bf16 once; 8 columns per thread.
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint4 *__restrict__ in, int64_t R, int64_t F8,
                                                         uint4 *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = R * F8;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = c / F8, j = c - row * F8;
    const uint4 g = __ldg(in + row * 2 * F8 + j), u = __ldg(in + row * 2 * F8 + F8 + j);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float g0 = __uint_as_float(gw[k] << 16), g1 = __uint_as_float(gw[k] & 0xFFFF0000u);
      const float u0 = __uint_as_float(uw[k] << 16), u1 = __uint_as_float(uw[k] & 0xFFFF0000u);
      const float h0 = g0 / (1.f + expf(-g0)) * u0, h1 = g1 / (1.f + expf(-g1)) * u1;
      __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
      o[k] = *reinterpret_cast<uint32_t *>(&b);
    }
    out[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// out[t, :] = sum over j < top_k of in[t * top_k + j, :], in fp32 (ascending j),
// rounded to bf16 once; 8 columns per thread.
__global__ void __launch_bounds__(256) topk_sum_kernel(const uint4 *__restrict__ in, int64_t T, int top_k,
                                                         int64_t H8, uint4 *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t n = T * H8;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = c / H8, j = c - t * H8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < top_k; ++k) {
      const uint4 v = __ldg(in + (t * top_k + k) * H8 + j);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += __uint_as_float(w[q] << 16);
        acc[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<uint32_t *>(&b);
    }
    out[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// fused_moe's routing, one warp per token: softmax over the E experts of the
// token's gating logits and the top_k largest probabilities, largest first.
// The selection compares the logits (softmax is increasing in each of them, so
// this picks the same experts without rounding ties), equal logits going to the
// lower expert id; the weights are exp(l - max) / sum, in fp32 with expf, and
// divided by their sum when renormalize.  Lane l holds experts l, l + 32, ...
// One warp routes token t; ids_sh, when given, receives the token's ids too.
template <int NV>
__device__ __forceinline__ void topk_softmax_token(const float *__restrict__ gating, int64_t t, int E, int top_k,
                                                   int renormalize, float *__restrict__ weights,
                                                   int32_t *__restrict__ ids, int32_t *ids_sh) {
  const int lane = threadIdx.x & 31;
  const float *row = gating + t * E;
  float v[NV];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? __ldg(row + e) : -INFINITY;
    m = fmaxf(m, v[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (lane + 32 * j < E) sum += expf(v[j] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  uint32_t taken = 0;
  float wsel = 0.f, wsum = 0.f;  // lane r keeps the weight of pick r
  int isel = 0;
  for (int r = 0; r < top_k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && (v[j] > bv || (v[j] == bv && e < bi))) {
        bv = v[j];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);  // the owner marks it
    const float w = expf(bv - m) / sum;
    wsum += w;
    if (lane == (r & 31)) {
      wsel = w;
      isel = bi;
    }
    if ((r & 31) == 31 || r == top_k - 1) {  // flush up to 32 picks
      const int r0 = r & ~31;
      if (lane <= r - r0) {
        ids[t * top_k + r0 + lane] = isel;
        if (ids_sh) ids_sh[t * top_k + r0 + lane] = isel;
        weights[t * top_k + r0 + lane] = wsel;  // renormalized below
      }
    }
  }
  if (renormalize) {
    __syncwarp();
    for (int r = lane; r < top_k; r += 32) weights[t * top_k + r] = weights[t * top_k + r] / wsum;
  }
}

template <int NV>
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float *__restrict__ gating, int64_t T, int E,
                                                             int top_k, int renormalize, float *__restrict__ weights,
                                                             int32_t *__restrict__ ids) {
  pdl_wait();
  pdl_trigger();
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // whole warps leave together
  topk_softmax_token<NV>(gating, t, E, top_k, renormalize, weights, ids, nullptr);
}

// mgemm_moe_route_align: the routing, the alignment and the args block of a
// batch of at most MGEMM_ROUTE_ALIGN_MAX_ENTRIES entries in one CTA, so that a
// decode-size batch takes one launch instead of five.  Each step computes what
// its own kernel above computes (the same device code for the routing; the
// same counts, scan, tail fill and round-wise stable placement for the
// alignment; the args fill of mgemm_fill_args with M = -1), so the results are
// the same bit for bit; the experts of the entries stay in shared memory
// between the steps.  Thread e owns expert e in the scan (E <= NT threads);
// the placement takes rounds of NT entries, one per thread.  NT is 128 or 256
// for the smallest batches (fewer threads make the many CTA barriers cheaper),
// else 1024.
__host__ __device__ constexpr size_t route_align_smem(int64_t n, int E, int NT) {
  return 4 * (size_t)n + 4 * (size_t)E * (3 + NT / 32);
}

template <int NV, int NT>
__global__ void __launch_bounds__(NT, 1)
    route_align_kernel(const float *__restrict__ gating, int T, int E, int top_k, int renormalize, int block,
                       int64_t cap, int max_blocks, float *__restrict__ weights, int32_t *__restrict__ ids,
                       int32_t *__restrict__ sorted_ids, int32_t *__restrict__ expert_ids,
                       int32_t *__restrict__ num_post, int64_t *__restrict__ group_sizes, uint8_t *__restrict__ args) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int ra_sm[];
  const int n = T * top_k;
  int32_t *s_e = ra_sm;                            // [n]: expert of each entry
  int *cnt = ra_sm + n;                            // [E]: entries of expert e
  int *first = cnt + E;                            // [E]: first sorted position of expert e
  int *run = first + E;                            // [E]: entries of e placed by earlier rounds
  uint32_t *wcnt = reinterpret_cast<uint32_t *>(run + E);  // [warps][E]: (round << 16) | count
  constexpr int kWarps = NT / 32;
  __shared__ int warp_sum[kWarps];
  __shared__ int total_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += NT) {
    cnt[e] = 0;
    run[e] = 0;
  }
  for (int i = tid; i < kWarps * E; i += NT) wcnt[i] = 0xFFFFFFFFu;  // no round matches
  // routing, one warp per token; or the caller's ids
  if (gating) {
    for (int t = warp; t < T; t += kWarps) topk_softmax_token<NV>(gating, t, E, top_k, renormalize, weights, ids, s_e);
  } else {
    for (int i = tid; i < n; i += NT) s_e[i] = ids[i];
  }
  __syncthreads();
  // counts (entries outside [0, E) are not placed)
  for (int i = tid; i < n; i += NT) {
    const int e = s_e[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  // padded counts and their exclusive scan over the experts
  const int c = tid < E ? cnt[tid] : 0;
  const int pc = tid < E ? (c + block - 1) / block * block : 0;
  int incl = pc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < kWarps ? warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane < kWarps) warp_sum[lane] = v;
    if (lane == 31) total_sh = v;
  }
  __syncthreads();
  const int start = incl - pc + (warp > 0 ? warp_sum[warp - 1] : 0);
  const int total = total_sh;
  if (tid < E) {
    first[tid] = start;
    for (int q = start + c; q < start + pc; ++q) sorted_ids[q] = n;  // the expert's padding
    for (int b = start / block; b < (start + pc) / block; ++b) expert_ids[b] = tid;
    if (group_sizes) group_sizes[tid] = pc;
  }
  if (tid == 0) *num_post = total;
  for (int64_t q = total + tid; q < cap; q += NT) sorted_ids[q] = n;
  for (int b = total / block + tid; b < max_blocks; b += NT) expert_ids[b] = -1;
  __syncthreads();
  // stable placement: an entry's place among its expert's entries is its rank
  // in its warp plus the counts of earlier warps of the round plus what
  // earlier rounds placed
  const uint32_t below = (1u << lane) - 1u;
  for (int r = 0; r * NT < n; ++r) {
    const int i = r * NT + tid;
    int e = -1;
    if (i < n) {
      e = s_e[i];
      if (e < 0 || e >= E) e = -1;
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
      sorted_ids[first[e] + run[e] + before + rank] = i;
    }
    __syncthreads();
    if (e >= 0 && leader) atomicAdd(&run[e], __popc(same));
    __syncthreads();
  }
  // the args block of the padded group sizes (M = -1: their sum)
  fill_args_body<NT>((int64_t)pc, E, -1, args);
}

template <int NV, int NT>
int launch_route_align(size_t smem, cudaStream_t s, const float *gating, int T, int E, int top_k, int renormalize,
                       int block, int64_t cap, int max_blocks, float *weights, int32_t *ids, int32_t *sorted_ids,
                       int32_t *expert_ids, int32_t *num_post, int64_t *group_sizes, uint8_t *args) {
  static bool attr_done[64] = {};
  int dev = 0;
  int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return MGEMM_EINVAL;
  if (!attr_done[dev]) {
    rc = cuda_rc(cudaFuncSetAttribute(route_align_kernel<NV, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)route_align_smem(MGEMM_ROUTE_ALIGN_MAX_ENTRIES, NT, NT)),
                 "cudaFuncSetAttribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  return launch_pdl(route_align_kernel<NV, NT>, dim3(1), dim3(NT), smem, s, 1, "mgemm_moe_route_align launch",
                    gating, T, E, top_k, renormalize, block, cap, max_blocks, weights, ids, sorted_ids, expert_ids,
                    num_post, group_sizes, args);
}

}  // namespace mgemm

using namespace mgemm;

extern "C" int mgemm_topk_softmax(const float *gating, int64_t T, int E, int top_k, int renormalize,
                                  float *topk_weights, int32_t *topk_ids, mgemm_stream_t stream) {
  if (T < 0 || E < 1 || E > MGEMM_MAX_EXPERTS || top_k < 1 || top_k > E) return MGEMM_EINVAL;
  if (T == 0) return MGEMM_OK;
  if (!gating || !topk_weights || !topk_ids) return MGEMM_EINVAL;
  if (((uintptr_t)gating & 3) || ((uintptr_t)topk_weights & 3) || ((uintptr_t)topk_ids & 3)) return MGEMM_EALIGN;
  const int64_t blocks = (T + 7) / 8;
  if (blocks >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  const int nv = (E + 31) / 32;
#define MGEMM_TOPK_LAUNCH(NV)                                                                                 \
  return launch_pdl(topk_softmax_kernel<NV>, dim3((unsigned)blocks), dim3(256), 0, s, 1, "mgemm_topk_softmax launch", \
                    gating, T, E, top_k, renormalize, topk_weights, topk_ids)
  if (nv <= 1) MGEMM_TOPK_LAUNCH(1);
  if (nv <= 2) MGEMM_TOPK_LAUNCH(2);
  if (nv <= 4) MGEMM_TOPK_LAUNCH(4);
  if (nv <= 8) MGEMM_TOPK_LAUNCH(8);
  if (nv <= 16) MGEMM_TOPK_LAUNCH(16);
  MGEMM_TOPK_LAUNCH(32);
#undef MGEMM_TOPK_LAUNCH
}

extern "C" int mgemm_topk_sum(const void *in, int64_t T, int top_k, int64_t H, void *out, mgemm_stream_t stream) {
  if (!in || !out || T < 0 || top_k < 1 || H < 0) return MGEMM_EINVAL;
  if (H % 8 || ((uintptr_t)in & 15) || ((uintptr_t)out & 15)) return MGEMM_EALIGN;
  if (T == 0 || H == 0) return MGEMM_OK;
  int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  const int64_t n = T * (H / 8);
  const int64_t want = (n + 255) / 256;
  const int blocks = (int)(want < (int64_t)sms * 32 ? want : (int64_t)sms * 32);
  return launch_pdl(topk_sum_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, 1, "mgemm_topk_sum launch",
                    (const uint4 *)in, T, top_k, H / 8, (uint4 *)out);
}

extern "C" int mgemm_gather_rows(const void *src, int64_t src_rows, int64_t row_bytes, int64_t src_ld_bytes,
                                 const int32_t *sorted_ids, const int32_t *num_post_padded, int64_t numel, int top_k,
                                 void *dst, int64_t dst_rows, int64_t dst_ld_bytes, mgemm_stream_t stream) {
  if (!src || !sorted_ids || !num_post_padded || !dst) return MGEMM_EINVAL;
  if (src_rows < 0 || dst_rows < 0 || numel < 0 || top_k < 1 || row_bytes <= 0) return MGEMM_EINVAL;
  if (src_ld_bytes < row_bytes || dst_ld_bytes < row_bytes) return MGEMM_EINVAL;
  if (row_bytes % 16 || src_ld_bytes % 16 || dst_ld_bytes % 16 || ((uintptr_t)src & 15) || ((uintptr_t)dst & 15) ||
      ((uintptr_t)sorted_ids & 3) || ((uintptr_t)num_post_padded & 3))
    return MGEMM_EALIGN;
  if (dst_rows == 0) return MGEMM_OK;
  int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  const int64_t want = (dst_rows + 7) / 8;
  const int blocks = (int)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
  return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, 1, "mgemm_gather_rows launch",
                    (const uint4 *)src, src_rows, row_bytes / 16, src_ld_bytes / 16, dst_ld_bytes / 16, sorted_ids,
                    num_post_padded, numel, top_k, (uint4 *)dst, dst_rows);
}

extern "C" int mgemm_silu_and_mul(const void *in, int64_t R, int64_t F, void *out, mgemm_stream_t stream) {
  if (!in || !out || R < 0 || F < 0) return MGEMM_EINVAL;
  if (F % 8 || ((uintptr_t)in & 15) || ((uintptr_t)out & 15)) return MGEMM_EALIGN;
  if (R == 0 || F == 0) return MGEMM_OK;
  int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  const int64_t n = R * (F / 8);
  const int64_t want = (n + 255) / 256;
  const int blocks = (int)(want < (int64_t)sms * 32 ? want : (int64_t)sms * 32);
  return launch_pdl(silu_mul_kernel, dim3(blocks), dim3(256), 0, (cudaStream_t)stream, 1, "mgemm_silu_and_mul launch",
                    (const uint4 *)in, R, F / 8, (uint4 *)out);
}

extern "C" int mgemm_moe_route_align(const float *gating, int64_t T, int E, int top_k, int renormalize,
                                     int block_size, float *topk_weights, int32_t *topk_ids, int32_t *sorted_ids,
                                     int32_t *expert_ids, int32_t *num_post_padded, int64_t *group_sizes, void *args,
                                     mgemm_stream_t stream) {
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (T < 0 || top_k < 1 || (gating && top_k > E) || block_size < 1 || block_size > 4096) return MGEMM_EINVAL;
  if (T > MGEMM_ROUTE_ALIGN_MAX_ENTRIES || T * top_k > MGEMM_ROUTE_ALIGN_MAX_ENTRIES) return MGEMM_EINVAL;
  const int64_t numel = T * top_k;
  const int64_t cap = numel + (int64_t)E * (block_size - 1);
  if (cap >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  // (no tokens: the ids and weights may be NULL)
  if (!sorted_ids || !expert_ids || !num_post_padded || !args || (numel > 0 && !topk_ids) ||
      (gating && numel > 0 && !topk_weights))
    return MGEMM_EINVAL;
  if (((uintptr_t)gating & 3) || ((uintptr_t)topk_weights & 3) || ((uintptr_t)topk_ids & 3) ||
      ((uintptr_t)sorted_ids & 3) || ((uintptr_t)expert_ids & 3) || ((uintptr_t)num_post_padded & 3) ||
      ((uintptr_t)group_sizes & 7) || ((uintptr_t)args & 15))
    return MGEMM_EALIGN;
  const int max_blocks = (int)(cap / block_size);
  cudaStream_t s = (cudaStream_t)stream;
  const int nv = (E + 31) / 32;
  uint8_t *a = static_cast<uint8_t *>(args);
  // 128 threads for at most 8 tokens (two per warp) over at most 128 experts, 256 for at most
  // 8 tokens over at most 256 experts
  const bool small = E <= 128 && T <= 8, mid = E <= 256 && T <= 8;
#define MGEMM_RA_LAUNCH(NV, NT)                                                                                   \
  return launch_route_align<NV, NT>(route_align_smem(numel, E, NT), s, gating, (int)T, E, top_k, renormalize,   \
                                    block_size, cap, max_blocks, topk_weights, topk_ids, sorted_ids, expert_ids, \
                                    num_post_padded, group_sizes, a)
  if (small) {
    if (nv <= 1) MGEMM_RA_LAUNCH(1, 128);
    if (nv <= 2) MGEMM_RA_LAUNCH(2, 128);
    MGEMM_RA_LAUNCH(4, 128);
  }
  if (mid) MGEMM_RA_LAUNCH(8, 256);
  if (nv <= 1) MGEMM_RA_LAUNCH(1, 1024);
  if (nv <= 2) MGEMM_RA_LAUNCH(2, 1024);
  if (nv <= 4) MGEMM_RA_LAUNCH(4, 1024);
  if (nv <= 8) MGEMM_RA_LAUNCH(8, 1024);
  if (nv <= 16) MGEMM_RA_LAUNCH(16, 1024);
  MGEMM_RA_LAUNCH(32, 1024);
#undef MGEMM_RA_LAUNCH
}

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
    int rc = launch_pdl(moe_align_count_kernel, dim3(nch), dim3(kAlignThreads), (size_t)E * 4, s, 1,
                        "moe_align count launch", topk_ids, numel, E, counts);
    if (rc) return rc;
  }
  int rc = launch_pdl(moe_align_scan_kernel, dim3(1), dim3(1024), 0, s, 1, "moe_align scan launch", counts, nch, E,
                      block_size, numel, cap, max_blocks, sorted_ids, expert_ids, num_post_padded, group_sizes);
  if (rc) return rc;
  if (nch > 0) {
    const size_t smem = (size_t)E * 4 * 9;  // run[E] + 8 warps x E counts: at most 36 KB
    rc = launch_pdl(moe_align_place_kernel, dim3(nch), dim3(kAlignThreads), smem, s, 1, "moe_align place launch",
                    topk_ids, numel, E, (const int32_t *)counts, sorted_ids);
  }
  return rc;
}
