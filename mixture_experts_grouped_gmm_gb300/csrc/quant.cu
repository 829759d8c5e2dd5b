// FP8 quantize kernels: rowwise, and per-group colwise (single and dual).
//
// Source: "[moe training] Optimize FP8 MoE backward pass: fused colwise
// kernel + AMD tuning" (pytorch/ao commit 34322b5): the fused rowwise
// scale+cast (one launch instead of three ops), the per-group colwise kernel
// of bench_colwise_block_configs.py (_colwise_kernel), and the dual colwise
// kernel that quantizes grad_output and A in one launch.
//
// Both kernels are HBM-bound; the design aims at reading the bf16 input once
// from DRAM with 16-byte coalesced loads and writing each fp8 byte once.
//   rowwise: one warp per row; a row of up to 24*256 elements stays in
//            registers between the amax and the cast, so it is read once.
//            Longer rows take a second pass (served by L2).
//   colwise: one 512-thread CTA per (tensor, group, 64-column block); pass 1
//            reduces the column amax over the group's rows, pass 2 re-reads
//            (from L2), casts, transposes 256-row chunks in shared memory and
//            writes each column's bytes contiguously (16-byte stores inside
//            the group, byte stores on the ragged group edges).  CTAs are
//            ordered by group size, largest first, so long groups start early.
#include "common.cuh"

namespace mgemm {

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ float amax8(const uint4 &v, float a) {
  a = fmaxf(a, fabsf(bf16_lo(v.x)));
  a = fmaxf(a, fabsf(bf16_hi(v.x)));
  a = fmaxf(a, fabsf(bf16_lo(v.y)));
  a = fmaxf(a, fabsf(bf16_hi(v.y)));
  a = fmaxf(a, fabsf(bf16_lo(v.z)));
  a = fmaxf(a, fabsf(bf16_hi(v.z)));
  a = fmaxf(a, fabsf(bf16_lo(v.w)));
  a = fmaxf(a, fabsf(bf16_hi(v.w)));
  return a;
}

// 8 bf16 -> 8 e4m3 bytes (x * s is exact: s is a power of two)
__device__ __forceinline__ uint2 cast8(const uint4 &v, float s) {
  uint2 o;
  o.x = (uint32_t)cvt_e4m3x2(bf16_lo(v.x) * s, bf16_hi(v.x) * s) |
        ((uint32_t)cvt_e4m3x2(bf16_lo(v.y) * s, bf16_hi(v.y) * s) << 16);
  o.y = (uint32_t)cvt_e4m3x2(bf16_lo(v.z) * s, bf16_hi(v.z) * s) |
        ((uint32_t)cvt_e4m3x2(bf16_lo(v.w) * s, bf16_hi(v.w) * s) << 16);
  return o;
}

// 8 bf16 -> 8 e4m3 bytes with one power-of-two scale per column
__device__ __forceinline__ uint2 cast8_scaled(const uint4 &v, const float (&s)[8]) {
  uint2 o;
  o.x = (uint32_t)cvt_e4m3x2(bf16_lo(v.x) * s[0], bf16_hi(v.x) * s[1]) |
        ((uint32_t)cvt_e4m3x2(bf16_lo(v.y) * s[2], bf16_hi(v.y) * s[3]) << 16);
  o.y = (uint32_t)cvt_e4m3x2(bf16_lo(v.z) * s[4], bf16_hi(v.z) * s[5]) |
        ((uint32_t)cvt_e4m3x2(bf16_lo(v.w) * s[6], bf16_hi(v.w) * s[7]) << 16);
  return o;
}

__device__ __forceinline__ float warp_max(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------ rowwise
// NCH = chunks of 8 elements per lane kept in registers (row length <= NCH*256);
// NCH = 0 selects the two-pass loop for any length.
template <int NCH>
__global__ void __launch_bounds__(256) quant_rowwise_kernel(const __nv_bfloat16 *__restrict__ in, int64_t R,
                                                            int64_t C, int64_t ld_in, uint8_t *__restrict__ out,
                                                            int64_t ld_out, float *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < R; row += warps_total) {
    const __nv_bfloat16 *src = in + row * ld_in;
    uint8_t *dst = out + row * ld_out;
    float a = 0.f;
    if constexpr (NCH > 0) {
      uint4 v[NCH];
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int64_t c = ((int64_t)j * 32 + lane) * 8;
        if (c < C) {
          v[j] = ldg_nc_v4(src + c);
          a = amax8(v[j], a);
        }
      }
      a = warp_max(a);
      const float s = pow2_scale_from_amax(a);
      if (lane == 0) scales[row] = s;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int64_t c = ((int64_t)j * 32 + lane) * 8;
        if (c < C) *reinterpret_cast<uint2 *>(dst + c) = cast8(v[j], s);
      }
    } else {
      for (int64_t c = (int64_t)lane * 8; c < C; c += 256) a = amax8(ldg_nc_v4(src + c), a);
      a = warp_max(a);
      const float s = pow2_scale_from_amax(a);
      if (lane == 0) scales[row] = s;
      for (int64_t c = (int64_t)lane * 8; c < C; c += 256)
        *reinterpret_cast<uint2 *>(dst + c) = cast8(*reinterpret_cast<const uint4 *>(src + c), s);
    }
  }
}

// ------------------------------------------------------------------ colwise
// One CTA of 512 threads per (tensor, group, 64-column block).  Warp w owns
// columns 8*(w % 8) .. +7 and, per 256-row chunk, rows 128*(w / 8) + 4*lane
// .. +3: each lane loads four 16-byte row pieces (the CTA keeps 64 KB of loads
// in flight), and in pass 2 writes each column's four codes with one 32-bit
// shared-memory store (consecutive lanes -> consecutive words, no bank
// conflicts).  Few, fat CTAs keep the set of group column blocks being read
// small enough that pass 2 re-reads them from L2.
constexpr int kColBlock = 64;                 // columns per CTA (128 bytes of bf16 per row)
constexpr int kColThreads = 512;
constexpr int kRowChunk = 256;                // rows per pass-2 transpose chunk
constexpr int kTPitch = kRowChunk + 16;       // bytes per transposed column in smem

struct ColTensor {
  const __nv_bfloat16 *in;
  uint8_t *out;
  float *sc;
  int64_t C;
  int ncb;  // column blocks
};

__device__ __forceinline__ void amax8_into(float (&a)[8], const uint4 &v) {
  a[0] = fmaxf(a[0], fabsf(bf16_lo(v.x)));
  a[1] = fmaxf(a[1], fabsf(bf16_hi(v.x)));
  a[2] = fmaxf(a[2], fabsf(bf16_lo(v.y)));
  a[3] = fmaxf(a[3], fabsf(bf16_hi(v.y)));
  a[4] = fmaxf(a[4], fabsf(bf16_lo(v.z)));
  a[5] = fmaxf(a[5], fabsf(bf16_hi(v.z)));
  a[6] = fmaxf(a[6], fabsf(bf16_lo(v.w)));
  a[7] = fmaxf(a[7], fabsf(bf16_hi(v.w)));
}

__global__ void __launch_bounds__(kColThreads) quant_colwise_kernel(const uint8_t *__restrict__ args, int E,
                                                                    int64_t M, ColTensor t1, ColTensor t2,
                                                                    int vec_ok) {
  __shared__ float red[2][kColBlock];
  __shared__ float s_scale[kColBlock];
  __shared__ __align__(16) uint8_t tile[kColBlock][kTPitch];

  const ArgsView av(args, E);
  if (*av.status != 0) return;
  const int per_group = t1.ncb + t2.ncb;
  const int item = blockIdx.x;
  const int g = av.wgrad_order[item / per_group];  // largest groups first
  int cb = item % per_group;
  const ColTensor &T = cb < t1.ncb ? t1 : t2;
  if (cb >= t1.ncb) cb -= t1.ncb;
  const int64_t rs = av.offsets[g], re = av.offsets[g + 1];
  const int64_t col0 = (int64_t)cb * kColBlock;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cchunk = warp & 7;          // 8 columns each
  const int rhalf = warp >> 3;          // 0..1
  const int64_t mycol = col0 + cchunk * 8;
  const bool col_ok = mycol < T.C;
  const __nv_bfloat16 *src = T.in + mycol;

  // pass 1: column amax over the group's rows (each lane: two 4-row quads, 8
  // loads in flight)
  float a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = 0.f;
  if (col_ok) {
    for (int64_t r0 = rs + rhalf * 128 + lane * 4; r0 < re; r0 += 512) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + (i & 3) + (i >> 2) * 256;
        if (r < re) v[i] = ldg_nc_v4(src + r * T.C);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (r0 + (i & 3) + (i >> 2) * 256 < re) amax8_into(a, v[i]);
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = warp_max(a[j]);
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) red[rhalf][cchunk * 8 + j] = a[j];
  }
  __syncthreads();
  if (tid < kColBlock) {
    const float s = pow2_scale_from_amax(fmaxf(red[0][tid], red[1][tid]));
    s_scale[tid] = s;
    if (col0 + tid < T.C) T.sc[(int64_t)g * T.C + col0 + tid] = s;
  }
  __syncthreads();
  if (re <= rs) return;

  float sc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) sc[j] = s_scale[cchunk * 8 + j];

  // pass 2: cast, transpose through shared memory, column-contiguous stores.
  // Chunks start on 16-row boundaries of the whole tensor so that interior
  // 16-byte segments of every column are aligned.
  const int64_t base0 = rs & ~(int64_t)15;
  const int lr0 = rhalf * 128 + lane * 4;  // this lane's first row within the chunk
  auto load_chunk = [&](uint4 (&v)[4], int64_t cr) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = cr + lr0 + i;
      v[i] = (col_ok && r >= rs && r < re) ? ldg_nc_v4(src + r * T.C) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 v[4];
  load_chunk(v, base0);
  for (int64_t cr = base0; cr < re; cr += kRowChunk) {
    // codes of column j for rows lr0..lr0+3, one byte per row
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 o = cast8_scaled(v[i], sc);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[j] |= ((o.x >> (8 * j)) & 0xFFu) << (8 * i);
        w[4 + j] |= ((o.y >> (8 * j)) & 0xFFu) << (8 * i);
      }
    }
    // next chunk's loads are in flight while this one is transposed and stored
    if (cr + kRowChunk < re) load_chunk(v, cr + kRowChunk);
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint32_t *>(&tile[cchunk * 8 + j][lr0]) = w[j];
    __syncthreads();
    // 64 columns x 16 segments of 16 rows
#pragma unroll
    for (int k = 0; k < (kColBlock * (kRowChunk / 16)) / kColThreads; ++k) {
      const int idx = tid + k * kColThreads;
      const int c = idx / (kRowChunk / 16);
      const int seg = idx % (kRowChunk / 16);
      const int64_t col = col0 + c;
      const int64_t r0 = cr + seg * 16;
      if (col >= T.C || r0 >= re || r0 + 16 <= rs) continue;
      uint8_t *dst = T.out + col * M + r0;
      const uint8_t *srcb = &tile[c][seg * 16];
      if (vec_ok && r0 >= rs && r0 + 16 <= re) {
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(srcb);
      } else {
        for (int j = 0; j < 16; ++j) {
          const int64_t r = r0 + j;
          if (r >= rs && r < re) dst[j] = srcb[j];
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace mgemm

using namespace mgemm;

template <int NCH>
static void launch_rowwise(const __nv_bfloat16 *in, int64_t R, int64_t C, int64_t ld_in, uint8_t *out,
                           int64_t ld_out, float *scales, cudaStream_t s) {
  const int64_t blocks_needed = (R + 7) / 8;
  int sms = mgemm_num_sms();
  if (sms <= 0) sms = 148;
  const int64_t cap = (int64_t)sms * 32;
  const int blocks = (int)(blocks_needed < cap ? blocks_needed : cap);
  quant_rowwise_kernel<NCH><<<blocks, 256, 0, s>>>(in, R, C, ld_in, out, ld_out, scales);
}

extern "C" int mgemm_quant_rowwise(const void *in, int64_t R, int64_t C, int64_t ld_in, uint8_t *out,
                                   int64_t ld_out, float *scales, mgemm_stream_t stream) {
  if (R < 0 || C < 0) return MGEMM_EINVAL;
  if (R == 0 || C == 0) return MGEMM_OK;
  if (!in || !out || !scales) return MGEMM_EINVAL;
  if (C % 8 || ld_in < C || ld_out < C) return MGEMM_EINVAL;
  if (((uintptr_t)in & 15) || ((uintptr_t)out & 15) || (ld_in % 8) || (ld_out % 16)) return MGEMM_EALIGN;
  const __nv_bfloat16 *x = (const __nv_bfloat16 *)in;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t nch = (C + 255) / 256;
  if (nch <= 1) launch_rowwise<1>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 2) launch_rowwise<2>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 4) launch_rowwise<4>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 6) launch_rowwise<6>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 8) launch_rowwise<8>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 12) launch_rowwise<12>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 16) launch_rowwise<16>(x, R, C, ld_in, out, ld_out, scales, s);
  else if (nch <= 24) launch_rowwise<24>(x, R, C, ld_in, out, ld_out, scales, s);
  else launch_rowwise<0>(x, R, C, ld_in, out, ld_out, scales, s);
  return cuda_rc(cudaGetLastError(), "mgemm_quant_rowwise launch");
}

extern "C" int mgemm_quant_colwise_grouped(const void *args, int E, int64_t M, const void *in1, int64_t C1,
                                           uint8_t *out1, float *sc1, const void *in2, int64_t C2,
                                           uint8_t *out2, float *sc2, mgemm_stream_t stream) {
  if (!args || !in1 || !out1 || !sc1) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || C1 <= 0 || C1 % 8) return MGEMM_EINVAL;
  if (((uintptr_t)args & 15) || ((uintptr_t)in1 & 15)) return MGEMM_EALIGN;
  ColTensor t1{(const __nv_bfloat16 *)in1, out1, sc1, C1, (int)((C1 + kColBlock - 1) / kColBlock)};
  ColTensor t2{nullptr, nullptr, nullptr, 0, 0};
  if (in2) {
    if (!out2 || !sc2 || C2 <= 0 || C2 % 8) return MGEMM_EINVAL;
    if ((uintptr_t)in2 & 15) return MGEMM_EALIGN;
    t2 = ColTensor{(const __nv_bfloat16 *)in2, out2, sc2, C2, (int)((C2 + kColBlock - 1) / kColBlock)};
  }
  const int vec_ok = (M % 16 == 0) && (((uintptr_t)out1 & 15) == 0) && (!in2 || (((uintptr_t)out2 & 15) == 0));
  const int64_t items = (int64_t)E * (t1.ncb + t2.ncb);
  if (items >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  quant_colwise_kernel<<<(unsigned)items, kColThreads, 0, (cudaStream_t)stream>>>((const uint8_t *)args, E, M,
                                                                                  t1, t2, vec_ok);
  return cuda_rc(cudaGetLastError(), "mgemm_quant_colwise_grouped launch");
}
