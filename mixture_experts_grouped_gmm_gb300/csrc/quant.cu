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
//   colwise: persistent CTAs (one per SM) fed by TMA through a 6-stage ring
//            of 256-row x 64-column boxes, over (group, tensor, column-block)
//            items in order of decreasing group size; 16 consumer warps read
//            the boxes with transposing ldmatrix, reduce the column magnitude
//            max (pass 1; the first 8 boxes are parked in tensor memory),
//            then convert two rows of one column per e4m3x2
//            conversion so the codes come out column-major (pass 2), stage
//            them in shared memory, and write them with TMA tensor stores,
//            each column's bytes contiguous.
#include "common.cuh"

namespace mgemm {

// ------------------------------------------------------------------ rowwise
// NCH = chunks of 8 elements per lane kept in registers (row length <= NCH*256);
// NCH = 0 selects the two-pass loop for any length.
template <int NCH>
__global__ void __launch_bounds__(256) quant_rowwise_kernel(const __nv_bfloat16 *__restrict__ in, int64_t R,
                                                            int64_t C, int64_t ld_in, uint8_t *__restrict__ out,
                                                            int64_t ld_out, float *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
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
      quant_row_two_pass(src, C, dst, scales + row, lane);
    }
  }
}

// ------------------------------------------------------------------ MX blocks
// One warp per row, 8 elements (16 bytes) per lane and chunk of 256 (NCH chunks'
// loads in flight per round, sized to the row on the host): lanes
// 4j .. 4j + 3 hold block j of the chunk, whose magnitude maximum two
// shuffles combine.  The scale is the rowwise rule applied per block; the
// e8m0 byte 127 - log2(s) is 254 minus s's biased exponent (s is a power of
// two, always normal).
// NCH chunks of 256 elements per round, their loads issued first (a row of up
// to NCH * 256 elements in one round).
template <int NCH>
__global__ void __launch_bounds__(256) quant_mx_kernel(const __nv_bfloat16 *__restrict__ in, int64_t R, int64_t C,
                                                       int64_t ld_in, uint8_t *__restrict__ out, int64_t ld_out,
                                                       uint8_t *__restrict__ sf, int64_t ld_sf) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < R; row += warps_total) {
    const __nv_bfloat16 *src = in + row * ld_in;
    uint8_t *dst = out + row * ld_out;
    for (int64_t c0 = 0; c0 < C; c0 += NCH * 256) {
      uint4 v[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int64_t c = c0 + i * 256 + lane * 8;
        v[i] = c < C ? ldg_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int64_t c = c0 + i * 256 + lane * 8;
        const bool live = c < C;  // C % 32 == 0: a block's four lanes agree
        float a = amax8(v[i], 0.f);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const float s = pow2_scale_from_amax(a);
        if (live) {
          *reinterpret_cast<uint2 *>(dst + c) = cast8(v[i], s);
          if ((lane & 3) == 0) sf[row * ld_sf + c / 32] = (uint8_t)(254u - (__float_as_uint(s) >> 23));
        }
      }
    }
  }
}

// ------------------------------------------------------------ INT4 blocks
// The weights of the FP8 x INT4 grouped GEMM ("F8I4 Grouped Gemm
// Optimization for Sparse M", FBGEMM PR #3854; the page gives no format, this
// is the library's reading): w [E, N, K] bf16, one warp per row (e, n), 8
// elements per lane and chunk of 256; lanes 4j .. 4j + 3 hold block j of 32.
// Per block: s = 2^floor(log2(fp32(7 / max(amax, 1e-12)))), q = clamp(
// round_half_even(w s), -8, 7) (w s is exact), nibbles packed two per byte
// along K (element 2i in the low nibble of byte i), and the e8m0 byte of the
// decode factor 1 / s (254 minus s's biased exponent) stored contraction-block
// major: sf[((e (K / 128) + k / 128) N + n) 4 + (k % 128) / 32], so that the
// scales of BN consecutive rows for one block of 128 are BN x 4 contiguous bytes.
__device__ __forceinline__ float int4_scale_from_amax(float amax) {
  const float s = __fdiv_rn(7.0f, fmaxf(amax, 1e-12f));
  return __uint_as_float(__float_as_uint(s) & 0x7F800000u);
}

__device__ __forceinline__ uint32_t nib(float v, float s) {
  const int q = min(7, max(-8, __float2int_rn(v * s)));
  return (uint32_t)q & 15u;
}

// 8 bf16 -> 8 packed nibbles (element 0 in bits 0-3)
__device__ __forceinline__ uint32_t pack8_int4(const uint4 &v, float s) {
  return nib(bf16_lo(v.x), s) | nib(bf16_hi(v.x), s) << 4 | nib(bf16_lo(v.y), s) << 8 | nib(bf16_hi(v.y), s) << 12 |
         nib(bf16_lo(v.z), s) << 16 | nib(bf16_hi(v.z), s) << 20 | nib(bf16_lo(v.w), s) << 24 |
         nib(bf16_hi(v.w), s) << 28;
}

template <int NCH>
__global__ void __launch_bounds__(256) quant_int4_kernel(const __nv_bfloat16 *__restrict__ in, int64_t R, int N, int K,
                                                         int64_t ld_in, uint8_t *__restrict__ out,
                                                         uint8_t *__restrict__ sf) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int kblocks = K / 128;
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < R; row += warps_total) {
    const int64_t e = row / N, n = row % N;
    const __nv_bfloat16 *src = in + row * ld_in;
    uint8_t *dst = out + row * (K / 2);
    for (int c0 = 0; c0 < K; c0 += NCH * 256) {
      uint4 v[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int c = c0 + i * 256 + lane * 8;
        v[i] = c < K ? ldg_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int c = c0 + i * 256 + lane * 8;
        float a = amax8(v[i], 0.f);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const float s = int4_scale_from_amax(a);
        if (c < K) {  // K % 128 == 0: a block's four lanes agree
          *reinterpret_cast<uint32_t *>(dst + c / 2) = pack8_int4(v[i], s);
          if ((lane & 3) == 0)
            sf[((e * kblocks + c / 128) * N + n) * 4 + (c % 128) / 32] = (uint8_t)(254u - (__float_as_uint(s) >> 23));
        }
      }
    }
  }
}

// ------------------------------------------------------------ MX colwise
// Per-group colwise MX blocks (the wgrad operands).  CTA (column block, j):
// rows 128 j .. 128 j + 127 of the padded column-major layout, which lie in
// one group g (every group spans a multiple of 128 padded rows), and 64
// columns of one tensor.  The bf16 tile is staged in shared memory ([128
// rows][64 columns], loaded 16 bytes per thread, rows past the group as
// zeros); thread (s, c) then takes column c's 32-row sub-block s: its
// magnitude maximum, the scale, 32 codes written as two 16-byte stores into
// the column, and one e8m0 byte at sf[(j C + c) 4 + s].
struct MxColTensor {
  const __nv_bfloat16 *in;
  uint8_t *out;
  uint8_t *sf;
  int64_t C;
  int ncb;  // 64-column blocks
};

__global__ void __launch_bounds__(256) quant_colwise_mx_kernel(const uint8_t *__restrict__ args, int E, int64_t ld,
                                                               MxColTensor t1, MxColTensor t2) {
  __shared__ __align__(16) __nv_bfloat16 tile[128][64];
  __shared__ __align__(16) uint8_t codes[64][144];  // [column][128 rows] + 16 bytes of padding (banks)
  pdl_wait();
  pdl_trigger();
  const ArgsView av(args, E);
  if (*av.status != 0) return;
  // CTA b: column block b % ncb (of both tensors), row block b / ncb, so that
  // CTAs running together read whole rows
  const int ncb = t1.ncb + t2.ncb;
  const int cb = (int)(blockIdx.x % (unsigned)ncb);
  const int64_t jb = (int64_t)(blockIdx.x / (unsigned)ncb);
  const int64_t r0p = jb * 128;  // first padded row of the block
  if (r0p >= __ldg(av.poffsets + E)) return;
  const bool second = cb >= t1.ncb;
  const MxColTensor &T = second ? t2 : t1;
  const int64_t col0 = (int64_t)(second ? cb - t1.ncb : cb) * 64;
  // the group holding padded row r0p
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(av.poffsets + mid) <= r0p) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int64_t lr0 = r0p - __ldg(av.poffsets + g);                        // row of the group
  const int64_t m = __ldg(av.offsets + g + 1) - __ldg(av.offsets + g);     // its rows
  const int64_t gr0 = __ldg(av.offsets + g) + lr0;                         // first input row
  const int t = threadIdx.x;
  // load: thread t covers columns 8 (t % 8) .. + 7 of rows t / 8 + 32 i
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = t / 8 + 32 * i;
    const int64_t c = col0 + 8 * (t % 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (lr0 + r < m && c < T.C) v = ldg_nc_v4(T.in + (gr0 + r) * T.C + c);
    *reinterpret_cast<uint4 *>(&tile[r][8 * (t % 8)]) = v;
  }
  __syncthreads();
  // convert: warp w takes sub-block s = w / 2 of columns 32 (w % 2) .. + 31
  const int w = t >> 5, lane = t & 31;
  const int sblk = w >> 1, cc = 32 * (w & 1) + lane;
  const int64_t col = col0 + cc;
  float a = 0.f;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __bfloat162float(tile[32 * sblk + i][cc]);
    a = fmaxf(a, fabsf(v[i]));
  }
  const float sc = pow2_scale_from_amax(a);
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    q[i] = (uint32_t)cvt_e4m3x2(v[4 * i] * sc, v[4 * i + 1] * sc) |
           ((uint32_t)cvt_e4m3x2(v[4 * i + 2] * sc, v[4 * i + 3] * sc) << 16);
  uint4 *cdst = reinterpret_cast<uint4 *>(&codes[cc][32 * sblk]);
  cdst[0] = make_uint4(q[0], q[1], q[2], q[3]);
  cdst[1] = make_uint4(q[4], q[5], q[6], q[7]);
  if (col < T.C) T.sf[(jb * T.C + col) * 4 + sblk] = (uint8_t)(254u - (__float_as_uint(sc) >> 23));
  __syncthreads();
  // store: 16-byte piece p of column c (chunk t + 256 i = 8 c + p), so a warp
  // writes four whole 128-byte column segments
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int id = t + 256 * i, c = id >> 3, part = id & 7;
    if (col0 + c < T.C)
      *reinterpret_cast<uint4 *>(T.out + (col0 + c) * ld + r0p + 16 * part) =
          *reinterpret_cast<const uint4 *>(&codes[c][16 * part]);
  }
}

// ------------------------------------------------------------------ colwise
// Persistent, TMA-fed.  Work item = (group, tensor, 64-column block), items
// in order of decreasing group size, handed out one at a time from a counter
// in the args block (dynamic scheduling keeps the CTAs balanced when group
// sizes are skewed).
//   warp 16 (one thread): streams boxes of 256 rows x 64 columns (32 KB,
//            128-byte swizzle) of the item's column block through a 6-stage
//            ring (192 KB of loads in flight per SM), running ahead across
//            items.  Boxes start at the group's first row and cover its rows
//            rounded up to kColPad (the padded length of its output column).
//   warps 0-15: warp w owns columns 8*(w % 8) .. +7 and rows 128*(w / 8) ..
//            +127 of each box.  ldmatrix.x4.trans reads 32 rows x 8 columns
//            (conflict-free under the swizzle) and hands lane t, in each of
//            its 4 registers, two consecutive rows of column t / 4.  Pass 1
//            keeps a packed bf16x2 running max of magnitudes; pass 2 scales
//            each register with one packed fp32 multiply and converts it to an
//            e4m3 pair that is already in column-major order, stores it as 16
//            bits into one of two tiles (two [64 columns][128 rows] halves,
//            16-byte chunks swizzled by the column); each warp's 8 columns x
//            128 rows form a 1 KB block of the tile, which the warp writes out
//            with its own TMA tensor store while it converts the next box into
//            the other tile -- no CTA-wide barrier per box.  Rows past the
//            group are cleared before the cast, so the padding of every
//            column is written as zero codes.  Between the passes the
//            first 8 boxes of an item wait in tensor memory (each warp parks
//            its 16 registers per box with tcgen05.st and reads them back in
//            pass 2), so every ring slot is freed right after pass 1 and the
//            loads of the next item stream meanwhile; boxes past the 8th are
//            read again, newest first.
// Output: the padded column-major layout -- column c of group g starts at
// out[c * ld + poffsets[g]] (poffsets from the args block), m_g codes then
// zeros up to a multiple of kColPad; every start is 128-byte aligned, so the
// FP8 wgrad reads whole, aligned 128-row blocks of every group.
// Consumer warps synchronize with a hardware barrier (see
// cw_consumer_barrier_any); every pipeline wait is bounded and gives up after about
// 1 s with MGEMM_STATUS_TIMEOUT.
constexpr int kCwRows = 256;
constexpr int kCwStages = 6;
constexpr int kCwConsumers = 16;
constexpr int kCwThreads = (kCwConsumers + 1) * 32;
constexpr int kCwBox = kCwRows * 128;   // 32 KB
constexpr int kCwTile = 64 * kCwRows;   // transposed tile: 2 halves of [64 columns][128 rows] codes
constexpr int kCwQueue = 4;  // item ids handed from the producer to the consumers
// Between the two passes the first kCwPark boxes of an item wait in tensor
// memory (16 columns per consumer warp per box: 8 boxes fill 512 columns), so
// every ring slot is freed as soon as pass 1 has read it; later boxes are read
// again.
constexpr int kCwPark = 8;
constexpr int kCwTmemCols = 512;
constexpr size_t kCwSmemFixed = 1024 + (size_t)kCwStages * kCwBox + 2 * kCwTile + 2 * 2 * 64 * 4 + 256;
static_assert(kCwSmemFixed <= 227 * 1024, "the ring, tiles and barriers fit one CTA's shared memory");
// (the group offsets, padded offsets and size order are read from the args
// block through the read-only cache, once per item)
__host__ __device__ constexpr size_t cw_smem_bytes(int) { return kCwSmemFixed; }

struct ColTensor {  // (the codes go out through the tensor maps)
  float *sc;
  int64_t C;
  int ncb;  // 64-column blocks
};

struct CwItem {
  int tensor, g, cb, nck;
  int64_t rs, re;  // the group's rows
  int64_t plen;    // its padded length (rows rounded up to kColPad)
  int64_t pos;     // where its rows start in each output column
};

__device__ __forceinline__ CwItem cw_decode(int item, const int64_t *off, const int64_t *poff, const int *order,
                                            const ColTensor &t1, const ColTensor &t2) {
  CwItem it;
  const int per_group = t1.ncb + t2.ncb;
  it.g = __ldg(order + item / per_group);
  const int cb = item % per_group;
  it.tensor = cb < t1.ncb ? 0 : 1;
  it.cb = it.tensor == 0 ? cb : cb - t1.ncb;
  it.rs = __ldg(off + it.g);
  it.re = __ldg(off + it.g + 1);
  it.plen = (it.re - it.rs + kColPad - 1) / kColPad * kColPad;
  it.pos = __ldg(poff + it.g);
  it.nck = (int)((it.plen + kCwRows - 1) / kCwRows);
  return it;
}

// Packed running max of magnitudes: each half of the result has magnitude
// max(|acc|, |v|) (its sign is meaningless; clear it before use).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t acc, uint32_t v) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(v));
  return r;
}

// Two bf16 values (one register) times a power-of-two scale (packed as {s, s})
// -> two e4m3 codes (round to nearest even, saturating), low element in the
// low byte.  One packed fp32 multiply serves both elements.
__device__ __forceinline__ uint16_t bf16x2_scaled_e4m3x2(uint32_t x, uint64_t s2) {
  uint16_t r;
  asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 p;\n\t"
      "shl.b32 lo, %1, 16;\n\t"
      "and.b32 hi, %1, 0xFFFF0000;\n\t"
      "mov.b64 p, {lo, hi};\n\t"
      "mul.rn.f32x2 p, p, %2;\n\t"
      "mov.b64 {lo, hi}, p;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 %0, hi, lo;\n\t}"
      : "=h"(r)
      : "r"(x), "l"(s2));
  return r;
}

// Four 8x8 b16 matrices (rows given by lanes 0-31), transposed on the way out.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Hardware barrier among the 16 consumer warps only (the producer warp never
// takes part), returning the OR of `flag` over all of them.  Every consumer warp
// executes every barrier: a warp whose bounded data wait gives up raises the
// abort flag and keeps going through the same steps; the decision to leave is
// taken by this barrier, so all consumer warps get the same answer and leave
// together.
__device__ __forceinline__ bool cw_consumer_barrier_any(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, p;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)flag), "n"(kCwConsumers * 32)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(kCwThreads, 1)
    quant_colwise_kernel(const __grid_constant__ CUtensorMap tm1, const __grid_constant__ CUtensorMap tm2,
                         const __grid_constant__ CUtensorMap tmo1, const __grid_constant__ CUtensorMap tmo2,
                         const uint8_t *__restrict__ args, int E, int64_t ld, ColTensor t1, ColTensor t2,
                         int items) {
  extern __shared__ uint8_t cw_smem_raw[];
  uint8_t *smem =
      reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(cw_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem;
  uint8_t *tiles = ring + kCwStages * kCwBox;                  // 2 x kCwTile
  float *red = reinterpret_cast<float *>(tiles + 2 * kCwTile);  // [2 items][2 halves][64]
  uint64_t *full = reinterpret_cast<uint64_t *>(red + 2 * 2 * 64);
  uint64_t *empty = full + kCwStages;
  uint64_t *qfull = empty + kCwStages;
  uint64_t *qempty = qfull + kCwQueue;
  int *abort_flag = reinterpret_cast<int *>(qempty + kCwQueue);
  int *s_item = abort_flag + 1;  // [kCwQueue]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(s_item + kCwQueue);

  pdl_wait();
  pdl_trigger();
  const ArgsView av(args, E);
  if (*av.status != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kCwStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCwConsumers);
    }
    for (int q = 0; q < kCwQueue; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], kCwConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kCwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int *vabort = abort_flag;
  uint32_t issued = 0;

  if (warp == kCwConsumers) {
    // ---- producer
    if (lane == 0) {
      tma_prefetch_desc(&tm1);
      tma_prefetch_desc(&tm2);
      tma_prefetch_desc(&tmo1);
      tma_prefetch_desc(&tmo2);
      int stage = 0, q = 0;
      uint32_t phase = 0, qphase = 0;
      // Items are taken from the args block's work counter in order of
      // decreasing group size, so every CTA stays busy until the end.  Each
      // CTA's last take returns a value >= items; the CTA whose last take is
      // the launch's final one (items + grid - 1) sets the counter back to 0:
      // no other CTA touches it after its own last take.
      while (true) {
        int item = atomicAdd(av.work, 1);
        const bool done = item >= items || *vabort;
        if (item == items + (int)gridDim.x - 1) atomicExch(av.work, 0);
        if (!mbar_wait(&qempty[q], qphase ^ 1, vabort)) {
          set_status(av.status, MGEMM_STATUS_TIMEOUT);
          *vabort = 1;
        }
        s_item[q] = done ? -1 : item;
        mbar_arrive(&qfull[q]);
        if (++q == kCwQueue) {
          q = 0;
          qphase ^= 1;
        }
        if (done) break;
        const CwItem it = cw_decode(item, av.offsets, av.poffsets, av.wgrad_order, t1, t2);
        const CUtensorMap *tm = it.tensor == 0 ? &tm1 : &tm2;
        // every box, then again, newest first, those not parked in tensor memory
        const int parked = it.nck < kCwPark ? it.nck : kCwPark;
        for (int i = 0; i < 2 * it.nck - parked && !*vabort; ++i) {
          const int k = i < it.nck ? i : it.nck - 1 - (i - it.nck);
          if (!mbar_wait(&empty[stage], phase ^ 1, vabort)) {
            set_status(av.status, MGEMM_STATUS_TIMEOUT);
            *vabort = 1;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kCwBox);
          ++issued;
          tma_load_2d(ring + stage * kCwBox, tm, &full[stage], it.cb * 64, (int)(it.rs + (int64_t)k * kCwRows));
          if (++stage == kCwStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else {
    // ---- consumers
    const int cc = warp & 7, rhalf = warp >> 3;
    const int lcol = cc * 8 + (lane >> 2);  // this lane's column within the block
    const int rpair = 2 * (lane & 3);       // row offset of its pair inside each 8-row matrix
    // this lane's column in a transposed half-tile: 128 bytes (rows) per
    // column, 16-byte chunks swizzled by the column (the 128-byte pattern the
    // output tensor maps store with)
    const uint32_t tsw = (uint32_t)(lcol & 7);
    int stage = 0, q = 0;
    uint32_t phase = 0, qphase = 0;
    uint32_t tile_par = 0;  // alternates with every pass-2 box, across items
    uint32_t item_par = 0;  // alternates with every item that has rows
    // a data wait that gives up marks the kernel aborted but does not leave the
    // step sequence, so barrier participation stays identical in every warp
    auto wait_full = [&]() {
      if (!mbar_wait_warp(&full[stage], phase, vabort) && lane == 0) {
        set_status(av.status, MGEMM_STATUS_TIMEOUT);
        *vabort = 1;
      }
    };
    // ldmatrix row address of this lane for 32-row block j of the warp's half of a box
    auto row_addr = [&](const uint8_t *box, int j) -> uint32_t {
      const int r = rhalf * 128 + j * 32 + lane;
      return smem_u32(box + r * 128 + ((cc ^ (r & 7)) << 4));
    };
    while (true) {
      // next item id from the producer (-1: no more work)
      int item = -1;
      if (mbar_wait_warp(&qfull[q], qphase, vabort)) {
        item = s_item[q];
      } else if (lane == 0) {  // gave up (or the kernel was aborted): report it, leave
        set_status(av.status, MGEMM_STATUS_TIMEOUT);
        *vabort = 1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[q]);
      if (++q == kCwQueue) {
        q = 0;
        qphase ^= 1;
      }
      // No barrier per item start: the one after pass 1 combines the column
      // maxima, and every warp leaves at a barrier too (here, or at that one
      // when any warp gave up), so all warps run the same number of barriers.
      if (item < 0) {  // no more work, or a wait that gave up: the exit barrier
        cw_consumer_barrier_any(true);
        break;
      }
      const CwItem it = cw_decode(item, av.offsets, av.poffsets, av.wgrad_order, t1, t2);
      const ColTensor &T = it.tensor == 0 ? t1 : t2;
      const int64_t col0 = (int64_t)it.cb * 64;
      if (it.nck == 0) {  // empty group: amax 0 -> scale 2^48, no data
        if (rhalf == 0 && (lane & 3) == 0 && col0 + lcol < T.C)
          T.sc[(int64_t)it.g * T.C + col0 + lcol] = pow2_scale_from_amax(0.f);
        continue;
      }
      const int parked = it.nck < kCwPark ? it.nck : kCwPark;  // boxes 0 .. parked - 1 wait in TMEM
      float *red_i = red + item_par * 128;
      item_par ^= 1;
      // this warp's 16 columns of TMEM slot k (its lane quarter is warp % 4)
      auto slot_addr = [&](int k) -> uint32_t {
        return tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(k * 64 + (warp >> 2) * 16);
      };
      // This lane's 16 values of box k (the ring stage at hand): ldmatrix j,
      // matrix m give rows 128 rhalf + 32 j + 8 m + rpair (low half) and + 1
      // (high half) of the box, column lcol.  Rows past the group are cleared
      // (only the boxes at the group's two ends hold rows of other groups) in
      // a separate pass over the registers that only such a box takes: a
      // compare inside the load loop cost about 10% of the kernel's time.
      auto read_box = [&](int k, uint32_t (&v)[16]) {
        const uint8_t *box = ring + stage * kCwBox;
        const bool edge = it.rs + (int64_t)(k + 1) * kCwRows > it.re;  // the box runs past the group
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t w[4];
          ldsm_x4_trans(row_addr(box, j), w);
#pragma unroll
          for (int m = 0; m < 4; ++m) v[4 * j + m] = w[m];
        }
        if (edge) {
          // rows of the warp's half at or past lim (relative to its pair) lie past the group
          const int lim = (int)(it.re - (it.rs + (int64_t)k * kCwRows + rhalf * 128)) - rpair;
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int gr = j * 32 + m * 8;
              if (gr >= lim) v[4 * j + m] &= 0xFFFF0000u;
              if (gr + 1 >= lim) v[4 * j + m] &= 0x0000FFFFu;
            }
        }
      };
      // pass 1: magnitude max of column lcol over this warp's rows; the first
      // kCwPark boxes are parked in TMEM, and every ring slot is freed at once
      uint32_t am = 0u;
      for (int k = 0; k < it.nck; ++k) {
        wait_full();
        uint32_t v[16];
        read_box(k, v);
#pragma unroll
        for (int r = 0; r < 16; ++r) am = bf16x2_absmax(am, v[r]);
        if (k < parked) tmem_st_32x32b_x16(slot_addr(k), v);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == kCwStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      tmem_st_wait();  // this thread's parked boxes are in TMEM before pass 2 reads them
      am = bf16x2_absmax(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = bf16x2_absmax(am, __shfl_xor_sync(0xffffffffu, am, 2));
      am &= 0x7FFF7FFFu;
      if ((lane & 3) == 0) red_i[rhalf * 64 + lcol] = fmaxf(bf16_lo(am), bf16_hi(am));
      if (cw_consumer_barrier_any(*vabort != 0)) break;
      const float sc = pow2_scale_from_amax(fmaxf(red_i[lcol], red_i[64 + lcol]));
      if (rhalf == 0 && (lane & 3) == 0 && col0 + lcol < T.C) T.sc[(int64_t)it.g * T.C + col0 + lcol] = sc;
      const uint64_t sc2 = ((uint64_t)__float_as_uint(sc) << 32) | __float_as_uint(sc);
      // pass 2: box k is converted into one tile while the stores of the
      // previous box drain from the other; one consumer barrier per box.  The
      // parked boxes come from TMEM, the rest from the ring, newest first, in
      // the order the producer loads them again.
      for (int i = 0; i < it.nck; ++i) {
        const bool from_tmem = i < parked;
        const int k = from_tmem ? i : it.nck - 1 - (i - parked);
        uint32_t v[16];
        if (from_tmem) {
          tmem_ld_32x32b_x16(slot_addr(k), v);
          tmem_ld_wait();
        } else {
          wait_full();
          read_box(k, v);
        }
        uint8_t *tile = tiles + tile_par * kCwTile;
        tile_par ^= 1;
        // this warp's block of the tile: its 8 columns x 128 rows (1 KB); the
        // store that read it two boxes ago has finished reading it
        uint8_t *wblk = tile + rhalf * (kCwTile / 2) + cc * 1024;
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        uint8_t *tcol = wblk + (lane >> 2) * 128 + rpair;
        // rows past the group were cleared: the padding of the column gets zero codes
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            // rows j*32 + m*8 + rpair, +1 of the half: chunk 2j + m/2, byte 8 (m & 1) + rpair
            const uint32_t chunk = (uint32_t)(2 * j + (m >> 1)) ^ tsw;
            *reinterpret_cast<uint16_t *>(tcol + chunk * 16 + (m & 1) * 8) =
                bf16x2_scaled_e4m3x2(v[4 * j + m], sc2);
          }
        }
        fence_proxy_async_smem();  // the codes are read by the tensor store below
        __syncwarp();
        if (!from_tmem) {
          if (lane == 0) mbar_arrive(&empty[stage]);  // box consumed; the codes live in the tile
          if (++stage == kCwStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        // the warp stores its own block: [8 columns][128 rows] to rows
        // pos + 256 k + 128 rhalf of columns col0 + 8 cc .. (only halves inside
        // the group's padded length, a multiple of 128; the map clips columns
        // past C).  No CTA barrier: a wait that gave up lets every warp run on
        // to the next item's barrier, where they all leave together.
        // (one bulk group per box, empty when there is nothing to store, so
        // "at most one group pending" always means the store of the last box)
        const int64_t q = (int64_t)k * kCwRows + rhalf * 128;
        if (lane == 0) {
          if (q < it.plen && col0 + cc * 8 < T.C)
            tma_store_2d(it.tensor == 0 ? &tmo1 : &tmo2, wblk, (int)(it.pos + q), (int)(col0 + cc * 8));
          bulk_commit();
        }
      }
    }
    tmem_st_wait();
    if (lane == 0) bulk_wait_all();  // the warp's tensor stores are complete before the CTA leaves
  }
  tc_fence_before();
  __syncthreads();
  if (*vabort && warp == kCwConsumers && lane == 0) {
    for (int s = 0; s < kCwStages; ++s) {  // wait for this CTA's copies in flight, bounded
      const uint32_t armed = issued / kCwStages + ((uint32_t)s < issued % kCwStages ? 1u : 0u);
      if (armed) mbar_wait_drain(&full[s], (armed - 1) & 1);
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCwTmemCols);
  }
}

}  // namespace mgemm

using namespace mgemm;

template <int NCH>
static int launch_rowwise(const __nv_bfloat16 *in, int64_t R, int64_t C, int64_t ld_in, uint8_t *out,
                          int64_t ld_out, float *scales, cudaStream_t s) {
  const int64_t blocks_needed = (R + 7) / 8;
  int sms = sm_count_cached();
  if (sms <= 0) sms = 148;
  const int64_t cap = (int64_t)sms * 32;
  const int blocks = (int)(blocks_needed < cap ? blocks_needed : cap);
  return launch_pdl(quant_rowwise_kernel<NCH>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_rowwise launch", in, R, C,
                    ld_in, out, ld_out, scales);
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
  if (nch <= 1) return launch_rowwise<1>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 2) return launch_rowwise<2>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 4) return launch_rowwise<4>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 6) return launch_rowwise<6>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 8) return launch_rowwise<8>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 12) return launch_rowwise<12>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 16) return launch_rowwise<16>(x, R, C, ld_in, out, ld_out, scales, s);
  if (nch <= 24) return launch_rowwise<24>(x, R, C, ld_in, out, ld_out, scales, s);
  return launch_rowwise<0>(x, R, C, ld_in, out, ld_out, scales, s);
}

extern "C" int mgemm_quant_mx(const void *in, int64_t R, int64_t C, int64_t ld_in, uint8_t *out, int64_t ld_out,
                              uint8_t *sf, int64_t ld_sf, mgemm_stream_t stream) {
  if (R < 0 || C < 0) return MGEMM_EINVAL;
  if (R == 0 || C == 0) return MGEMM_OK;
  if (!in || !out || !sf) return MGEMM_EINVAL;
  if (C % 32 || ld_in < C || ld_out < C || ld_sf < C / 32) return MGEMM_EINVAL;
  if (((uintptr_t)in & 15) || ((uintptr_t)out & 15) || ((uintptr_t)sf & 15) || (ld_in % 8) || (ld_out % 16) ||
      (ld_sf % 16))
    return MGEMM_EALIGN;
  const int64_t blocks_needed = (R + 7) / 8;
  int sms = sm_count_cached();
  if (sms <= 0) sms = 148;
  const int64_t cap = (int64_t)sms * 32;
  const int blocks = (int)(blocks_needed < cap ? blocks_needed : cap);
  const __nv_bfloat16 *x = (const __nv_bfloat16 *)in;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t nch = (C + 255) / 256;
  if (nch <= 2)
    return launch_pdl(quant_mx_kernel<2>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_mx launch", x, R, C, ld_in,
                      out, ld_out, sf, ld_sf);
  if (nch <= 4)
    return launch_pdl(quant_mx_kernel<4>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_mx launch", x, R, C, ld_in,
                      out, ld_out, sf, ld_sf);
  if (nch <= 6)
    return launch_pdl(quant_mx_kernel<6>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_mx launch", x, R, C, ld_in,
                      out, ld_out, sf, ld_sf);
  return launch_pdl(quant_mx_kernel<8>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_mx launch", x, R, C, ld_in, out,
                    ld_out, sf, ld_sf);
}

extern "C" int mgemm_quant_int4(const void *w, int E, int N, int K, int64_t ld_in, uint8_t *packed, uint8_t *sf,
                                mgemm_stream_t stream) {
  if (E < 1 || N < 1 || K < 1 || K % 128 || ld_in < K) return MGEMM_EINVAL;
  if ((int64_t)E * N >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (!w || !packed || !sf) return MGEMM_EINVAL;
  if (((uintptr_t)w & 15) || ((uintptr_t)packed & 15) || ((uintptr_t)sf & 15) || (ld_in % 8)) return MGEMM_EALIGN;
  const int64_t R = (int64_t)E * N;
  const int64_t blocks_needed = (R + 7) / 8;
  int sms = sm_count_cached();
  if (sms <= 0) sms = 148;
  const int64_t cap = (int64_t)sms * 32;
  const int blocks = (int)(blocks_needed < cap ? blocks_needed : cap);
  const __nv_bfloat16 *x = (const __nv_bfloat16 *)w;
  cudaStream_t s = (cudaStream_t)stream;
  const int nch = (K + 255) / 256;
  if (nch <= 2)
    return launch_pdl(quant_int4_kernel<2>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_int4 launch", x, R, N, K,
                      ld_in, packed, sf);
  if (nch <= 4)
    return launch_pdl(quant_int4_kernel<4>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_int4 launch", x, R, N, K,
                      ld_in, packed, sf);
  return launch_pdl(quant_int4_kernel<8>, dim3(blocks), dim3(256), 0, s, 1, "mgemm_quant_int4 launch", x, R, N, K, ld_in,
                    packed, sf);
}

extern "C" int mgemm_quant_colwise_mx(const void *args, int E, int64_t M, const void *in1, int64_t C1, uint8_t *out1,
                                      uint8_t *sf1, const void *in2, int64_t C2, uint8_t *out2, uint8_t *sf2,
                                      int64_t ld, mgemm_stream_t stream) {
  if (!args || !in1 || !out1 || !sf1) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || C1 <= 0 || C1 % 8) return MGEMM_EINVAL;
  if (ld < mgemm_colwise_ld(M, E)) return MGEMM_EINVAL;
  if (((uintptr_t)args & 15) || ((uintptr_t)in1 & 15) || ((uintptr_t)out1 & 15) || ((uintptr_t)sf1 & 15) || ld % 128)
    return MGEMM_EALIGN;
  if (in2) {
    if (!out2 || !sf2 || C2 <= 0 || C2 % 8) return MGEMM_EINVAL;
    if (((uintptr_t)in2 & 15) || ((uintptr_t)out2 & 15) || ((uintptr_t)sf2 & 15)) return MGEMM_EALIGN;
  }
  if (M == 0) return MGEMM_OK;
  MxColTensor t1{(const __nv_bfloat16 *)in1, out1, sf1, C1, (int)((C1 + 63) / 64)};
  MxColTensor t2{(const __nv_bfloat16 *)in2, out2, sf2, in2 ? C2 : 0, in2 ? (int)((C2 + 63) / 64) : 0};
  const int64_t nblk = ld / 128 * (t1.ncb + t2.ncb);
  if (nblk >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  const dim3 grid((unsigned)nblk);
  return launch_pdl(quant_colwise_mx_kernel, grid, dim3(256), 0, (cudaStream_t)stream, 1,
                    "mgemm_quant_colwise_mx launch", (const uint8_t *)args, E, ld, t1, t2);
}

extern "C" int mgemm_quant_colwise_grouped(const void *args, int E, int64_t M, const void *in1, int64_t C1,
                                           uint8_t *out1, float *sc1, const void *in2, int64_t C2,
                                           uint8_t *out2, float *sc2, int64_t ld, mgemm_stream_t stream) {
  if (!args || !in1 || !out1 || !sc1) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || C1 <= 0 || C1 % 8) return MGEMM_EINVAL;
  if (ld < mgemm_colwise_ld(M, E)) return MGEMM_EINVAL;
  if (((uintptr_t)args & 15) || ((uintptr_t)in1 & 15) || ((uintptr_t)out1 & 15) || ld % 16) return MGEMM_EALIGN;
  if (in2) {
    if (!out2 || !sc2 || C2 <= 0 || C2 % 8) return MGEMM_EINVAL;
    if (((uintptr_t)in2 & 15) || ((uintptr_t)out2 & 15)) return MGEMM_EALIGN;
  }
  int rc = ensure_context();
  if (rc) return rc;
  // rows of a zero-row tensor are never loaded; the map only needs valid dims
  const uint64_t Mm = M > 0 ? (uint64_t)M : 1;
  CUtensorMap tm1, tm2;
  {
    const uint64_t d[2] = {(uint64_t)C1, Mm};
    const uint64_t st[1] = {(uint64_t)C1 * 2};
    const uint32_t box[2] = {64, kCwRows};
    if (!make_tensor_map(&tm1, false, 2, in1, d, st, box)) return MGEMM_ECUDA;
  }
  if (in2) {
    const uint64_t d[2] = {(uint64_t)C2, Mm};
    const uint64_t st[1] = {(uint64_t)C2 * 2};
    const uint32_t box[2] = {64, kCwRows};
    if (!make_tensor_map(&tm2, false, 2, in2, d, st, box)) return MGEMM_ECUDA;
  } else {
    tm2 = tm1;
  }
  // the outputs: column c of the padded layout is row c of a [C][ld] byte
  // matrix; boxes of 8 columns x 128 rows (bytes): one consumer warp's block
  CUtensorMap tmo1, tmo2;
  {
    const uint64_t d[2] = {(uint64_t)ld, (uint64_t)C1};
    const uint64_t st[1] = {(uint64_t)ld};
    const uint32_t box[2] = {128, 8};
    if (!make_tensor_map(&tmo1, true, 2, out1, d, st, box)) return MGEMM_ECUDA;
  }
  if (in2) {
    const uint64_t d[2] = {(uint64_t)ld, (uint64_t)C2};
    const uint64_t st[1] = {(uint64_t)ld};
    const uint32_t box[2] = {128, 8};
    if (!make_tensor_map(&tmo2, true, 2, out2, d, st, box)) return MGEMM_ECUDA;
  } else {
    tmo2 = tmo1;
  }
  ColTensor t1{sc1, C1, (int)((C1 + 63) / 64)};
  ColTensor t2{sc2, in2 ? C2 : 0, in2 ? (int)((C2 + 63) / 64) : 0};
  const int64_t items = (int64_t)E * (t1.ncb + t2.ncb);
  if (items >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  const int sms = sm_count_cached();
  if (sms <= 0) return MGEMM_ECUDA;
  const int grid = (int)(items < sms ? items : sms);
  static bool attr_done[64] = {};
  int dev = 0;
  if ((rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice"))) return rc;
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if ((rc = cuda_rc(cudaFuncSetAttribute(quant_colwise_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)cw_smem_bytes(MGEMM_MAX_EXPERTS)),
                      "cudaFuncSetAttribute")))
      return rc;
    attr_done[dev] = true;
  }
  return launch_pdl(quant_colwise_kernel, dim3(grid), dim3(kCwThreads), cw_smem_bytes(E), (cudaStream_t)stream, 1,
                    "mgemm_quant_colwise_grouped launch", tm1, tm2, tmo1, tmo2, (const uint8_t *)args, E, ld, t1,
                    t2, (int)items);
}
