// mgemm_fill_args: device group sizes -> args block, in one CTA.
//
// "Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21): a
// single-threadblock kernel replaces the host roundtrip of the batch sizes;
// one thread per expert (<= 1024); a block scan over the sizes; problems sorted
// by k descending when k is dynamic.  "F8I4 Grouped Gemm Optimization for
// Sparse M" (FBGEMM PR #3854): only the non-empty groups are scheduled.
//
// This kernel: warp-shuffle block scans (int64 offsets, int32 compaction and
// tile prefix), and a rank sort for the wgrad order (each thread counts the
// experts that precede it: larger size, or equal size and smaller id), which is
// deterministic and needs no temporary storage.  The block size is bucketed by
// E (32, 128, 1024 threads) since the cost of a single-CTA kernel grows with
// its thread count.
#include <cudaTypedefs.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "fill_args.cuh"

namespace mgemm {

template <int NT>
__global__ void __launch_bounds__(NT) fill_args_kernel(const int64_t *__restrict__ sizes, int E, int64_t M,
                                                       uint8_t *__restrict__ args) {
  pdl_wait();
  pdl_trigger();
  fill_args_body<NT>(threadIdx.x < E ? sizes[threadIdx.x] : 0, E, M, args);
}

// mgemm_fill_args and mgemm_quant_rowwise of the token rows in one launch: CTA
// 0 fills the args block while the other CTAs cast rows (one warp per row,
// two passes over the row), so the two independent steps run side by side.
template <int NT, int NCH>
__global__ void __launch_bounds__(NT) fill_quant_kernel(const int64_t *__restrict__ sizes, int E, int64_t M,
                                                        uint8_t *__restrict__ args, int64_t R,
                                                        const __nv_bfloat16 *__restrict__ x, int64_t C,
                                                        int64_t ld_in, uint8_t *__restrict__ q, int64_t ld_out,
                                                        float *__restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0) {
    fill_args_body<NT>(threadIdx.x < E ? sizes[threadIdx.x] : 0, E, M, args);
    return;
  }
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31;
  const int64_t step = (int64_t)(gridDim.x - 1) * W;
  for (int64_t row = (int64_t)(blockIdx.x - 1) * W + (threadIdx.x >> 5); row < R; row += step) {
    if constexpr (NCH > 0)
      quant_row_regs<NCH>(x + row * ld_in, C, q + row * ld_out, scales + row, lane);
    else
      quant_row_two_pass(x + row * ld_in, C, q + row * ld_out, scales + row, lane);
  }
}

namespace {
thread_local char g_last_error[192] = "";
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}
}  // namespace

bool make_tensor_map(CUtensorMap *m, bool byte_elems, int rank, const void *base, const uint64_t *dims,
                     const uint64_t *strides, const uint32_t *box, bool swizzle128) {
  auto enc = encode_fn();
  if (!enc) {
    note_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", 0);
    return false;
  }
  const uint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r =
      enc(m, byte_elems ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    note_error("cuTensorMapEncodeTiled", (int)r);
    return false;
  }
  return true;
}

int ensure_context() {
  thread_local bool done = false;
  if (done) return MGEMM_OK;
  int dev = 0;
  int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  rc = cuda_rc(cudaSetDevice(dev), "cudaSetDevice");
  if (rc) return rc;
  done = true;
  return MGEMM_OK;
}

int sm_count_cached() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (!cached[dev]) cached[dev] = mgemm_num_sms();
  return cached[dev];
}

void note_error(const char *where, int code) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: error %d (%s)", where, code,
           cudaGetErrorString((cudaError_t)code));
}

}  // namespace mgemm

using namespace mgemm;

extern "C" const char *mgemm_last_error(void) { return g_last_error; }

extern "C" int64_t mgemm_colwise_ld(int64_t M, int E) {
  if (M < 0 || E < 1 || E > MGEMM_MAX_EXPERTS) return -1;
  const int64_t groups = M < E ? M : E;  // at most this many non-empty groups, each padded by < kColPad rows
  const int64_t rows = M + (int64_t)(kColPad - 1) * groups;
  return (rows + kColPad - 1) / kColPad * kColPad;
}

extern "C" size_t mgemm_args_bytes(int E) {
  if (E < 1 || E > MGEMM_MAX_EXPERTS) return 0;
  return args_layout(E).bytes;
}

extern "C" int mgemm_args_layout(int E, size_t *off_offsets, size_t *off_active, size_t *off_mtile_start,
                                 size_t *off_wgrad_order) {
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  ArgsLayout L = args_layout(E);
  if (off_offsets) *off_offsets = L.offsets;
  if (off_active) *off_active = L.active;
  if (off_mtile_start) *off_mtile_start = L.mtile_start;
  if (off_wgrad_order) *off_wgrad_order = L.wgrad_order;
  return MGEMM_OK;
}

extern "C" int mgemm_fill_args(const int64_t *group_sizes, int E, int64_t M, void *args, mgemm_stream_t stream) {
  if (!group_sizes || !args) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < -1 || M >= (int64_t(1) << 31)) return MGEMM_EINVAL;
  if (((uintptr_t)args & 15) || ((uintptr_t)group_sizes & 7)) return MGEMM_EALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t *a = (uint8_t *)args;
  if (E <= 32) return launch_pdl(fill_args_kernel<32>, dim3(1), dim3(32), 0, s, 1, "mgemm_fill_args launch", group_sizes, E, M, a);
  if (E <= 128)
    return launch_pdl(fill_args_kernel<128>, dim3(1), dim3(128), 0, s, 1, "mgemm_fill_args launch", group_sizes, E, M, a);
  return launch_pdl(fill_args_kernel<1024>, dim3(1), dim3(1024), 0, s, 1, "mgemm_fill_args launch", group_sizes, E, M, a);
}

extern "C" int mgemm_fill_args_quant_rowwise(const int64_t *group_sizes, int E, int64_t M, void *args, const void *x,
                                             int64_t K, int64_t ld_x, uint8_t *xq, int64_t ld_q, float *sx,
                                             mgemm_stream_t stream) {
  if (!group_sizes || !args) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0 || M >= (int64_t(1) << 31) || K < 0 || ld_x < K || ld_q < K) return MGEMM_EINVAL;
  if (M > 0 && K > 0 && (!x || !xq || !sx)) return MGEMM_EINVAL;
  if (((uintptr_t)args & 15) || ((uintptr_t)group_sizes & 7)) return MGEMM_EALIGN;
  if (M > 0 && K > 0 && (((uintptr_t)x & 15) || ((uintptr_t)xq & 7) || ((uintptr_t)sx & 3) || K % 8 || ld_x % 8 ||
                         ld_q % 8))
    return MGEMM_EALIGN;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t *a = (uint8_t *)args;
  const __nv_bfloat16 *xb = (const __nv_bfloat16 *)x;
  const int64_t rows = K > 0 ? M : 0;  // no columns: nothing to cast (the scales stay unwritten)
  int sms = sm_count_cached();
  if (sms <= 0) sms = 148;
  auto blocks = [&](int w) -> unsigned {
    const int64_t need = (rows + w - 1) / w, cap = (int64_t)sms * 8;
    return 1u + (unsigned)(need < cap ? need : cap);
  };
  // rows of up to 24 x 256 elements stay in registers (one read) with the
  // 32- and 128-thread blocks; the 1024-thread block reads its rows twice
  const bool regs = K <= 24 * 256;
  if (E <= 32)
    return regs ? launch_pdl(fill_quant_kernel<32, 24>, dim3(blocks(1)), dim3(32), 0, s, 1,
                             "fill + rowwise cast launch", group_sizes, E, M, a, rows, xb, K, ld_x, xq, ld_q, sx)
                : launch_pdl(fill_quant_kernel<32, 0>, dim3(blocks(1)), dim3(32), 0, s, 1,
                             "fill + rowwise cast launch", group_sizes, E, M, a, rows, xb, K, ld_x, xq, ld_q, sx);
  if (E <= 128)
    return regs ? launch_pdl(fill_quant_kernel<128, 24>, dim3(blocks(4)), dim3(128), 0, s, 1,
                             "fill + rowwise cast launch", group_sizes, E, M, a, rows, xb, K, ld_x, xq, ld_q, sx)
                : launch_pdl(fill_quant_kernel<128, 0>, dim3(blocks(4)), dim3(128), 0, s, 1,
                             "fill + rowwise cast launch", group_sizes, E, M, a, rows, xb, K, ld_x, xq, ld_q, sx);
  return launch_pdl(fill_quant_kernel<1024, 0>, dim3(blocks(32)), dim3(1024), 0, s, 1, "fill + rowwise cast launch",
                    group_sizes, E, M, a, rows, xb, K, ld_x, xq, ld_q, sx);
}

extern "C" int mgemm_num_sms(void) {
  int dev = 0, n = 0;
  int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  rc = cuda_rc(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  return rc ? rc : n;
}

extern "C" const char *mgemm_error_string(int code) {
  switch (code) {
    case MGEMM_OK: return "ok";
    case MGEMM_EINVAL: return "invalid argument";
    case MGEMM_EALIGN: return "pointer or stride not 16-byte aligned";
    case MGEMM_ETOOMANY: return "too many experts";
    case MGEMM_ECUDA: return "CUDA call failed";
    case MGEMM_ENOTSUP: return "combination not supported";
    case MGEMM_STATUS_NEGATIVE_SIZE: return "device status: negative group size";
    case MGEMM_STATUS_SUM_MISMATCH: return "device status: group sizes do not sum to M";
    case MGEMM_STATUS_TIMEOUT: return "device status: pipeline wait timed out";
    default: return "unknown code";
  }
}

extern "C" int mgemm_version(void) { return 100; }
