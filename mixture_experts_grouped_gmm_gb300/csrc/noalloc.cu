// mgemm_fwd_noalloc: the grouped forward GEMM for callers that cannot
// allocate device memory.
//
// The forward pass needs an args block (the tile schedule that
// mgemm_fill_args derives from the group sizes) besides its inputs and
// output.  Most callers allocate it themselves.  Some cannot: code that runs
// inside another framework's launch callback with no allocator of its own,
// code that must not call cudaMalloc because that can synchronize the device
// in a latency-critical loop, or runtimes that only hand out a fixed
// workspace decided ahead of time.  For them this entry point keeps the args
// block in a statically sized device array that lives in this library.
//
// The array holds an args block for up to MGEMM_NOALLOC_MAX_EXPERTS experts
// (about 33 KB); every GPU that loads the library keeps it until the process
// exits.  All calls share it, so calls whose work overlaps on the GPU (for
// example on two streams) race on it.  Each call rewrites every part of it
// that the forward kernel reads (mgemm_fill_args writes the whole header,
// the offsets, the active-group list and the tile prefix), so nothing from
// an earlier call leaks into the next.
#include <mutex>

#include "gemm_launch.cuh"

namespace {

constexpr size_t noalloc_args_bytes() { return mgemm::args_layout(MGEMM_NOALLOC_MAX_EXPERTS).bytes; }

static __device__ __align__(256) uint8_t g_noalloc_args[noalloc_args_bytes()];

// the args block of every E up to the stated maximum fits the array (the
// layout grows with E)
static_assert(mgemm::args_layout(MGEMM_NOALLOC_MAX_EXPERTS).bytes <= sizeof(g_noalloc_args),
              "the static args block holds MGEMM_NOALLOC_MAX_EXPERTS experts");
static_assert(MGEMM_NOALLOC_MAX_EXPERTS <= MGEMM_MAX_EXPERTS, "the fill kernel serves every E the array holds");

// Device address of g_noalloc_args, looked up once per device with that
// device current (in host code the symbol is only a stand-in, not an address
// the GPU can use).  The address is cached for the life of the process, so
// the library must not be used across a cudaDeviceReset of that device.
void *noalloc_args_ptr(int *rc) {
  static void *ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  *rc = mgemm::cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (*rc) return nullptr;
  if (dev < 0 || dev >= 64) {
    *rc = MGEMM_EINVAL;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    *rc = mgemm::cuda_rc(cudaGetSymbolAddress(&p, g_noalloc_args), "cudaGetSymbolAddress");
    if (*rc) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" int mgemm_fwd_noalloc(const int64_t *group_sizes, int E, int dtype, int trans_b, const void *x,
                                 const float *sx, const void *w, const float *sw, void *out, int64_t M, int K, int N,
                                 mgemm_stream_t stream) {
  // Every check of mgemm_fill_args and mgemm_fwd comes first: a call that is
  // rejected launches nothing and leaves the shared array as it was.
  if (!group_sizes) return MGEMM_EINVAL;
  if (E < 1) return MGEMM_EINVAL;
  if (E > MGEMM_NOALLOC_MAX_EXPERTS) return MGEMM_ETOOMANY;
  if (M < 0) return MGEMM_EINVAL;  // (mgemm_fill_args' M = -1 form has no use here)
  if ((uintptr_t)group_sizes & 7) return MGEMM_EALIGN;
  int rc = mgemm::fwd_checks(dtype, trans_b, x, sx, w, sw, out, M, K, N, E);
  if (rc) return rc;
  if (M == 0) return MGEMM_OK;  // no rows: nothing to schedule or compute
  void *args = noalloc_args_ptr(&rc);
  if (rc) return rc;
  rc = mgemm_fill_args(group_sizes, E, M, args, stream);
  if (rc) return rc;
  return mgemm_fwd(args, dtype, trans_b, x, sx, w, sw, out, M, K, N, E, stream);
}
