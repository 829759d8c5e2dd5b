// Host-side launch of one GemmCfg instantiation (shared by the bf16 and fp8
// translation units) and the declarations the entry points call.
#pragma once

#include "gemm.cuh"

namespace mgemm {

// The host-side argument checks of mgemm_fwd other than those of the args
// block (pointers, alignment, dtype and layout, sizes); MGEMM_OK or the code
// mgemm_fwd would return.  Makes no CUDA call.
int fwd_checks(int dtype, int trans_b, const void *x, const float *sx, const void *w, const float *sw,
               const void *out, int64_t M, int K, int N, int E);

template <class C>
int launch_gemm(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p_in, int grid,
                cudaStream_t s, const CUtensorMap *sfa = nullptr, const CUtensorMap *sfb = nullptr) {
  GemmParams p = p_in;
  size_t smem = C::SMEM_BYTES;
  if constexpr (C::DynRing) {
    // as many [A slot | B slot] stages as fit next to the staging buffers and barriers
    p.stage_bytes = C::KC * (p.a_rows + p.bn) * 128;
    const size_t room = (size_t)227 * 1024 - C::FIXED_BYTES;
    const int fit = (int)(room / (size_t)p.stage_bytes);
    p.stages = fit < C::STAGES ? fit : C::STAGES;
    if (p.a_rows % 8 || p.stages < 2) return MGEMM_EINVAL;
    smem = C::FIXED_BYTES + (size_t)p.stages * p.stage_bytes;
  }
  static bool attr_done[64] = {};
  int dev = 0;
  int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return MGEMM_EINVAL;
  if (!attr_done[dev]) {
    rc = cuda_rc(cudaFuncSetAttribute(mgemm_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)C::SMEM_BYTES),
                 "cudaFuncSetAttribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  // CTA pairs: clusters of two CTAs (grid is even); every CTA of the grid is resident
  return launch_pdl(mgemm_gemm_kernel<C>, dim3((unsigned)grid), dim3(C::THREADS), smem, s, C::Pair ? 2u : 1u,
                    C::Pair ? "grouped GEMM launch (CTA pairs)" : "grouped GEMM launch", a, b, o, sfa ? *sfa : a,
                    sfb ? *sfb : a, p);
}

// Two GEMMs in one launch (mgemm_dual_kernel): split CTAs for the first, the
// rest of grid for the second
template <class C0, class C1>
int launch_dual(const CUtensorMap &a0, const CUtensorMap &b0, const CUtensorMap &o0, const GemmParams &p0,
                const CUtensorMap &a1, const CUtensorMap &b1, const CUtensorMap &o1, const GemmParams &p1, int split,
                int grid, cudaStream_t s) {
  static_assert(!C0::DynRing && !C1::DynRing, "fixed rings");
  constexpr size_t smem = C0::SMEM_BYTES > C1::SMEM_BYTES ? C0::SMEM_BYTES : C1::SMEM_BYTES;
  if (split < 1 || split >= grid) return MGEMM_EINVAL;
  static bool attr_done[64] = {};
  int dev = 0;
  int rc = cuda_rc(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 0 || dev >= 64) return MGEMM_EINVAL;
  if (!attr_done[dev]) {
    rc = cuda_rc(cudaFuncSetAttribute(mgemm_dual_kernel<C0, C1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem),
                 "cudaFuncSetAttribute");
    if (rc) return rc;
    attr_done[dev] = true;
  }
  return launch_pdl(mgemm_dual_kernel<C0, C1>, dim3((unsigned)grid), dim3(C0::THREADS), smem, s, 1u,
                    "grouped GEMM launch (two GEMMs)", a0, b0, o0, a1, b1, o1, p0, p1, split);
}

// bf16 dgrad (w [E, K, N]; the 64-, 128- or 256-wide form by pd.bn) and wgrad in one launch
int gemm_bf16_dgrad_wgrad(const CUtensorMap &da, const CUtensorMap &db, const CUtensorMap &dout, const GemmParams &pd,
                          const CUtensorMap &wa, const CUtensorMap &wb, const CUtensorMap &wout, const GemmParams &pw,
                          int split, int grid, cudaStream_t s);
// MXFP8: e4m3 x [M, K] and w [E, N, K] with e8m0 scale rows (maps sfa, sfb), 128-wide tiles
int gemm_fp8_rows_mx(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                     const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s);
int gemm_fp8_rows_mx192(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s);
int gemm_fp8_rows_mx256(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s);
// MXFP8 wgrad: padded column-major x^T [K, ld] and grad_out^T [N, ld] with k-block-major scale rows
int gemm_fp8_experts_mx(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s);
int gemm_fp8_experts_mx256(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s);
// bf16 routed rows with few per group: run-time rings (A slot of a_rows rows), K-major w
int gemm_bf16_rows_few_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s);
int gemm_bf16_rows_few_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                           int grid, cudaStream_t s);
int gemm_bf16_rows_few_wide(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                            int grid, cudaStream_t s);
// the same in k-chunk boxes (K % 64 == 0; the gated form's B map has a gate / up dimension)
int gemm_bf16_rows_few_narrow_kc(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                                 const GemmParams &p, int grid, cudaStream_t s);
int gemm_bf16_rows_few_mid_kc(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s);
int gemm_bf16_rows_few_mid_kc4(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s);
int gemm_bf16_rows_few_wide_kc(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                               int grid, cudaStream_t s);
// bf16: A K-major rows, B MN-major ([E, K, N] weights)
int gemm_bf16_rows_bmn(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s);
// bf16: A K-major rows, B K-major ([E, N, K] weights, or dgrad on [E, K, N])
int gemm_bf16_rows_bk(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s);
// bf16 wgrad: both operands MN-major (row-major x and grad_out)
int gemm_bf16_experts(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s);
// mid (BN <= 128, 6-stage) and narrow (BN <= 64, 8-stage) forms of the rows-mode kernels
int gemm_bf16_rows_bmn_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                           int grid, cudaStream_t s);
int gemm_bf16_rows_bmn_w192(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                            int grid, cudaStream_t s);
int gemm_bf16_rows_bk_w192(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                           int grid, cudaStream_t s);
int gemm_bf16_rows_bk_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                          int grid, cudaStream_t s);
int gemm_fp8_rows_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                      int grid, cudaStream_t s);
int gemm_bf16_rows_bmn_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s);
int gemm_bf16_rows_bk_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                             int grid, cudaStream_t s);
int gemm_fp8_rows_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                         int grid, cudaStream_t s);
// fp8 forward / dgrad: both K-major, scaled epilogue
int gemm_fp8_rows(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s);
// the same with a run-time ring sized to the launch's token rows (fewer than 128), by tile width
int gemm_fp8_rows_few(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                      cudaStream_t s);
int gemm_fp8_rows_few_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                          int grid, cudaStream_t s);
int gemm_fp8_rows_few_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                             int grid, cudaStream_t s);
// fp8 wgrad: column-major quantized operands (K-major), scaled epilogue
int gemm_fp8_experts(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s);
// fp8 forward / dgrad with at least 128 token rows on CTA pairs (256-row tiles inside a group; grid even)
int gemm_fp8_rows_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s);
// the same on CTA pairs (256-row tiles of K, cta_group::2; grid even)
int gemm_fp8_experts_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                          int grid, cudaStream_t s);

}  // namespace mgemm
