// bf16 instantiations of the persistent grouped GEMM (kind::f16 tensor cores).
#include "gemm_launch.cuh"

namespace mgemm {

int gemm_bf16_rows_bmn(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, true, kModeRows>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_bk(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows>>(a, b, o, p, grid, s);
}
int gemm_bf16_experts(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s) {
  return launch_gemm<GemmCfg<false, true, true, kModeExperts, 256, 3, 4>>(a, b, o, p, grid, s);
}
int gemm_bf16_dgrad_wgrad(const CUtensorMap &da, const CUtensorMap &db, const CUtensorMap &dout, const GemmParams &pd,
                          const CUtensorMap &wa, const CUtensorMap &wb, const CUtensorMap &wout, const GemmParams &pw,
                          int split, int grid, cudaStream_t s) {
  // the dgrad half takes the form mgemm_dgrad would launch for its tile width
  // (a deeper ring for narrower tiles: more weight bytes in flight per SM)
  using W = GemmCfg<false, true, true, kModeExperts, 256, 3, 4>;
  if (pd.bn <= 64)
    return launch_dual<GemmCfg<false, false, false, kModeRows, 64, 8>, W>(da, db, dout, pd, wa, wb, wout, pw, split,
                                                                          grid, s);
  if (pd.bn <= 128)
    return launch_dual<GemmCfg<false, false, false, kModeRows, 128, 6>, W>(da, db, dout, pd, wa, wb, wout, pw, split,
                                                                           grid, s);
  return launch_dual<GemmCfg<false, false, false, kModeRows>, W>(da, db, dout, pd, wa, wb, wout, pw, split, grid, s);
}
int gemm_bf16_rows_bmn_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, true, kModeRows, 64, 8>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_bk_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                             int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 64, 8>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_bmn_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                           int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, true, kModeRows, 128, 6>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_bmn_w192(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                            int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, true, kModeRows, 192, 5, 1>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_bk_w192(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                           int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 192, 5, 1>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_bk_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                          int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 128, 6>>(a, b, o, p, grid, s);
}

// routed rows with few per group (decode-size batches): run-time rings whose A
// slot holds only those rows, K-major w, four epilogue warps (the gated and
// scattered epilogues)
int gemm_bf16_rows_few_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 64, 24, 1, false, 4, true, 1>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_few_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                           int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 128, 24, 1, false, 4, true, 1>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_few_wide(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                            int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 256, 24, 1, false, 4, true, 1>>(a, b, o, p, grid, s);
}
// the same with K % 64 == 0: each operand's contraction blocks of a stage in one box of
// consecutive 128-byte k-chunks (4 / 2 / 2 blocks per stage at 64 / 128 / 256 columns)
int gemm_bf16_rows_few_narrow_kc(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                                 const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 64, 24, 1, false, 4, true, 4>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_few_mid_kc(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                              int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 128, 24, 1, false, 4, true, 2>>(a, b, o, p, grid, s);
}
// 128 columns with at most 8 rows per group: four blocks per stage (three 68 KB stages)
int gemm_bf16_rows_few_mid_kc4(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                               const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 128, 24, 1, false, 4, true, 4>>(a, b, o, p, grid, s);
}
int gemm_bf16_rows_few_wide_kc(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                               int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<false, false, false, kModeRows, 256, 24, 1, false, 4, true, 2>>(a, b, o, p, grid, s);
}

}  // namespace mgemm
