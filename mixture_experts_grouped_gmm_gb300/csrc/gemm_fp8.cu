// e4m3 instantiations of the persistent grouped GEMM (kind::f8f6f4 tensor
// cores, fp32 accumulation, power-of-two scales divided out in the epilogue).
#include "gemm_launch.cuh"

namespace mgemm {

int gemm_fp8_rows(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows>>(a, b, o, p, grid, s);
}
int gemm_fp8_experts(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeExperts, 256, 4, 1, false, 8>>(a, b, o, p, grid, s);
}
int gemm_fp8_rows_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                       cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 256, 6, 1, true, 8>>(a, b, o, p, grid, s);
}
int gemm_fp8_experts_pair(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                          int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeExperts, 256, 6, 1, true, 8>>(a, b, o, p, grid, s);
}
int gemm_fp8_rows_few(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p, int grid,
                      cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 256, 24, 1, false, 8, true, 1>>(a, b, o, p, grid, s);
}
int gemm_fp8_rows_few_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                          int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 128, 24, 1, false, 8, true, 2>>(a, b, o, p, grid, s);
}
int gemm_fp8_rows_few_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                             int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 64, 24, 1, false, 8, true, 4>>(a, b, o, p, grid, s);
}
int gemm_fp8_rows_narrow(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                         int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 64, 8, 1, false, 8>>(a, b, o, p, grid, s);
}
int gemm_fp8_rows_mid(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const GemmParams &p,
                      int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 128, 6>>(a, b, o, p, grid, s);
}

int gemm_fp8_rows_mx(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                     const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 128, 5, 2, false, 4, false, 1, true>>(a, b, o, p, grid, s,
                                                                                                  &sfa, &sfb);
}

int gemm_fp8_rows_mx192(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 192, 4, 2, false, 4, false, 1, true>>(a, b, o, p, grid, s,
                                                                                                  &sfa, &sfb);
}

// 256-wide tiles with one TMEM accumulator (three stages, eight epilogue warps)
int gemm_fp8_rows_mx256(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeRows, 256, 3, 1, false, 8, false, 1, true>>(a, b, o, p, grid, s,
                                                                                                 &sfa, &sfb);
}

int gemm_fp8_experts_mx256(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                           const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeExperts, 256, 3, 1, false, 8, false, 1, true>>(
      a, b, o, p, grid, s, &sfa, &sfb);
}

int gemm_fp8_experts_mx(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const CUtensorMap &sfa,
                        const CUtensorMap &sfb, const GemmParams &p, int grid, cudaStream_t s) {
  return launch_gemm<GemmCfg<true, false, false, kModeExperts, 192, 4, 2, false, 4, false, 1, true>>(
      a, b, o, p, grid, s, &sfa, &sfb);
}

}  // namespace mgemm
