"""GB300-native Mixture-of-Experts grouped GEMM (sm_103a)."""
