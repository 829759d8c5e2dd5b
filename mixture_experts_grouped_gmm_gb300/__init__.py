"""GB300-native Mixture-of-Experts grouped GEMM (sm_103a).

The compute path is libmgemm.so (hand-written CUDA for sm_103a, C ABI in
include/mgemm.h); ``binding`` marshals torch tensors into it and ``gmm``
wraps forward/backward as an autograd op.  ``workloads`` draws the seeded
synthetic inputs.
"""

from . import binding  # noqa: F401
from .gmm import gmm, gmm_fp8  # noqa: F401
