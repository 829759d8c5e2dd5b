"""``gmm(x, w, group_sizes)``: the grouped GEMM as a differentiable op.

"Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21), benchmark
script: ``out = gmm(x, w, batch_sizes)`` followed by ``out.sum().backward()``,
with batch_sizes resident on the GPU so nothing waits on the host.

Forward: one ``mgemm_fill_args`` (the args block is kept for the backward
pass) and one ``mgemm_fwd``.  Backward: ``mgemm_dgrad`` and ``mgemm_wgrad``
reuse the same args block.  This module only allocates outputs with torch and
calls the binding; every step runs in the CUDA library.
"""

import torch

from . import binding as B


class GroupedGemm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, group_sizes, trans_b):
        if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
            raise B.MgemmError("gmm takes bf16 x and w")
        x = x.contiguous()
        w = w.contiguous()
        E = w.shape[0]
        M, K = x.shape
        N = w.shape[1] if trans_b else w.shape[2]
        args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=x.device)
        B.mgemm_fill_args(group_sizes, E, M, args)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
        B.mgemm_fwd(args, B.MGEMM_BF16, trans_b, x, None, w, None, out, M, K, N, E)
        ctx.save_for_backward(x, w, args)
        ctx.dims = (M, K, N, E, trans_b)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        x, w, args = ctx.saved_tensors
        M, K, N, E, trans_b = ctx.dims
        go = grad_out.contiguous()
        gx = gw = None
        if ctx.needs_input_grad[0]:
            gx = torch.empty(M, K, dtype=torch.bfloat16, device=x.device)
            if trans_b:   # w[e] is [N, K]: grad_x = grad_out . w[e]
                B.mgemm_fwd(args, B.MGEMM_BF16, 0, go, None, w, None, gx, M, N, K, E)
            else:         # w[e] is [K, N]: grad_x = grad_out . w[e]^T
                B.mgemm_dgrad(args, B.MGEMM_BF16, go, None, w, None, gx, M, K, N, E)
        if ctx.needs_input_grad[1]:
            if trans_b:   # grad_w[e] [N, K] = grad_out_e^T . x_e
                gw = torch.empty(E, N, K, dtype=torch.bfloat16, device=x.device)
                B.mgemm_wgrad(args, B.MGEMM_BF16, go, None, x, None, gw, M, N, K, E)
            else:
                gw = torch.empty(E, K, N, dtype=torch.bfloat16, device=x.device)
                B.mgemm_wgrad(args, B.MGEMM_BF16, x, None, go, None, gw, M, K, N, E)
        return gx, gw, None, None


def gmm(x, w, group_sizes, trans_b=False):
    """out[rows of group e] = x[rows of group e] @ w[e]  (w[e]^T with trans_b).

    x: bf16 [M, K] on the GPU, rows contiguous by expert; w: bf16 [E, K, N]
    ([E, N, K] with trans_b); group_sizes: int64 [E] on the GPU, summing to M.
    """
    return GroupedGemm.apply(x, w, group_sizes, bool(trans_b))
