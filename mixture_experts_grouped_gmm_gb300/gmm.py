"""``gmm(x, w, group_sizes)``: the grouped GEMM as a differentiable op.

"Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21), benchmark
script: ``out = gmm(x, w, batch_sizes)`` followed by ``out.sum().backward()``,
with batch_sizes resident on the GPU so nothing waits on the host.

Forward: one ``mgemm_fill_args`` (the args block is kept for the backward
pass) and one ``mgemm_fwd``.  Backward: ``mgemm_dgrad_wgrad`` when both
gradients are wanted and w is [E, K, N] (one launch where the two GEMMs
overlap), else ``mgemm_dgrad`` / ``mgemm_fwd`` and ``mgemm_wgrad``; all reuse
the same args block.  This module only allocates outputs with torch and
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
        if ctx.needs_input_grad[0] and ctx.needs_input_grad[1] and not trans_b:
            gx = torch.empty(M, K, dtype=torch.bfloat16, device=x.device)
            gw = torch.empty(E, K, N, dtype=torch.bfloat16, device=x.device)
            B.mgemm_dgrad_wgrad(args, go, w, x, gx, gw, M, K, N, E)
            return gx, gw, None, None
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


# --------------------------------------------------------------------- FP8
# The group sizes of the weights viewed [E K, N] (E groups of K rows) depend
# only on (device, E, K) and are made once.  Their args block is filled per
# call: the colwise cast hands out its work through the block's counter, so a
# block shared by calls on two streams would race.
_WEIGHT_GROUPS = {}


def _weight_group_args(device, E, K):
    key = (str(device), E, K)
    sizes = _WEIGHT_GROUPS.get(key)
    if sizes is None:
        sizes = _WEIGHT_GROUPS[key] = torch.full((E,), K, dtype=torch.int64, device=device)
    args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=device)
    B.mgemm_fill_args(sizes, E, E * K, args)
    return args


class GroupedGemmFp8(torch.autograd.Function):
    """The FP8 training step of "[moe training] Optimize FP8 MoE backward pass:
    fused colwise kernel + AMD tuning" (pytorch/ao commit 34322b5), as an
    autograd op over the bf16 master tensors x [M, K] and w [E, K, N]:

    forward   fill + rowwise cast of x (one launch), per-(e, n) cast of w over K
              (the per-group colwise kernel on w viewed [E K, N], groups of K
              rows), FP8 grouped GEMM reading those codes in place
    backward  rowwise cast of grad_out, rowwise cast of w per (e, k) over N,
              FP8 dgrad; one dual per-group colwise cast of grad_out and x,
              FP8 wgrad (the commit message's 5 -> 2 launches)

    Every step runs in the CUDA library; outputs are bf16."""

    @staticmethod
    def forward(ctx, x, w, group_sizes):
        if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
            raise B.MgemmError("gmm_fp8 takes bf16 x and w")
        x = x.contiguous()
        w = w.contiguous()
        E, K, N = w.shape
        M = x.shape[0]
        dev = x.device
        u8, f32 = torch.uint8, torch.float32
        args = torch.empty(B.mgemm_args_bytes(E), dtype=u8, device=dev)
        xq = torch.empty(M, K, dtype=u8, device=dev)
        sx = torch.empty(M, dtype=f32, device=dev)
        B.mgemm_fill_args_quant_rowwise(group_sizes, E, M, args, x, xq, sx)
        ldw = B.mgemm_colwise_ld(E * K, E)
        wq = torch.empty(N * ldw, dtype=u8, device=dev)
        sw = torch.empty(E * N, dtype=f32, device=dev)
        B.mgemm_quant_colwise_grouped(_weight_group_args(dev, E, K), E, E * K, w.view(E * K, N), wq, sw, ld=ldw)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        B.mgemm_fwd_fp8_strided(args, xq, sx, wq, ldw, -(-K // 128) * 128, sw, out, M, K, N, E)
        ctx.save_for_backward(x, w, args)
        ctx.dims = (M, K, N, E)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        x, w, args = ctx.saved_tensors
        M, K, N, E = ctx.dims
        dev = x.device
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        go = grad_out.contiguous().to(bf)
        gx = gw = None
        if ctx.needs_input_grad[0]:
            goq = torch.empty(M, N, dtype=u8, device=dev)
            sgo = torch.empty(M, dtype=f32, device=dev)
            B.mgemm_quant_rowwise(go, goq, sgo)
            wdq = torch.empty(E * K, N, dtype=u8, device=dev)
            swd = torch.empty(E * K, dtype=f32, device=dev)
            B.mgemm_quant_rowwise(w.view(E * K, N), wdq, swd)
            gx = torch.empty(M, K, dtype=bf, device=dev)
            B.mgemm_dgrad(args, B.MGEMM_FP8_E4M3, goq, sgo, wdq, swd, gx, M, K, N, E)
        if ctx.needs_input_grad[1]:
            ld = B.mgemm_colwise_ld(M, E)
            goqt = torch.empty(N * ld, dtype=u8, device=dev)
            xqt = torch.empty(K * ld, dtype=u8, device=dev)
            sgoc = torch.empty(E * N, dtype=f32, device=dev)
            sxc = torch.empty(E * K, dtype=f32, device=dev)
            B.mgemm_quant_colwise_grouped(args, E, M, go, goqt, sgoc, x, xqt, sxc, ld=ld)
            gw = torch.empty(E, K, N, dtype=bf, device=dev)
            B.mgemm_wgrad(args, B.MGEMM_FP8_E4M3, xqt, sxc, goqt, sgoc, gw, M, K, N, E, ld=ld)
        return gx, gw, None


def gmm_fp8(x, w, group_sizes):
    """The grouped GEMM with FP8 (e4m3, power-of-two scales) operands in forward
    and backward: x bf16 [M, K], w bf16 [E, K, N], group_sizes int64 [E] on the
    GPU.  Forward: x rowwise, w per (e, n) over K; dgrad: grad_out rowwise, w per
    (e, k) over N; wgrad: grad_out and x per group and column.  K % 16 == 0 and
    N % 16 == 0."""
    return GroupedGemmFp8.apply(x, w, group_sizes)
