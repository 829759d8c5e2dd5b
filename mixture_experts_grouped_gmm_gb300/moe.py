"""The routed MoE layer (``fused_moe``) on this library's kernels.

pytorch-labs/applied-ai issue 24 (the column-major fused MoE script, built on
vLLM's fused_moe.py), ``fused_moe``: the top-k expert ids are aligned to the
block size (``moe_align_block_size``); the first GEMM multiplies each (token,
slot) entry by its expert's w1 and writes row ``entry`` of a [T * top_k, 2F]
cache; ``silu_and_mul`` gates it to [T * top_k, F]; the second GEMM multiplies
each entry by its expert's w2, scaled by its routed weight; the top_k rows of
each token are summed.

Here the steps are:
  mgemm_moe_align    sorted entries, block experts, padded group sizes
  mgemm_fill_args    args block of the sorted rows (M = -1: the padded total)
  mgemm_gather_rows  the token rows in sorted order (zeros for padding)
  mgemm_fwd_gated    first GEMM over the sorted rows with silu_and_mul in its
                     epilogue (gate and up columns of w1 in one accumulator),
                     output kept in sorted order: exactly the rows the second
                     GEMM reads (padding rows give zeros)
  mgemm_fwd_scatter  second GEMM, each row times its routed weight and stored
                     at its (token, slot) entry
  mgemm_topk_sum     the sum over each token's top_k entries
The page's layer writes the first GEMM's [T * top_k, 2F] output, gates it in a
second pass and gathers it again for the second GEMM; here the gate is applied
before the first rounding and the gated rows stay in sorted order, so neither
the 2F-wide cache nor the second gather exists.
``fused_moe`` starts from the gating logits, as the page's does: the routing
(softmax over the experts, top-k, optional renormalization) is
``mgemm_topk_softmax``.  ``fused_experts`` starts from routing weights and ids
the caller already has.  For decode-size batches the routing, the alignment and
the args block come from one launch (``mgemm_moe_route_align``, the same
results bit for bit), and for at most 32 entries (a hidden size that is a
multiple of 64) the first GEMM reads the token rows through the sorted ids
itself (``mgemm_fwd_gated_gather``), so the layer takes four launches.  This
module only
allocates buffers with torch and calls the binding; every step runs in the
CUDA library, and nothing waits on the host.
"""

import torch

from . import binding as B

BLOCK = B.MGEMM_TILE_M  # rows per block: the GEMM's row tile
# fused_moe routes batches of at most this many tokens in the one-CTA launch
# (mgemm_moe_route_align, one warp per token); larger batches use the routing
# kernel's one warp per token over many CTAs
ROUTE_ALIGN_TOKENS = 16


def align(topk_ids, E, block=BLOCK):
    """mgemm_moe_align with freshly allocated outputs: (sorted_ids,
    expert_ids, num_post_padded, group_sizes)."""
    dev = topk_ids.device
    ids = topk_ids.to(torch.int32).contiguous()
    n = ids.numel()
    cap, max_blocks = B.moe_align_buffer_sizes(n, E, block)
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(max_blocks, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    gs = torch.empty(E, dtype=torch.int64, device=dev)
    ws = torch.empty(B.mgemm_moe_align_workspace_bytes(n, E), dtype=torch.uint8, device=dev)
    B.mgemm_moe_align(ids, E, block, sorted_ids, expert_ids, npp, ws, gs)
    return sorted_ids, expert_ids, npp, gs


def route(gating_output, topk, renormalize):
    """mgemm_topk_softmax: (topk_weights float32 [T, topk], topk_ids int32 [T, topk])."""
    g = gating_output.to(torch.float32).contiguous()
    T = g.shape[0]
    w = torch.empty(T, topk, dtype=torch.float32, device=g.device)
    i = torch.empty(T, topk, dtype=torch.int32, device=g.device)
    B.mgemm_topk_softmax(g, topk, renormalize, w, i)
    return w, i


def route_align(gating_output, topk, renormalize, block=BLOCK):
    """mgemm_moe_route_align from gating logits [T, E], with freshly allocated
    outputs: (topk_weights, topk_ids, sorted_ids, expert_ids, num_post_padded,
    group_sizes, args)."""
    g = gating_output.to(torch.float32).contiguous()
    T, E = g.shape
    w = torch.empty(T, topk, dtype=torch.float32, device=g.device)
    ids = torch.empty(T, topk, dtype=torch.int32, device=g.device)
    return _route_align(g, w, ids, T, E, topk, renormalize, block)


def align_args(topk_ids, E, block=BLOCK):
    """mgemm_moe_route_align on given ids: (sorted_ids, expert_ids,
    num_post_padded, group_sizes, args)."""
    ids = topk_ids.to(torch.int32).contiguous()
    T, topk = ids.shape
    r = _route_align(None, None, ids, T, E, topk, False, block)
    return r[2:]


def _route_align(g, w, ids, T, E, topk, renormalize, block):
    dev = ids.device
    n = T * topk
    cap, max_blocks = B.moe_align_buffer_sizes(n, E, block)
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(max_blocks, dtype=torch.int32, device=dev)
    npp = torch.empty(1, dtype=torch.int32, device=dev)
    gs = torch.empty(E, dtype=torch.int64, device=dev)
    args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=dev)
    B.mgemm_moe_route_align(g, T, E, topk, renormalize, block, w, ids, sorted_ids, expert_ids, npp, args, gs)
    return w, ids, sorted_ids, expert_ids, npp, gs, args


def _check_layer(hidden_states, w1, w2):
    if hidden_states.dtype != torch.bfloat16 or w1.dtype != torch.bfloat16 or w2.dtype != torch.bfloat16:
        raise B.MgemmError("fused_moe takes bf16 activations and weights")


def fused_moe(hidden_states, w1, w2, gating_output, topk, renormalize):
    """The page's fused_moe: route by gating_output [T, E] (top-k of the
    softmax, renormalized when asked), then fused_experts."""
    T = gating_output.shape[0]
    if T <= ROUTE_ALIGN_TOKENS and T * topk <= B.MGEMM_ROUTE_ALIGN_MAX_ENTRIES:
        _check_layer(hidden_states, w1, w2)
        tw, _, sorted_ids, _, npp, _, args = route_align(gating_output, topk, renormalize)
        return _experts(hidden_states, w1, w2, tw, sorted_ids, npp, args, T, topk)
    topk_weights, topk_ids = route(gating_output, topk, renormalize)
    return fused_experts(hidden_states, w1, w2, topk_weights, topk_ids)


def fused_experts(hidden_states, w1, w2, topk_weights, topk_ids):
    """hidden_states bf16 [T, H]; w1 bf16 [E, 2F, H]; w2 bf16 [E, H, F];
    topk_weights float32 [T, top_k]; topk_ids int [T, top_k], every id in
    [0, E) (as in fused_moe, whose caches are uninitialized: an entry that is
    not placed leaves its rows undefined).  Returns bf16 [T, H]."""
    _check_layer(hidden_states, w1, w2)
    T, top_k = topk_ids.shape
    E = w1.shape[0]
    n = T * top_k
    if n <= B.MGEMM_ROUTE_ALIGN_MAX_ENTRIES:
        sorted_ids, _, npp, _, args = align_args(topk_ids, E)
    else:
        sorted_ids, _, npp, gs = align(topk_ids, E)
        args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=sorted_ids.device)
        B.mgemm_fill_args(gs, E, -1, args)
    return _experts(hidden_states, w1, w2, topk_weights, sorted_ids, npp, args, T, top_k)


def _experts(hidden_states, w1, w2, topk_weights, sorted_ids, npp, args, T, top_k):
    """The gather, the two GEMMs and the top-k sum over aligned entries."""
    x = hidden_states.contiguous()
    w1 = w1.contiguous()
    w2 = w2.contiguous()
    H = x.shape[1]
    E, F2, _ = w1.shape
    F = F2 // 2
    n = T * top_k
    dev = x.device
    cap = sorted_ids.numel()
    # rows the GEMMs may see: every entry, plus the padding of at most
    # min(E, n) experts (a bound known on the host; it sizes their tiles)
    rows = min(cap, n + min(E, n) * (BLOCK - 1))
    bf = torch.bfloat16
    a2 = torch.empty(cap, F, dtype=bf, device=dev)  # rows past the padded total are never read
    # every group holds at most n routed rows (decode-size batches: n < 128)
    if n <= 32 and H % 64 == 0:
        # the first GEMM reads the token rows through the sorted ids itself
        B.mgemm_fwd_gated_gather(args, x, sorted_ids, n, top_k, w1, a2, rows, H, F, E, n)
    else:
        a1 = torch.empty(cap, H, dtype=bf, device=dev)
        B.mgemm_gather_rows(x, sorted_ids, npp, n, top_k, a1)
        B.mgemm_fwd_gated(args, a1, w1, a2, rows, H, F, E, n)
    c3 = torch.empty(n, H, dtype=bf, device=dev)
    wts = topk_weights.to(torch.float32).contiguous().view(-1)
    B.mgemm_fwd_scatter(args, B.MGEMM_BF16, 1, a2, w2, c3, sorted_ids, n, wts, rows, F, H, E)
    out = torch.empty(T, H, dtype=bf, device=dev)
    B.mgemm_topk_sum(c3, T, top_k, out)
    return out
