"""Routing-side steps of the fused MoE layer, restated as plain Python (oracle;
test infrastructure only).

Source: pytorch-labs/applied-ai issue 24 (the column-major fused MoE script,
built on vLLM's fused_moe.py): the docstring of ``moe_align_block_size`` and
its worked example, the docstring and body of ``fused_moe_kernel``, and
``fused_moe``.

What ``moe_align_block_size`` computes (docstring): the flat list of
(token, slot) entries of ``topk_ids`` (row-major, so entry i belongs to token
i // top_k) is grouped by expert; each expert's entries are padded with the
id ``numel`` up to a multiple of ``block_size``; ``expert_ids`` names the expert
of every block and ``num_tokens_post_padded`` is the padded total.

Readings (where the page is silent or garbled):
* Order inside an expert: ascending flat index (stable); the worked example
  shows exactly that.
* The worked example names experts 1..4 under ``num_experts = 4``; read as
  0-based expert ids with five experts, expert 0 receiving no entries.  An
  expert with no entries gets no block (padding rounds 0 up to 0).
* Experts appear in ascending id.
* Buffer sizes are the page's: ``sorted_token_ids`` holds
  ``numel + num_experts * (block_size - 1)`` entries, pre-filled with ``numel``
  (so every position past the padded total also reads ``numel``).
  ``expert_ids`` is sized here to the largest possible block count,
  ``(numel + num_experts * (block_size - 1)) // block_size``; the page leaves
  the unused tail uninitialized, here it holds -1.
* Entries outside [0, num_experts) are not placed anywhere (the page does not
  say; vLLM would index out of bounds).
* ``group_sizes`` (not on the page) is each expert's padded count, the row
  count the grouped GEMM of this library takes per expert.
"""


def buffer_sizes(numel, num_experts, block_size):
    """(entries of sorted_token_ids, entries of expert_ids)."""
    cap = numel + num_experts * (block_size - 1)
    return cap, cap // block_size


def moe_align_block_size(topk_ids, block_size, num_experts):
    """topk_ids: nested list / array of expert ids, any shape (flattened
    row-major).  Returns (sorted_token_ids, expert_ids, num_tokens_post_padded,
    group_sizes) as Python lists / int."""
    flat = [int(v) for v in _flatten(topk_ids)]
    numel = len(flat)
    cap, max_blocks = buffer_sizes(numel, num_experts, block_size)
    per_expert = [[] for _ in range(num_experts)]
    for i, e in enumerate(flat):
        if 0 <= e < num_experts:
            per_expert[e].append(i)
    sorted_ids = []
    expert_ids = []
    group_sizes = []
    for e in range(num_experts):
        ids = per_expert[e]
        padded = -(-len(ids) // block_size) * block_size
        sorted_ids += ids + [numel] * (padded - len(ids))
        expert_ids += [e] * (padded // block_size)
        group_sizes.append(padded)
    total = len(sorted_ids)
    sorted_ids += [numel] * (cap - total)
    expert_ids += [-1] * (max_blocks - len(expert_ids))
    return sorted_ids, expert_ids, total, group_sizes


def _flatten(x):
    if hasattr(x, "tolist"):
        x = x.tolist()
    if isinstance(x, (list, tuple)):
        out = []
        for v in x:
            out += _flatten(v)
        return out
    return [x]


def fused_moe_gemm(A, B, sorted_ids, expert_ids, num_post, numel, top_k, block_size, topk_weights=None):
    """One launch of fused_moe_kernel, in float64: for every position s below
    num_post whose id = sorted_ids[s] is a real entry (id < numel), row id of
    the output is A[id // top_k] . B[e]^T with e = expert_ids[s // block_size],
    times topk_weights[id] when weights are given (MUL_ROUTED_WEIGHT).
    A [rows, K], B [E, N, K] (the kernel's b_ptr strides: expert, n, k).
    Returns [numel, N] with NaN in rows no position writes."""
    import numpy as np

    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    N = B.shape[1]
    out = np.full((numel, N), np.nan)
    for s in range(int(num_post)):
        i = int(sorted_ids[s])
        if i >= numel:
            continue  # padding: masked loads and stores
        e = int(expert_ids[s // block_size])
        row = A[i // top_k] @ B[e].T
        if topk_weights is not None:
            row = row * float(topk_weights[i])
        out[i] = row
    return out


def silu_and_mul(x):
    """vLLM's silu_and_mul as fused_moe uses it: for [rows, 2F] input,
    silu(x[:, :F]) * x[:, F:] with silu(v) = v / (1 + exp(-v)), in float64."""
    import numpy as np

    x = np.asarray(x, dtype=np.float64)
    F = x.shape[1] // 2
    g, u = x[:, :F], x[:, F:]
    return g / (1.0 + np.exp(-g)) * u


def gather_rows(src, sorted_ids, num_post, numel, top_k):
    """Row s of the result is src[sorted_ids[s] // top_k] for the real entries
    below num_post, zero for padding (the rows fused_moe_kernel's masked loads
    see)."""
    import numpy as np

    src = np.asarray(src)
    out = np.zeros((int(num_post), src.shape[1]), dtype=np.float64)
    for s in range(int(num_post)):
        i = int(sorted_ids[s])
        if i < numel:
            out[s] = src[i // top_k]
    return out


def topk_softmax(gating_output, top_k, renormalize):
    """fused_moe's routing: softmax over the experts of each token's gating
    logits, the top_k largest probabilities (largest first) and their expert
    ids, divided by their sum when renormalize.  float64.

    Readings: the selection is made on the logits (softmax is strictly
    increasing in each logit, so the top_k probabilities are those of the
    top_k logits); equal logits go to the lower expert id first (the order a
    stable descending sort gives)."""
    import numpy as np

    g = np.asarray(gating_output, dtype=np.float64)
    T, E = g.shape
    ids = np.empty((T, top_k), dtype=np.int64)
    wts = np.empty((T, top_k), dtype=np.float64)
    for t in range(T):
        row = g[t]
        m = row.max()
        ex = np.exp(row - m)
        p = ex / ex.sum()
        order = sorted(range(E), key=lambda e: (-row[e], e))[:top_k]
        ids[t] = order
        wts[t] = p[order]
        if renormalize:
            wts[t] = wts[t] / wts[t].sum()
    return wts, ids


def fused_moe_token(x_row, w1, w2, expert_ids, weights):
    """One token's output of the fused_moe layer, float64: the sum over its
    top-k entries (expert e, routed weight a) of
    a * silu_and_mul(x . w1[e]^T) . w2[e]^T, with w1[e] [2F, H] and w2[e] [H, F]
    (w1, w2: arrays [E, ...] or mappings from expert id to its matrix).
    What fused_moe computes for that token, without the rest of the batch."""
    import numpy as np

    x = np.asarray(x_row, dtype=np.float64)
    out = None
    for e, a in zip(expert_ids, weights):
        up = np.asarray(w1[int(e)], dtype=np.float64) @ x
        h = silu_and_mul(up[None, :])[0]
        y = float(a) * (np.asarray(w2[int(e)], dtype=np.float64) @ h)
        out = y if out is None else out + y
    return out
