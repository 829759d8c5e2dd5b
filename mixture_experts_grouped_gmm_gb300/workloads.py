"""Seeded synthetic inputs for the grouped GEMM workloads.

This module only draws random inputs; it holds none of the grouped GEMM's
arithmetic (no scan, no quantization, no product).  Both the CUDA path and the
CPU oracle consume what it returns, so the two sides always see the same bytes.

Shapes and distributions follow the workloads on the source pages:

* ``tiny``   -- E=4, M=64, K=128, N=256; group sizes multinomial(64, uniform
  over 4); x, w ~ U[0, 1) bf16.  A variant forces one empty group.
* ``grin``   -- the GRIN-MoE benchmark script of "Support GPU-resident batch
  sizes" (tgale96/grouped_gemm PR #21): M=1024, K=4096, N=6400, E=8, batch
  sizes [M/E]*E (int64, on the device), x[M, K] and w[E, K, N] from
  ``torch.rand`` in bf16 after ``manual_seed(0)``.
* ``sparse_m`` -- "F8I4 Grouped Gemm Optimization for Sparse M" (FBGEMM PR
  #3854): total_M tokens each routed to a uniformly random one of E=128
  experts; K=5120, N=8192; x ~ N(0, 1), w ~ N(0, 0.02) in bf16 (the FP8 path
  quantizes both).
* ``mixtral`` -- the routed layer of the column-major fused MoE page
  (pytorch-labs/applied-ai issue 24): T tokens, hidden 4096, E=8, top-2 of the
  softmax of N(0, 1) gating logits, token copies sorted by expert and each
  group padded to a multiple of 128 rows (the moe_align_block_size layout, with
  padding rows set to zero); w1[E, 4096, 2*14336], w2[E, 14336, 4096] ~ N(0, 0.02).
* ``deepseek`` -- the DeepSeek-MoE-16B backward shapes of "[moe training]
  Optimize FP8 MoE backward pass" (pytorch/ao commit 34322b5): 16384 tokens,
  hidden 2048, expert ffn 1408, E=64, top-6 experts per token drawn without
  replacement from a Zipf(s=1.2) popularity over a seeded permutation, with 4
  seeded experts at popularity 0 so that several groups are empty.

Every generator takes a ``device`` and draws with a ``torch.Generator`` on it,
so large workloads are created directly in HBM.  All tensors are contiguous.
"""

import torch

BF16 = torch.bfloat16


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _counts(expert_ids, E):
    return torch.bincount(expert_ids.reshape(-1).to(torch.int64).cpu(), minlength=E).to(torch.int64)


def tiny(seed=0, zero_group=False, device="cpu", E=4, M=64, K=128, N=256):
    gh = _gen("cpu", seed)
    if zero_group:
        sizes = torch.tensor([0, 20, 20, 24][:E], dtype=torch.int64)
        sizes[-1] += M - int(sizes.sum())
    else:
        picks = torch.multinomial(torch.full((E,), 1.0 / E), M, replacement=True, generator=gh)
        sizes = _counts(picks, E)
    g = _gen(device, seed)
    x = torch.rand(M, K, generator=g, device=device, dtype=torch.float32).to(BF16)
    w = torch.rand(E, K, N, generator=g, device=device, dtype=torch.float32).to(BF16)
    return dict(x=x, w=w, group_sizes=sizes.to(device), E=E, M=M, K=K, N=N)


def grin(seed=0, device="cpu", M=1024, K=4096, N=6400, E=8):
    g = _gen(device, seed)
    x = torch.rand(M, K, generator=g, device=device, dtype=torch.float32).to(BF16)
    w = torch.rand(E, K, N, generator=g, device=device, dtype=torch.float32).to(BF16)
    sizes = torch.tensor([M // E] * E, dtype=torch.int64, device=device)
    return dict(x=x, w=w, group_sizes=sizes, E=E, M=M, K=K, N=N)


def sparse_m(total_m, E=128, K=5120, N=8192, seed=None, device="cpu", with_weights=True):
    """Token rows sorted by expert; w is [E, N, K] (the FP8 forward layout)."""
    seed = total_m if seed is None else seed
    gh = _gen("cpu", seed)
    experts = torch.randint(0, E, (total_m,), generator=gh)
    sizes = _counts(experts, E)
    g = _gen(device, seed)
    x = torch.randn(total_m, K, generator=g, device=device, dtype=torch.float32).to(BF16)
    out = dict(x=x, group_sizes=sizes.to(device), E=E, M=total_m, K=K, N=N)
    if with_weights:
        w = torch.empty(E, N, K, device=device, dtype=BF16)
        for e in range(E):          # per expert, to bound the fp32 temporary
            w[e] = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02).to(BF16)
        out["w_nk"] = w
    return out


def _normal_weights(shape, g, device, std=0.02):
    w = torch.empty(shape, device=device, dtype=BF16)
    for e in range(shape[0]):
        w[e] = (torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32) * std).to(BF16)
    return w


def mixtral(seed=0, device="cpu", T=4096, H=4096, F=14336, E=8, topk=2, pad=128, with_weights=True):
    gh = _gen("cpu", seed)
    logits = torch.randn(T, E, generator=gh)
    probs = torch.softmax(logits, dim=-1)
    topw, topi = torch.topk(probs, topk, dim=-1)
    flat_e = topi.reshape(-1)
    order = torch.sort(flat_e, stable=True).indices            # token copies grouped by expert
    counts = _counts(flat_e, E)
    padded = ((counts + pad - 1) // pad) * pad
    M = int(padded.sum())
    src_token = torch.full((M,), -1, dtype=torch.int64)         # -1 marks a zero padding row
    starts = torch.cumsum(padded, 0) - padded
    pos = 0
    for e in range(E):
        c = int(counts[e])
        src_token[int(starts[e]):int(starts[e]) + c] = order[pos:pos + c] // topk
        pos += c
    g = _gen(device, seed)
    hidden = torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(BF16)
    idx = src_token.to(device)
    x = torch.zeros(M, H, device=device, dtype=BF16)
    valid = idx >= 0
    x[valid] = hidden[idx[valid]]
    out = dict(x=x, group_sizes=padded.to(device), counts=counts, src_token=src_token,
               topk_weights=topw, topk_ids=topi, E=E, M=M, T=T, H=H, F=F)
    if with_weights:
        out["w1"] = _normal_weights((E, H, 2 * F), g, device)
        out["w2"] = _normal_weights((E, F, H), g, device)
    return out


def deepseek(seed=0, device="cpu", T=16384, H=2048, F=1408, E=64, topk=6, zipf_s=1.2, n_dead=4,
             with_weights=True):
    gh = _gen("cpu", seed)
    perm = torch.randperm(E, generator=gh)
    pop = torch.empty(E, dtype=torch.float64)
    pop[perm] = 1.0 / torch.arange(1, E + 1, dtype=torch.float64) ** zipf_s
    dead = torch.randperm(E, generator=gh)[:n_dead]
    pop[dead] = 0.0
    choice = torch.multinomial((pop / pop.sum()).float().expand(T, E), topk, replacement=False, generator=gh)
    sizes = _counts(choice, E)
    M = int(sizes.sum())
    g = _gen(device, seed)
    x = torch.randn(M, H, generator=g, device=device, dtype=torch.float32).to(BF16)
    grad_out = torch.randn(M, F, generator=g, device=device, dtype=torch.float32).to(BF16)
    out = dict(x=x, grad_out=grad_out, group_sizes=sizes.to(device), E=E, M=M, K=H, N=F, dead=dead)
    if with_weights:
        out["w"] = _normal_weights((E, H, F), g, device)            # [E, K, N] master layout
    return out
