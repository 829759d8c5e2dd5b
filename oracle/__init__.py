"""Plain CPU oracle for the MoE grouped GEMM hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports, calls or links anything here, and nothing here imports the product.

Every routine is slow and obviously correct: numpy in float64, loops over
groups, a library matmul as the only contraction primitive.  Each function
cites the passage of the source pages it restates:

* "Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21) -- the
  gmm(x, w, batch_sizes) benchmark script, the review of
  csrc/fill_arguments.cuh (kDynamicK sort, block scan) and of
  csrc/grouped_gemm.cu (trans_a / trans_b templates, k=0 outputs).
* "F8I4 Grouped Gemm Optimization for Sparse M" (pytorch/FBGEMM PR #3854),
  Summary -- run only over the non-empty groups.
* "[moe training] Optimize FP8 MoE backward pass: fused colwise kernel + AMD
  tuning" (pytorch/ao commit 34322b5) -- the commit message (rowwise 3-op
  sequence, dual colwise kernel; the MXFP8 path and its 32-row group
  padding) and bench_colwise_block_configs.py (_colwise_kernel,
  run_experiment).
* "F8I4 Grouped Gemm Optimization for Sparse M" (pytorch/FBGEMM PR #3854),
  title and Summary -- FP8 activations times INT4 weights (f8i4).
* pytorch-labs/applied-ai issue 24 (the column-major fused MoE script on
  vLLM's fused_moe.py) -- moe_align_block_size and its worked example,
  fused_moe_kernel, silu_and_mul, topk_softmax, the fused_moe layer.

Modules:
  formats -- FP8 e4m3fn decode / saturating round-to-nearest-even encode, bf16 rounding
  args   -- group-size scan, active-group compaction, tile prefix, wgrad order
  quant  -- power-of-two absmax scales, rowwise and per-group colwise quantize
  gmm    -- forward, dgrad and wgrad for bf16 and FP8-scaled operands
  mx     -- MXFP8: 32-element block scales (e8m0), row and per-group column block quantize, block-scaled fwd and wgrad
  f8i4   -- FP8 x INT4: 32-element INT4 block quantize (e8m0 scales), nibble packing, the grouped forward
  routing -- moe_align_block_size, gather, topk_softmax, silu_and_mul and the fused_moe layer of the routed path

Parity status: every function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``; none is "parity unpinned".
"""

from . import args, f8i4, formats, gmm, mx, quant, routing  # noqa: F401
