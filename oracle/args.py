"""Device-side argument fill, restated as plain Python (oracle; test infrastructure only).

Sources:
* "Support GPU-resident batch sizes" (tgale96/grouped_gemm PR #21),
  description: a single-threadblock kernel turns the list of batch sizes that
  lives on the GPU into the per-problem GEMM arguments, so the sizes never
  travel to the host; at most 1024 experts (one thread per expert).
* same page, review of csrc/fill_arguments.cuh: "If k is dynamic, we sort the
  problems by k in descending order. Otherwise, m is dynamic, and no sorting
  happens" (kDynamicK), and the block scan over batch sizes.
* same page, review of ZeroOutK0Outputs / IgnoreK0Problems: problems whose
  contraction length is 0 (wgrad of an empty expert) must produce zeros.
* "F8I4 Grouped Gemm Optimization for Sparse M" (pytorch/FBGEMM PR #3854),
  Summary: set up the grouped GEMM over min(total_M, groups) problems so that
  empty groups cost nothing.

Readings (where the pages are silent):
* offsets are exclusive prefix sums, offsets[0] = 0, offsets[E] = M; group e
  owns rows [offsets[e], offsets[e+1]).
* the active list holds exactly the non-empty groups in ascending expert id;
  its length is <= min(M, E).
* the tile prefix counts row tiles of ``tile_m`` rows per active group;
  column tiles are multiplied in by each GEMM since they depend on its N.
* the wgrad order is a stable sort by size, descending: equal sizes keep
  ascending expert id; empty experts come last (they still get a zero block).
* errors: any negative size -> status 1 (checked first); sizes that do not sum
  to M -> status 2; otherwise 0.  With a non-zero status the other fields are
  unspecified.
"""

STATUS_OK = 0
STATUS_NEGATIVE_SIZE = 1
STATUS_SUM_MISMATCH = 2


def fill_args(group_sizes, M, tile_m=128):
    """Return a dict with status, offsets, active, mtile_start, wgrad_order."""
    sizes = [int(s) for s in group_sizes]
    E = len(sizes)
    status = STATUS_OK
    if any(s < 0 for s in sizes):
        status = STATUS_NEGATIVE_SIZE
    elif sum(sizes) != int(M):
        status = STATUS_SUM_MISMATCH

    offsets = [0]
    for s in sizes:                       # sequential exclusive scan
        offsets.append(offsets[-1] + s)

    active = [e for e in range(E) if sizes[e] > 0]
    mtile_start = [0]
    for e in active:
        mtile_start.append(mtile_start[-1] + (sizes[e] + tile_m - 1) // tile_m)

    # stable sort by descending size (Python's sort is stable)
    wgrad_order = sorted(range(E), key=lambda e: -sizes[e])

    return {
        "status": status,
        "offsets": offsets,
        "n_active": len(active),
        "active": active,
        "mtile_start": mtile_start,
        "wgrad_order": wgrad_order,
    }
