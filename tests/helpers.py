"""Shared test helpers: host copies, tolerances, args-block parsing, sentinels."""

import numpy as np
import torch

BF16_TOL = 1e-2   # max|err| <= 1e-2 * max|ref| for bf16 GEMM outputs
FP8_TOL = 3e-2    # max|err| <= 3e-2 * max|ref| for FP8-operand GEMM outputs
SENTINEL_BF16 = 0x7FC1  # a NaN payload no kernel produces


def to_np(t):
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.detach().double().cpu().numpy()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    err = np.max(np.abs(got - ref)) if ref.size else 0.0
    return err, scale


def assert_close(got, ref, tol, what=""):
    err, scale = rel_err(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    assert err <= tol * scale + 1e-30, (f"{what}: max|err| {err:.4g} > {tol} * max|ref| {scale:.4g} "
                                        f"(ratio {err / max(scale, 1e-300):.3g})")


def parse_args(args, E):
    from mixture_experts_grouped_gmm_gb300 import binding as B

    lay = B.mgemm_args_layout(E)
    raw = args.cpu().numpy().tobytes()
    hdr = np.frombuffer(raw[:16], dtype=np.int32)
    out = dict(status=int(hdr[0]), n_active=int(hdr[1]), E=int(hdr[2]),
               M=int(np.frombuffer(raw[16:24], dtype=np.int64)[0]))
    out["offsets"] = np.frombuffer(raw[lay["offsets"]:lay["offsets"] + 8 * (E + 1)], dtype=np.int64).tolist()
    out["active"] = np.frombuffer(raw[lay["active"]:lay["active"] + 4 * E], dtype=np.int32).tolist()
    out["mtile_start"] = np.frombuffer(raw[lay["mtile_start"]:lay["mtile_start"] + 4 * (E + 1)],
                                       dtype=np.int32).tolist()
    out["wgrad_order"] = np.frombuffer(raw[lay["wgrad_order"]:lay["wgrad_order"] + 4 * E], dtype=np.int32).tolist()
    P = (lay["wgrad_order"] + 4 * E + 7) // 8 * 8           # header: W + 4E rounded up to 8
    out["poffsets"] = np.frombuffer(raw[P:P + 8 * (E + 1)], dtype=np.int64).tolist()
    Q = P + 8 * (E + 1)
    out["ptile_start"] = np.frombuffer(raw[Q:Q + 4 * (E + 1)], dtype=np.int32).tolist()
    return out


COL_PAD = 128  # MGEMM_COL_PAD


def padded_offsets(sizes, pad=COL_PAD):
    """Where each group starts in the padded column-major FP8 layout (the header's
    poffsets): the prefix sum of the group sizes, each rounded up to pad."""
    p = [0]
    for m in sizes:
        p.append(p[-1] + -(-int(m) // pad) * pad)
    return p


def unpad_colwise(buf, C, ld, sizes):
    """[C, ld] padded column-major codes -> [C, M] (the groups' rows only)."""
    a = np.asarray(buf).reshape(C, ld)
    po = padded_offsets(sizes)
    parts = [a[:, po[g]:po[g] + int(m)] for g, m in enumerate(sizes)]
    return np.concatenate(parts, axis=1) if parts else a[:, :0]


def colwise_padding(buf, C, ld, sizes):
    """The padding bytes of every group and column (must all be zero codes)."""
    a = np.asarray(buf).reshape(C, ld)
    po = padded_offsets(sizes)
    parts = [a[:, po[g] + int(m):po[g + 1]] for g, m in enumerate(sizes)]
    return np.concatenate(parts, axis=1) if parts else a[:, :0]


def new_args(E, device):
    from mixture_experts_grouped_gmm_gb300 import binding as B

    return torch.zeros(B.mgemm_args_bytes(E), dtype=torch.uint8, device=device)


def sentinel_bf16(shape, device):
    return torch.full(shape, SENTINEL_BF16, dtype=torch.int16, device=device).view(torch.bfloat16)


def is_sentinel(t):
    return bool((t.contiguous().view(torch.int16) == SENTINEL_BF16).all())


def rows_by_expert(sizes, rows):
    """Group sorted sample rows by expert: returns sub-group sizes for oracle calls."""
    off = np.cumsum(sizes)
    e_of = np.searchsorted(off, rows, side="right")
    return [int(np.sum(e_of == e)) for e in range(len(sizes))]
