"""Thin Python binding of libmgemm.so (the C ABI in include/mgemm.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU (or None), passes their data pointers, sizes and the current
CUDA stream to the C entry point of the same name, and raises
``MgemmError`` on a negative return code.  No arithmetic of the path happens
here, and there is no fallback: if the library is missing the first call
raises.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmgemm.so")

MGEMM_OK = 0
MGEMM_BF16 = 0
MGEMM_FP8_E4M3 = 1
MGEMM_MAX_EXPERTS = 1024
MGEMM_TILE_M = 128
MGEMM_COL_PAD = 128
STATUS = {0: "ok", 1: "negative group size", 2: "group sizes do not sum to M", 4: "pipeline wait timed out"}

_lib = None


class MgemmError(RuntimeError):
    pass


_SIGS = {
    "mgemm_args_bytes": (ctypes.c_size_t, [ctypes.c_int]),
    "mgemm_args_layout": (ctypes.c_int, [ctypes.c_int] + [ctypes.POINTER(ctypes.c_size_t)] * 4),
    "mgemm_fill_args": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_void_p]),
    "mgemm_quant_rowwise": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_quant_colwise_grouped": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_void_p]),
    "mgemm_quant_mx": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p]),
    "mgemm_fwd_mx": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mgemm_quant_colwise_mx": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                              ctypes.c_void_p]),
    "mgemm_wgrad_mx": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int64, ctypes.c_void_p]),
    "mgemm_fill_args_quant_rowwise": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_fwd_fp8_strided": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_void_p]),
    "mgemm_fwd_fp8_sparse": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mgemm_quant_int4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_fwd_f8i4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_void_p]),
    "mgemm_colwise_ld": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int]),
    "mgemm_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mgemm_dgrad": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mgemm_wgrad": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p]),
    "mgemm_dgrad_wgrad": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mgemm_dgrad_wgrad_split": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "mgemm_fwd_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "mgemm_moe_align_workspace_bytes": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int]),
    "mgemm_moe_align": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_gather_rows": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "mgemm_fwd_scatter": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p]),
    "mgemm_fwd_gated": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_void_p]),
    "mgemm_fwd_gated_gather": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int64, ctypes.c_void_p]),
    "mgemm_silu_and_mul": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                          ctypes.c_void_p]),
    "mgemm_topk_sum": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_topk_softmax": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_moe_route_align": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p]),
    "mgemm_num_sms": (ctypes.c_int, []),
    "mgemm_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mgemm_version": (ctypes.c_int, []),
    "mgemm_last_error": (ctypes.c_char_p, []),
}


def lib():
    """Load libmgemm.so once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MgemmError(f"{LIB_PATH} is missing; build it with mixture_experts_grouped_gmm_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t=None):
    dev = t.device if t is not None else None
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(rc, what):
    if rc != MGEMM_OK:
        detail = lib().mgemm_last_error().decode() if rc == -4 else ""
        raise MgemmError(f"{what} failed: {rc} ({lib().mgemm_error_string(rc).decode()}) {detail}")


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise MgemmError("mgemm kernels take device tensors only")


def mgemm_args_bytes(E):
    return int(lib().mgemm_args_bytes(int(E)))


def mgemm_args_layout(E):
    vals = [ctypes.c_size_t() for _ in range(4)]
    _check(lib().mgemm_args_layout(int(E), *[ctypes.byref(v) for v in vals]), "mgemm_args_layout")
    return dict(zip(("offsets", "active", "mtile_start", "wgrad_order"), (v.value for v in vals)))


def mgemm_fill_args(group_sizes, E, M, args):
    _cuda(group_sizes, args)
    _check(lib().mgemm_fill_args(_p(group_sizes), int(E), int(M), _p(args), _stream(args)), "mgemm_fill_args")


def mgemm_quant_rowwise(inp, out, scales):
    _cuda(inp, out, scales)
    R, C = inp.shape
    _check(lib().mgemm_quant_rowwise(_p(inp), R, C, inp.stride(0), _p(out), out.stride(0), _p(scales),
                                     _stream(inp)), "mgemm_quant_rowwise")


MX_BLOCK = 32


def mx_ld_sf(C):
    """Bytes per scale row of mgemm_quant_mx for C columns: C / 32 rounded up to 16."""
    return -(-(C // MX_BLOCK) // 16) * 16


def mgemm_quant_mx(inp, out, sf):
    """inp bf16 [R, C] -> out e4m3 [R, C] (uint8) and sf e8m0 [R, ld_sf] (uint8)."""
    _cuda(inp, out, sf)
    R, C = inp.shape
    _check(lib().mgemm_quant_mx(_p(inp), R, C, inp.stride(0), _p(out), out.stride(0), _p(sf), sf.stride(0),
                                _stream(inp)), "mgemm_quant_mx")


def mgemm_fwd_mx(args, x, sx, w, sw, out, M, K, N, E):
    """MXFP8 grouped GEMM: x e4m3 [M, K] + sx [M, ld_sf]; w e4m3 [E, N, K] + sw [E * N, ld_sf]."""
    _cuda(args, x, sx, w, sw, out)
    _check(lib().mgemm_fwd_mx(_p(args), _p(x), _p(sx), _p(w), _p(sw), sx.stride(0), _p(out), int(M), int(K), int(N),
                              int(E), _stream(out)), "mgemm_fwd_mx")


def mgemm_quant_colwise_mx(args, E, M, x1, out1, sf1, x2=None, out2=None, sf2=None, ld=None):
    """Per-group colwise MX blocks of x1 [M, C1] (and x2 [M, C2]) into the padded
    column-major codes out1 [C1 * ld] and scale rows sf1 [ld / 128 * C1 * 4]."""
    _cuda(args, x1, out1, sf1, x2, out2, sf2)
    ld = ld or mgemm_colwise_ld(M, E)
    C2 = x2.shape[1] if x2 is not None else 0
    _check(lib().mgemm_quant_colwise_mx(_p(args), int(E), int(M), _p(x1), x1.shape[1], _p(out1), _p(sf1), _p(x2),
                                        int(C2), _p(out2), _p(sf2), int(ld), _stream(x1)),
           "mgemm_quant_colwise_mx")


def mgemm_wgrad_mx(args, x, sx, go, sgo, grad_w, M, K, N, E, ld=None):
    """MXFP8 wgrad on the outputs of mgemm_quant_colwise_mx -> grad_w bf16 [E, K, N]."""
    _cuda(args, x, sx, go, sgo, grad_w)
    ld = mgemm_colwise_ld(M, E) if ld is None else ld
    _check(lib().mgemm_wgrad_mx(_p(args), _p(x), _p(sx), _p(go), _p(sgo), _p(grad_w), int(M), int(K), int(N), int(E),
                                int(ld), _stream(grad_w)), "mgemm_wgrad_mx")


def mgemm_fill_args_quant_rowwise(group_sizes, E, M, args, x, xq, sx):
    """mgemm_fill_args(group_sizes, E, M, args) and mgemm_quant_rowwise(x, xq, sx) in one launch."""
    _cuda(group_sizes, args, x, xq, sx)
    R, K = x.shape
    if R != M:
        raise MgemmError("x must hold the M token rows")
    _check(lib().mgemm_fill_args_quant_rowwise(_p(group_sizes), int(E), int(M), _p(args), _p(x), K, x.stride(0),
                                               _p(xq), xq.stride(0), _p(sx), _stream(x)),
           "mgemm_fill_args_quant_rowwise")


def mgemm_fwd_fp8_strided(args, x, sx, w, ld_wn, ld_we, sw, out, M, K, N, E):
    """FP8 forward with the e4m3 weights w[e, n, k] at byte e * ld_we + n * ld_wn + k of w."""
    _cuda(args, x, sx, w, sw, out)
    _check(lib().mgemm_fwd_fp8_strided(_p(args), _p(x), _p(sx), _p(w), int(ld_wn), int(ld_we), _p(sw), _p(out), int(M),
                                       int(K), int(N), int(E), _stream(out)), "mgemm_fwd_fp8_strided")


SPARSE_MAX_ROWS = 16


def mgemm_fwd_fp8_sparse(group_sizes, E, x, w, sw, out, status):
    """fill + rowwise cast of x + FP8 forward in one launch, for at most 16 token rows.
    x bf16 [M, K]; w e4m3 [E, N, K] (uint8); sw fp32 [E * N]; out bf16 [M, N]; status int32 [1]."""
    _cuda(group_sizes, x, w, sw, out, status)
    M, K = x.shape
    N = out.shape[1]
    _check(lib().mgemm_fwd_fp8_sparse(_p(group_sizes), int(E), _p(x), x.stride(0), _p(w), _p(sw), _p(out), _p(status),
                                      int(M), int(K), int(N), _stream(out)), "mgemm_fwd_fp8_sparse")


def int4_scale_bytes(E, N, K):
    """Bytes of mgemm_quant_int4's scale array: one e8m0 byte per 32 elements."""
    return E * (K // 128) * N * 4


def mgemm_quant_int4(w, packed, sf):
    """w bf16 [E, N, K] -> packed uint8 [E, N, K // 2], sf uint8 [int4_scale_bytes]."""
    _cuda(w, packed, sf)
    E, N, K = w.shape
    if w.stride(2) != 1 or w.stride(0) != N * w.stride(1):
        raise MgemmError("mgemm_quant_int4 takes w [E, N, K] with rows (e, n) at a common stride")
    _check(lib().mgemm_quant_int4(_p(w), E, N, K, w.stride(1), _p(packed), _p(sf), _stream(w)), "mgemm_quant_int4")


def mgemm_fwd_f8i4(args, x, sx, w_packed, w_scales, out, M, K, N, E):
    _cuda(args, x, sx, w_packed, w_scales, out)
    _check(lib().mgemm_fwd_f8i4(_p(args), _p(x), _p(sx), _p(w_packed), _p(w_scales), _p(out), int(M), int(K), int(N),
                                int(E), _stream(out)), "mgemm_fwd_f8i4")


def mgemm_colwise_ld(M, E):
    """Bytes per column of the padded column-major FP8 layout (a multiple of 128)."""
    return int(lib().mgemm_colwise_ld(int(M), int(E)))


def mgemm_quant_colwise_grouped(args, E, M, in1, out1, sc1, in2=None, out2=None, sc2=None, ld=None):
    """out1 / out2: C * ld bytes (ld defaults to their size / C), padded column-major."""
    _cuda(args, in1, out1, sc1, in2, out2, sc2)
    C1 = in1.shape[1]
    C2 = in2.shape[1] if in2 is not None else 0
    if ld is None:
        ld = out1.numel() // C1
    _check(lib().mgemm_quant_colwise_grouped(_p(args), int(E), int(M), _p(in1), C1, _p(out1), _p(sc1),
                                             _p(in2), C2, _p(out2), _p(sc2), int(ld), _stream(in1)),
           "mgemm_quant_colwise_grouped")


def mgemm_fwd(args, dtype, trans_b, x, sx, w, sw, out, M, K, N, E):
    _cuda(args, x, sx, w, sw, out)
    _check(lib().mgemm_fwd(_p(args), int(dtype), int(trans_b), _p(x), _p(sx), _p(w), _p(sw), _p(out), int(M),
                           int(K), int(N), int(E), _stream(out)), "mgemm_fwd")


def mgemm_dgrad(args, dtype, grad_out, sgo, w, sw, grad_x, M, K, N, E):
    _cuda(args, grad_out, sgo, w, sw, grad_x)
    _check(lib().mgemm_dgrad(_p(args), int(dtype), _p(grad_out), _p(sgo), _p(w), _p(sw), _p(grad_x), int(M),
                             int(K), int(N), int(E), _stream(grad_x)), "mgemm_dgrad")


def mgemm_wgrad(args, dtype, x, sx, grad_out, sgo, grad_w, M, K, N, E, ld=None):
    """FP8: x [K, ld] and grad_out [N, ld] padded column-major (ld defaults to x's size / K)."""
    _cuda(args, x, sx, grad_out, sgo, grad_w)
    if ld is None:
        ld = x.numel() // K if dtype == MGEMM_FP8_E4M3 and x is not None else 0
    _check(lib().mgemm_wgrad(_p(args), int(dtype), _p(x), _p(sx), _p(grad_out), _p(sgo), _p(grad_w), int(M),
                             int(K), int(N), int(E), int(ld), _stream(grad_w)), "mgemm_wgrad")


def mgemm_dgrad_wgrad(args, grad_out, w, x, grad_x, grad_w, M, K, N, E):
    """bf16 backward with w [E, K, N]: grad_x (as mgemm_dgrad) and grad_w (as mgemm_wgrad), in one launch
    where the two share the GPU better than they take turns."""
    _cuda(args, grad_out, w, x, grad_x, grad_w)
    _check(lib().mgemm_dgrad_wgrad(_p(args), _p(grad_out), _p(w), _p(x), _p(grad_x), _p(grad_w), int(M), int(K),
                                   int(N), int(E), _stream(grad_w)), "mgemm_dgrad_wgrad")


def mgemm_dgrad_wgrad_split(M, K, N, E):
    """CTAs mgemm_dgrad_wgrad gives dgrad in one launch (0: two launches in turn)."""
    rc = lib().mgemm_dgrad_wgrad_split(int(M), int(K), int(N), int(E))
    if rc < 0:
        _check(rc, "mgemm_dgrad_wgrad_split")
    return rc


def mgemm_fwd_noalloc(group_sizes, dtype, trans_b, x, sx, w, sw, out, M, K, N, E):
    """Forward pass without a caller-provided args block (for callers that
    cannot allocate device memory; the library keeps the block in a static
    device array shared by all calls)."""
    _cuda(group_sizes, x, sx, w, sw, out)
    _check(lib().mgemm_fwd_noalloc(_p(group_sizes), int(E), int(dtype), int(trans_b), _p(x), _p(sx), _p(w), _p(sw),
                                   _p(out), int(M), int(K), int(N), _stream(out)), "mgemm_fwd_noalloc")


def mgemm_moe_align_workspace_bytes(numel, E):
    return int(lib().mgemm_moe_align_workspace_bytes(int(numel), int(E)))


def moe_align_buffer_sizes(numel, E, block_size):
    """(entries of sorted_ids, entries of expert_ids) for mgemm_moe_align."""
    cap = int(numel) + int(E) * (int(block_size) - 1)
    return cap, cap // int(block_size)


def mgemm_moe_align(topk_ids, E, block_size, sorted_ids, expert_ids, num_post_padded, workspace, group_sizes=None):
    """moe_align_block_size on the device: topk_ids int32 (any shape, flattened
    row-major); outputs as laid out in mgemm.h."""
    _cuda(topk_ids, sorted_ids, expert_ids, num_post_padded, workspace, group_sizes)
    _check(lib().mgemm_moe_align(_p(topk_ids), int(topk_ids.numel()), int(E), int(block_size), _p(sorted_ids),
                                 _p(expert_ids), _p(num_post_padded), _p(group_sizes), _p(workspace),
                                 _stream(sorted_ids)), "mgemm_moe_align")


def mgemm_gather_rows(src, sorted_ids, num_post_padded, numel, top_k, dst):
    """dst row s = src row sorted_ids[s] // top_k (zeros for padding entries), s < *num_post_padded."""
    _cuda(src, sorted_ids, num_post_padded, dst)
    rb = src.shape[1] * src.element_size()
    _check(lib().mgemm_gather_rows(_p(src), src.shape[0], rb, src.stride(0) * src.element_size(), _p(sorted_ids),
                                   _p(num_post_padded), int(numel), int(top_k), _p(dst), dst.shape[0],
                                   dst.stride(0) * dst.element_size(), _stream(dst)), "mgemm_gather_rows")


def mgemm_fwd_scatter(args, dtype, trans_b, x, w, out, row_map, map_limit, row_weight, M, K, N, E):
    _cuda(args, x, w, out, row_map, row_weight)
    _check(lib().mgemm_fwd_scatter(_p(args), int(dtype), int(trans_b), _p(x), _p(w), _p(out), _p(row_map),
                                   int(map_limit), _p(row_weight), int(M), int(K), int(N), int(E), _stream(out)),
           "mgemm_fwd_scatter")


def mgemm_fwd_gated(args, x, w, out, M, K, F, E, group_rows_max=0):
    """out [M, F] = silu(x . w_gate^T) * (x . w_up^T), w [E, 2F, K] bf16."""
    _cuda(args, x, w, out)
    _check(lib().mgemm_fwd_gated(_p(args), _p(x), _p(w), _p(out), int(M), int(K), int(F), int(E),
                                 int(group_rows_max), _stream(out)),
           "mgemm_fwd_gated")


def mgemm_fwd_gated_gather(args, x, sorted_ids, numel, top_k, w, out, M, K, F, E, group_rows_max):
    """mgemm_fwd_gated over the token rows x [T, K] read through sorted_ids
    (row sorted_ids[i] // top_k; ids >= numel are padding)."""
    _cuda(args, x, sorted_ids, w, out)
    _check(lib().mgemm_fwd_gated_gather(_p(args), _p(x), x.shape[0], _p(sorted_ids), int(numel), int(top_k), _p(w),
                                        _p(out), int(M), int(K), int(F), int(E), int(group_rows_max), _stream(out)),
           "mgemm_fwd_gated_gather")


def mgemm_silu_and_mul(inp, out):
    _cuda(inp, out)
    R, F2 = inp.shape
    _check(lib().mgemm_silu_and_mul(_p(inp), R, F2 // 2, _p(out), _stream(out)), "mgemm_silu_and_mul")


def mgemm_topk_sum(inp, T, top_k, out):
    _cuda(inp, out)
    _check(lib().mgemm_topk_sum(_p(inp), int(T), int(top_k), inp.shape[-1], _p(out), _stream(out)),
           "mgemm_topk_sum")


def mgemm_topk_softmax(gating, top_k, renormalize, topk_weights, topk_ids):
    """gating float32 [T, E] -> topk_weights float32 [T, top_k], topk_ids int32 [T, top_k]."""
    _cuda(gating, topk_weights, topk_ids)
    T, E = gating.shape
    _check(lib().mgemm_topk_softmax(_p(gating), T, E, int(top_k), int(bool(renormalize)), _p(topk_weights),
                                    _p(topk_ids), _stream(gating)), "mgemm_topk_softmax")


MGEMM_ROUTE_ALIGN_MAX_ENTRIES = 4096


def mgemm_moe_route_align(gating, T, E, top_k, renormalize, block_size, topk_weights, topk_ids, sorted_ids,
                          expert_ids, num_post_padded, args, group_sizes=None):
    """mgemm_topk_softmax + mgemm_moe_align + mgemm_fill_args(M = -1) in one
    launch (T * top_k <= MGEMM_ROUTE_ALIGN_MAX_ENTRIES).  gating float32 [T, E],
    or None: topk_ids int32 [T, top_k] is then the input."""
    _cuda(gating, topk_weights, topk_ids, sorted_ids, expert_ids, num_post_padded, args, group_sizes)
    _check(lib().mgemm_moe_route_align(_p(gating), int(T), int(E), int(top_k), int(bool(renormalize)),
                                       int(block_size), _p(topk_weights), _p(topk_ids), _p(sorted_ids),
                                       _p(expert_ids), _p(num_post_padded), _p(group_sizes), _p(args),
                                       _stream(sorted_ids)), "mgemm_moe_route_align")


def mgemm_num_sms():
    return int(lib().mgemm_num_sms())


def args_status(args):
    """Read the device status word (synchronizes the args tensor's stream)."""
    return int(args[:4].view(torch.int32).item())
