"""CPU-only checks of the C ABI: the library builds, loads without a GPU,
exports every entry point include/mgemm.h declares, reports the documented
args-block layout, and rejects bad arguments on the host before any CUDA call.
Also checks that the product package never imports the oracle."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mgemm.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_grouped_gmm_gb300 import binding, build

    build.build()
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mgemm_\w+)\s*\(", src)))


def test_header_declares_the_six_hot_path_calls():
    names = declared_functions()
    for n in ("mgemm_fill_args", "mgemm_quant_rowwise", "mgemm_quant_colwise_grouped", "mgemm_fwd",
              "mgemm_dgrad", "mgemm_wgrad"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(os.path.join(ROOT, "mixture_experts_grouped_gmm_gb300", "libmgemm.so"))
    for n in declared_functions():
        assert hasattr(raw, n), n


def test_args_layout_matches_header(lib):
    from mixture_experts_grouped_gmm_gb300 import binding as B

    for E in (1, 4, 8, 64, 128, 1000, 1024):
        lay = B.mgemm_args_layout(E)
        A = 24 + 8 * (E + 1)
        T = A + 4 * E
        W = T + 4 * (E + 1)
        assert lay == dict(offsets=24, active=A, mtile_start=T, wgrad_order=W)
        nbytes = B.mgemm_args_bytes(E)
        assert nbytes >= W + 4 * E and nbytes % 16 == 0
    assert B.mgemm_args_bytes(0) == 0 and B.mgemm_args_bytes(1025) == 0


def test_version_and_error_strings(lib):
    assert lib.mgemm_version() >= 100
    for code in (0, -1, -2, -3, -4, -5, 1, 2, 4):
        assert lib.mgemm_error_string(code).decode() != "unknown code"


P = ctypes.c_void_p


def test_host_checks_fill_args(lib):
    good = P(0x10000)
    assert lib.mgemm_fill_args(None, 4, 64, good, None) == -1
    assert lib.mgemm_fill_args(good, 0, 64, good, None) == -1
    assert lib.mgemm_fill_args(good, 1025, 64, good, None) == -3
    assert lib.mgemm_fill_args(good, 4, -2, good, None) == -1  # M = -1 means "the sum of the sizes"
    assert lib.mgemm_fill_args(good, 4, 64, P(0x10008), None) == -2   # args must be 16-byte aligned


def test_host_checks_gemms(lib):
    a, x, w, o = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    s = P(0x50000)
    assert lib.mgemm_fwd(None, 0, 0, x, None, w, None, o, 64, 128, 256, 4, None) == -1
    assert lib.mgemm_fwd(a, 7, 0, x, None, w, None, o, 64, 128, 256, 4, None) == -1        # dtype
    assert lib.mgemm_fwd(a, 0, 0, x, None, w, None, o, 64, 130, 256, 4, None) == -2        # K % 8
    assert lib.mgemm_fwd(a, 1, 1, x, s, w, s, o, 64, 136, 256, 4, None) == -2              # fp8 K % 16
    assert lib.mgemm_fwd(a, 1, 0, x, s, w, s, o, 64, 128, 256, 4, None) == -5              # fp8 needs [E,N,K]
    assert lib.mgemm_fwd(a, 1, 1, x, None, w, s, o, 64, 128, 256, 4, None) == -1           # scales required
    assert lib.mgemm_fwd(a, 0, 0, P(0x20008), None, w, None, o, 64, 128, 256, 4, None) == -2
    assert lib.mgemm_fwd(a, 0, 0, x, None, w, None, o, 64, 128, 256, 2000, None) == -3
    assert lib.mgemm_fwd(a, 0, 0, x, None, w, None, o, 0, 128, 256, 4, None) == 0          # M = 0: nothing to do
    assert lib.mgemm_dgrad(a, 0, x, None, w, None, None, 64, 128, 256, 4, None) == -1
    assert lib.mgemm_wgrad(a, 1, x, s, w, s, o, 64, 128, 256, 4, 64, None) == -1           # fp8 ld < colwise_ld
    assert lib.mgemm_wgrad(a, 1, x, s, w, s, o, 64, 128, 256, 4, 648, None) == -2          # fp8 ld % 16
    assert lib.mgemm_wgrad(a, 0, x, None, w, None, None, 64, 128, 256, 4, 0, None) == -1
    dw = lib.mgemm_dgrad_wgrad
    g, gx, gw = P(0x60000), P(0x70000), P(0x80000)
    assert dw(None, g, w, x, gx, gw, 64, 128, 256, 4, None) == -1                           # no args block
    assert dw(a, g, None, x, gx, gw, 64, 128, 256, 4, None) == -1                           # no weights
    assert dw(a, g, w, x, None, gw, 64, 128, 256, 4, None) == -1                            # no grad_x
    assert dw(a, g, w, x, gx, P(0x80008), 64, 128, 256, 4, None) == -2                      # grad_w alignment
    assert dw(a, g, w, x, gx, gw, 64, 130, 256, 4, None) == -2                              # K % 8
    assert dw(a, g, w, x, gx, gw, 64, 128, 256, 2000, None) == -3                           # too many experts
    assert dw(a, None, w, None, None, None, 0, 128, 256, 4, None) == -1                     # M = 0: grad_w needed
    sp = lib.mgemm_dgrad_wgrad_split
    assert sp(64, 128, 256, 0) == -1 and sp(-1, 128, 256, 4) == -1 and sp(64, 128, 256, 2000) == -3
    f = lib.mgemm_fwd_scatter
    m = P(0x60000)
    assert f(a, 1, 1, x, w, o, m, 64, None, 64, 128, 256, 4, None) == -5                  # fp8: not provided
    assert f(a, 0, 1, x, w, o, None, 64, None, 64, 128, 256, 4, None) == -1               # no row map
    assert f(a, 0, 1, x, w, o, P(0x60002), 64, None, 64, 128, 256, 4, None) == -2         # row map alignment
    assert f(a, 0, 1, x, w, o, m, -1, None, 64, 128, 256, 4, None) == -1                  # map_limit < 0
    assert lib.mgemm_fwd_gated(a, x, w, o, 64, 128, 100, 4, 0, None) == -2               # F % 8
    assert lib.mgemm_fwd_gated(a, x, w, o, 64, 128, 0, 4, 0, None) == -1                 # F < 1
    assert lib.mgemm_fwd_gated(a, x, w, o, 64, 128, 64, 4, -1, None) == -1               # group_rows_max < 0


def test_host_checks_quant(lib):
    i, o, s = P(0x10000), P(0x20000), P(0x30000)
    assert lib.mgemm_quant_rowwise(i, 4, 12, 12, o, 16, s, None) == -1                    # C % 8
    assert lib.mgemm_quant_rowwise(i, 4, 16, 16, o, 24, s, None) == -2                    # ld_out % 16
    assert lib.mgemm_quant_rowwise(i, 0, 16, 16, o, 16, s, None) == 0                     # empty: no launch
    assert lib.mgemm_quant_colwise_grouped(None, 4, 64, i, 64, o, s, None, 0, None, None, 640, None) == -1
    assert lib.mgemm_quant_colwise_grouped(i, 4, 64, i, 60, o, s, None, 0, None, None, 640, None) == -1  # C % 8
    assert lib.mgemm_quant_colwise_grouped(i, 4, 64, i, 64, o, s, None, 0, None, None, 512, None) == -1  # ld small
    assert lib.mgemm_quant_colwise_grouped(i, 4, 64, i, 64, o, s, None, 0, None, None, 648, None) == -2  # ld % 16


def test_host_checks_mx(lib):
    i, o, s, a = P(0x10000), P(0x20000), P(0x30000), P(0x40000)
    q = lib.mgemm_quant_mx
    assert q(i, 4, 48, 48, o, 48, s, 16, None) == -1           # C % 32
    assert q(i, 4, 64, 64, o, 64, s, 8, None) == -2            # ld_sf % 16
    assert q(i, 4, 64, 64, o, 64, s, 0, None) == -1            # ld_sf < C / 32
    assert q(i, 0, 64, 64, o, 64, s, 16, None) == 0            # empty: no launch
    assert q(P(0x10008), 4, 64, 64, o, 64, s, 16, None) == -2  # input alignment
    f = lib.mgemm_fwd_mx
    assert f(a, i, s, i, s, 16, o, 64, 192, 256, 4, None) == -1     # K % 128
    assert f(a, i, s, i, s, 16, o, 64, 1024, 256, 4, None) == -1    # ld_sf < K / 32
    assert f(a, i, s, i, s, 24, o, 64, 512, 256, 4, None) == -2     # ld_sf % 16
    assert f(a, i, s, i, s, 16, o, 64, 512, 252, 4, None) == -1     # N % 8
    assert f(a, i, s, i, s, 16, o, 64, 512, 256, 1025, None) == -3  # E
    assert f(a, None, s, i, s, 16, o, 64, 512, 256, 4, None) == -1  # no x
    assert f(a, i, s, i, s, 16, o, 0, 512, 256, 4, None) == 0       # M = 0: nothing to do
    c = lib.mgemm_quant_colwise_mx
    assert c(a, 4, 64, i, 60, o, s, None, 0, None, None, 640, None) == -1   # C % 8
    assert c(a, 4, 64, i, 64, o, s, None, 0, None, None, 512, None) == -1   # ld < colwise_ld
    assert c(a, 4, 64, i, 64, o, s, None, 0, None, None, 656, None) == -2   # ld % 128
    assert c(a, 0, 64, i, 64, o, s, None, 0, None, None, 640, None) == -1   # E < 1
    wg = lib.mgemm_wgrad_mx
    assert wg(a, i, s, i, s, o, 64, 120, 256, 4, 640, None) == -1           # K % 16
    assert wg(a, i, s, i, s, o, 64, 128, 256, 4, 512, None) == -1           # ld < colwise_ld
    assert wg(a, i, s, i, s, o, 64, 128, 256, 4, 656, None) == -2           # ld % 128
    assert wg(a, None, s, i, s, o, 64, 128, 256, 4, 640, None) == -1        # no x


def test_host_checks_moe_align(lib):
    # rejected on the host before any CUDA call, so these run without a GPU
    p = ctypes.c_void_p(0x10000)
    f = lib.mgemm_moe_align
    assert f(p, 12, 0, 4, p, p, p, None, p, None) == -1          # E < 1
    assert f(p, 12, 1025, 4, p, p, p, None, p, None) == -3       # E > MGEMM_MAX_EXPERTS
    assert f(p, 12, 4, 0, p, p, p, None, p, None) == -1          # block_size < 1
    assert f(p, -1, 4, 4, p, p, p, None, p, None) == -1          # numel < 0
    assert f(p, (1 << 31) - 10, 4, 4, p, p, p, None, p, None) == -1  # numel + E (block - 1) >= 2^31
    assert f(None, 12, 4, 4, p, p, p, None, p, None) == -1       # no topk_ids
    assert f(p, 12, 4, 4, None, p, p, None, p, None) == -1       # no sorted_ids
    assert f(p, 12, 4, 4, p, p, p, None, ctypes.c_void_p(0x10008), None) == -2  # workspace not 16-aligned
    assert f(p, 12, 4, 4, p, p, p, ctypes.c_void_p(0x10004), p, None) == -2      # group_sizes not 8-aligned
    ws = lib.mgemm_moe_align_workspace_bytes
    assert ws(0, 4) == 16 and ws(2048, 4) == 16 and ws(2049, 64) == 2 * 64 * 4 and ws(10, 0) == -1


def test_host_checks_topk_softmax(lib):
    p = ctypes.c_void_p(0x10000)
    f = lib.mgemm_topk_softmax
    assert f(p, 4, 0, 1, 0, p, p, None) == -1      # E < 1
    assert f(p, 4, 1025, 1, 0, p, p, None) == -1   # E > MGEMM_MAX_EXPERTS
    assert f(p, 4, 8, 9, 0, p, p, None) == -1      # top_k > E
    assert f(p, 4, 8, 0, 0, p, p, None) == -1      # top_k < 1
    assert f(None, 4, 8, 2, 0, p, p, None) == -1   # no logits
    assert f(ctypes.c_void_p(0x10002), 4, 8, 2, 0, p, p, None) == -2  # misaligned
    assert f(None, 0, 8, 2, 0, None, None, None) == 0   # no tokens: nothing to do


def test_host_checks_moe_route_align(lib):
    p = ctypes.c_void_p(0x10000)
    f = lib.mgemm_moe_route_align
    # (gating, T, E, top_k, renormalize, block, weights, ids, sorted, experts, npp, sizes, args, stream)
    assert f(p, 4, 0, 1, 0, 128, p, p, p, p, p, None, p, None) == -1          # E < 1
    assert f(p, 4, 1025, 1, 0, 128, p, p, p, p, p, None, p, None) == -3       # E > MGEMM_MAX_EXPERTS
    assert f(p, 4, 8, 9, 0, 128, p, p, p, p, p, None, p, None) == -1         # top_k > E with logits
    assert f(p, 4, 8, 0, 0, 128, p, p, p, p, p, None, p, None) == -1         # top_k < 1
    assert f(p, 4, 8, 2, 0, 0, p, p, p, p, p, None, p, None) == -1           # block_size < 1
    assert f(p, 4, 8, 2, 0, 4097, p, p, p, p, p, None, p, None) == -1        # block_size > 4096
    assert f(p, -1, 8, 2, 0, 128, p, p, p, p, p, None, p, None) == -1        # T < 0
    assert f(p, 2049, 8, 2, 0, 128, p, p, p, p, p, None, p, None) == -1      # T * top_k > 4096 entries
    assert f(p, 4097, 8, 1, 0, 128, p, p, p, p, p, None, p, None) == -1      # T > 4096
    assert f(p, 4, 8, 2, 0, 128, None, p, p, p, p, None, p, None) == -1      # logits without weights
    assert f(p, 4, 8, 2, 0, 128, p, p, p, p, p, None, None, None) == -1      # no args block
    assert f(None, 4, 8, 2, 0, 128, None, None, p, p, p, None, p, None) == -1  # no ids
    assert f(p, 4, 8, 2, 0, 128, p, p, p, p, p, None, ctypes.c_void_p(0x10008), None) == -2  # args not 16-aligned
    assert f(p, 4, 8, 2, 0, 128, p, p, p, p, p, ctypes.c_void_p(0x10004), p, None) == -2     # sizes not 8-aligned
    # given ids (no logits): top_k may exceed E
    assert f(None, 4, 2, 3, 0, 128, None, p, p, p, p, None, ctypes.c_void_p(0x10008), None) == -2


def test_host_checks_fwd_gated_gather(lib):
    p = ctypes.c_void_p(0x10000)
    f = lib.mgemm_fwd_gated_gather
    # (args, x, x_rows, sorted_ids, numel, top_k, w, out, M, K, F, E, group_rows_max, stream)
    assert f(p, p, 4, None, 8, 2, p, p, 512, 256, 64, 8, 8, None) == -1     # no sorted ids
    assert f(p, p, 0, p, 8, 2, p, p, 512, 256, 64, 8, 8, None) == -1        # no token rows
    assert f(p, p, 4, p, 8, 0, p, p, 512, 256, 64, 8, 8, None) == -1        # top_k < 1
    assert f(p, p, 4, ctypes.c_void_p(0x10002), 8, 2, p, p, 512, 256, 64, 8, 8, None) == -2  # ids misaligned
    assert f(p, p, 4, p, 8, 2, p, p, 512, 256, 60, 8, 8, None) == -2        # F % 8 != 0
    assert f(p, p, 4, p, 80, 2, p, p, 512, 256, 64, 8, 33, None) == -5      # more than 32 rows per group
    assert f(p, p, 4, p, 8, 2, p, p, 512, 256, 64, 8, 0, None) == -5        # no bound on the rows


def test_colwise_ld_bounds_the_padded_layout():
    # M rows in at most min(M, E) non-empty groups, each padded by fewer than
    # MGEMM_COL_PAD rows, rounded up to MGEMM_COL_PAD
    from mixture_experts_grouped_gmm_gb300 import binding as B

    pad = B.MGEMM_COL_PAD
    for M, E in ((64, 4), (0, 4), (1, 1), (1, 128), (98304, 64), (1000, 1024), (5, 3)):
        want = -(-(M + (pad - 1) * min(M, E)) // pad) * pad
        assert B.mgemm_colwise_ld(M, E) == want, (M, E)
        # enough for the worst split: min(M, E) groups of one row each, the rest in one group
        g = min(M, E)
        worst = (g - 1) * pad + (-(-(M - g + 1) // pad) * pad if M else 0) if g else 0
        assert B.mgemm_colwise_ld(M, E) >= worst
    assert B.mgemm_colwise_ld(-1, 4) == -1 and B.mgemm_colwise_ld(10, 0) == -1 and B.mgemm_colwise_ld(10, 1025) == -1


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "mixture_experts_grouped_gmm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f
                assert "oracle/" not in src, f


def test_mx_scale_row_bytes():
    # C / 32 scale bytes per row, rounded up to a multiple of 16 (the TMA stride rule)
    from mixture_experts_grouped_gmm_gb300 import binding as B

    for C, want in ((32, 16), (512, 16), (544, 32), (1408, 48), (2048, 64), (5120, 160), (96, 16)):
        assert B.mx_ld_sf(C) == want, C
        assert B.mx_ld_sf(C) >= C // 32 and B.mx_ld_sf(C) % 16 == 0


def test_library_exports_only_the_c_abi():
    # Only the C ABI (mgemm_*) is exported: C++ template instantiations and their
    # function-local statics stay local, so two builds of the library in one
    # process (the wait-probe test build and the product) share no symbol.
    import shutil
    import subprocess

    from mixture_experts_grouped_gmm_gb300 import binding as B

    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm (binutils) not available")
    out = subprocess.run([nm, "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    names = [ln.split()[-1] for ln in out.splitlines() if ln.strip()]
    assert names and all(n.startswith("mgemm_") for n in names), [n for n in names if not n.startswith("mgemm_")]
