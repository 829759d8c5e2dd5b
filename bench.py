#!/usr/bin/env python3
"""Benchmark of the MoE grouped-GEMM hot path on GB300.

Headline (one JSON line on stdout, rank 0): the GRIN-MoE-shaped bf16
``gmm(x, w, group_sizes)`` forward + backward step of "Support GPU-resident
batch sizes" (tgale96/grouped_gemm PR #21): M=1024, K=4096, N=6400, E=8,
group sizes [128]*8 on the device, x and w from U[0, 1), loss = out.sum() so
grad_out = 1.  One step = mgemm_fill_args + mgemm_fwd + mgemm_dgrad_wgrad
(both gradients in one launch; 161.1 GFLOP).  metric = TFLOP/s of the whole
job.

The same line carries: per-kernel times and roofline fractions measured with
CUDA events inside the timed region, SM clocks sampled during it, an
end-to-end number through the public ``gmm`` op with host-resident inputs
copied every step, the CPU oracle timed on a bounded sample, and secondary
measurements: p50 latency of the sparse-M FP8 forward (E=128, K=5120,
N=8192), the DeepSeek-MoE-16B-shaped FP8 training step (quantize kernels as
GB/s against HBM) and the Mixtral-shaped bf16 up/down projections.

``--impl reference`` times the CPU oracle instead (the reference arm).
Multi-GPU: one process per GPU, independent replicas (the path needs no
exchange), weak scaling, max time over ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

GRIN = dict(M=1024, K=4096, N=6400, E=8)
FLOP_GEMM = 2 * GRIN["M"] * GRIN["K"] * GRIN["N"]
FLOP_STEP = 3 * FLOP_GEMM
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CONFIG = {"workload": "GRIN-MoE gmm fwd+bwd bf16", "M": 1024, "K": 4096, "N": 6400, "E": 8,
          "group_sizes": "[128]*8 (int64, on device)", "inputs": "x, w ~ U[0,1) bf16, seed 0; grad_out = 1",
          "l2": "inputs larger than L2 (w 419 MB, grad_w 419 MB per step)", "parallelism": "replicas"}


# The pages' own figures for this path, quoted with their hardware (context,
# not targets: none was measured on this GPU).
PAGES_CONTEXT = [
    {"what": "total kernel time of 30 GRIN-MoE gmm fwd+bwd iterations (M=1024, K=4096, N=6400, E=8, bf16): "
             "batch sizes on the host (a device-to-host roundtrip per call) vs on the device",
     "value": "68 ms -> 60 ms (with device sizes about 2.0 ms, 80 TFLOP/s per iteration)",
     "hardware": "A100",
     "source": "Support GPU-resident batch sizes (tgale96/grouped_gemm PR #21), timing table"},
    {"what": "latency of the FP8 x INT4 grouped GEMM at total_M = 1 with 128 groups, with problems set up for "
             "min(total_M, groups) groups instead of all groups",
     "value": "about 3x lower",
     "hardware": "not stated",
     "source": "F8I4 Grouped Gemm Optimization for Sparse M (FBGEMM PR #3854), Summary"},
]


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-extras", action="store_true", help="headline step only")
    p.add_argument("--workload", choices=["all", "sparse", "deepseek", "mxfp8", "mixtral", "decode"], default="all",
                   help="'all': headline line with every block; otherwise run only that block (profiling)")
    p.add_argument("--tokens", type=int, default=16384,
                   help="DeepSeek-shaped block: tokens (x top-6 rows); decode block: tokens of the batch")
    p.add_argument("--experts", type=int, default=128, help="sparse-M block: number of experts")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i",
                 str(self.index), "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 6]
        if not rows:
            return None
        mhz = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": float(rows[0][1]), "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- our arm
class Step:
    """The GRIN step through the C ABI; with events given, one is recorded
    before every launch and one after the last."""

    def __init__(self, torch, B, dev):
        from mixture_experts_grouped_gmm_gb300 import workloads

        self.torch, self.B = torch, B
        d = workloads.grin(device=dev)
        M, K, N, E = d["M"], d["K"], d["N"], d["E"]
        self.d, self.M, self.K, self.N, self.E = d, M, K, N, E
        bf = torch.bfloat16
        self.args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=dev)
        self.out = torch.empty(M, N, dtype=bf, device=dev)
        self.gx = torch.empty(M, K, dtype=bf, device=dev)
        self.gw = torch.empty(E, K, N, dtype=bf, device=dev)
        self.go = torch.ones(M, N, dtype=bf, device=dev)

    def fill_args(self):
        self.B.mgemm_fill_args(self.d["group_sizes"], self.E, self.M, self.args)

    def fwd(self):
        B, d = self.B, self.d
        B.mgemm_fwd(self.args, B.MGEMM_BF16, 0, d["x"], None, d["w"], None, self.out, self.M, self.K, self.N, self.E)

    def dgrad(self):
        B, d = self.B, self.d
        B.mgemm_dgrad(self.args, B.MGEMM_BF16, self.go, None, d["w"], None, self.gx, self.M, self.K, self.N, self.E)

    def wgrad(self):
        B, d = self.B, self.d
        B.mgemm_wgrad(self.args, B.MGEMM_BF16, d["x"], None, self.go, None, self.gw, self.M, self.K, self.N, self.E)

    def dgrad_wgrad(self):
        B, d = self.B, self.d
        B.mgemm_dgrad_wgrad(self.args, self.go, d["w"], d["x"], self.gx, self.gw, self.M, self.K, self.N, self.E)

    def run(self):
        self.fill_args()
        self.fwd()
        self.dgrad_wgrad()


def time_events(torch, fn, reps, scrub=None):
    """p50 / mean of fn() over reps, each timed with events on the current stream;
    an optional L2 scrub runs (untimed) before every rep."""
    ts = []
    for _ in range(reps):
        if scrub is not None:
            scrub.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    ts.sort()
    return {"p50_us": ts[len(ts) // 2], "p10_us": ts[len(ts) // 10], "p90_us": ts[(9 * len(ts)) // 10],
            "mean_us": sum(ts) / len(ts)}


def time_back_to_back(torch, ops, reps):
    """Average time in us of each (name, fn) of ops: fn launched reps times back
    to back between two events on the current stream (no event, and so no host
    gap, between two launches of the same kernel)."""
    t = {}
    for n, fn in ops:
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record()
        for _ in range(reps):
            fn()
        k1.record()
        torch.cuda.synchronize()
        t[n] = k0.elapsed_time(k1) * 1e3 / reps
    return t


def sparse_m_extra(torch, B, dev, pk, E=128, reps=100):
    from mixture_experts_grouped_gmm_gb300 import workloads

    K, N = 5120, 8192
    w = workloads.sparse_m(1, E=E, K=K, N=N, device=dev)["w_nk"]
    wq = torch.empty(E * N, K, dtype=torch.uint8, device=dev)
    sw = torch.empty(E * N, dtype=torch.float32, device=dev)
    B.mgemm_quant_rowwise(w.view(E * N, K), wq, sw)
    # the same weights as INT4 blocks (the F8I4 path)
    wp = torch.empty(E, N, K // 2, dtype=torch.uint8, device=dev)
    wsf = torch.empty(B.int4_scale_bytes(E, N, K), dtype=torch.uint8, device=dev)
    B.mgemm_quant_int4(w, wp, wsf)
    del w
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {"shape": f"E={E} K=5120 N=8192 fp8 e4m3, rowwise scales; cold L2 (256 MB scrub between reps); "
                    f"{reps} reps, each timed alone (the event clock ticks every ~2 us: the mean resolves finer); "
                    "f8i4: the same weights as INT4 blocks of 32 with e8m0 scales (mgemm_quant_int4), "
                    "x rowwise FP8 (mgemm_fwd_f8i4)",
           "points": []}
    for tm in (1, 2, 4, 16, 64, 256):
        d = workloads.sparse_m(tm, E=E, K=K, N=N, device=dev, with_weights=False)
        gs = d["group_sizes"]
        n_touched = int((gs > 0).sum())
        args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=dev)
        xq = torch.empty(tm, K, dtype=torch.uint8, device=dev)
        sx = torch.empty(tm, dtype=torch.float32, device=dev)
        out = torch.empty(tm, N, dtype=torch.bfloat16, device=dev)

        def full():
            B.mgemm_fill_args(gs, E, tm, args)
            B.mgemm_quant_rowwise(d["x"], xq, sx)
            B.mgemm_fwd(args, B.MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, tm, K, N, E)

        full()

        def fwd_only():
            B.mgemm_fwd(args, B.MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, tm, K, N, E)

        def fused_full():  # fill and token cast in one launch, then the forward
            B.mgemm_fill_args_quant_rowwise(gs, E, tm, args, d["x"], xq, sx)
            B.mgemm_fwd(args, B.MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, tm, K, N, E)

        def f8i4_full():
            B.mgemm_fill_args_quant_rowwise(gs, E, tm, args, d["x"], xq, sx)
            B.mgemm_fwd_f8i4(args, xq, sx, wp, wsf, out, tm, K, N, E)

        def f8i4_only():
            B.mgemm_fwd_f8i4(args, xq, sx, wp, wsf, out, tm, K, N, E)

        t_full = time_events(torch, full, reps, scrub)
        t_fwd = time_events(torch, fwd_only, reps, scrub)
        t_one = None
        if tm <= B.SPARSE_MAX_ROWS:  # scan + token cast + forward in one launch
            def one_launch():
                B.mgemm_fwd_fp8_sparse(gs, E, d["x"], wq, sw, out, st)

            one_launch()
            t_one = time_events(torch, one_launch, reps, scrub)
        fused_full()
        t_fused = time_events(torch, fused_full, reps, scrub)
        f8i4_full()
        t_i4_full = time_events(torch, f8i4_full, reps, scrub)
        t_i4 = time_events(torch, f8i4_only, reps, scrub)
        byts = n_touched * K * N + n_touched * N * 4 + tm * (K + 4 + 2 * N)
        byts_i4 = n_touched * K * N // 2 + n_touched * N * K // 32 + tm * (K + 4 + 2 * N)
        res["points"].append({"total_M": tm, "experts_touched": n_touched,
                              "p50_us_fill_quant_fwd": round(t_full["p50_us"], 2),
                              "p50_us_fwd": round(t_fwd["p50_us"], 2),
                              "p50_us_fused_fill_quant_then_fwd": round(t_fused["p50_us"], 2),
                              "p50_us_single_launch": round(t_one["p50_us"], 2) if t_one else None,
                              "mean_us_single_launch": round(t_one["mean_us"], 2) if t_one else None,
                              "mean_us_fused_fill_quant_then_fwd": round(t_fused["mean_us"], 2),
                              "fwd_hbm_frac": round(byts / (t_fwd["p50_us"] * 1e-6) / 1e9 / pk["hbm_gbs"], 3),
                              "f8i4": {"p50_us_fused_fill_quant_then_fwd": round(t_i4_full["p50_us"], 2),
                                       "p50_us_fwd": round(t_i4["p50_us"], 2),
                                       "fwd_hbm_frac": round(byts_i4 / (t_i4["p50_us"] * 1e-6) / 1e9 / pk["hbm_gbs"],
                                                             3),
                                       "fwd_vs_fp8": round(t_i4["p50_us"] / t_fwd["p50_us"], 3)}})
    # flat in E: one token, E experts (a prefix of the same weights)
    sweep = []
    d = workloads.sparse_m(1, E=8, K=K, N=N, device=dev, with_weights=False)
    for Ee in [e for e in (8, 16, 32, 64, 128) if e <= E]:
        gs = torch.zeros(Ee, dtype=torch.int64, device=dev)
        gs[Ee // 2] = 1
        args = torch.empty(B.mgemm_args_bytes(Ee), dtype=torch.uint8, device=dev)
        xq = torch.empty(1, K, dtype=torch.uint8, device=dev)
        sx = torch.empty(1, dtype=torch.float32, device=dev)
        out = torch.empty(1, N, dtype=torch.bfloat16, device=dev)

        def full():
            B.mgemm_fill_args(gs, Ee, 1, args)
            B.mgemm_quant_rowwise(d["x"], xq, sx)
            B.mgemm_fwd(args, B.MGEMM_FP8_E4M3, 1, xq, sx, wq, sw, out, 1, K, N, Ee)

        full()

        def one_launch():
            B.mgemm_fwd_fp8_sparse(gs, Ee, d["x"], wq, sw, out, st)

        one_launch()
        t3, t1 = time_events(torch, full, reps, scrub), time_events(torch, one_launch, reps, scrub)
        sweep.append({"E": Ee, "p50_us_fill_quant_fwd": round(t3["p50_us"], 2),
                      "p50_us_single_launch": round(t1["p50_us"], 2), "mean_us_single_launch": round(t1["mean_us"], 2)})
    res["E_sweep_total_M_1"] = sweep
    del wq, wp, wsf, scrub
    return res


def deepseek_extra(torch, B, dev, pk, tokens=16384, reps=10, hidden=2048, ffn=1408, down_proj=False):
    """The DeepSeek-shaped FP8 step on the up projection (K = hidden 2048 -> N = ffn 1408), or
    with down_proj on the down projection (K = ffn 1408 -> N = hidden 2048), same routing."""
    from mixture_experts_grouped_gmm_gb300 import workloads

    d = workloads.deepseek(device=dev, T=tokens, H=ffn if down_proj else hidden, F=hidden if down_proj else ffn)
    M, K, N, E = d["M"], d["K"], d["N"], d["E"]
    u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
    w_kn = d["w"]   # the master weights [E, K, N]: both FP8 weight operands are cast from it in the step
    ld = B.mgemm_colwise_ld(M, E)  # padded column-major FP8 layout of the colwise outputs
    # the forward operand (one scale per (e, n) over K): the per-group colwise cast of w viewed
    # [E K, N] with E groups of K rows, read in place by the strided forward
    ldw = B.mgemm_colwise_ld(E * K, E)
    Kp = -(-K // 128) * 128
    wargs = torch.empty(B.mgemm_args_bytes(E), dtype=u8, device=dev)
    B.mgemm_fill_args(torch.full((E,), K, dtype=torch.int64, device=dev), E, E * K, wargs)  # constant: once
    T = dict(args=torch.empty(B.mgemm_args_bytes(E), dtype=u8, device=dev),
             xq=torch.empty(M, K, dtype=u8, device=dev), sx=torch.empty(M, dtype=f32, device=dev),
             goq=torch.empty(M, N, dtype=u8, device=dev), sgo=torch.empty(M, dtype=f32, device=dev),
             wq=torch.empty(N * ldw, dtype=u8, device=dev), sw=torch.empty(E * N, dtype=f32, device=dev),
             wdq=torch.empty(E * K, N, dtype=u8, device=dev), swd=torch.empty(E * K, dtype=f32, device=dev),
             xqt=torch.empty(K * ld, dtype=u8, device=dev), sxc=torch.empty(E * K, dtype=f32, device=dev),
             goqt=torch.empty(N * ld, dtype=u8, device=dev), sgoc=torch.empty(E * N, dtype=f32, device=dev),
             out=torch.empty(M, N, dtype=bf, device=dev), gx=torch.empty(M, K, dtype=bf, device=dev),
             gw=torch.empty(E, K, N, dtype=bf, device=dev))
    x, go = d["x"], d["grad_out"]
    ops = [
        ("fill", lambda: B.mgemm_fill_args(d["group_sizes"], E, M, T["args"])),
        ("quant_w", lambda: (B.mgemm_quant_colwise_grouped(wargs, E, E * K, w_kn.view(E * K, N), T["wq"], T["sw"],
                                                           ld=ldw),
                             B.mgemm_quant_rowwise(w_kn.view(E * K, N), T["wdq"], T["swd"]))),
        ("quant_x_rowwise", lambda: B.mgemm_quant_rowwise(x, T["xq"], T["sx"])),
        ("fwd", lambda: B.mgemm_fwd_fp8_strided(T["args"], T["xq"], T["sx"], T["wq"], ldw, Kp, T["sw"], T["out"], M,
                                                K, N, E)),
        ("quant_go_rowwise", lambda: B.mgemm_quant_rowwise(go, T["goq"], T["sgo"])),
        ("colwise_dual", lambda: B.mgemm_quant_colwise_grouped(T["args"], E, M, go, T["goqt"], T["sgoc"], x, T["xqt"],
                                                               T["sxc"])),
        ("dgrad", lambda: B.mgemm_dgrad(T["args"], 1, T["goq"], T["sgo"], T["wdq"], T["swd"], T["gx"], M, K, N, E)),
        ("wgrad", lambda: B.mgemm_wgrad(T["args"], 1, T["xqt"], T["sxc"], T["goqt"], T["sgoc"], T["gw"], M, K, N, E)),
    ]
    names = [n for n, _ in ops]

    def step():
        for _, fn in ops:
            fn()

    for _ in range(min(3, reps)):
        step()
    torch.cuda.synchronize()
    t = time_back_to_back(torch, ops, reps)
    # the whole step, back to back with no event between launches
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for r in range(reps):
        step()
    s1.record()
    torch.cuda.synchronize()
    step_us = s0.elapsed_time(s1) * 1e3 / reps
    fl = 2 * M * K * N
    fp8_peak = 2 * pk["bf16_tflops"]
    byts = {"quant_w": 2 * (E * N * K * 3 + E * N * 4), "quant_x_rowwise": M * K * 3 + M * 4,
            "quant_go_rowwise": M * N * 3 + M * 4, "colwise_dual": M * (K + N) * 3 + E * (K + N) * 4}
    kern = {}
    for n in names:
        k = {"us": round(t[n], 2)}
        if n in ("fwd", "dgrad", "wgrad"):
            k["tflops"] = round(fl / (t[n] * 1e-6) / 1e12, 1)
            k["tensor_frac_fp8"] = round(fl / (t[n] * 1e-6) / 1e12 / fp8_peak, 3)
        if n in byts:
            gbs = byts[n] / (t[n] * 1e-6) / 1e9
            k["gbs"] = round(gbs, 1)
            k["hbm_frac"] = round(gbs / pk["hbm_gbs"], 3)
        kern[n] = k
    total = sum(t.values())
    out = {"shape": f"M={M} (16384 tokens x top-6, Zipf 1.2, {int((d['group_sizes'] == 0).sum())} empty groups) "
                    f"K={K} N={N} E={E} ({'down' if down_proj else 'up'} projection), e4m3 operands, bf16 outputs; both weight casts run in the timed step from "
                    "the one bf16 master w [E, K, N] (forward operand: per-group colwise cast of w viewed [E K, N], "
                    "read in place by mgemm_fwd_fp8_strided; dgrad operand: rowwise cast); the weight groups' args "
                    "block (E groups of K rows, constant) is filled once outside it",
           "kernels_timing": "each kernel launched reps times back to back between two events",
           "step_us": round(step_us, 1), "sum_of_kernels_us": round(total, 1), "gemm_tflops": round(3 * fl / (sum(t[n] for n in ('fwd', 'dgrad', 'wgrad'))
                                                                    * 1e-6) / 1e12, 1),
           "fp8_peak_tflops": round(fp8_peak, 1), "kernels": kern}
    del T, d, wargs
    return out


def deepseek_mx_extra(torch, B, dev, pk, tokens=16384, reps=10):
    """MXFP8 on the DeepSeek shapes: the block casts (one e8m0 scale per 32
    contraction elements) of x, grad_out and both weight layouts, and the
    block-scaled fwd and dgrad GEMMs."""
    from mixture_experts_grouped_gmm_gb300 import workloads

    d = workloads.deepseek(device=dev, T=tokens)
    M, K, N, E = d["M"], d["K"], d["N"], d["E"]
    u8, bf = torch.uint8, torch.bfloat16
    w_kn = d["w"]
    w_nk = w_kn.transpose(1, 2).contiguous()
    x, go = d["x"], d["grad_out"]
    lk, ln = B.mx_ld_sf(K), B.mx_ld_sf(N)
    T = dict(args=torch.empty(B.mgemm_args_bytes(E), dtype=u8, device=dev),
             xq=torch.empty(M, K, dtype=u8, device=dev), sx=torch.empty(M, lk, dtype=u8, device=dev),
             goq=torch.empty(M, N, dtype=u8, device=dev), sgo=torch.empty(M, ln, dtype=u8, device=dev),
             wq=torch.empty(E * N, K, dtype=u8, device=dev), sw=torch.empty(E * N, lk, dtype=u8, device=dev),
             wdq=torch.empty(E * K, N, dtype=u8, device=dev), swd=torch.empty(E * K, ln, dtype=u8, device=dev),
             out=torch.empty(M, N, dtype=bf, device=dev), gx=torch.empty(M, K, dtype=bf, device=dev))
    ld = B.mgemm_colwise_ld(M, E)  # padded column-major layout of the wgrad operands
    T.update(xqt=torch.empty(K * ld, dtype=u8, device=dev), sxc=torch.empty(ld // 128 * K * 4, dtype=u8, device=dev),
             gqt=torch.empty(N * ld, dtype=u8, device=dev), sgc=torch.empty(ld // 128 * N * 4, dtype=u8, device=dev),
             gw=torch.empty(E, K, N, dtype=bf, device=dev))
    ops = [
        ("fill", lambda: B.mgemm_fill_args(d["group_sizes"], E, M, T["args"])),
        ("quant_w", lambda: (B.mgemm_quant_mx(w_nk.view(E * N, K), T["wq"], T["sw"]),
                             B.mgemm_quant_mx(w_kn.view(E * K, N), T["wdq"], T["swd"]))),
        ("quant_x", lambda: B.mgemm_quant_mx(x, T["xq"], T["sx"])),
        ("fwd", lambda: B.mgemm_fwd_mx(T["args"], T["xq"], T["sx"], T["wq"].view(E, N, K), T["sw"], T["out"], M, K,
                                       N, E)),
        ("quant_go", lambda: B.mgemm_quant_mx(go, T["goq"], T["sgo"])),
        ("dgrad", lambda: B.mgemm_fwd_mx(T["args"], T["goq"], T["sgo"], T["wdq"].view(E, K, N), T["swd"], T["gx"], M,
                                         N, K, E)),
        ("colwise_dual", lambda: B.mgemm_quant_colwise_mx(T["args"], E, M, go, T["gqt"], T["sgc"], x, T["xqt"],
                                                          T["sxc"], ld)),
        ("wgrad", lambda: B.mgemm_wgrad_mx(T["args"], T["xqt"], T["sxc"], T["gqt"], T["sgc"], T["gw"], M, K, N, E,
                                           ld)),
    ]
    names = [n for n, _ in ops if n != "fill"]

    def step():
        for _, fn in ops:
            fn()

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    t = time_back_to_back(torch, ops, reps)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for r in range(reps):
        step()
    s1.record()
    torch.cuda.synchronize()
    step_us = s0.elapsed_time(s1) * 1e3 / reps
    fl = 2 * M * K * N
    fp8_peak = 2 * pk["bf16_tflops"]
    byts = {"quant_w": 2 * E * N * K * 3 + E * (N * lk + K * ln), "quant_x": M * K * 3 + M * lk,
            "quant_go": M * N * 3 + M * ln, "colwise_dual": M * (K + N) * 3 + M // 32 * (K + N)}
    kern = {}
    for n in names:
        k = {"us": round(t[n], 2)}
        if n in ("fwd", "dgrad", "wgrad"):
            k["tflops"] = round(fl / (t[n] * 1e-6) / 1e12, 1)
            k["tensor_frac_fp8"] = round(fl / (t[n] * 1e-6) / 1e12 / fp8_peak, 3)
        if n in byts:
            gbs = byts[n] / (t[n] * 1e-6) / 1e9
            k["gbs"] = round(gbs, 1)
            k["hbm_frac"] = round(gbs / pk["hbm_gbs"], 3)
        kern[n] = k
    out = {"shape": f"M={M} K={K} N={N} E={E} (the DeepSeek step's routing), e4m3 codes, one e8m0 scale per "
                    "32 contraction elements, bf16 outputs; the forward's bf16 weight copy in the [E, N, K] layout "
                    "is made once outside the timed step (both block casts of the weights are timed in it)",
           "step_us": round(step_us, 1), "gemm_tflops": round(3 * fl / (sum(t[n] for n in ("fwd", "dgrad", "wgrad"))
                                                                    * 1e-6) / 1e12, 1),
           "fp8_peak_tflops": round(fp8_peak, 1), "kernels": kern}
    del T, d, w_nk
    return out


def mixtral_extra(torch, B, dev, pk):
    from mixture_experts_grouped_gmm_gb300 import workloads

    d = workloads.mixtral(device=dev)
    M, H, F, E = d["M"], d["H"], d["F"], d["E"]
    args = torch.empty(B.mgemm_args_bytes(E), dtype=torch.uint8, device=dev)
    B.mgemm_fill_args(d["group_sizes"], E, M, args)
    up = torch.empty(M, 2 * F, dtype=torch.bfloat16, device=dev)
    h = torch.randn(M, F, device=dev).to(torch.bfloat16)
    down = torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    t_up = time_events(torch, lambda: B.mgemm_fwd(args, 0, 0, d["x"], None, d["w1"], None, up, M, H, 2 * F, E), 10)
    t_dn = time_events(torch, lambda: B.mgemm_fwd(args, 0, 0, h, None, d["w2"], None, down, M, F, H, E), 10)
    real = int(d["counts"].sum())
    f_up, f_dn = 2 * M * H * 2 * F, 2 * M * F * H
    res = {"shape": f"T=4096 top-2, E=8, padded M={M} ({real} routed rows), up [4096 -> 28672], down [14336 -> 4096]"}
    for n, t, f in (("up", t_up, f_up), ("down", t_dn, f_dn)):
        tf = f / (t["p50_us"] * 1e-6) / 1e12
        res[n] = {"p50_us": round(t["p50_us"], 1), "tflops_padded_rows": round(tf, 1),
                  "tensor_frac": round(tf / pk["bf16_tflops"], 3),
                  "tflops_routed_rows": round(tf * real / M, 1)}
    res["routed_layer"] = routed_layer(torch, B, dev, pk, d)
    del d
    return res


def routed_layer(torch, B, dev, pk, d):
    """The routed layer (moe.fused_experts: device alignment, gather, up GEMM
    with silu_and_mul in its epilogue, down GEMM with routed weights scattered to
    the entries, top-k sum) on the same routing and weights (viewed in the [E, N, K] layout of
    fused_moe; the values do not affect the time)."""
    from mixture_experts_grouped_gmm_gb300 import moe

    T, H, F, E = d["T"], d["H"], d["F"], d["E"]
    w1 = d["w1"].view(E, 2 * F, H)
    w2 = d["w2"].view(E, H, F)
    g = torch.Generator(device=dev).manual_seed(1)
    x = torch.randn(T, H, generator=g, device=dev).to(torch.bfloat16)
    tw = d["topk_weights"].to(dev)
    tid = d["topk_ids"].to(dev).to(torch.int32)
    t = time_events(torch, lambda: moe.fused_experts(x, w1, w2, tw, tid), 10)
    routed = T * tid.shape[1]
    flop = 2 * routed * H * 2 * F + 2 * routed * F * H
    tf = flop / (t["p50_us"] * 1e-6) / 1e12
    res = {"what": "moe.fused_experts(x, w1, w2, topk_weights, topk_ids), all steps on the device",
           "p50_us": round(t["p50_us"], 1), "tflops_routed_rows": round(tf, 1),
           "tensor_frac_routed": round(tf / pk["bf16_tflops"], 3)}
    res["decode_graph"] = decode_layer(torch, dev, pk, d, g)
    return res


def decode_layer(torch, dev, pk, d, g, sizes=(1, 4, 16, 64)):
    """Decode-size batches of the whole layer from gating logits (routing
    included), replayed from a CUDA graph: the weights of the touched experts
    against HBM."""
    from mixture_experts_grouped_gmm_gb300 import moe

    H, F, E = d["H"], d["F"], d["E"]
    w1 = d["w1"].view(E, 2 * F, H)
    w2 = d["w2"].view(E, H, F)
    dec = []
    for Td in sizes:
        xd = torch.randn(Td, H, generator=g, device=dev).to(torch.bfloat16)
        gd = torch.randn(Td, E, generator=g, device=dev)
        f = lambda: moe.fused_moe(xd, w1, w2, gd, 2, True)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                f()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            f()
        td = time_events(torch, graph.replay, 20)
        # ten layers back to back in one graph: the steady rate of a decode loop
        # (a replay timed alone also holds the graph's launch from the host)
        graph10 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph10):
            for _ in range(10):
                f()
        graph10.replay()
        t10 = time_events(torch, graph10.replay, 10)
        _, tidd = moe.route(gd, 2, True)
        touched = int((torch.bincount(tidd.view(-1).long(), minlength=E) > 0).sum())
        wb = touched * 3 * F * H * 2
        b2b = t10["mean_us"] / 10
        dec.append({"tokens": Td, "experts_touched": touched, "p50_us": round(td["p50_us"], 1),
                    "hbm_frac": round(wb / (td["p50_us"] * 1e-6) / 1e9 / pk["hbm_gbs"], 3),
                    "us_per_layer_back_to_back": round(b2b, 1),
                    "hbm_frac_back_to_back": round(wb / (b2b * 1e-6) / 1e9 / pk["hbm_gbs"], 3)})
        del graph, graph10
    return dec


def cpu_baseline_grin(seconds=10.0):
    """The oracle (numpy float64) on one expert's group of the GRIN step."""
    import numpy as np
    import torch

    from mixture_experts_grouped_gmm_gb300 import workloads
    from oracle import gmm as og

    d = workloads.grin(device="cpu")
    K, N = d["K"], d["N"]
    rows = 128
    x = d["x"][:rows].double().numpy()
    w = d["w"][:1].double().numpy()
    go = np.ones((rows, N))
    sizes = [rows]
    t0 = time.perf_counter()
    n = 0
    while True:
        og.gmm_fwd(x, w, sizes)
        og.gmm_dgrad(go, w, sizes)
        og.gmm_wgrad(x, go, sizes)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    flops = n * 3 * 2 * rows * K * N
    del torch
    return {"value": round(flops / dt / 1e12, 5), "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"{n} x (fwd+dgrad+wgrad) of one 128-row expert group (1/8 of the step), float64 numpy",
            "seconds": round(dt, 2)}


def _time_cpu(fn, min_seconds):
    """Run fn until min_seconds have passed (at least once); seconds per call and calls."""
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            return dt / n, n


def cpu_baselines(seconds=3.0):
    """The oracle (numpy float64, as it stands) on each workload, on the host
    cores: in full where it finishes in seconds, else on a row sample whose
    time is also extrapolated to the full workload by FLOP count (labelled)."""
    import numpy as np
    import torch

    from mixture_experts_grouped_gmm_gb300 import workloads
    from oracle import args as oa
    from oracle import gmm as og
    from oracle import quant as oq
    from oracle import routing as orr

    cores = host_cores()
    res = []
    bf = torch.bfloat16

    def npy(t):
        return t.double().numpy()

    # tiny bf16: the whole step (fill, fwd, dgrad, wgrad)
    d = workloads.tiny(device="cpu")
    x, w, sizes = npy(d["x"]), npy(d["w"]), d["group_sizes"].tolist()
    go = np.ones((d["M"], d["N"]))
    fl = 3 * 2 * d["M"] * d["K"] * d["N"]

    def tiny_step():
        oa.fill_args(sizes, d["M"])
        og.gmm_fwd(x, w, sizes), og.gmm_dgrad(go, w, sizes), og.gmm_wgrad(x, go, sizes)

    dt, n = _time_cpu(tiny_step, seconds / 3)
    res.append({"config": "tiny bf16 gmm fwd+dgrad+wgrad (E=4, M=64, K=128, N=256)", "kind": "oracle",
                "cores": cores, "sample": "the whole step", "calls": n, "us_per_step": round(dt * 1e6, 1),
                "value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s"})

    # GRIN: one expert's 128-row group of the step (1/8 of its work)
    g = cpu_baseline_grin(seconds)
    g = dict(g, config="GRIN-MoE gmm fwd+bwd bf16 (M=1024, K=4096, N=6400, E=8)",
             extrapolated_full_step_ms=round(8 * 3 * 2 * 128 * 4096 * 6400 / (g["value"] * 1e12) * 1e3, 1))
    res.append(g)

    # sparse-M FP8: fill + rowwise cast of the tokens + forward over the touched experts, in full
    K, N, E = 5120, 8192, 128
    for tm in (1,):
        d = workloads.sparse_m(tm, E=E, K=K, N=N, with_weights=False)
        sizes = d["group_sizes"].tolist()
        touched = [e for e in range(E) if sizes[e] > 0]
        gen = torch.Generator().manual_seed(tm)
        wt = (torch.randn(len(touched), N, K, generator=gen) * 0.02).to(bf).double().numpy()
        qs = [oq.quant_rowwise(wt[i]) for i in range(len(touched))]
        wq, sw = np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])
        del wt, qs
        xs = npy(d["x"])
        sub = [sizes[e] for e in touched]       # the touched experts' groups, in expert order

        def sparse_step():
            oa.fill_args(sizes, tm)
            xq, sx = oq.quant_rowwise(xs)
            og.gmm_fwd_fp8(xq, sx, wq, sw, sub)

        dt, n = _time_cpu(sparse_step, seconds / 2)
        res.append({"config": f"sparse-M FP8 fwd (E=128, K=5120, N=8192), total_M={tm}", "kind": "oracle",
                    "cores": cores, "calls": n,
                    "sample": f"the whole call: fill, rowwise cast of {tm} token rows, forward over the "
                              f"{len(touched)} touched experts (weights pre-quantized, as on the GPU)",
                    "value": round(dt * 1e6, 1), "unit": "us (latency)"})
        del wq, sw

    # Mixtral bf16: 128 routed rows of one expert through up, silu_and_mul and down
    H, F = 4096, 14336
    gen = torch.Generator().manual_seed(4)
    rows = 128
    xs = (torch.randn(rows, H, generator=gen)).to(bf).double().numpy()
    w1 = (torch.randn(1, H, 2 * F, generator=gen) * 0.02).to(bf).double().numpy()
    w2 = (torch.randn(1, F, H, generator=gen) * 0.02).to(bf).double().numpy()

    def mix_step():
        up = og.gmm_fwd(xs, w1, [rows])
        og.gmm_fwd(orr.silu_and_mul(up), w2, [rows])

    dt, n = _time_cpu(mix_step, seconds / 2)
    del w1, w2
    fl = 2 * rows * H * 2 * F + 2 * rows * F * H
    routed = 4096 * 2
    res.append({"config": "Mixtral-shaped routed layer bf16 (T=4096, top-2, E=8, H=4096, F=14336)", "kind": "oracle",
                "cores": cores, "calls": n,
                "sample": "128 routed rows of one expert: up GEMM, silu_and_mul, down GEMM (row sample)",
                "sample_ms": round(dt * 1e3, 2), "value": round(fl / dt / 1e12, 5), "unit": "TFLOP/s",
                "extrapolated_full_ms": round(dt * routed / rows * 1e3, 1),
                "extrapolation": "by FLOP count to the 8192 routed rows"})

    # DeepSeek FP8 step: 512 rows of one expert group through every step of the FP8 training path
    Hd, Fd = 2048, 1408
    gen = torch.Generator().manual_seed(5)
    rows = 512
    xs = torch.randn(rows, Hd, generator=gen).to(bf).double().numpy()
    gos = torch.randn(rows, Fd, generator=gen).to(bf).double().numpy()
    wkn = (torch.randn(1, Hd, Fd, generator=gen) * 0.02).to(bf).double().numpy()
    offs = np.array([0, rows])

    def ds_step():
        wq, sw = oq.quant_rowwise(wkn[0].T)                   # forward weights, per (e, n) over K
        wdq, swd = oq.quant_rowwise(wkn[0])                   # dgrad weights, per (e, k) over N
        xq, sx = oq.quant_rowwise(xs)
        og.gmm_fwd_fp8(xq, sx, wq[None], sw, [rows])
        goq, sgo = oq.quant_rowwise(gos)
        (gqt, sgc), (xqt, sxc) = oq.quant_colwise_grouped_dual(gos, xs, offs)
        og.gmm_dgrad_fp8(goq, sgo, wdq[None], swd, [rows])
        og.gmm_wgrad_fp8(xqt, sxc, gqt, sgc, [rows])

    dt, n = _time_cpu(ds_step, seconds / 2)
    fl = 3 * 2 * rows * Hd * Fd
    res.append({"config": "DeepSeek-MoE-16B-shaped FP8 training step (98304 rows, K=2048, N=1408, E=64)",
                "kind": "oracle", "cores": cores, "calls": n,
                "sample": "512 rows of one expert group: the weight casts of both layouts, rowwise casts of x and "
                          "grad_out, the dual colwise cast, fwd, dgrad and wgrad (row sample)",
                "sample_ms": round(dt * 1e3, 2), "value": round(fl / dt / 1e12, 5), "unit": "TFLOP/s",
                "extrapolated_full_ms": round(dt * 98304 / rows * 1e3, 1),
                "extrapolation": "by row count to the 98304 routed rows (the weight casts, per expert, "
                                 "are over-counted by it)"})
    return res


def run_block(a):
    """One secondary block alone (used for profiling a workload's kernels)."""
    import torch

    from mixture_experts_grouped_gmm_gb300 import binding as B
    from mixture_experts_grouped_gmm_gb300 import build as _build

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    pk, _ = peaks()
    if a.workload == "sparse":
        out = sparse_m_extra(torch, B, dev, pk, E=a.experts, reps=max(1, a.steps))
    elif a.workload == "deepseek":
        out = deepseek_extra(torch, B, dev, pk, tokens=a.tokens, reps=max(1, a.steps))
    elif a.workload == "mxfp8":
        out = deepseek_mx_extra(torch, B, dev, pk, tokens=a.tokens, reps=max(1, a.steps))
    elif a.workload == "decode":
        from mixture_experts_grouped_gmm_gb300 import workloads

        d = workloads.mixtral(device=dev)
        out = decode_layer(torch, dev, pk, d, torch.Generator(device=dev).manual_seed(1), sizes=(a.tokens,))
    else:
        out = mixtral_extra(torch, B, dev, pk)
    print(json.dumps({"workload": a.workload, a.workload: out}), flush=True)


def run_ours(a):
    import torch
    import torch.distributed as dist

    from mixture_experts_grouped_gmm_gb300 import binding as B
    from mixture_experts_grouped_gmm_gb300 import build as _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0 or world == 1:
        _build.build()
    if world > 1:
        dist.barrier()
    B.lib()
    pk, pk_src = peaks()

    def barrier():
        if world > 1:
            dist.barrier()

    st = Step(torch, B, dev)
    for _ in range(a.warmup):
        st.run()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.15)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(a.steps):
        st.run()
    t_end.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    ms = max_over_ranks(t_start.elapsed_time(t_end) / a.steps, world, dist, dev)
    # status after the timed region (sync point outside timing)
    assert B.args_status(st.args) == 0
    # per-kernel times: each kernel of the step launched `steps` times back to
    # back between two events on the launching stream.  An event recorded
    # between two launches would break the programmatic overlap of launch
    # latency and charge the host's gap to the next kernel; here the launches
    # follow each other as in the step, so a kernel's average is its own time.
    # (dgrad and wgrad alone are not launches of the step: they show what the
    # one-launch backward saves)
    names = ["fill_args", "fwd", "dgrad_wgrad", "dgrad", "wgrad"]
    per = {}
    barrier()
    torch.cuda.synchronize()
    for n in names:
        fn = getattr(st, n)
        fn()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record()
        for i in range(a.steps):
            fn()
        k1.record()
        torch.cuda.synchronize()
        per[n] = k0.elapsed_time(k1) * 1e3 / a.steps
    assert B.args_status(st.args) == 0
    # the same step captured once in a CUDA graph and replayed: no call reads
    # anything on the host, so the replays run back to back
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph):
        st.run()
    for _ in range(3):
        step_graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(a.steps):
        step_graph.replay()
    g1.record()
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1) / a.steps, world, dist, dev)
    assert B.args_status(st.args) == 0
    del step_graph

    gemm_bytes = (GRIN["E"] * GRIN["K"] * GRIN["N"] + GRIN["M"] * GRIN["K"] + GRIN["M"] * GRIN["N"]) * 2
    alg_bytes = {"fill_args": 8 * 8 + 24 + 8 * 9 + 4 * (8 + 9 + 8), "fwd": gemm_bytes,
                 "dgrad_wgrad": 2 * gemm_bytes, "dgrad": gemm_bytes, "wgrad": gemm_bytes}
    flops = {"fwd": FLOP_GEMM, "dgrad_wgrad": 2 * FLOP_GEMM, "dgrad": FLOP_GEMM, "wgrad": FLOP_GEMM}
    kernels = {}
    for n in names:
        us = per[n]
        k = {"us": round(us, 2), "gbs": round(alg_bytes[n] / (us * 1e-6) / 1e9, 1)}
        if n != "fill_args":
            k["tflops"] = round(flops[n] / (us * 1e-6) / 1e12, 1)
            k["hbm_frac"] = round(k["gbs"] / pk["hbm_gbs"], 3)
            k["tensor_frac"] = round(k["tflops"] / pk["bf16_tflops_sustained"], 3)
        if n in ("dgrad", "wgrad"):
            k["in_step"] = False
        kernels[n] = k
    dom = max(("fwd", "dgrad_wgrad"), key=lambda n: per[n])
    achieved = alg_bytes[dom] / (per[dom] * 1e-6) / 1e9
    traffic, traffic_note = None, None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            from mixture_experts_grouped_gmm_gb300.build import gemm_source_hash

            tj = json.load(open(tpath))
            ent = tj.get(dom)
            if ent and ent.get("gemm_source_hash") == gemm_source_hash():
                traffic = ent.get("dram_bytes_per_launch")
                traffic_note = ent.get("note")
        except Exception:
            traffic = None
    value = job_tflops(world, FLOP_STEP, ms)

    line = {"metric": "grouped-GEMM TFLOP/s (GRIN-MoE gmm fwd+bwd)", "value": round(value, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": dict(CONFIG), "gpu_launches": 3 * a.steps,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                         "peak_source": pk_src, "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 3),
                         "traffic": traffic, "traffic_note": traffic_note, "alg_bytes_per_launch": alg_bytes[dom],
                         "kernel_choice": "the step's longest GEMM launch by its back-to-back average (the one-launch "
                                          "backward: dgrad and wgrad on disjoint CTAs; bytes of both)"},
            "kernels": kernels,
            "kernels_timing": "each kernel launched `steps` times back to back between two events on its stream",
            "pages_context": PAGES_CONTEXT,
            "clocks": clk,
            "graph": {"ms_per_step": round(graph_ms, 5), "value": round(job_tflops(world, FLOP_STEP, graph_ms), 2),
                      "unit": "TFLOP/s", "what": "the same step captured once in a CUDA graph, replayed"}}

    # end to end through the public op with host-resident inputs
    if rank == 0 or True:
        from mixture_experts_grouped_gmm_gb300 import gmm

        xh = st.d["x"].cpu().pin_memory()
        wh = st.d["w"].cpu().pin_memory()
        gh = st.d["group_sizes"].cpu().pin_memory()
        e2e_steps = max(3, min(a.steps, 50))

        # Each step's inputs are copied on a copy stream into one of two device
        # buffers while the previous step computes (a training loop's prefetch):
        # every timed step still copies its x, w and sizes from pinned memory and
        # reads its loss back.
        copy_stream = torch.cuda.Stream(device=dev)
        bufs = [tuple(torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (xh, wh, gh)) for _ in range(2)]
        landed = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        for ev in freed:
            ev.record()

        def prefetch(i):
            b = i % 2
            copy_stream.wait_event(freed[b])  # step i - 2 no longer reads the buffer
            with torch.cuda.stream(copy_stream):
                for dst, src in zip(bufs[b], (xh, wh, gh)):
                    dst.copy_(src, non_blocking=True)
            landed[b].record(copy_stream)

        def e2e_steps_from(i0, n):
            prefetch(i0)
            for i in range(i0, i0 + n):
                b = i % 2
                torch.cuda.current_stream().wait_event(landed[b])
                if i + 1 < i0 + n:
                    prefetch(i + 1)
                xb, wb, gb = bufs[b]
                x = xb.detach().requires_grad_(True)
                w = wb.detach().requires_grad_(True)
                out = gmm(x, w, gb)
                loss = out.float().sum()
                loss.backward()
                freed[b].record()
                loss.item()

        e2e_steps_from(0, 2)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        e2e_steps_from(2, e2e_steps)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / e2e_steps, world, dist, dev)
        line["e2e"] = {"value": round(job_tflops(world, FLOP_STEP, e2e_ms), 2), "unit": "TFLOP/s",
                       "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                       "h2d_bytes_per_step": xh.numel() * 2 + wh.numel() * 2 + gh.numel() * 8,
                       "d2h_bytes_per_step": 4,
                       "path": "gmm(x, w, group_sizes) autograd op; pinned host x, w, sizes copied in every step "
                               "(on a copy stream, into two device buffers in turn, each copy overlapping the "
                               "previous step's compute); loss.item() read back every step"}
        del xh, wh

    if not a.no_extras:
        del st
        torch.cuda.empty_cache()
        line["sparse_m_fp8"] = sparse_m_extra(torch, B, dev, pk)
        torch.cuda.empty_cache()
        line["deepseek_fp8_step"] = deepseek_extra(torch, B, dev, pk)
        torch.cuda.empty_cache()
        line["deepseek_fp8_step_down_proj"] = deepseek_extra(torch, B, dev, pk, down_proj=True)
        torch.cuda.empty_cache()
        line["deepseek_mxfp8"] = deepseek_mx_extra(torch, B, dev, pk)
        torch.cuda.empty_cache()
        line["mixtral_bf16"] = mixtral_extra(torch, B, dev, pk)
    if rank == 0 and world == 1 and not a.no_cpu:
        cb = cpu_baseline_grin()
        cb["configs"] = cpu_baselines()
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def max_over_ranks(value, world, dist, device):
    """The largest of every rank's value (the job's time is its slowest
    rank's); the value itself with one rank."""
    if world <= 1:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flop_per_rank_step, ms_per_step):
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return world * flop_per_rank_step / (ms_per_step * 1e-3) / 1e12


def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    from mixture_experts_grouped_gmm_gb300 import workloads
    from oracle import gmm as og

    d = workloads.grin(device="cpu")
    K, N = d["K"], d["N"]
    xall = d["x"].double().numpy()
    w0 = d["w"][:1].double().numpy()

    def make(rows):
        x = xall[:rows]
        go = np.ones((rows, N))

        def step():
            og.gmm_fwd(x, w0, [rows])
            og.gmm_dgrad(go, w0, [rows])
            og.gmm_wgrad(x, go, [rows])
        return step

    rows = 128
    step = make(rows)
    t0 = time.perf_counter()
    step()
    t1 = time.perf_counter() - t0
    budget = 120.0 / max(1, a.steps + a.warmup)            # seconds per step
    if t1 > budget:
        rows = max(8, int(rows * budget / t1))
        step = make(rows)
    for _ in range(a.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        step()
    dt = (time.perf_counter() - t0) / a.steps
    flops = 3 * 2 * rows * K * N
    value = flops / dt / 1e12
    sample = f"per step: fwd+dgrad+wgrad of {rows} rows of one expert group (float64 numpy oracle)"
    line = {"impl": "reference", "metric": "grouped-GEMM TFLOP/s (GRIN-MoE gmm fwd+bwd)",
            "value": round(value, 5), "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", a.gpus)),
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": dict(CONFIG),
            "cpu_baseline": {"kind": "oracle", "cores": host_cores(), "sample": sample, "value": round(value, 5)},
            "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.workload != "all":
        run_block(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
