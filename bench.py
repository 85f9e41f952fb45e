"""Benchmark of the MoE expert layer on GB300.

One step = one pass of the whole hot path over one batch: route + sort,
permute, grouped GEMM gate_up with fused SwiGLU, grouped GEMM down, weighted
combine (FP8 workloads add the activation quantiser and use the quantising
epilogue).  --gather folds the permute into the gate_up GEMM.  Default
workload: the 32-expert top-4 layer (T=4096, H=I=2880, bf16, biased routing).
Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

--impl reference times the CPU oracle (a deliberately plain program) on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; grouped-GEMM TFLOP/s as % of GB300 tensor peak"
DEFAULT_WORKLOAD = "32e-top4-h2880"
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="measure the headline workload only (skip the other workloads' record)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels one by one instead of replaying a CUDA graph")
    ap.add_argument("--grad", action="store_true",
                    help="time the grouped GEMMs' gradients (dgrad, wgrad) instead of the forward step")
    ap.add_argument("--gather", action="store_true",
                    help="gather the gate_up GEMM's rows from token order inside the GEMM "
                         "(moe_forward's MOE_FWD_GATHER) instead of a separate permute")
    ap.add_argument("--fused-combine", action="store_true",
                    help="fold the weighted combine into the down GEMM (moe_forward's "
                         "MOE_FWD_FUSED_COMBINE; bf16 workloads)")
    ap.add_argument("--ncu", action="store_true",
                    help="profiler mode: W warm-up steps then K steps, nothing else (no clock "
                         "pre-roll, end-to-end pass or CPU baseline), so launches can be counted")
    ap.add_argument("--experts", type=int, default=0,
                    help="shrink the workload to this many experts, tokens scaled alike "
                         "(same rows per expert; for small profiler captures)")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def write_peak(torch):
    """Write-only HBM bandwidth measured here: a 1 GiB fill of a float32 buffer
    (4-byte stores; torch's fills of 1- and 2-byte elements stop near half of
    this), timed with CUDA events, median of 10 after 3 warm-up runs."""
    buf = torch.empty((1 << 30) // 4, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        buf.zero_()
    ts = []
    for _ in range(10):
        e0.record()
        buf.zero_()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    del buf
    return (1 << 30) / (statistics.median(ts) * 1e-3) / 1e9


def route_kernels(T: int, E: int, k: int) -> int:
    """Kernels moe_route_sort launches: two, or one for a small batch -- a
    single sort block (T*k <= 1024) with at most four (tokens per warp) x
    (logits per lane) of routing work, the library's rule."""
    nv = 1 if E <= 32 else 2 if E <= 64 else 4 if E <= 128 else 8
    return 1 if T * k <= 1024 and -(-T // 32) * nv <= 4 else 2


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, v in enumerate(flags) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ ranks
def flush_l2(buf, i):
    """Evict L2 between timed steps: write a buffer larger than L2, then read
    it back, so that L2 is left holding clean lines and the next step does not
    pay for writing the flush's dirty lines back to HBM."""
    buf.fill_(i & 0xFF)
    buf.max()


def cross_rank_max(value: float, dist, device) -> float:
    """The largest per-rank value (the slowest rank's time); identity on one rank."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of independent replicas: every rank's tokens over
    the slowest rank's step time."""
    return tokens_per_rank * world / (ms_max * 1e-3)


# ------------------------------------------------------------------ inputs
def make_layer(wl, torch, moe, synth):
    """Seeded synthetic layer resident on the device (weights drawn on the host
    expert by expert, copied once; FP8 weights quantised by the library)."""
    t0 = time.time()
    dev = torch.device("cuda")

    def bf16_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    L = {}
    L["x_host"] = synth.hidden_states(wl)
    L["logits_host"] = synth.router_logits(wl)
    bias = synth.expert_bias(wl)
    L["bias_host"] = bias
    L["x"] = bf16_dev(L["x_host"])
    L["logits"] = torch.from_numpy(L["logits_host"]).to(dev)
    L["bias"] = None if bias is None else torch.from_numpy(bias).to(dev)
    mask = synth.sentinel_mask(wl)
    L["mask"] = None if mask is None else torch.from_numpy(mask).to(dev)
    fp8 = wl.dtype == "fp8"
    for which, (n, kdim) in (("w1", (2 * wl.I, wl.H)), ("w2", (wl.H, wl.I))):
        if not fp8:
            L[which] = bf16_dev(synth.expert_weights(wl, which))
            continue
        q = torch.empty((wl.E, n, kdim), dtype=torch.uint8, device=dev)
        s = torch.empty((wl.E, (n + 127) // 128, kdim // 128), dtype=torch.float32, device=dev)
        chunk = 16
        for e0 in range(0, wl.E, chunk):
            ex = list(range(e0, min(wl.E, e0 + chunk)))
            wb = bf16_dev(synth.expert_weights(wl, which, experts=ex))
            moe.moe_weight_quant_fp8(wb, len(ex), n, kdim, q[e0:e0 + len(ex)], s[e0:e0 + len(ex)])
            torch.cuda.synchronize()
            del wb
        L[which], L[which + "_s"] = q, s
    L["setup_s"] = time.time() - t0
    return L


class Step:
    """The hot path as the chain of C-ABI calls moe_forward enqueues, with
    CUDA events between kernels on the launching stream."""

    def __init__(self, wl, L, torch, moe, separate_scatter=True, fused_combine=False):
        self.wl, self.L, self.torch, self.moe = wl, L, torch, moe
        self.scatter = separate_scatter
        self.fused = fused_combine and wl.dtype != "fp8"
        T, E, k, H, I = wl.T, wl.E, wl.k, wl.H, wl.I
        R = T * k
        self.fp8 = wl.dtype == "fp8"
        dev = torch.device("cuda")
        z = lambda *s, dt=torch.uint8: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        self.ids, self.w = z(T, k, dt=torch.int32), z(T, k, dt=torch.float32)
        self.sr, self.rp, self.off = z(R, dt=torch.int32), z(R, dt=torch.int32), z(E + 1, dt=torch.int32)
        self.rws_bytes = moe.moe_route_sort_workspace_size(T, E, k)
        self.rws = z(max(self.rws_bytes, 16))
        if self.fp8:
            self.xq, self.xs = z(T, H), z(T, H // 128, dt=torch.float32)
            if self.scatter:
                self.xp, self.xps = z(R, H), z(H // 128, R, dt=torch.float32)
            self.h, self.hs = z(R, I), z(I // 128, R, dt=torch.float32)
        else:
            if self.scatter:
                self.xp = z(R, H, dt=torch.bfloat16)
            self.h = z(R, I, dt=torch.bfloat16)
        self.y2 = z(R, H, dt=torch.bfloat16)
        self.out = z(T, H, dt=torch.bfloat16)
        self.names = (["route_sort"] + (["act_quant"] if self.fp8 else []) +
                      (["permute"] if self.scatter else []) + ["gemm_gate_up_swiglu", "gemm_down"] +
                      ([] if self.fused else ["combine"]))
        if self.fused:
            self.cws_bytes = moe.moe_grouped_gemm_combine_workspace_size(T, H)
            self.cws = z(self.cws_bytes)
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(self.names) + 1)]
        self.times = {n: [] for n in self.names}

    def launches_per_step(self):
        return len(self.names) - 1 + route_kernels(self.wl.T, self.wl.E, self.wl.k)

    def run(self, record=False):
        wl, L, moe = self.wl, self.L, self.moe
        T, E, k, H, I = wl.T, wl.E, wl.k, wl.H, wl.I
        R = T * k
        ev = iter(self.ev)
        mark = (lambda: next(ev).record()) if record else (lambda: None)
        mark()
        moe.moe_route_sort(L["logits"], L["bias"], L["mask"], self.ids, self.w, T, E, k, wl.renormalize,
                           self.sr, self.rp, self.off, self.rws, self.rws_bytes)
        mark()
        if self.fp8:
            moe.moe_act_quant_fp8(L["x"], T, H, self.xq, self.xs)
            mark()
            if self.scatter:
                moe.moe_permute(moe.MOE_FP8_E4M3_B128, self.xq, self.xs, T, H, k, self.sr, self.off, E, R,
                                self.xp, self.xps)
                mark()
                moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, self.xp, self.xps, L["w1"], L["w1_s"], self.off, E,
                                     R, 2 * I, H, moe.MOE_EPI_SWIGLU_QUANT_FP8, self.h, self.hs)
            else:
                moe.moe_grouped_gemm_gather(moe.MOE_FP8_E4M3_B128, self.xq, self.xs, T, k, self.sr, L["w1"],
                                            L["w1_s"], self.off, E, R, 2 * I, H, moe.MOE_EPI_SWIGLU_QUANT_FP8,
                                            self.h, self.hs)
            mark()
            moe.moe_grouped_gemm(moe.MOE_FP8_E4M3_B128, self.h, self.hs, L["w2"], L["w2_s"], self.off, E, R,
                                 H, I, moe.MOE_EPI_STORE, self.y2, None)
        else:
            if self.scatter:
                moe.moe_permute(moe.MOE_BF16, L["x"], None, T, H, k, self.sr, self.off, E, R, self.xp, None)
                mark()
                moe.moe_grouped_gemm(moe.MOE_BF16, self.xp, None, L["w1"], None, self.off, E, R, 2 * I, H,
                                     moe.MOE_EPI_SWIGLU, self.h, None)
            else:
                moe.moe_grouped_gemm_gather(moe.MOE_BF16, L["x"], None, T, k, self.sr, L["w1"], None, self.off,
                                            E, R, 2 * I, H, moe.MOE_EPI_SWIGLU, self.h, None)
            mark()
            if self.fused:
                moe.moe_grouped_gemm_combine(self.h, L["w2"], self.off, E, R, H, I, self.ids, self.w, self.sr, self.rp,
                                             T, k, self.y2, self.out, self.cws, self.cws_bytes)
            else:
                moe.moe_grouped_gemm(moe.MOE_BF16, self.h, None, L["w2"], None, self.off, E, R, H, I,
                                     moe.MOE_EPI_STORE, self.y2, None)
        mark()
        if not self.fused:
            moe.moe_combine(self.y2, self.ids, self.w, self.rp, T, k, H, E, self.out)
            mark()

    def collect(self):
        for i, n in enumerate(self.names):
            self.times[n].append(self.ev[i].elapsed_time(self.ev[i + 1]))
        return self.ev[0].elapsed_time(self.ev[-1])


def flops_bytes(wl, live_rows, experts_live, separate_scatter=False):
    """Algorithmic work of one step: GEMM FLOPs on live rows and the minimum
    HBM bytes of each kernel (weights of experts with rows, with their block
    scales for FP8; activations once).  The gathered gate_up GEMM reads x
    itself: each token row once at least."""
    T, E, k, H, I = wl.T, wl.E, wl.k, wl.H, wl.I
    R = T * k
    fp8 = wl.dtype == "fp8"
    wb = 1 if fp8 else 2
    ab = 1 if fp8 else 2
    w1 = 2 * I * H * wb + (2 * I // 128) * (H // 128) * 4 * fp8
    w2 = H * I * wb + -(-H // 128) * (I // 128) * 4 * fp8
    sa = (H // 128) * 4 * fp8          # activation scales per row of x (FP8)
    sh = (I // 128) * 4 * fp8          # ... of h
    f1 = 2.0 * live_rows * (2 * I) * H
    f2 = 2.0 * live_rows * H * I
    b1 = (experts_live * w1 + (live_rows if separate_scatter else T) * (H * ab + sa)
          + live_rows * (I * ab + sh) + (R - live_rows) * (I * ab + sh))
    b2 = experts_live * w2 + live_rows * (I * ab + sh) + R * H * 2
    bp = T * (H * ab + sa) + live_rows * (H * ab + sa)
    bc = live_rows * H * 2 + R * 12 + T * H * 2
    bq = T * H * 2 + T * H + T * (H // 128) * 4
    br = T * E * 4 + R * 20
    # the part of each data-movement kernel's bytes that is written
    wr = dict(permute_bytes=live_rows * (H * ab + sa), combine_bytes=T * H * 2,
              act_quant_bytes=T * H + T * (H // 128) * 4, route_bytes=R * 20)
    return dict(gemm1_flop=f1, gemm2_flop=f2, gemm1_bytes=b1, gemm2_bytes=b2, permute_bytes=bp,
                combine_bytes=bc, act_quant_bytes=bq, route_bytes=br, written=wr)


def layer_summary(wl, step, step_ms, separate, pk):
    """Per-layer figures from the timed steps: step time and tokens/s, and per
    kernel its time with its fraction of the bound that applies -- the tensor
    peak (bf16, or 2 x bf16 for FP8) and the HBM copy bandwidth for the grouped
    GEMMs (and the larger of the two as the roofline), HBM for the data-movement
    kernels."""
    off = step.off.cpu().numpy()
    live = int(off[-1])
    experts_live = int((np.diff(off) > 0).sum())
    fb = flops_bytes(wl, live, experts_live, separate)
    kt = {n: statistics.fmean(v) for n, v in step.times.items()}
    fp8 = wl.dtype == "fp8"
    tpeak = pk["bf16_tflops"] * (2.0 if fp8 else 1.0)
    hbm = pk["hbm_gbs"]
    gemm = {}
    for name, key, fl, by in (("gate_up", "gemm_gate_up_swiglu", fb["gemm1_flop"], fb["gemm1_bytes"]),
                              ("down", "gemm_down", fb["gemm2_flop"], fb["gemm2_bytes"])):
        t = kt[key] * 1e-3
        gemm[name] = {"ms": kt[key], "tflops": fl / t / 1e12, "tensor_frac": fl / t / 1e12 / tpeak,
                      "hbm_gbs": by / t / 1e9, "hbm_frac": by / t / 1e9 / hbm,
                      "roofline_frac": max(fl / (tpeak * 1e12), by / (hbm * 1e9)) / t,
                      "algorithmic_flop": fl, "algorithmic_bytes": by}
    # DRAM traffic per launch from an ncu capture of this workload, where
    # profiles/ holds one (null otherwise)
    tp = os.path.join(ROOT, "profiles", f"traffic_{wl.name}.json")
    if os.path.exists(tp) and separate:
        with open(tp) as f:
            tr = json.load(f)
        gemm["gate_up"]["traffic"] = tr.get("gemm_gate_up_swiglu_bytes")
        gemm["down"]["traffic"] = tr.get("gemm_down_bytes")
    data = {}
    for name, key in (("route_sort", "route_bytes"), ("act_quant", "act_quant_bytes"),
                      ("permute", "permute_bytes"), ("combine", "combine_bytes")):
        if name in kt:
            gbs = fb[key] / (kt[name] * 1e-3) / 1e9
            data[name] = {"ms": kt[name], "gbs": gbs, "hbm_frac": gbs / hbm, "algorithmic_bytes": fb[key]}
            if pk.get("write_gbs"):
                wgbs = fb["written"][key] / (kt[name] * 1e-3) / 1e9
                data[name].update({"written_bytes": fb["written"][key], "write_gbs": wgbs,
                                   "write_frac": wgbs / pk["write_gbs"]})
    ms = statistics.fmean(step_ms)
    return {"ms_per_step": ms, "tokens_per_s": wl.T / (ms * 1e-3), "live_rows": live,
            "experts_with_rows": experts_live, "kernels_ms": kt, "gemm": gemm, "data_movement": data,
            "peaks": {"tensor_tflops": tpeak, "hbm_gbs": hbm, "write_gbs": pk.get("write_gbs"),
                      "tensor_source": ("fp8 = 2 x " if fp8 else "") + "measured bf16 burst (cuBLAS)"},
            "_fb": fb}


# ------------------------------------------------------------------ CPU oracle
# multiply-adds of the oracle's budget for one timed sample: all-core and one core
CPU_MACS_ALL = 40e9
CPU_MACS_ONE = 3e9


def oracle_weights(wl, synth, used, chunk=16):
    """Host weights for the oracle: full [E, ...] stacks of which only the
    experts in `used` are drawn (the others are never written, and never read:
    the oracle runs only the experts its tokens pick).  FP8 weights are
    quantised by the oracle, chunk by chunk."""
    import oracle
    fp8 = wl.dtype == "fp8"
    out = []
    for which, (n, kdim) in (("w1", (2 * wl.I, wl.H)), ("w2", (wl.H, wl.I))):
        W = np.empty((wl.E, n, kdim), np.uint8 if fp8 else np.uint16)
        S = np.empty((wl.E, -(-n // 128), kdim // 128), np.float32) if fp8 else None
        for i in range(0, len(used), chunk):
            ex = np.asarray(used[i:i + chunk])
            bf = synth.expert_weights(wl, which, experts=ex)
            if fp8:
                W[ex], S[ex] = oracle.quant_weight_fp8(bf)
            else:
                W[ex] = bf
        out += [W, S]
    return out[0], out[2], out[1], out[3]


def oracle_layer_rate(wl, synth, n_one=None, n_all=None):
    """The oracle, as it stands, on the first tokens of the workload: one
    whole layer (route, sort, [quantise], permute, both GEMMs, combine) per
    call, timed on one core (one-core build) and on every host core (OpenMP
    build).  Sample sizes follow a fixed multiply-add budget unless given."""
    import oracle
    macs = wl.k * 3 * wl.H * wl.I
    n_all = n_all or int(min(wl.T, max(8, CPU_MACS_ALL // macs)))
    n_one = n_one or int(min(wl.T, max(2, CPU_MACS_ONE // macs)))
    if wl.dtype == "fp8":
        # the experts the sample picks are drawn and quantised first (about 80
        # of the 256-expert layer's for 12 tokens): that setup dominates
        n_all, n_one = min(n_all, 12), min(n_one, 4)
    n = max(n_all, n_one)
    x, logits, bias = synth.hidden_states(wl)[:n], synth.router_logits(wl)[:n], synth.expert_bias(wl)
    prev = oracle.use_openmp(True)
    try:
        ids, _ = oracle.route_topk(logits, bias, wl.k, wl.renormalize)
        W1, W2, s1, s2 = oracle_weights(wl, synth, np.unique(ids))
        res = {}
        for label, omp, m in (("all", True, n_all), ("one", False, n_one)):
            oracle.use_openmp(omp)
            reps, dt = 0, 0.0
            while dt < 0.5 or reps == 0:          # repeat a tiny sample to at least 0.5 s
                t0 = time.perf_counter()
                oracle.moe_forward(x[:m], W1, W2, E=wl.E, k=wl.k, logits=logits[:m], bias=bias,
                                   renormalize=wl.renormalize, W1_scales=s1, W2_scales=s2)
                dt += time.perf_counter() - t0
                reps += 1
            res[label] = (m * reps / dt, m, reps, dt, oracle.threads())
    finally:
        oracle.use_openmp(prev)
    return res


def cpu_baseline_record(wl, synth):
    cores, model = cpu_info()
    r = oracle_layer_rate(wl, synth)
    v, m, reps, dt, thr = r["all"]
    v1, m1, reps1, dt1, _ = r["one"]
    return {"value": v, "unit": "tokens/s", "cores": thr, "kind": "oracle",
            "sample": (f"first {m} of {wl.T} tokens of {wl.name}, x{reps} ({dt:.1f} s), "
                       f"OpenMP build over rows on {thr} threads"),
            "single_core": {"value": v1, "unit": "tokens/s", "cores": 1,
                            "sample": f"first {m1} tokens, x{reps1} ({dt1:.1f} s), one-core build"},
            "cpu": model, "host_cores": cores}


def cpu_info():
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return cores, model


def reference_main(args, wl, synth):
    """The reference arm: the CPU oracle, as it stands, on every host core
    (its OpenMP build), each step one layer over a bounded window of the
    workload's tokens."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    macs = wl.k * 3 * wl.H * wl.I
    per_step = int(max(1, min(wl.T, 4e9 // macs)))
    starts = [(i * per_step) % max(1, wl.T - per_step + 1) for i in range(args.warmup + args.steps)]
    x, logits, bias = synth.hidden_states(wl), synth.router_logits(wl), synth.expert_bias(wl)
    prev = oracle.use_openmp(True)
    try:
        ids, _ = oracle.route_topk(np.concatenate([logits[j:j + per_step] for j in starts]), bias, wl.k,
                                   wl.renormalize)
        W1, W2, s1, s2 = oracle_weights(wl, synth, np.unique(ids))
        threads = oracle.threads()

        def one(j):
            oracle.moe_forward(x[j:j + per_step], W1, W2, E=wl.E, k=wl.k, logits=logits[j:j + per_step],
                               bias=bias, renormalize=wl.renormalize, W1_scales=s1, W2_scales=s2)

        for j in starts[:args.warmup]:
            one(j)
        t0 = time.perf_counter()
        for j in starts[args.warmup:]:
            one(j)
        dt = time.perf_counter() - t0
    finally:
        oracle.use_openmp(prev)
    value = per_step * args.steps / dt
    cores, model = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy draws)",
        "config": {"workload": wl.name, "T": wl.T, "E": wl.E, "k": wl.k, "H": wl.H, "I": wl.I,
                   "layer_dtype": wl.dtype, "step": f"{per_step} tokens of the workload per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": (f"{per_step} tokens per step x {args.steps} steps of {wl.name}, "
                                    f"OpenMP build over rows on {threads} threads"),
                         "cpu": model, "host_cores": cores},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ sweep
SWEEP_NAME = "sweep-128e-h2048-i768-m16384"


def sweep_measure(steps, warmup, synth, torch, moe, pk):
    """Both grouped GEMMs over 16384 permuted rows of 128 experts (H=2048,
    I=768, bf16) with 100 / 50 / 12.5 % of the rows live: split equally over
    all experts, and concentrated on the first live/128 experts (128 rows
    each).  Sentinel rows are NaN on input; the GEMMs write them as zeros."""
    base = synth.Sweep()
    wl = base.workload

    def bf16_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)

    W1 = bf16_dev(synth.expert_weights(wl, "w1"))
    W2 = bf16_dev(synth.expert_weights(wl, "w2"))
    M, E, H, I = base.M_cap, base.E, base.H, base.I
    h = torch.empty((M, I), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    rows = []
    for live in (16384, 8192, 2048):
        sw = synth.Sweep(live=live)
        A = bf16_dev(synth.sweep_rows(sw))
        for layout in ("equal", "concentrated"):
            if layout == "equal":
                off_np = synth.sweep_offsets(sw)
            else:
                n_exp = live // 128
                off_np = np.minimum(np.arange(E + 1) * 128, live).astype(np.int32)
                assert off_np[n_exp] == live
            off = torch.from_numpy(off_np).cuda()

            def run():
                moe.moe_grouped_gemm(moe.MOE_BF16, A, None, W1, None, off, E, M, 2 * I, H, moe.MOE_EPI_SWIGLU,
                                     h, None)
                ev[1].record()
                moe.moe_grouped_gemm(moe.MOE_BF16, h, None, W2, None, off, E, M, H, I, moe.MOE_EPI_STORE, y2,
                                     None)

            for _ in range(max(3, warmup)):
                run()
            torch.cuda.synchronize()
            t1, t2 = [], []
            for i in range(steps):
                flush_l2(flush, i)
                ev[0].record()
                run()
                ev[2].record()
                torch.cuda.synchronize()
                t1.append(ev[0].elapsed_time(ev[1]))
                t2.append(ev[1].elapsed_time(ev[2]))
            if moe.moe_get_device_error() != 0:
                raise SystemExit("device error in sweep")
            g1, g2 = statistics.fmean(t1), statistics.fmean(t2)
            n_live_exp = int((np.diff(off_np) > 0).sum())
            flop = 2.0 * live * (2 * I * H + H * I)
            wbytes = n_live_exp * (2 * I * H + H * I) * 2
            abytes = live * (H + 2 * I) * 2 + M * H * 2
            t = (g1 + g2) * 1e-3
            rows.append({"live": live, "layout": layout, "experts_live": n_live_exp, "gate_up_ms": g1,
                         "down_ms": g2, "pair_ms": g1 + g2, "pair_tflops": flop / t / 1e12,
                         "tensor_frac": flop / t / 1e12 / pk["bf16_tflops"],
                         "pair_hbm_gbs": (wbytes + abytes) / t / 1e9,
                         "hbm_frac": (wbytes + abytes) / t / 1e9 / pk["hbm_gbs"],
                         "hbm_roofline_ms": (wbytes + abytes) / (pk["hbm_gbs"] * 1e9) * 1e3,
                         "tensor_roofline_ms": flop / (pk["bf16_tflops"] * 1e12) * 1e3})
    full = {r["layout"]: r["pair_ms"] for r in rows if r["live"] == 16384}
    for r in rows:
        r["time_vs_full"] = r["pair_ms"] / full[r["layout"]]
    del W1, W2, h, y2, flush
    torch.cuda.empty_cache()
    return rows


def sweep_cpu_baseline(synth):
    """The oracle's grouped GEMM pair (gate_up, silu * up, bf16 h, down) on
    sampled live rows of the 2048-live sweep: rows/s on every core (OpenMP
    build) and on one core."""
    import oracle
    sw = synth.Sweep(live=2048)
    wl = sw.workload
    A, off = synth.sweep_rows(sw), synth.sweep_offsets(sw)
    W1, W2 = synth.expert_weights(wl, "w1"), synth.expert_weights(wl, "w2")
    cores, model = cpu_info()
    res = {}
    prev = oracle.use_openmp(True)
    try:
        for label, omp, n in (("all", True, 2048), ("one", False, 128)):
            oracle.use_openmp(omp)
            rows = np.linspace(0, sw.live - 1, n).astype(np.int32)
            t0 = time.perf_counter()
            hb = np.zeros((sw.M_cap, sw.I), np.uint16)
            hb[rows] = oracle.bf16_round(oracle.swiglu(oracle.grouped_gemm_bf16(A, W1, off, rows=rows), n))
            oracle.grouped_gemm_bf16(hb, W2, off, rows=rows)
            dt = time.perf_counter() - t0
            res[label] = (n / dt, n, dt, oracle.threads())
    finally:
        oracle.use_openmp(prev)
    v, n, dt, thr = res["all"]
    v1, n1, dt1, _ = res["one"]
    return {"value": v, "unit": "rows/s", "cores": thr, "kind": "oracle",
            "sample": f"{n} of the 2048 live rows ({dt:.1f} s), OpenMP build over rows on {thr} threads",
            "single_core": {"value": v1, "unit": "rows/s", "cores": 1,
                            "sample": f"{n1} live rows ({dt1:.1f} s), one-core build"},
            "cpu": model, "host_cores": cores}


def sweep_main(args, synth, torch, moe):
    pk, pk_kind = peaks()
    rows = sweep_measure(args.steps, args.warmup, synth, torch, moe, pk)
    print(json.dumps({"metric": "grouped GEMM pair time vs live rows (sentinel sweep)", "unit": "ms",
                      "config": {"workload": SWEEP_NAME, "dtype": "bf16",
                                 "l2": "flushed between steps", "steps": args.steps},
                      "peaks": {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"], "kind": pk_kind},
                      "rows": rows}))
    return 0


# ------------------------------------------------------------------ gradients
def grad_main(args, wl, synth, torch, moe):
    """Forward, dgrad (dA = dC B[e]) and wgrad (dB[e] = dC_e^T A_e) of both
    grouped GEMMs of a bf16 layer, on the layer's own routing (the library's
    route + sort), random activations and output gradients; L2 flushed
    between timed calls.  Gradients cost the forward's FLOPs each."""
    if wl.dtype != "bf16":
        raise SystemExit("--grad: bf16 layers only")
    pk, pk_kind = peaks()
    dev = torch.device("cuda")
    T, E, k, H, I = wl.T, wl.E, wl.k, wl.H, wl.I
    R = T * k

    def bf16_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    r = moe.route_sort_t(E, k, logits=torch.from_numpy(synth.router_logits(wl)).to(dev),
                         expert_bias=None if synth.expert_bias(wl) is None else
                         torch.from_numpy(synth.expert_bias(wl)).to(dev), renormalize=wl.renormalize)
    off = r["offsets"]
    live = int(off[-1].item())
    g = torch.Generator(device="cuda").manual_seed(1)
    X = torch.randn((R, H), device=dev, generator=g).bfloat16()
    h = torch.randn((R, I), device=dev, generator=g).bfloat16()
    dY1 = torch.randn((R, 2 * I), device=dev, generator=g).bfloat16()
    dY2 = torch.randn((R, H), device=dev, generator=g).bfloat16()
    W1, W2 = bf16_dev(synth.expert_weights(wl, "w1")), bf16_dev(synth.expert_weights(wl, "w2"))
    out1 = torch.empty((R, 2 * I), dtype=torch.bfloat16, device=dev)
    out2 = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
    dX, dh = torch.empty_like(X), torch.empty_like(h)
    dW1, dW2 = torch.empty_like(W1), torch.empty_like(W2)
    ws_n = max(moe.moe_grouped_gemm_dgrad_workspace_size(E, 2 * I, H), moe.moe_grouped_gemm_dgrad_workspace_size(E, H, I),
               moe.moe_grouped_gemm_wgrad_workspace_size(E, R, 2 * I, H), moe.moe_grouped_gemm_wgrad_workspace_size(E, R, H, I))
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    ops = {
        "gate_up forward": lambda: moe.moe_grouped_gemm(moe.MOE_BF16, X, None, W1, None, off, E, R, 2 * I, H,
                                                        moe.MOE_EPI_STORE, out1, None),
        "gate_up dgrad": lambda: moe.moe_grouped_gemm_dgrad(dY1, W1, off, E, R, 2 * I, H, dX, ws, ws_n),
        "gate_up wgrad": lambda: moe.moe_grouped_gemm_wgrad(X, dY1, off, E, R, 2 * I, H, dW1, ws, ws_n),
        "down forward": lambda: moe.moe_grouped_gemm(moe.MOE_BF16, h, None, W2, None, off, E, R, H, I,
                                                     moe.MOE_EPI_STORE, out2, None),
        "down dgrad": lambda: moe.moe_grouped_gemm_dgrad(dY2, W2, off, E, R, H, I, dh, ws, ws_n),
        "down wgrad": lambda: moe.moe_grouped_gemm_wgrad(h, dY2, off, E, R, H, I, dW2, ws, ws_n),
    }
    flop = {"gate_up": 2.0 * live * 2 * I * H, "down": 2.0 * live * H * I}
    # wgrad writes the whole dB (E * N * K bf16): its write rate against the
    # write-only bandwidth measured here as a fill of the gate_up dB buffer
    # viewed as float32 (4-byte stores), timed like the ops
    out_bytes = {"gate_up": dW1.numel() * 2, "down": dW2.numel() * 2}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(f):
        for _ in range(max(3, args.warmup)):
            f()
        torch.cuda.synchronize()
        ts = []
        for i in range(args.steps):
            flush_l2(flush, i)
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.fmean(ts)

    write_gbs = out_bytes["gate_up"] / (timed(lambda: dW1.view(torch.float32).zero_()) * 1e-3) / 1e9
    rows = []
    for name, f in ops.items():
        ms = timed(f)
        tf = flop[name.split()[0]] / (ms * 1e-3) / 1e12
        row = {"op": name, "ms": ms, "tflops": tf, "frac": tf / pk["bf16_tflops"]}
        if name.endswith("wgrad"):
            wgbs = out_bytes[name.split()[0]] / (ms * 1e-3) / 1e9
            row.update({"out_bytes": out_bytes[name.split()[0]], "write_gbs": wgbs, "write_frac": wgbs / write_gbs})
        rows.append(row)
    if moe.moe_get_device_error() != 0:
        raise SystemExit("device error in the gradient bench")
    print(json.dumps({"metric": "grouped GEMM forward and gradients", "unit": "TFLOP/s",
                      "config": {"workload": wl.name, "live_rows": live, "l2": "flushed between timed calls",
                                 "steps": args.steps, "note": "dgrad reads the weights in place; wgrad reads the "
                                 "activations and output gradients in place and includes the copy of "
                                 "each expert's partial last 64 rows"},
                      "peak": {"bf16_tflops": pk["bf16_tflops"], "kind": pk_kind,
                               "write_gbs": write_gbs,
                               "write_kind": "float32 fill of the gate_up dB buffer, measured here"},
                      "rows": rows}))
    return 0


# ------------------------------------------------------------------ timing
def prepare_step(step, args, torch, moe):
    """W warm-up steps, then (unless --no-graph) the step's C-ABI calls
    captured once into a CUDA graph and replayed, as a serving loop would, so
    that host launch gaps between its short kernels stay out of the step time.
    Returns (run_step, graph or None)."""
    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    if moe.moe_get_device_error() != 0:
        raise SystemExit(f"device error during warm-up ({step.wl.name})")
    if args.no_graph:
        return step.run, None
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step.run()                        # one eager pass on the capture stream
        with torch.cuda.graph(graph, stream=side):
            step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    if moe.moe_get_device_error() != 0:
        raise SystemExit(f"device error in the captured step ({step.wl.name})")
    return graph.replay, graph


def timed_steps(run_step, step, flush, steps, torch):
    """K steps timed with CUDA events on the launching stream, L2 flushed
    (untimed) before each; then K eager steps with events between the kernels
    for the per-kernel durations.  Returns (step_ms, wall seconds of the
    first loop)."""
    step_ms = []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush_l2(flush, i)
        s0.record()
        run_step()
        s1.record()
        torch.cuda.synchronize()
        step_ms.append(s0.elapsed_time(s1))
    wall = time.perf_counter() - wall0
    for i in range(steps):
        flush_l2(flush, i)
        step.run(record=True)
        torch.cuda.synchronize()
        step.collect()
    return step_ms, wall


def preroll(run_step, torch, seconds):
    """Untimed steps so that the 200 ms clock samples see the GPU under this load."""
    t_pre = time.perf_counter()
    while time.perf_counter() - t_pre < seconds:
        run_step()
        torch.cuda.synchronize()


# the other workloads measured in the same run, beside the headline one
CONFIG_WORKLOADS = ("tiny-8e-top2", "128e-top8-h2048-zipf", "256e-top8-h7168-fp8")


def measure_config(wl, args, torch, moe, synth, pk, flush, device_index):
    """One more layer workload with the headline's protocol (graph replay, L2
    flushed between timed steps, per-kernel events), its CPU baseline beside
    it; its buffers are freed before returning."""
    L = make_layer(wl, torch, moe, synth)
    step = Step(wl, L, torch, moe)
    run_step, graph = prepare_step(step, args, torch, moe)
    with ClockSampler(device_index) as clk:
        preroll(run_step, torch, 0.3)
        step_ms, wall = timed_steps(run_step, step, flush, args.steps, torch)
    if moe.moe_get_device_error() != 0:
        raise SystemExit(f"device error in the timed steps of {wl.name}")
    rec = layer_summary(wl, step, step_ms, True, pk)
    rec.pop("_fb")
    rec["config"] = {"T": wl.T, "E": wl.E, "k": wl.k, "H": wl.H, "I": wl.I, "dtype": wl.dtype,
                     "bias": wl.bias, "sentinel_slots": wl.n_sentinel}
    rec["steps"] = args.steps
    rec["setup_s"] = L["setup_s"]
    rec["clocks"] = clk.summary()
    del graph, run_step, step, L
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline_record(wl, synth)
    return rec


# ------------------------------------------------------------------ main
def main():
    args = parse()
    from grouped_gemm_serving_gb300 import synth
    if args.workload == "sweep":
        import torch
        from grouped_gemm_serving_gb300 import build as gbuild
        gbuild.build()
        from grouped_gemm_serving_gb300 import moe
        return sweep_main(args, synth, torch, moe)
    if args.workload in synth.WORKLOADS:
        wl = synth.WORKLOADS[args.workload]
    else:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(synth.WORKLOADS)}")
    if args.experts:
        wl = wl.with_(name=f"{wl.name}-scaled-e{args.experts}", E=args.experts,
                      T=max(1, wl.T * args.experts // wl.E))
    if args.impl == "reference":
        return reference_main(args, wl, synth)

    import torch
    from grouped_gemm_serving_gb300 import build as gbuild
    gbuild.build()
    if args.grad:
        from grouped_gemm_serving_gb300 import moe
        return grad_main(args, wl, synth, torch, moe)
    from grouped_gemm_serving_gb300 import moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()

    L = make_layer(wl, torch, moe, synth)
    separate = not (args.gather and (wl.H * (1 if wl.dtype == "fp8" else 2)) % 128 == 0)
    step = Step(wl, L, torch, moe, separate_scatter=separate, fused_combine=args.fused_combine)
    if args.ncu:
        for _ in range(args.warmup + args.steps):
            step.run()
        torch.cuda.synchronize()
        err = moe.moe_get_device_error()
        print(json.dumps({"mode": "ncu", "workload": wl.name, "launches_per_step": step.launches_per_step(),
                          "steps": args.warmup + args.steps, "device_error": err}))
        return 1 if err else 0
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    run_step, graph = prepare_step(step, args, torch, moe)

    # ---- timed region: K steps, L2 flushed between steps (untimed)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        preroll(run_step, torch, 1.0)
        barrier()
        step_ms, wall = timed_steps(run_step, step, flush, args.steps, torch)
    torch.cuda.synchronize()
    barrier()
    if moe.moe_get_device_error() != 0:
        raise SystemExit("device error in the timed region")
    ms = statistics.fmean(step_ms)
    ms_max = cross_rank_max(ms, dist, "cuda")

    # ---- e2e: moe_forward with host buffers (pinned), copies inside the timed region
    x_pin = torch.from_numpy(L["x_host"].view(np.int16)).pin_memory()
    lg_pin = torch.from_numpy(L["logits_host"]).pin_memory()
    out_pin = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    fa_dtype = moe.MOE_FP8_E4M3_B128 if wl.dtype == "fp8" else moe.MOE_BF16
    fa = moe.forward_args(dtype=fa_dtype, T=wl.T, E=wl.E,
                          k=wl.k, H=wl.H, I=wl.I, x=x_pin, W1=L["w1"], W2=L["w2"], W1_scales=L.get("w1_s"),
                          W2_scales=L.get("w2_s"), out=out_pin, logits=lg_pin, expert_bias=L["bias"],
                          sentinel_mask=L["mask"],
                          renormalize=wl.renormalize, host_io=True, gather=not separate,
                          fused_combine=step.fused)
    nws = moe.moe_forward_workspace_size(fa)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        moe.moe_forward(fa, ws, nws)
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.steps):
        flush_l2(flush, i)
        e0.record()
        moe.moe_forward(fa, ws, nws)
        e1.record()
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_mean = statistics.fmean(e2e_ms)
    e2e_serial_max = cross_rank_max(e2e_mean, dist, "cuda")
    if moe.moe_get_device_error() != 0:
        raise SystemExit("device error in the e2e region")

    # ---- e2e, serving loop: a stream of batches from pinned host memory.
    # Each batch's input copy runs on one copy stream and its output read on
    # another, so they overlap the neighbouring batches' kernels (two device
    # staging buffers each way); moe_forward runs on the compute stream with
    # device pointers.  Every batch's copies lie inside the timed region, which
    # ends when the last batch's output has reached host memory.
    d_x = [torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda") for _ in range(2)]
    d_lg = [torch.empty((wl.T, wl.E), dtype=torch.float32, device="cuda") for _ in range(2)]
    d_out = [torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda") for _ in range(2)]
    outs_pin = [torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory() for _ in range(2)]
    fa_dev = [moe.forward_args(dtype=fa_dtype, T=wl.T, E=wl.E, k=wl.k, H=wl.H, I=wl.I, x=d_x[i],
                               W1=L["w1"], W2=L["w2"], W1_scales=L.get("w1_s"), W2_scales=L.get("w2_s"),
                               out=d_out[i], logits=d_lg[i], expert_bias=L["bias"], sentinel_mask=L["mask"],
                               renormalize=wl.renormalize,
                               gather=not separate, fused_combine=step.fused) for i in range(2)]
    s_comp, s_in, s_out = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in_ready", "in_free", "out_ready", "out_free")}
    # each staging slot's moe_forward call captured once, like the step above
    forward = [lambda i=i: moe.moe_forward(fa_dev[i], ws, nws) for i in range(2)]
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(s_comp)
        graphs = [torch.cuda.CUDAGraph() for _ in range(2)]
        with torch.cuda.stream(side):
            for i in range(2):
                moe.moe_forward(fa_dev[i], ws, nws)
                with torch.cuda.graph(graphs[i], stream=side):
                    moe.moe_forward(fa_dev[i], ws, nws)
        s_comp.wait_stream(side)
        torch.cuda.synchronize()
        forward = [g.replay for g in graphs]

    def serve(n_batches):
        s_in.wait_stream(s_comp)
        for b in range(n_batches):
            i = b & 1
            if b >= 2:
                s_in.wait_event(ev["in_free"][i])        # batch b-2 has finished with d_x[i]
            with torch.cuda.stream(s_in):
                d_x[i].copy_(x_pin, non_blocking=True)
                d_lg[i].copy_(lg_pin, non_blocking=True)
            ev["in_ready"][i].record(s_in)
            s_comp.wait_event(ev["in_ready"][i])
            if b >= 2:
                s_comp.wait_event(ev["out_free"][i])     # batch b-2's output has been read
            with torch.cuda.stream(s_comp):
                forward[i]()
            ev["in_free"][i].record(s_comp)
            ev["out_ready"][i].record(s_comp)
            s_out.wait_event(ev["out_ready"][i])
            with torch.cuda.stream(s_out):
                outs_pin[i].copy_(d_out[i], non_blocking=True)
            ev["out_free"][i].record(s_out)
        s_comp.wait_stream(s_out)

    serve(3)
    torch.cuda.synchronize()
    n_serve = max(args.steps, 8)
    e0.record(s_comp)
    serve(n_serve)
    e1.record(s_comp)
    torch.cuda.synchronize()
    e2e_max = cross_rank_max(e0.elapsed_time(e1) / n_serve, dist, "cuda")
    if moe.moe_get_device_error() != 0:
        raise SystemExit("device error in the serving loop")
    if not np.array_equal(outs_pin[(n_serve - 1) & 1].numpy(), out_pin.numpy()):
        raise SystemExit("serving-loop output differs from moe_forward with host buffers")

    # ---- e2e, serving loop through the C-ABI's host path: moe_forward with
    # MOE_FWD_HOST_IO | MOE_FWD_STAGED_OUT on pinned buffers, batches
    # alternating over two streams (a workspace and a set of pinned buffers
    # each), so that one batch's host copies (the library's side-stream copy of
    # x, the logits, the output's copy back) overlap its neighbour's kernels.
    # The timed region ends when both streams are done.
    h_x = [torch.from_numpy(L["x_host"].view(np.int16)).pin_memory() for _ in range(2)]
    h_lg = [torch.from_numpy(L["logits_host"]).pin_memory() for _ in range(2)]
    h_out = [torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory() for _ in range(2)]
    fa_h = [moe.forward_args(dtype=fa_dtype, T=wl.T, E=wl.E, k=wl.k, H=wl.H, I=wl.I, x=h_x[i], W1=L["w1"],
                             W2=L["w2"], W1_scales=L.get("w1_s"), W2_scales=L.get("w2_s"), out=h_out[i],
                             logits=h_lg[i], expert_bias=L["bias"], sentinel_mask=L["mask"],
                             renormalize=wl.renormalize, host_io=True, gather=not separate,
                             fused_combine=step.fused, staged_out=True) for i in range(2)]
    ws_h = [ws, torch.empty(nws, dtype=torch.uint8, device="cuda")]
    h_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    # eager calls: the library chains the kernels of successive host-I/O calls
    # (not under stream capture), so the two streams' kernels do not compete
    h_forward = [lambda i=i: moe.moe_forward(fa_h[i], ws_h[i], nws) for i in range(2)]

    def serve_capi(n_batches):
        for st in h_streams:
            st.wait_stream(s_comp)
        for b in range(n_batches):
            with torch.cuda.stream(h_streams[b & 1]):
                h_forward[b & 1]()
        for st in h_streams:
            s_comp.wait_stream(st)

    serve_capi(3)
    torch.cuda.synchronize()
    e0.record(s_comp)
    serve_capi(n_serve)
    e1.record(s_comp)
    torch.cuda.synchronize()
    e2e_capi_max = cross_rank_max(e0.elapsed_time(e1) / n_serve, dist, "cuda")
    if moe.moe_get_device_error() != 0:
        raise SystemExit("device error in the C-ABI serving loop")
    for i in range(2):
        if not np.array_equal(h_out[i].numpy(), out_pin.numpy()):
            raise SystemExit("C-ABI serving-loop output differs from moe_forward with host buffers")

    if rank != 0:
        dist.destroy_process_group()
        return 0

    # ---- roofline of the dominant kernel (the gate_up grouped GEMM)
    pk, pk_kind = peaks()
    pk = dict(pk, write_gbs=write_peak(torch))
    summ = layer_summary(wl, step, step_ms, separate, pk)
    fb = summ.pop("_fb")
    live, experts_live = summ["live_rows"], summ["experts_with_rows"]
    g = summ["gemm"]["gate_up"]
    fp8 = wl.dtype == "fp8"
    peak_note = (f"fp8 = 2 x {pk_kind} bf16 burst" if fp8 else f"{pk_kind} bf16 burst (cuBLAS)")
    traffic = None
    tp = os.path.join(ROOT, "profiles", f"traffic_{wl.name}.json")
    if os.path.exists(tp):
        with open(tp) as f:
            traffic = json.load(f).get("gemm_gate_up_swiglu_bytes" if separate
                                       else "gemm_gate_up_swiglu_gather_bytes")
    kernel_name = ("grouped GEMM gate_up + fused SwiGLU" + (" + FP8 quantisation of h" if fp8 else "")
                   if separate else "grouped GEMM gate_up, A gathered from token order, + fused SwiGLU")
    if fb["gemm1_bytes"] / (pk["hbm_gbs"] * 1e9) > fb["gemm1_flop"] / (summ["peaks"]["tensor_tflops"] * 1e12):
        roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": g["hbm_gbs"], "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": g["hbm_frac"], "peak_source": f"{pk_kind} HBM copy bandwidth",
                    "traffic": traffic, "tensor_frac": g["tensor_frac"], "tensor_peak_source": peak_note}
    else:
        roofline = {"bound": "tensor", "kernel": kernel_name, "achieved": g["tflops"],
                    "peak": summ["peaks"]["tensor_tflops"], "unit": "TFLOP/s", "frac": g["tensor_frac"],
                    "peak_source": peak_note, "traffic": traffic}
    roofline.update(algorithmic_flop=fb["gemm1_flop"], algorithmic_bytes=fb["gemm1_bytes"])
    clocks = clk.summary()
    cpu = None
    configs = None
    if world == 1:
        if not args.no_cpu_baseline:
            cpu = cpu_baseline_record(wl, synth)
        if not args.no_configs:
            # the other workloads, each with its own CPU baseline; these run
            # after the timed region above and are not part of its steps
            configs = {}
            for name in CONFIG_WORKLOADS:
                if name != wl.name:
                    configs[name] = measure_config(synth.WORKLOADS[name], args, torch, moe, synth, pk, flush,
                                                   local)
            with ClockSampler(local) as sclk:
                rows = sweep_measure(args.steps, args.warmup, synth, torch, moe, pk)
            configs[SWEEP_NAME] = {"rows": rows, "steps": args.steps, "clocks": sclk.summary(),
                                   "l2": "flushed between steps"}
            if not args.no_cpu_baseline:
                configs[SWEEP_NAME]["cpu_baseline"] = sweep_cpu_baseline(synth)
    line = {
        "metric": METRIC, "value": job_tokens_per_s(wl.T, world, ms_max), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded numpy draws; random-init weights N(0,0.02))",
        "config": {"workload": wl.name, "T": wl.T, "E": wl.E, "k": wl.k, "H": wl.H, "I": wl.I,
                   "bias": wl.bias, "live_rows": live, "experts_with_rows": experts_live,
                   "parallelism": f"replicas x{world} (no collective)",
                   "scatter": "separate kernel" if separate else "gathered inside the gate_up GEMM",
                   "combine": "fused into the down GEMM" if step.fused else "separate kernel",
                   "l2": "flushed between timed steps (256 MiB write, then read back; untimed)",
                   "launch": "eager C-ABI calls" if args.no_graph else "CUDA graph of the step's C-ABI calls"},
        "roofline": roofline,
        "gemm": {"gate_up_tflops": summ["gemm"]["gate_up"]["tflops"],
                 "down_tflops": summ["gemm"]["down"]["tflops"],
                 "gate_up_frac": summ["gemm"]["gate_up"]["tensor_frac"],
                 "down_frac": summ["gemm"]["down"]["tensor_frac"],
                 "pair_tflops": (fb["gemm1_flop"] + fb["gemm2_flop"]) /
                 ((summ["kernels_ms"]["gemm_gate_up_swiglu"] + summ["kernels_ms"]["gemm_down"]) * 1e-3) / 1e12,
                 "detail": summ["gemm"]},
        "kernels_ms": summ["kernels_ms"],
        "hbm": {"permute_gbs": summ["data_movement"].get("permute", {}).get("gbs"),
                "combine_gbs": summ["data_movement"].get("combine", {}).get("gbs"),
                "peak_gbs": pk["hbm_gbs"], "write_peak_gbs": pk["write_gbs"],
                "write_peak_source": "1 GiB float32 fill timed in this run (write-only HBM bandwidth)",
                "detail": summ["data_movement"]},
        "e2e": {"value": job_tokens_per_s(wl.T, world, e2e_capi_max), "unit": "tokens/s",
                "h2d_bytes_per_step": wl.T * wl.H * 2 + wl.T * wl.E * 4,
                "d2h_bytes_per_step": wl.T * wl.H * 2,
                "mode": ("serving loop through the C ABI: moe_forward with MOE_FWD_HOST_IO | "
                         "MOE_FWD_STAGED_OUT on pinned host buffers, batches alternating over two streams "
                         "(one workspace and pinned buffer set each, eager calls, the library running the "
                         "calls' kernels in call order), so one batch's host copies overlap its neighbours' "
                         "kernels; all copies inside the timed region"),
                "batches": n_serve,
                "staged_value": job_tokens_per_s(wl.T, world, e2e_max),
                "staged_mode": ("the caller stages the batches instead: input copies and output reads on two "
                                "copy streams around moe_forward on device buffers (" +
                                ("eager" if args.no_graph else "one CUDA graph per staging slot") + ")"),
                "serial_value": job_tokens_per_s(wl.T, world, e2e_serial_max),
                "serial_mode": ("moe_forward with MOE_FWD_HOST_IO on pinned buffers, one batch at a time: x "
                                "copied in on the library's side stream while the batch is routed, the "
                                "combine writing the pinned output in place")},
        "gpu_launches": step.launches_per_step() * args.steps * 2,   # graph replays + eager steps
        "clocks": clocks,
        "cpu_baseline": cpu,
        "configs": configs,
        "wall_s_timed": wall,
        "setup_s": L["setup_s"],
    }
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
