#!/usr/bin/env python
"""Benchmark of the ragged grouped SwiGLU expert layer on GB300.

One step = the whole hot path over one batch of the large workload (T = 16384 tokens, E = 256
experts, top-8, d = 2048, h = 512, M = 131072 routed rows): route histogram + offsets +
placement, permute, grouped up/gate GEMM with fused SwiGLU, grouped down GEMM, weighted
combine, and the backward (combine backward, down dgrad with fused SwiGLU backward and the
routing-weight gradient, up dgrad, both wgrads, permute backward). Every step is a library
kernel called through the C ABI.

Metric: useful expert TFLOP/s, 18*M*d*h per forward+backward step (6*M*d*h forward), M counting
routed rows only. Prints one JSON line. `--impl reference` times the CPU fp64 oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "useful expert TFLOP/s (6*M*d*h fwd, 18*M*d*h fwd+bwd), fwd+bwd step"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_NOTE = "inputs larger than L2 (129 MB): xp 512 MB, weights 1.6 GB; no flush"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="large")
    p.add_argument("--config", type=int, choices=range(5), default=None,
                   help="a named workload by index (0 toy, 1 balanced, 2 finegrained, 3 skew, 4 large); "
                        "overrides --workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-variants", action="store_true")
    p.add_argument("--sweep", choices=["capacity", "histogram", "configs", "precision", "oracle", "accumulation"],
                   default=None,
                   help="studies instead of the step: capacity (grouped vs capacity-padded BMM over "
                        "routed-row counts), histogram (throughput vs load imbalance), configs "
                        "(forward and training GEMMs on every workload), precision (the wgrads with "
                        "and without the low half of the activation operand), oracle (the CPU "
                        "baseline on every workload, all cores and one), accumulation (the error of "
                        "long contractions against fp32 sums rounded to nearest and toward zero)")
    args = p.parse_args()
    if args.config is not None:
        args.workload = ("toy", "balanced", "finegrained", "skew", "large")[args.config]
    return args


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's `value` (the slowest replica sets the job's time)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job throughput of `world` replicas that each did `flops_per_rank` in `ms` (max over
    ranks): weak scaling, the work grows with the replicas."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------------------ CPU oracle timing
class OracleSampler:
    """Times the oracle as it stands on a bounded sample of the workload: the route (histogram,
    offsets, placement) over all slots, then, expert by expert, the permute of that expert's
    rows, its forward and its backward (combine backward as a scaled permute), until about
    `seconds` of CPU time. Weight and input generation is not timed."""

    def __init__(self, wl):
        self.wl = wl
        self.x = wl.x()
        self.dout = wl.dout()
        self.next_expert = 0

    def run(self, seconds: float):
        import numpy as np
        from oracle import moe_oracle as O
        wl = self.wl
        t0 = time.perf_counter()
        r = O.route_offsets(wl.ids, wl.E)
        elapsed = time.perf_counter() - t0
        segs = O.segments(r["offsets"])
        picked, rows, flops = 0, 0, 0
        for _ in range(wl.E):
            e = self.next_expert
            self.next_expert = (e + 1) % wl.E
            s, t = segs[e]
            if t == s:
                continue
            wu, wd = wl.w_ug(e), wl.w_down(e)
            src = r["sorted_src"][s:t]
            one = np.array([t - s])
            t0 = time.perf_counter()
            xp = O.permute(self.x, src, t - s, wl.k)
            y, u, a, _ = O.expert_forward(xp, one, lambda i: wu, lambda i: wd)
            dy = O.permute(self.dout, src, t - s, wl.k, row_scale=wl.weights)
            O.expert_backward(dy, xp, u, one, lambda i: wu, lambda i: wd)
            # routing-weight gradient of this expert's slots: <dOut[token], unweighted y row>
            O.routing_weight_grad(O.permute(self.dout, src, t - s, wl.k), y, np.arange(t - s), t - s, 1)
            elapsed += time.perf_counter() - t0
            picked += 1
            rows += t - s
            flops += O.flops_fwd_bwd(t - s, wl.d, wl.h)
            if elapsed >= seconds:
                break
        desc = (f"route over all {wl.n} slots, then {picked} of {wl.E} experts ({rows} of {r['M']} rows): "
                f"permute + fp64 forward + backward (incl. routing-weight gradient) per expert")
        return flops, elapsed, desc


def blas_threads():
    """Threads of numpy's BLAS pool: threadpoolctl's report when it is installed, else the
    OPENBLAS/OMP thread variables, else the host's cores (OpenBLAS's default)."""
    try:
        from threadpoolctl import threadpool_info
        n = [p["num_threads"] for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count()


SINGLE_THREAD_CHILD = """
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
from ragged_grouped_gemm_device_gb300 import workloads as W
flops, el, desc = bench.OracleSampler(W.make(sys.argv[2])).run(float(sys.argv[3]))
print(json.dumps({"value": flops / el / 1e12, "sample": desc, "blas_threads": bench.blas_threads()}))
"""


def oracle_single_thread(workload: str, seconds: float):
    """The same oracle sample on one core: a child process whose BLAS pools are pinned to one
    thread before numpy loads (fork + exec: the child touches no CUDA state)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        res = subprocess.run([sys.executable, "-c", SINGLE_THREAD_CHILD, ROOT, workload, str(seconds)],
                             env=env, capture_output=True, text=True, timeout=300)
        return json.loads(res.stdout.strip().splitlines()[-1])
    except Exception as exc:  # reported, never fatal: the GPU numbers stand without it
        return {"error": f"{type(exc).__name__}: {exc}"[:200]}


def oracle_rates(wl, seconds: float) -> dict:
    """The oracle as it stands on a bounded sample of one workload, forward and forward +
    backward separately: expert by expert (in index order, empty experts skipped), the permute
    of its rows and its fp64 forward (6*M_e*d*h), or forward + backward (18*M_e*d*h), until about
    `seconds` of CPU time each. Weight generation is not timed."""
    import numpy as np
    from oracle import moe_oracle as O
    x, dout = wl.x(), wl.dout()
    r = O.route_offsets(wl.ids, wl.E)
    segs = O.segments(r["offsets"])
    order = [e for e in range(wl.E) if segs[e][1] > segs[e][0]]
    out = {}
    for mode in ("fwd", "fwd_bwd"):
        el, fl, rows, nexp = 0.0, 0, 0, 0
        for e in order:
            s, t = segs[e]
            wu, wd = wl.w_ug(e), wl.w_down(e)
            src = r["sorted_src"][s:t]
            one = np.array([t - s])
            t0 = time.perf_counter()
            xp = O.permute(x, src, t - s, wl.k)
            _, u, _, _ = O.expert_forward(xp, one, lambda i: wu, lambda i: wd)
            if mode == "fwd_bwd":
                dy = O.permute(dout, src, t - s, wl.k, row_scale=wl.weights)
                O.expert_backward(dy, xp, u, one, lambda i: wu, lambda i: wd)
            el += time.perf_counter() - t0
            fl += (O.flops_fwd_bwd if mode == "fwd_bwd" else O.flops_fwd)(t - s, wl.d, wl.h)
            rows += t - s
            nexp += 1
            if el >= seconds:
                break
        out[mode] = {"tflops": fl / el / 1e12, "experts": nexp, "rows": rows, "seconds": round(el, 2)}
    return out


ORACLE_SWEEP = ("balanced", "finegrained", "skew", "large")
ORACLE_SWEEP_CHILD = """
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
from ragged_grouped_gemm_device_gb300 import workloads as W
print(json.dumps({n: bench.oracle_rates(W.make(n), float(sys.argv[2])) for n in bench.ORACLE_SWEEP}))
"""


def run_sweep_oracle(args):
    """The CPU baseline on every mid-size and large workload: the oracle's forward and forward +
    backward rates on all host cores (numpy's BLAS pool) and, in a child process whose BLAS pools
    are pinned to one thread, on one core. No GPU is used."""
    from ragged_grouped_gemm_device_gb300 import workloads as W
    seconds = 3.0
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    child = subprocess.run([sys.executable, "-c", ORACLE_SWEEP_CHILD, ROOT, str(seconds)], env=env,
                           capture_output=True, text=True, timeout=900)
    single = json.loads(child.stdout.strip().splitlines()[-1]) if child.returncode == 0 else {}
    for name in ORACLE_SWEEP:
        wl = W.make(name)
        row = {"sweep": "oracle", "workload": name, "T": wl.T, "top_k": wl.k, "E": wl.E, "d": wl.d, "h": wl.h,
               "cores": os.cpu_count(), "blas_threads": blas_threads(), "all_cores": oracle_rates(wl, seconds),
               "single_thread": single.get(name, {"error": child.stderr[-300:]})}
        print(json.dumps(row), flush=True)
    return 0


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from ragged_grouped_gemm_device_gb300 import workloads as W
    wl = W.make(args.workload)
    cores = os.cpu_count()
    sampler = OracleSampler(wl)
    vals = []
    desc = ""
    # each step is a bounded sample: 2 s of oracle work, less when many steps are asked for,
    # so that the whole reference run stays near two minutes
    per_step = min(2.0, 120.0 / max(1, args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        flops, el, desc = sampler.run(per_step)
        if i >= args.warmup:
            vals.append((flops, el))
    tot_f = sum(f for f, _ in vals)
    tot_t = sum(t for _, t in vals)
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / len(vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "blas_threads": blas_threads(),
                         "kind": "oracle", "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl):
    import numpy as np
    ids = wl.ids.reshape(-1)
    counts = np.bincount(ids[(ids >= 0) & (ids < wl.E)], minlength=wl.E)
    M = int(counts.sum())
    p = counts[counts > 0] / M
    ih = 1.0 + float((p * np.log(p)).sum()) / float(np.log(wl.E))
    scheduled = int(sum(-(-int(c) // 128) * 128 for c in counts))
    return {"workload": f"{wl.name}: T={wl.T} tokens, E={wl.E} experts, top_k={wl.k}, d={wl.d}, h={wl.h}, SwiGLU",
            "T": wl.T, "top_k": wl.k, "E": wl.E, "d": wl.d, "h": wl.h, "M": M,
            "rows_per_expert": {"mean": M / wl.E, "max": int(counts.max()), "min": int(counts.min()),
                                "empty": int((counts == 0).sum())},
            "I_H": ih, "scheduled_rows_128": scheduled, "useful_rows": M, "l2": L2_NOTE}


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1])); mx.append(float(r[2])); pw.append(float(r[3]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(pw),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ our arm
GEMM_SOURCES = ("common.cuh", "grouped_gemm.cu", "internal.h", "moe_gg.cu")


def _code_only(text):
    """C++ source without its comments, blank lines and layout whitespace: what the compiler sees."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def kernel_source_hash():
    """Hash of the grouped GEMM's code (device code, launch arguments and tensor maps; comments
    and layout whitespace left out): DRAM traffic taken by the profiler is valid only for it. The routing and
    row-movement kernels (route.cu, permute.cu) do not enter it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ragged_grouped_gemm_device_gb300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_traffic():
    """DRAM bytes per launch (large workload) from the committed ncu summaries, for the kernels
    unchanged since their capture: a summary's `traffic_per_launch_large:` line holds a JSON
    object with the source hash and the bytes per kernel; lines whose hash is not the current
    one are ignored."""
    out = {}
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return out
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith(".md"):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for line in f:
                if line.startswith("traffic_per_launch_large:"):
                    t = json.loads(line.split(":", 1)[1])
                    if t.get("source_hash") == kernel_source_hash():
                        out.update(t.get("kernels", {}))
    return out


def kernel_work(M, T, k, E, d, h):
    """Per launch of each step kernel on a workload with M routed rows: (useful FLOPs, compulsory
    DRAM bytes, FLOPs the tensor cores execute). Bytes count every operand read once and every
    output written once under the library's data contract: bf16 rows and weights, the saved U at
    3 bytes a value,
    bf16 low halves of P and dU (the wgrads' second operand half), fp32 weight gradients, int32
    indices, fp32 routing weights. The wgrads execute twice their useful FLOPs (both halves)."""
    mdh = float(M) * d * h
    np_ = 2 * ((h + 255) // 256)  # routing-gradient partials per row
    wd = E * h * d * 2.0          # one [E, h, d] bf16 weight
    w = {
        "route": (0, T * k * 4 * 4.0, 0),                       # ids read twice, placement + inverse map written
        "permute": (0, T * d * 2.0 + M * d * 2.0 + M * 4.0, 0),
        "up_swiglu": (4 * mdh, M * d * 2.0 + 2 * wd + M * h * 2.0 * 2 + M * 2 * h * 3.0 + M * 8.0, 4 * mdh),
        "down": (2 * mdh, M * h * 2.0 + wd + M * d * 2.0, 2 * mdh),
        "combine": (0, M * d * 2.0 + T * d * 2.0 + T * k * 4.0, 0),
        "combine_bwd": (0, T * d * 2.0 + M * d * 2.0 + M * 4.0, 0),
        "down_dgrad_swiglu": (2 * mdh, M * d * 2.0 + wd + M * 2 * h * 3.0 + M * 2 * h * 2.0 * 2 + M * np_ * 4.0
                              + M * 8.0, 2 * mdh),
        "routing_weight_grad": (0, M * np_ * 4.0 + T * k * 8.0, 0),
        "up_dgrad": (4 * mdh, M * 2 * h * 2.0 + 2 * wd + M * d * 2.0, 4 * mdh),
        # down: P high + low [M, h], dy [M, d] -> dW_down fp32; up: dU high + low [M, 2h], xp -> dW_ug fp32
        "wgrad_dual": (6 * mdh, M * h * 4.0 + M * d * 2.0 + E * h * d * 4.0 + M * 2 * h * 4.0 + M * d * 2.0
                       + E * 2 * h * d * 4.0, 12 * mdh),
        "permute_bwd": (0, M * d * 2.0 + T * d * 2.0 + T * k * 4.0, 0),
    }
    return w


def kernel_rooflines(per_call, work, peaks, peak_src):
    """Each kernel against its roofline. The tensor peak is the measured burst bf16 rate (the
    timed region is tens of milliseconds, not the seconds-long loop the sustained figure comes
    from); the memory peak the measured copy rate. A kernel is tensor-bound when its FLOPs per
    compulsory byte reach the ridge peak_tflops / peak_hbm, else memory-bound; `floor_ms` is
    the larger of its two floors and `frac` = floor / measured time. Returns (breakdown, the
    slowest kernel, the roofline object of that kernel)."""
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ridge = peak_tf * 1e12 / (peak_hbm * 1e9)
    out = {}
    for name, ms in per_call.items():
        fl, by, ex = work[name]
        sec = ms * 1e-3
        b = {"ms": round(ms, 4), "bytes": int(by), "gbs": round(by / sec / 1e9, 1),
             "hbm_frac": round(by / sec / 1e9 / peak_hbm, 3)}
        if fl:
            b["tflops"] = round(fl / sec / 1e12, 1)
            b["tensor_frac"] = round(fl / sec / 1e12 / peak_tf, 3)
            b["intensity"] = round(fl / by, 1)
            b["bound"] = "tensor" if fl / by >= ridge else "hbm"
            if ex != fl:
                b["mma_executed_tflops"] = round(ex / sec / 1e12, 1)
        else:
            b["bound"] = "hbm"
        floor = max(fl / (peak_tf * 1e12), by / (peak_hbm * 1e9))
        b["floor_ms"] = round(floor * 1e3, 4)
        b["frac"] = round(floor / sec, 3)
        out[name] = b
    dom = max(per_call, key=per_call.get)
    fl, by, ex = work[dom]
    sec = per_call[dom] * 1e-3
    if out[dom]["bound"] == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": fl / sec / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": fl / sec / 1e12 / peak_tf, "peak_source": f"bf16_tflops ({peak_src}, burst)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": by / sec / 1e9, "peak": peak_hbm, "unit": "GB/s",
                "frac": by / sec / 1e9 / peak_hbm, "peak_source": f"hbm_gbs ({peak_src})"}
    roof["algorithmic_bytes"] = int(by)
    roof["useful_flops"] = fl
    roof["tensor_frac_of_burst"] = fl / sec / 1e12 / peak_tf if fl else 0.0
    roof["mma_executed_tflops"] = ex / sec / 1e12 if ex else 0.0
    roof["ridge_flop_per_byte"] = round(ridge, 1)
    return out, dom, roof


VARIANT_CONFIGS = ("balanced", "finegrained", "skew")


def config_variants(L, names=VARIANT_CONFIGS):
    """Forward of the SwiGLU expert on the mid-size workloads: the grouped composite call, the
    in-library capacity-padded BMM at C = ceil(1.25 M/E) (same kernels, rows beyond C dropped
    and counted) and the host-scheduled per-expert loop. Grouped and BMM: mean of 20 launches
    queued in a CUDA graph after 10 warm-ups; loop: wall time of one call (it copies the counts
    to the host and waits), mean of 3 after one warm-up. Weights and inputs are drawn on the
    device (values do not change the timing); the routing is the workload's."""
    import torch
    from ragged_grouped_gemm_device_gb300 import workloads as W
    dev, bf, i32 = "cuda", torch.bfloat16, torch.int32
    res = {}
    for name in names:
        wl = W.make(name)
        T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
        gen = torch.Generator(device=dev).manual_seed(1)
        x = torch.randn(T, d, device=dev, generator=gen).to(bf)
        w_ug = (torch.randn(E, 2 * h, d, device=dev, generator=gen) * d ** -0.5).to(bf)
        w_down = (torch.randn(E, h, d, device=dev, generator=gen) * h ** -0.5).to(bf)
        ids = torch.from_numpy(wl.ids).to(dev)
        counts, offsets = torch.empty(E, dtype=i32, device=dev), torch.empty(E, dtype=i32, device=dev)
        ss, inv = torch.empty(n, dtype=i32, device=dev), torch.empty(n, dtype=i32, device=dev)
        rws = torch.empty(max(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), 1), dtype=torch.uint8, device=dev)
        xp = torch.empty(n, d, dtype=bf, device=dev)
        L.moe_route_offsets(ids, T, k, E, counts, offsets, ss, inv, rws)
        L.moe_permute(x, ss, offsets, None, T, k, E, d, xp)
        torch.cuda.synchronize()
        M = int(offsets[-1].item())
        C = -(-(5 * M) // (4 * E))
        dropped = int(torch.clamp(counts.long() - C, min=0).sum().item())
        y = torch.empty(n, d, dtype=bf, device=dev)
        a = torch.empty(n, h, dtype=bf, device=dev)
        status = torch.zeros(1, dtype=i32, device=dev)
        bws = torch.empty(L.moe_workspace_bytes(L.OP_PADDED_BMM, T, k, E, d, h, C), dtype=torch.uint8, device=dev)
        t_g = queued_mean_ms(lambda: L.moe_grouped_swiglu_fwd(xp, offsets, None, None, E, n, d, h, w_ug, w_down, y,
                                                               a, None, None, status))
        t_b = queued_mean_ms(lambda: L.moe_padded_bmm_swiglu_fwd(xp, offsets, E, n, d, h, C, w_ug, w_down, y, bws,
                                                                  status))
        top1 = None
        if k == 1:
            # the layer forward after the permute: grouped forward + combine, against the down
            # projection writing the token rows itself
            out = torch.empty(T, d, dtype=bf, device=dev)
            wts = torch.from_numpy(wl.weights.reshape(-1)).to(dev)
            t_sep = queued_mean_ms(lambda: (L.moe_grouped_swiglu_fwd(xp, offsets, ss, wts, E, n, d, h, w_ug, w_down, y,
                                                                     a, None, None, status),
                                            L.moe_unpermute_combine(y, inv, None, T, k, d, out)))
            t_fus = queued_mean_ms(lambda: L.moe_grouped_swiglu_fwd_top1_combine(xp, offsets, ss, inv, wts, E, T, d, h,
                                                                                 w_ug, w_down, out, a, None, status))
            top1 = {"forward_then_combine_ms": round(t_sep, 4), "fused_combine_ms": round(t_fus, 4),
                    "speedup": round(t_sep / t_fus, 3)}
            del out, wts
        loop = lambda: L.moe_loop_swiglu_fwd(xp, offsets, E, n, d, h, w_ug, w_down, y, a, None, status)
        loop()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(3):
            loop()
        torch.cuda.synchronize()
        t_l = (time.perf_counter() - t0) * 1e3 / 3
        assert status.item() == 0, f"device status {status.item()}"
        fl = 6.0 * M * d * h
        res[name] = {"T": T, "top_k": k, "E": E, "d": d, "h": h, "M": M,
                     "grouped": {"ms": round(t_g, 4), "tflops": round(fl / t_g / 1e9, 1)},
                     "padded_bmm": {"ms": round(t_b, 4), "tflops": round(fl / t_b / 1e9, 1), "C": C,
                                    "rows_multiplied": E * C, "rows_dropped": dropped},
                     "host_loop": {"ms": round(t_l, 4), "tflops": round(fl / t_l / 1e9, 1)},
                     "grouped_vs_bmm": round(t_b / t_g, 3), "grouped_vs_loop": round(t_l / t_g, 3)}
        if top1 is not None:
            res[name]["top1_fused_combine"] = top1
        del x, w_ug, w_down, xp, y, a, bws
        torch.cuda.empty_cache()
    return res


class TrainingStep:
    """One training step of the hot path as the benchmark times it: every row a1-a14 as one C-ABI
    call per kernel (13 launches), on buffers allocated once for T tokens, top_k slots, E experts
    and widths d, h. `calls(x, ids, weights, dout)` lists (name, launches, thunk) in step order:
    route, gather, up/gate + SwiGLU, down, combine, dOut gather, down dgrad + SwiGLU backward with
    the routing-gradient partials, their reduction, up/gate dgrad, both wgrads in one launch,
    input-gradient combine. The full-size parity test runs these same calls."""

    def __init__(self, L, T, k, E, d, h, w_ug, w_down, dev):
        import torch
        self.L, self.T, self.k, self.E, self.d, self.h = L, T, k, E, d, h
        self.n = n = T * k
        self.w_ug, self.w_down = w_ug, w_down
        bf, i32, f32, u8 = torch.bfloat16, torch.int32, torch.float32, torch.uint8
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E, dtype=i32, device=dev)
        self.sorted_src = torch.empty(n, dtype=i32, device=dev)
        self.inv_map = torch.empty(n, dtype=i32, device=dev)
        self.route_ws = torch.empty(max(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), 1), dtype=u8, device=dev)
        self.xp = torch.empty(n, d, dtype=bf, device=dev)
        self.a = torch.empty(n, h, dtype=bf, device=dev)
        self.y = torch.empty(n, d, dtype=bf, device=dev)
        self.saved = torch.empty(L.moe_workspace_bytes(L.OP_SAVED, T, k, E, d, h), dtype=u8, device=dev)
        self.out = torch.empty(T, d, dtype=bf, device=dev)
        self.dy = torch.empty(n, d, dtype=bf, device=dev)
        self.du_hi = torch.empty(n, 2 * h, dtype=bf, device=dev)
        self.du_lo = torch.empty(n, 2 * h, dtype=bf, device=dev)
        self.dxp = torch.empty(n, d, dtype=bf, device=dev)
        self.dx = torch.empty(T, d, dtype=bf, device=dev)
        self.dw_ug = torch.empty(E, 2 * h, d, dtype=f32, device=dev)
        self.dw_down = torch.empty(E, h, d, dtype=f32, device=dev)
        self.dw_part = torch.empty(n, L.routing_grad_parts(h), dtype=f32, device=dev)
        self.dw_route = torch.empty(T, k, dtype=f32, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        _, self.p_lo = L.saved_views(self.saved, n, h)

    def calls(self, xin, idin, win, doin):
        L, T, k, E, d, h, n = self.L, self.T, self.k, self.E, self.d, self.h, self.n
        w_ug, w_down, status = self.w_ug, self.w_down, self.status
        counts, offsets, sorted_src, inv_map = self.counts, self.offsets, self.sorted_src, self.inv_map
        xp, a, y, saved, out, dy = self.xp, self.a, self.y, self.saved, self.out, self.dy
        du_hi, du_lo, dxp, dx, dw_part = self.du_hi, self.du_lo, self.dxp, self.dx, self.dw_part
        return [
            ("route", 3, lambda: L.moe_route_offsets(idin, T, k, E, counts, offsets, sorted_src, inv_map,
                                                     self.route_ws)),
            ("permute", 1, lambda: L.moe_permute(xin, sorted_src, offsets, None, T, k, E, d, xp)),
            ("up_swiglu", 1, lambda: L.moe_grouped_up_swiglu(xp, offsets, sorted_src, win, E, n, d, h, w_ug, a,
                                                             saved, status)),
            ("down", 1, lambda: L.moe_grouped_down(a, offsets, E, n, d, h, w_down, y, status)),
            ("combine", 1, lambda: L.moe_unpermute_combine(y, inv_map, None, T, k, d, out)),
            ("combine_bwd", 1, lambda: L.moe_permute(doin, sorted_src, offsets, None, T, k, E, d, dy)),
            ("down_dgrad_swiglu", 1, lambda: L.moe_grouped_down_dgrad_swiglu(dy, saved, offsets, sorted_src, win, E,
                                                                             n, d, h, w_down, du_hi, du_lo, status,
                                                                             dw_part=dw_part)),
            ("routing_weight_grad", 1, lambda: L.moe_routing_weight_grad(dw_part, inv_map, T, k, h, self.dw_route)),
            ("up_dgrad", 1, lambda: L.moe_grouped_up_dgrad(du_hi, offsets, E, n, d, h, w_ug, dxp, status)),
            # both weight gradients (down, then up/gate) in one persistent launch
            ("wgrad_dual", 1, lambda: L.moe_grouped_wgrad_dual(a, self.p_lo, h, dy, d, self.dw_down, du_hi, du_lo,
                                                               2 * h, xp, d, self.dw_ug, offsets, E, n, status)),
            ("permute_bwd", 1, lambda: L.moe_unpermute_combine(dxp, inv_map, None, T, k, d, dx)),
        ]


def run_ours(args):
    import numpy as np
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from ragged_grouped_gemm_device_gb300 import _lib
    from ragged_grouped_gemm_device_gb300 import workloads as W
    L = _lib
    L.load()

    wl = W.make(args.workload)
    T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
    dev = torch.device("cuda", local_rank)
    bf = torch.bfloat16
    x_h = torch.from_numpy(wl.x()).to(bf)
    dout_h = torch.from_numpy(wl.dout()).to(bf)
    ids_h = torch.from_numpy(wl.ids)
    wts_h = torch.from_numpy(wl.weights)
    w_ug = torch.empty(E, 2 * h, d, dtype=bf, device=dev)
    w_down = torch.empty(E, h, d, dtype=bf, device=dev)
    for e in range(E):
        w_ug[e].copy_(torch.from_numpy(wl.w_ug(e)).to(bf))
        w_down[e].copy_(torch.from_numpy(wl.w_down(e)).to(bf))
    x, dout, ids, wts = x_h.to(dev), dout_h.to(dev), ids_h.to(dev), wts_h.to(dev)

    step = TrainingStep(L, T, k, E, d, h, w_ug, w_down, dev)
    counts, offsets, sorted_src, inv_map = step.counts, step.offsets, step.sorted_src, step.inv_map
    xp, a, y, saved, out, dy = step.xp, step.a, step.y, step.saved, step.out, step.dy
    du_hi, du_lo, dxp, dx, dw_ug, dw_down = step.du_hi, step.du_lo, step.dxp, step.dx, step.dw_ug, step.dw_down
    dw_part, dw_route, status = step.dw_part, step.dw_route, step.status
    stream = torch.cuda.current_stream()

    def inputs():
        return x, ids, wts, dout

    step_calls = step.calls

    calls = step_calls(*inputs())
    launches_per_step = sum(c[1] for c in calls)
    for _ in range(args.warmup):
        for _, _, fn in calls:
            fn()
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"

    # ---- timed region: K steps, events between the calls on the launching stream
    nc = len(calls)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        ev = evs[s]
        for i, (_, _, fn) in enumerate(calls):
            ev[i].record(stream)
            fn()
        ev[nc].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    per_call = {}
    for i, (name, _, _) in enumerate(calls):
        per_call[name] = statistics.mean(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps))
    assert status.item() == 0, f"device status {status.item()}"

    M = int(offsets[-1].item())
    ms_step = elapsed_ms / args.steps
    fwdbwd_flops = 18.0 * M * d * h
    value = job_tflops(world, fwdbwd_flops, ms_step)
    peaks, peak_src = load_peaks()
    mdh = float(M) * d * h
    breakdown, dom, roofline = kernel_rooflines(per_call, kernel_work(M, T, k, E, d, h), peaks, peak_src)
    traffic = load_traffic().get(dom)
    roofline["traffic"] = traffic
    fwd_ms = per_call["up_swiglu"] + per_call["down"]
    # the forward layer a1-a8: routing, gather, both projections and the combine
    fwd_layer_ms = sum(per_call[c] for c in ("route", "permute", "up_swiglu", "down", "combine"))
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))

    # ---- end to end through the public calls with host buffers (pinned), copies inside. As a
    # training loop would: the inputs of a step go host -> device on one copy stream into one of
    # two device buffers while the GPU computes the step before, and out / dx come back on a
    # second copy stream while the backward (or the next step) runs. Every step's copies lie
    # between the start and end events: the copy streams wait on the start event, and the end
    # event waits on the last read-back.
    xh, doh = x_h.pin_memory(), dout_h.pin_memory()
    idh, wh = ids_h.pin_memory(), wts_h.pin_memory()
    out_h = torch.empty(T, d, dtype=bf).pin_memory()
    dx_h = torch.empty(T, d, dtype=bf).pin_memory()
    bufs = [(torch.empty_like(x), torch.empty_like(ids), torch.empty_like(wts), torch.empty_like(dout))
            for _ in range(2)]
    calls_b = [step_calls(*b) for b in bufs]
    n_fwd = [c[0] for c in calls].index("combine") + 1  # calls up to the combine produce out
    cs_in, cs_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ev_in, ev_free = [ev(), ev()], [ev(), ev()]
    ev_out, ev_dx, ev_outcp, ev_dxcp = ev(), ev(), ev(), ev()

    def h2d(j, after):
        with torch.cuda.stream(cs_in):
            cs_in.wait_event(after)
            for dst, src in zip(bufs[j], (xh, idh, wh, doh)):
                dst.copy_(src, non_blocking=True)
            ev_in[j].record(cs_in)

    def e2e_run(n_steps, start_ev):
        start_ev.record(stream)
        for j in range(min(2, n_steps)):
            h2d(j, start_ev)
        for i in range(n_steps):
            j = i % 2
            stream.wait_event(ev_in[j])
            if i > 0:
                stream.wait_event(ev_outcp)  # the previous step's out has been read back
            for _, _, fn in calls_b[j][:n_fwd]:
                fn()
            ev_out.record(stream)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(ev_out)
                out_h.copy_(out, non_blocking=True)
                ev_outcp.record(cs_out)
            if i > 0:
                stream.wait_event(ev_dxcp)
            for _, _, fn in calls_b[j][n_fwd:]:
                fn()
            ev_dx.record(stream)
            ev_free[j].record(stream)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(ev_dx)
                dx_h.copy_(dx, non_blocking=True)
                ev_dxcp.record(cs_out)
            if i + 2 < n_steps:
                h2d(j, ev_free[j])
        stream.wait_event(ev_outcp)
        stream.wait_event(ev_dxcp)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(3, e0)
    torch.cuda.synchronize()
    e_steps = max(20, args.steps)  # as many steps as the device-timed loop: one host stall weighs less
    e2e_run(e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    e2e_ms = e0.elapsed_time(e1) / e_steps
    h2d = x_h.numel() * 2 + dout_h.numel() * 2 + ids_h.numel() * 4 + wts_h.numel() * 4
    d2h = 2 * T * d * 2
    e2e_ms = max_over_ranks(e2e_ms, world, dev)

    # ---- forward comparison variants (same kernels): padded BMM at ceil(1.25 M/E), host loop
    variants = None
    if not args.no_variants:
        C = -(-(5 * M) // (4 * E))
        bmm_ws = torch.empty(L.moe_workspace_bytes(L.OP_PADDED_BMM, T, k, E, d, h, C), dtype=torch.uint8, device=dev)
        y2 = torch.empty_like(y)

        def time_fn(fn, reps=10):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for _ in range(reps):
                fn()
            b1.record(stream)
            torch.cuda.synchronize()
            return b0.elapsed_time(b1) / reps, (time.perf_counter() - t0) * 1e3 / reps

        g_ms, _ = time_fn(lambda: L.moe_grouped_swiglu_fwd(xp, offsets, None, None, E, n, d, h, w_ug, w_down, y2,
                                                           a, None, None, status))
        b_ms, _ = time_fn(lambda: L.moe_padded_bmm_swiglu_fwd(xp, offsets, E, n, d, h, C, w_ug, w_down, y2, bmm_ws,
                                                              status))
        l_dev, l_wall = time_fn(lambda: L.moe_loop_swiglu_fwd(xp, offsets, E, n, d, h, w_ug, w_down, y2, a, None,
                                                              status), reps=5)
        fw = 6.0 * mdh
        # MXFP8 variant (scaled forward and dgrad, BF16 wgrads) against the bf16 training calls:
        # the forward includes its activation quantizations; the weight preparation (once per
        # weight update) is timed on its own
        mxw = torch.empty(L.moe_workspace_bytes(L.OP_MX_WEIGHTS, T, k, E, d, h), dtype=torch.uint8, device=dev)
        mfws = torch.empty(L.moe_workspace_bytes(L.OP_MX_FWD, T, k, E, d, h), dtype=torch.uint8, device=dev)
        mbws = torch.empty(L.moe_workspace_bytes(L.OP_MX_BWD, T, k, E, d, h), dtype=torch.uint8, device=dev)
        bbws = torch.empty(L.moe_workspace_bytes(L.OP_BWD, T, k, E, d, h), dtype=torch.uint8, device=dev)
        wp_ms, _ = time_fn(lambda: L.moe_mx_prepare_weights(w_ug, w_down, E, d, h, mxw))
        # each side from token rows: the gather (fused with the quantization on the MXFP8 side)
        # and the composite call; the backward from dOut through its gather
        sfb = L.moe_workspace_bytes(L.OP_MX_ROW_SCALES, T, k, E, d, h)
        xq, xsf = (torch.empty(n, d, dtype=torch.uint8, device=dev), torch.empty(sfb, dtype=torch.uint8, device=dev))
        dyq, dysf = (torch.empty(n, d, dtype=torch.uint8, device=dev), torch.empty(sfb, dtype=torch.uint8, device=dev))

        def mx_fwd():
            L.moe_permute_mxfp8(x, sorted_src, offsets, T, k, E, d, xp, xq, xsf, status)
            L.moe_grouped_swiglu_fwd_mxfp8(None, offsets, sorted_src, wts, E, n, d, h, mxw, y2, a, saved, mfws, status,
                                           xq=xq, xsf=xsf)

        def mx_bwd():
            L.moe_permute_mxfp8(dout, sorted_src, offsets, T, k, E, d, dy, dyq, dysf, status)
            L.moe_grouped_bwd_mxfp8(dy, xp, a, saved, offsets, sorted_src, wts, E, n, d, h, mxw, dxp, dw_ug, dw_down,
                                    mbws, status, dyq=dyq, dysf=dysf)

        def bf_fwd():
            L.moe_permute(x, sorted_src, offsets, None, T, k, E, d, xp)
            L.moe_grouped_swiglu_fwd(xp, offsets, sorted_src, wts, E, n, d, h, w_ug, w_down, y2, a, saved, None,
                                     status)

        def bf_bwd():
            L.moe_permute(dout, sorted_src, offsets, None, T, k, E, d, dy)
            L.moe_grouped_bwd(dy, xp, a, saved, offsets, sorted_src, wts, E, n, d, h, w_ug, w_down, dxp, dw_ug,
                              dw_down, bbws, status)

        mf_ms, _ = time_fn(mx_fwd)
        mb_ms, _ = time_fn(mx_bwd)
        tf_ms, _ = time_fn(bf_fwd)
        tb_ms, _ = time_fn(bf_bwd)
        del xq, xsf, dyq, dysf
        mxfp8 = {"weight_prep_ms": wp_ms, "fwd_ms": mf_ms, "fwd_tflops": fw / (mf_ms * 1e-3) / 1e12,
                 "bwd_ms": mb_ms, "fwd_bwd_tflops": 3 * fw / ((mf_ms + mb_ms) * 1e-3) / 1e12,
                 "bf16_training_fwd_ms": tf_ms, "bf16_bwd_ms": tb_ms,
                 "bf16_fwd_bwd_tflops": 3 * fw / ((tf_ms + tb_ms) * 1e-3) / 1e12,
                 "note": "from token rows, saved state written; MXFP8 forward = gather fused with the "
                         "quantization of xp, scaled up/gate GEMM quantizing P in its epilogue, scaled down "
                         "GEMM; backward = gather of dOut fused with its quantization, scaled dgrad quantizing "
                         "dU in its epilogue, scaled up dgrad, BF16 wgrads; bf16 = gather + the composite"}
        del mxw, mfws, mbws, bbws
        variants = {"grouped_fwd": {"ms": g_ms, "tflops": fw / (g_ms * 1e-3) / 1e12},
                    "padded_bmm_fwd": {"ms": b_ms, "tflops": fw / (b_ms * 1e-3) / 1e12, "C": C,
                                       "rows_multiplied": E * C, "rho_pad": 1 - M / (E * C)},
                    "host_loop_fwd": {"ms": l_wall, "tflops": fw / (l_wall * 1e-3) / 1e12,
                                      "note": "wall time incl. the D2H count copy and host wait"},
                    "mxfp8": mxfp8}
        del bmm_ws, y2
        torch.cuda.synchronize()
        assert status.item() == 0, f"device status {status.item()}"

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; random-init weights)",
        "config": workload_config(wl),
        "fwd": {"ms": fwd_ms, "tflops": 6.0 * mdh / (fwd_ms * 1e-3) / 1e12,
                "frac_of_burst_peak": 6.0 * mdh / (fwd_ms * 1e-3) / 1e12 / peak_tf,
                "peak_source": f"bf16_tflops ({peak_src}, burst: the timed region lasts well under a second)"},
        "fwd_layer": {"ms": fwd_layer_ms, "tflops": 6.0 * mdh / (fwd_layer_ms * 1e-3) / 1e12,
                      "span": "route, permute, up/gate + SwiGLU, down, combine (in the training step)"},
        "roofline": roofline,
        "e2e": {"value": job_tflops(world, fwdbwd_flops, e2e_ms), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "breakdown": breakdown,
        "variants": variants,
        "variants_by_config": config_variants(L) if (not args.no_variants and world == 1) else None,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        flops, el, desc = OracleSampler(wl).run(12.0)
        line["cpu_baseline"] = {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                                "blas_threads": blas_threads(), "kind": "oracle", "sample": desc,
                                "single_thread": oracle_single_thread(args.workload, 6.0)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# ------------------------------------------------------------------------------ projection sweeps
PROJ_E, PROJ_K, PROJ_N = 16, 4096, 4096


def queued_mean_ms(fn, warmup=10, samples=20):
    """Mean device time of `fn` over `samples` launches queued back to back: one CUDA graph of
    the launches, replayed once between two events, after `warmup` plain calls."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(samples):
            fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g.replay()  # first replay uploads the graph
    torch.cuda.synchronize()
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / samples


def median_ms(fn, warmup=3, samples=50):
    """Median device time of `fn` over `samples` launches, each timed alone between two events
    on the current stream and synchronised (the pages' median of 50)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def projection_setup(max_rows, seed=0):
    """Device inputs of the square projection: X [max_rows, K] ~ N(0, 1) and W [E, K, N] ~
    N(0, 1/sqrt(K)), bf16, drawn on the device from a seeded generator (the values do not
    change the timing; the parity tests draw the same shapes from workloads.py)."""
    import torch
    gen = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(max_rows, PROJ_K, device="cuda", generator=gen).to(torch.bfloat16)
    w = (torch.randn(PROJ_E, PROJ_K, PROJ_N, device="cuda", generator=gen) * PROJ_K ** -0.5).to(torch.bfloat16)
    return x, w


def spearman(a, b):
    import numpy as np
    ra = np.argsort(np.argsort(a)).astype(np.float64)
    rb = np.argsort(np.argsort(b)).astype(np.float64)
    return float(np.corrcoef(ra, rb)[0, 1])


def run_sweep_capacity(args):
    """Fig. 38 of "Section 09: Grouped GEMM" on GB300: one bf16 square expert projection
    (16 experts, d = h = 4096), balanced routing, total routed rows M = 64 ... 128K. Grouped:
    the exact-row grouped kernel over the rowwise buffer. Padded BMM: the same kernel over
    capacity C = 1.25 M/16 rows per expert (the padded layout, as a uniform problem list), and
    cuBLAS batched GEMM (torch.bmm) on the same padded shapes. Useful TFLOP/s counts valid rows."""
    import torch
    from ragged_grouped_gemm_device_gb300 import _lib as L
    from ragged_grouped_gemm_device_gb300 import workloads as W
    E, K, N = PROJ_E, PROJ_K, PROJ_N
    Ms = [64 << i for i in range(12)]
    Cmax = -(-5 * Ms[-1] // (4 * E))
    x, w = projection_setup(max(Ms[-1], E * Cmax))
    y = torch.empty(max(Ms[-1], E * Cmax), N, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = []
    for M in Ms:
        offs = torch.from_numpy(W.balanced_counts(M, E).cumsum().astype("int32")).cuda()
        C = -(-5 * M // (4 * E))
        uoffs = torch.arange(1, E + 1, dtype=torch.int32, device="cuda") * C
        xpad = x[: E * C].view(E, C, K)
        ypad = torch.empty(E, C, N, dtype=torch.bfloat16, device="cuda")
        t_g = queued_mean_ms(lambda: L.moe_grouped_down(x, offs, E, M, N, K, w, y, status))
        t_b = queued_mean_ms(lambda: L.moe_grouped_down(x, uoffs, E, E * C, N, K, w, y, status))
        t_c = queued_mean_ms(lambda: torch.bmm(xpad, w, out=ypad))
        fl = 2.0 * M * K * N
        row = {"sweep": "capacity", "M": M, "rows_per_expert": M / E, "C": C,
               "grouped_ms": t_g, "padded_same_kernel_ms": t_b, "padded_cublas_bmm_ms": t_c,
               "grouped_tflops": fl / t_g / 1e9, "padded_same_kernel_tflops": fl / t_b / 1e9,
               "padded_cublas_bmm_tflops": fl / t_c / 1e9,
               "speedup_vs_same_kernel": t_b / t_g, "speedup_vs_cublas_bmm": t_c / t_g}
        rows.append(row)
        print(json.dumps(row), flush=True)
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    cross = next((r["M"] for r in rows if r["speedup_vs_cublas_bmm"] > 1.0
                  and all(q["speedup_vs_cublas_bmm"] > 1.0 for q in rows if q["M"] >= r["M"])), None)
    print(json.dumps({"sweep": "capacity", "summary": True, "experts": E, "d": K, "h": N,
                      "timing": "mean of 20 launches queued in a CUDA graph after 10 warm-ups",
                      "grouped_faster_than_cublas_bmm_from_M": cross,
                      "grouped_never_slower_than_same_kernel_padded": all(
                          r["speedup_vs_same_kernel"] >= 0.98 for r in rows)}), flush=True)
    return 0


def run_sweep_histogram(args):
    """Fig. 40 of "Section 09: Grouped GEMM" on GB300: the same projection at M = 65536 rows over
    100 fixed-work load histograms stratified by I_H (Eq. 18); each histogram timed under 4
    expert-index permutations in a seeded random order, a balanced control before every ten
    cases and at the end. Reports the Spearman correlation of I_H with throughput, a
    histogram-level bootstrap 95% interval and the median throughput normalised to the
    balanced controls per I_H range."""
    import numpy as np
    import torch
    from ragged_grouped_gemm_device_gb300 import _lib as L
    from ragged_grouped_gemm_device_gb300 import workloads as W
    E, K, N, M = PROJ_E, PROJ_K, PROJ_N, 65536
    hists = W.dirichlet_histograms(M=M, E=E)
    perms = W.expert_permutations(E, 4)
    x, w = projection_setup(M)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fl = 2.0 * M * K * N

    def tput(counts):
        offs = torch.from_numpy(np.cumsum(counts).astype("int32")).cuda()
        return fl / queued_mean_ms(lambda: L.moe_grouped_down(x, offs, E, M, N, K, w, y, status)) / 1e9

    balanced = W.balanced_counts(M, E)
    conds = [(i, j) for i in range(len(hists)) for j in range(len(perms))]
    order = np.random.default_rng([args.steps, 40]).permutation(len(conds))
    per_hist = [[] for _ in hists]
    controls = []
    for n, ci in enumerate(order):
        if n % 10 == 0:
            controls.append(tput(balanced))
        i, j = conds[ci]
        per_hist[i].append((tput(hists[i][0][perms[j]]), len(controls) - 1))
    controls.append(tput(balanced))
    torch.cuda.synchronize()
    assert status.item() == 0, f"device status {status.item()}"
    # each case normalised by the mean of the two controls that bracket it
    norm = [float(np.mean([t / (0.5 * (controls[c] + controls[c + 1])) for t, c in v])) for v in per_hist]
    raw = [float(np.mean([t for t, _ in v])) for v in per_hist]
    ih = np.array([h[1] for h in hists])
    rho = spearman(ih, np.array(raw))
    rng = np.random.default_rng(7)
    boot = []
    for _ in range(2000):
        idx = rng.integers(0, len(hists), len(hists))
        boot.append(spearman(ih[idx], np.array(raw)[idx]))
    lo, hi = np.percentile(boot, [2.5, 97.5])
    edges = np.linspace(0.0, ih.max() + 1e-12, 11)
    med = [float(np.median([norm[k] for k in range(len(hists)) if edges[b] <= ih[k] < edges[b + 1]] or [float("nan")]))
           for b in range(10)]
    print(json.dumps({"sweep": "histogram", "experts": E, "M": M, "d": K, "h": N, "histograms": len(hists),
                      "permutations": len(perms), "balanced_tflops": float(np.mean(controls)),
                      "spearman_IH_vs_tflops": rho, "bootstrap_95": [float(lo), float(hi)],
                      "median_normalised_by_IH_range": med,
                      "IH_range_edges": [round(float(e), 4) for e in edges],
                      "cases": [{"I_H": float(ih[k]), "tflops": raw[k], "normalised": norm[k],
                                 "max_rows": int(hists[k][0].max())} for k in range(len(hists))]}), flush=True)
    return 0


def run_sweep_configs(args):
    """Forward of the SwiGLU expert on each named workload: the grouped composite call against
    the in-library capacity-padded BMM (C = ceil(1.25 M/E), same kernels) and the host-scheduled
    per-expert loop (wall time, including its count copy and host wait). Grouped and BMM: mean
    of 20 launches queued in a CUDA graph after 10 warm-ups, and the median of 50 launches each
    timed alone; loop: mean of 5 calls. Workloads with a backward also time the grouped GEMMs of
    a training step (a6-a7 with the saved state, then a10-a13 from dY at the grouped boundary,
    the two composite calls; 18*M*d*h useful FLOPs), graph-queued."""
    import torch
    from ragged_grouped_gemm_device_gb300 import _lib as L
    from ragged_grouped_gemm_device_gb300 import workloads as W
    dev, bf, i32 = "cuda", torch.bfloat16, torch.int32
    rows = []
    for name in ("toy", "balanced", "finegrained", "skew", "large"):
        wl = W.make(name)
        T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
        gen = torch.Generator(device=dev).manual_seed(1)
        x = torch.randn(T, d, device=dev, generator=gen).to(bf)
        w_ug = (torch.randn(E, 2 * h, d, device=dev, generator=gen) * d ** -0.5).to(bf)
        w_down = (torch.randn(E, h, d, device=dev, generator=gen) * h ** -0.5).to(bf)
        ids = torch.from_numpy(wl.ids).to(dev)
        counts, offsets = torch.empty(E, dtype=i32, device=dev), torch.empty(E, dtype=i32, device=dev)
        ss, inv = torch.empty(n, dtype=i32, device=dev), torch.empty(n, dtype=i32, device=dev)
        rws = torch.empty(max(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), 1), dtype=torch.uint8, device=dev)
        xp = torch.empty(n, d, dtype=bf, device=dev)
        L.moe_route_offsets(ids, T, k, E, counts, offsets, ss, inv, rws)
        L.moe_permute(x, ss, offsets, None, T, k, E, d, xp)
        torch.cuda.synchronize()
        M = int(offsets[-1].item())
        C = -(-(5 * M) // (4 * E))
        dropped = int(torch.clamp(counts.long() - C, min=0).sum().item())  # rows the padded BMM drops
        y = torch.empty(n, d, dtype=bf, device=dev)
        a = torch.empty(n, h, dtype=bf, device=dev)
        status = torch.zeros(1, dtype=i32, device=dev)
        bws = torch.empty(L.moe_workspace_bytes(L.OP_PADDED_BMM, T, k, E, d, h, C), dtype=torch.uint8, device=dev)
        fwd_g = lambda: L.moe_grouped_swiglu_fwd(xp, offsets, None, None, E, n, d, h, w_ug, w_down, y, a, None,
                                                 None, status)
        fwd_b = lambda: L.moe_padded_bmm_swiglu_fwd(xp, offsets, E, n, d, h, C, w_ug, w_down, y, bws, status)
        t_g, t_b = queued_mean_ms(fwd_g), queued_mean_ms(fwd_b)
        m_g, m_b = median_ms(fwd_g), median_ms(fwd_b)
        train = None
        if wl.has_bwd:
            sv = torch.empty(L.moe_workspace_bytes(L.OP_SAVED, T, k, E, d, h), dtype=torch.uint8, device=dev)
            bw = torch.empty(max(L.moe_workspace_bytes(L.OP_BWD, T, k, E, d, h), 1), dtype=torch.uint8,
                             device=dev)
            dyb = torch.randn(n, d, device=dev, generator=gen).to(bf)
            dxp = torch.empty(n, d, dtype=bf, device=dev)
            dwu = torch.empty(E, 2 * h, d, device=dev)
            dwd = torch.empty(E, h, d, device=dev)
            fwd_t = lambda: L.moe_grouped_swiglu_fwd(xp, offsets, None, None, E, n, d, h, w_ug, w_down, y, a,
                                                     sv, None, status)
            bwd_t = lambda: L.moe_grouped_bwd(dyb, xp, a, sv, offsets, None, None, E, n, d, h, w_ug, w_down,
                                              dxp, dwu, dwd, bw, status)
            t_ft, t_bt = queued_mean_ms(fwd_t), queued_mean_ms(bwd_t)
            train = {"fwd_ms": t_ft, "bwd_ms": t_bt,
                     "fwd_bwd_tflops": 18.0 * M * d * h / (t_ft + t_bt) / 1e9,
                     "bwd_tflops": 12.0 * M * d * h / t_bt / 1e9}
            del sv, bw, dyb, dxp, dwu, dwd
        loop = lambda: L.moe_loop_swiglu_fwd(xp, offsets, E, n, d, h, w_ug, w_down, y, a, None, status)
        for _ in range(2):
            loop()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(5):
            loop()
        torch.cuda.synchronize()
        t_l = (time.perf_counter() - t0) * 1e3 / 5
        assert status.item() == 0, f"device status {status.item()}"
        fl = 6.0 * M * d * h
        row = {"sweep": "configs", "workload": name, "T": T, "top_k": k, "E": E, "d": d, "h": h, "M": M,
               "C": C, "padded_bmm_dropped_rows": dropped, "grouped_ms": t_g, "padded_bmm_ms": t_b,
               "host_loop_ms": t_l,
               "grouped_tflops": fl / t_g / 1e9, "padded_bmm_tflops": fl / t_b / 1e9,
               "host_loop_tflops": fl / t_l / 1e9, "speedup_vs_bmm": t_b / t_g, "speedup_vs_loop": t_l / t_g,
               "grouped_median50_ms": m_g, "padded_bmm_median50_ms": m_b,
               "grouped_median50_tflops": fl / m_g / 1e9, "padded_bmm_median50_tflops": fl / m_b / 1e9,
               "training_gemms": train}
        rows.append(row)
        print(json.dumps(row), flush=True)
        del x, w_ug, w_down, xp, y, a, bws
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "configs", "summary": True,
                      "grouped_beats_padded_bmm_everywhere": all(r["speedup_vs_bmm"] > 1 for r in rows),
                      "grouped_beats_host_loop_everywhere": all(r["speedup_vs_loop"] > 1 for r in rows)}),
          flush=True)
    return 0


def run_sweep_precision(args):
    """Price of the wgrads' precision scheme: the dual wgrad launch (dW_down and dW_ug) with both
    bf16 halves of its activation operand (P = w*A for the down projection, dU for the up/gate
    projection; two MMAs per K step) against the high half only (one MMA per K step), on the
    workloads with a backward. Operands come from the library's own forward and dgrad on the
    workload's routing with device-drawn N(0,1) inputs; mean of 20 launches queued in a CUDA
    graph after 10 warm-ups. The accuracy side of the trade is a GPU test against the oracle."""
    import torch
    from ragged_grouped_gemm_device_gb300 import _lib as L
    from ragged_grouped_gemm_device_gb300 import workloads as W
    L.load()
    dev, bf, i32 = "cuda", torch.bfloat16, torch.int32
    for name in ("finegrained", "skew", "large"):
        wl = W.make(name)
        T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
        gen = torch.Generator(device=dev).manual_seed(2)
        x = torch.randn(T, d, device=dev, generator=gen).to(bf)
        w_ug = (torch.randn(E, 2 * h, d, device=dev, generator=gen) * d ** -0.5).to(bf)
        w_down = (torch.randn(E, h, d, device=dev, generator=gen) * h ** -0.5).to(bf)
        ids = torch.from_numpy(wl.ids).to(dev)
        counts, offsets = torch.empty(E, dtype=i32, device=dev), torch.empty(E, dtype=i32, device=dev)
        ss, inv = torch.empty(n, dtype=i32, device=dev), torch.empty(n, dtype=i32, device=dev)
        rws = torch.empty(max(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), 1), dtype=torch.uint8, device=dev)
        xp = torch.empty(n, d, dtype=bf, device=dev)
        status = torch.zeros(1, dtype=i32, device=dev)
        L.moe_route_offsets(ids, T, k, E, counts, offsets, ss, inv, rws)
        L.moe_permute(x, ss, offsets, None, T, k, E, d, xp)
        a = torch.empty(n, h, dtype=bf, device=dev)
        sv = torch.empty(L.moe_workspace_bytes(L.OP_SAVED, T, k, E, d, h), dtype=torch.uint8, device=dev)
        L.moe_grouped_up_swiglu(xp, offsets, None, None, E, n, d, h, w_ug, a, sv, status)
        dy = torch.randn(n, d, device=dev, generator=gen).to(bf)
        du_hi, du_lo = torch.empty(n, 2 * h, dtype=bf, device=dev), torch.empty(n, 2 * h, dtype=bf, device=dev)
        L.moe_grouped_down_dgrad_swiglu(dy, sv, offsets, None, None, E, n, d, h, w_down, du_hi, du_lo, status)
        _, p_lo = L.saved_views(sv, n, h)
        dwd = torch.empty(E, h, d, device=dev)
        dwu = torch.empty(E, 2 * h, d, device=dev)
        t_hl = queued_mean_ms(lambda: L.moe_grouped_wgrad_dual(a, p_lo, h, dy, d, dwd, du_hi, du_lo, 2 * h, xp, d,
                                                               dwu, offsets, E, n, status))
        t_hi = queued_mean_ms(lambda: L.moe_grouped_wgrad_dual(a, None, h, dy, d, dwd, du_hi, None, 2 * h, xp, d,
                                                               dwu, offsets, E, n, status))
        torch.cuda.synchronize()
        assert status.item() == 0, f"device status {status.item()}"
        M = int(offsets[-1].item())
        fl = 6.0 * M * d * h
        # bytes the scheme adds per step beyond bf16 saved state: the low half of P written by the
        # forward and read by the down wgrad, U at 3 bytes instead of 2 (written by the forward,
        # read by the dgrad), the low half of dU written by the dgrad and read by the up wgrad
        extra = M * h * 2 * 2 + M * 2 * h * 1 * 2 + M * 2 * h * 2 * 2
        print(json.dumps({"sweep": "precision", "workload": name, "M": M, "E": E, "d": d, "h": h,
                          "wgrad_hi_lo_ms": t_hl, "wgrad_hi_only_ms": t_hi,
                          "wgrad_hi_lo_useful_tflops": fl / t_hl / 1e9, "wgrad_hi_only_tflops": fl / t_hi / 1e9,
                          "extra_state_bytes_per_step": extra,
                          "timing": "mean of 20 launches queued in a CUDA graph after 10 warm-ups"}), flush=True)
        del x, w_ug, w_down, xp, a, sv, dy, du_hi, du_lo, dwd, dwu
        torch.cuda.empty_cache()
    return 0


def run_sweep_accumulation(args):
    """How the fp32 accumulation of long contractions behaves: one expert of K rows through the
    bf16 wgrad (fp32 out, K = the rows), N(0,1) bf16 operands, against the exact sum (fp64) and
    two fp32 emulations that add each 16-product MMA step's partial sum into the accumulator
    rounded to nearest (RN) or toward zero (RZ). Up to K = 8192 the library's accumulator is the
    tensor core's own; longer contractions are summed in segments of 8192 added in RN fp32."""
    import numpy as np
    import torch
    from ragged_grouped_gemm_device_gb300 import _lib as L
    L.load()
    dev = "cuda"
    P = Q = 16
    rng = np.random.default_rng(1)
    for lg in (10, 12, 13, 14, 16, 18, 20):
        K = 1 << lg
        ta = torch.from_numpy(rng.standard_normal((K, P)).astype(np.float32)).to(torch.bfloat16)
        tb = torch.from_numpy(rng.standard_normal((K, Q)).astype(np.float32)).to(torch.bfloat16)
        a64, b64 = ta.double().numpy(), tb.double().numpy()
        offs = torch.tensor([K], dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        dw = torch.full((1, P, Q), float("nan"), device=dev)
        L.moe_grouped_wgrad(ta.to(dev), None, P, tb.to(dev), Q, offs, 1, K, dw, st)
        torch.cuda.synchronize()
        assert st.item() == 0, f"device status {st.item()}"
        got = dw[0].cpu().double().numpy()
        ref = a64.T @ b64
        rn = np.zeros((P, Q), np.float32)
        rz = np.zeros((P, Q), np.float32)
        for k0 in range(0, K, 16):
            part = a64[k0:k0 + 16].T @ b64[k0:k0 + 16]
            rn = (rn.astype(np.float64) + part).astype(np.float32)
            s_ = rz.astype(np.float64) + part
            f = s_.astype(np.float32)
            over = np.abs(f.astype(np.float64)) > np.abs(s_)
            f[over] = np.nextafter(f[over], np.float32(0))
            rz = f
        rms = lambda e: float(np.sqrt((e ** 2).mean()))
        print(json.dumps({"sweep": "accumulation", "K": K, "segmented": K > 8192,
                          "ref_rms": rms(ref), "gpu_err_rms": rms(got - ref),
                          "fp32_rn_err_rms": rms(rn.astype(np.float64) - ref),
                          "fp32_rz_err_rms": rms(rz.astype(np.float64) - ref),
                          "gpu_err_max": float(np.abs(got - ref).max())}), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep == "capacity":
        return run_sweep_capacity(args)
    if args.sweep == "histogram":
        return run_sweep_histogram(args)
    if args.sweep == "configs":
        return run_sweep_configs(args)
    if args.sweep == "oracle":
        return run_sweep_oracle(args)
    if args.sweep == "precision":
        return run_sweep_precision(args)
    if args.sweep == "accumulation":
        return run_sweep_accumulation(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
