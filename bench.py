"""Benchmark of the NVFP4 W4A4 linear on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch: the four decoder
linears of a Qwen3-32B-shaped layer (qkv 5120->10240, o 8192->5120,
gate_up 5120->51200, down 25600->5120) at M = 16384 tokens, activations with
0.1% outlier channels scaled x50, each through nvfp4_linear (activation
quantization + block-scaled FP4 GEMM with the alpha/bias/bf16 epilogue).  This
is the largest layer workload that fits one GPU.  Weights are prepared once,
outside the timed region.  --workload llama times the Llama-3.1-8B-shaped
layer (qkv 4096->6144, o 4096->4096, gate_up 4096->28672, down 14336->4096)
at M = 8192 instead; the default line also carries that step as
`llama_m8192`.

  value      whole-job NVFP4-linear throughput, sum(2*M*N*K) / time, with the
             inputs resident in HBM (per-rank inputs of 1.4 GB: larger than L2)
  roofline   the GEMM kernel: its algorithmic FLOPs / its own CUDA-event time,
             against the dense-FP4 peak (measured burst bf16 peak x the
             nominal FP4:bf16 ratio 13.5/2.25 = 6: the kernel is timed by CUDA
             events inside a sub-second region)
  act_quant  the activation quantizer: algorithmic bytes / its CUDA-event time
             with a cold, clean L2 (a 256 MB read before each launch), against the
             measured HBM copy bandwidth; `in_pipeline` gives the same kernel timed
             right after the previous layer's GEMM
  e2e        the same metric through nvfp4_linear with the activation copied in
             from pinned host memory and the output copied back, every step
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
             (sampled rows x sampled output columns of each linear), one
             single-threaded process per host core

--suite prints, instead of the headline line, one JSON line per layer problem
of every workload (Llama / Qwen / padded-K / transform: quantizer, GEMM and
nvfp4_linear timed alone with a cold L2) and per point of the sweeps
(quantizer, transform quantizer at large M, dynamic global scale, MXFP4
quantizer).  --case runs one kernel a few times on synthetic data, for ncu.

--impl reference times that oracle as the reference arm.  Under torchrun
(N > 1) every rank runs its own batch (weak scaling, no data-path collective);
only the barrier and the max-over-ranks time reduction touch the network.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 linear TFLOP/s (frac of FP4 peak); act-quant GB/s (frac of HBM peak)"
# name -> (description, default tokens per GPU, problem generator of synthetic.py)
WORKLOADS = {
    "qwen": ("qwen3-32b decoder linears qkv/o/gate_up/down, 0.1% outlier channels x50", 16384, "qwen"),
    "llama": ("llama3.1-8b decoder linears qkv/o/gate_up/down", 8192, "llama"),
}
DEFAULT_WORKLOAD = "qwen"
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 : bf16 tensor rate of GB300
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CPU_SAMPLE_ROWS = 16                 # cpu_baseline sample: rows x columns of every linear
CPU_SAMPLE_COLS = 1024
REF_STEP_ROWS = CPU_SAMPLE_ROWS      # reference arm: the cpu_baseline sample, one per step
REF_STEP_COLS = CPU_SAMPLE_COLS
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "gemm_qwen_gate_up_m16384_traffic.txt")


# ------------------------------------------------------------ host logic ----

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--m", type=int, default=None, help="tokens per rank (default: the workload's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--case", choices=["quant", "gemm", "linear", "step"],
                    help="run one kernel on synthetic data a few times and exit (for ncu captures): "
                         "--m/--k/--n/--bs choose the shape, --steps the launches; 'step': the --workload's "
                         "layers at --m through nvfp4_linear, --steps times")
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--bs", type=int, default=0, help="--case: transform block size (0 = none)")
    ap.add_argument("--suite", action="store_true",
                    help="instead of the headline line: one JSON line per layer problem of every workload "
                         "(Llama/Qwen/padded-K/transform) and per point of the quantization sweep")
    a = ap.parse_args(argv)
    a.warmup = max(a.warmup, 3)
    if a.m is None:
        a.m = WORKLOADS[a.workload][1] if a.case in (None, "step") else 8192
    return a


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_seed(seed: int, rank: int) -> int:
    """Each rank draws its own activations (data-parallel over tokens)."""
    return seed + 7919 * rank


def max_over_ranks(v: float, device) -> float:
    """Slowest rank's time (all ranks call this; a no-op without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    return per_rank_units * world / max_seconds


def layer_problems(workload: str, m: int, rank: int = 0):
    from nvfp4_quantized_linear_gb300 import synthetic as syn
    make = getattr(syn, WORKLOADS[workload][2])
    return [syn.Problem(p.workload, p.name, p.m, p.k, p.n, seed=rank_seed(p.seed, rank), x_kind=p.x_kind)
            for p in make([m])]


def workload_label(workload: str, m: int) -> str:
    return f"{WORKLOADS[workload][0]}, M={m} tokens per GPU"


def quant_bytes(m: int, k: int) -> int:
    """Algorithmic bytes of one activation quantization: bf16 read, packed FP4
    and tiled scales written."""
    kp = (k + 31) // 32 * 32
    mp = (m + 127) // 128 * 128
    nbp = (kp // 16 + 3) // 4 * 4
    return 2 * m * k + m * kp // 2 + mp * nbp


def gemm_bytes(p) -> int:
    """Algorithmic bytes of one GEMM launch: packed operands, their scales, bf16 output."""
    kp = (p.k + 31) // 32 * 32
    nbp = (kp // 16 + 3) // 4 * 4
    mp, np_ = (p.m + 127) // 128 * 128, (p.n + 127) // 128 * 128
    return p.m * kp // 2 + mp * nbp + p.n * kp // 2 + np_ * nbp + 2 * p.m * p.n_keep


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "MEASURED_PEAKS.json (measured)"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "profiling-recipe fallback"


def gemm_source_hash() -> str:
    """Fingerprint of the headline's dominant kernel (the CTA-pair GEMM): its
    translation unit and the headers it includes."""
    h = hashlib.sha256()
    for name in ("gemm_pair.cu", "gemm_common.cuh", "ptx.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "nvfp4_quantized_linear_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic_record(path: str = None):
    """(gemm_source_hash, DRAM bytes per launch) of a committed ncu traffic
    summary, or None if it is missing or unreadable."""
    try:
        with open(path or PROFILE_TRAFFIC) as f:
            kv = dict(line.split(":", 1) for line in f if ":" in line and not line.startswith("#"))
        return kv["gemm_source_hash"].strip(), float(kv["dram_bytes_per_launch"].strip())
    except (OSError, KeyError, ValueError):
        return None


def recorded_traffic():
    """DRAM bytes of one gate_up GEMM launch of the headline workload from the
    committed ncu summary, if it was taken on the current GEMM source; else
    None (a record of another kernel revision says nothing about this one)."""
    rec = read_traffic_record()
    if rec is None or rec[0] != gemm_source_hash():
        return None
    return rec[1]


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=10)
        self.file.flush()

    def summary(self):
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None),
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- oracle ----

class OracleSample:
    """The CPU oracle on `rows` activation rows x `cols` output columns of each
    linear (weights of the sampled columns quantized once, untimed)."""

    def __init__(self, problems, rows: int, cols: int, seed: int = 0):
        import numpy as np
        import oracle
        from nvfp4_quantized_linear_gb300 import synthetic as syn
        oracle.build()
        self.oracle, self.np = oracle, np
        self.layers = []
        rng = np.random.default_rng(seed)
        for p in problems:
            # the sampled activation rows and weight rows are drawn with the
            # layer's own generators, so they are the same tensors the GPU sees
            x = syn.make_activation(p, device="cpu", m=min(p.m, 4 * rows))
            w = syn.bf16_normal((p.n, p.k), 0.02, p.seed + 100_000)
            c = np.sort(rng.choice(p.n, size=min(cols, p.n), replace=False))
            gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
            b, sb = oracle.quantize(syn.bf16_bits(w[c]), gs_w)
            self.layers.append(dict(p=p, x=syn.bf16_bits(x), b=b, sb=sb, gs_x=gs_x, alpha=syn.alpha_of(gs_x, gs_w),
                                    ncols=len(c)))
        self.rows = rows

    def flops(self) -> int:
        return sum(2 * self.rows * L["ncols"] * L["p"].k for L in self.layers)

    def run(self, step: int = 0):
        for L in self.layers:
            n = L["x"].shape[0]
            r = [(step * self.rows + i) % n for i in range(self.rows)]
            a, sa = self.oracle.quantize(L["x"][r], L["gs_x"])
            self.oracle.gemm(a, sa, L["b"], L["sb"], L["alpha"])


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_pass(layers, rows: int, step: int):
    """One pass of the oracle over its sample (the body of OracleSample.run)."""
    import oracle
    for L in layers:
        n = L["x"].shape[0]
        r = [(step * rows + i) % n for i in range(rows)]
        a, sa = oracle.quantize(L["x"][r], L["gs_x"])
        oracle.gemm(a, sa, L["b"], L["sb"], L["alpha"])


def _oracle_worker(layers, rows, steps, warmup, min_seconds, barrier, results):
    """A spawned oracle process: warm-up passes, then (after every process is
    ready) `steps` timed passes, or passes for min_seconds when steps is None."""
    for s in range(warmup):
        _oracle_pass(layers, rows, s)
    barrier.wait()
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_pass(layers, rows, warmup + reps)
        reps += 1
        el = time.perf_counter() - t0
        if (steps is not None and reps >= steps) or (steps is None and (el >= min_seconds or reps >= 200)):
            break
    results.put((reps, el))


def time_oracle(sample: OracleSample, procs: int, steps: int | None = None, warmup: int = 1,
                min_seconds: float = 10.0):
    """The oracle as it stands, in `procs` spawned processes at once, one per
    host core, each running the same sample.  Returns (TFLOP/s of all of them
    over the slowest one's time, that time, passes per process)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")                 # never fork a process that has touched the GPU
    barrier, results = ctx.Barrier(procs), ctx.Queue()
    # only arrays and scalars go to the processes (no torch import there)
    layers = [{key: L[key] for key in ("x", "b", "sb", "gs_x", "alpha")} for L in sample.layers]
    ps = [ctx.Process(target=_oracle_worker, args=(layers, sample.rows, steps, warmup, min_seconds, barrier, results))
          for _ in range(procs)]
    for p in ps:
        p.start()
    out = [results.get(timeout=1800) for _ in ps]
    for p in ps:
        p.join(timeout=60)
    el = max(e for _, e in out)
    reps = min(r for r, _ in out)
    return sample.flops() * sum(r for r, _ in out) / el / 1e12, el, reps


# ------------------------------------------------------------------ GPU ----

def setup_layers(problems, dev):
    """Device tensors of every layer problem: activation, prepared weight,
    scales, workspace (whose head doubles as the quantizer's output in the
    per-kernel pass) and output."""
    import torch

    import nvfp4_quantized_linear_gb300 as nv
    from nvfp4_quantized_linear_gb300 import synthetic as syn
    layers = []
    for p in problems:
        L = syn.make_layer(p, device=dev)
        gs_x = torch.tensor([L.gs_x], dtype=torch.float32, device=dev)
        gs_w = torch.tensor([L.gs_w], dtype=torch.float32, device=dev)
        alpha = torch.tensor([L.alpha], dtype=torch.float32, device=dev)
        w_fp4, w_sf = nv.prepare_weight(L.w, gs_w)
        ws = torch.empty(nv.nvfp4_linear_workspace_bytes(p.m, p.k, p.n), dtype=torch.uint8, device=dev)
        kp = nv.padded_k(p.k)
        a_fp4 = ws[:p.m * kp // 2]
        a_sf = ws[(p.m * kp // 2 + 255) // 256 * 256:]
        out = torch.empty((p.m, p.n), dtype=torch.bfloat16, device=dev)
        layers.append(dict(p=p, x=L.x, gs_x=gs_x, alpha=alpha, w_fp4=w_fp4, w_sf=w_sf, ws=ws, a_fp4=a_fp4,
                           a_sf=a_sf, out=out))
        del L
    torch.cuda.synchronize()
    return layers


def measure_step(layers, args, stream, barrier):
    """(A) the step through nvfp4_linear, K times: its time per step; (B) the
    same kernels launched one by one, each bracketed by CUDA events on the
    launching stream: per-kernel durations; (C) the quantizer alone with a
    cold, clean L2.  Returns the times in seconds."""
    import torch

    import nvfp4_quantized_linear_gb300 as nv

    def linear(l):
        p = l["p"]
        nv.nvfp4_linear(l["x"], p.m, p.k, p.k, l["gs_x"], None, 0, l["w_fp4"], l["w_sf"], p.n, p.n, l["alpha"],
                        None, l["out"], p.n, l["ws"], l["ws"].numel(), stream)

    def split(l, ev):
        p = l["p"]
        ev[0].record()
        nv.nvfp4_quant_act(l["x"], p.m, p.k, p.k, l["gs_x"], None, 0, l["a_fp4"], l["a_sf"], stream)
        ev[1].record()
        nv.nvfp4_gemm(l["a_fp4"], l["a_sf"], p.m, l["w_fp4"], l["w_sf"], p.n, p.n, p.k, l["alpha"], None,
                      l["out"], p.n, stream)
        ev[2].record()

    for _ in range(args.warmup):
        for l in layers:
            linear(l)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    # (A)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        for l in layers:
            linear(l)
    e1.record()
    torch.cuda.synchronize()
    barrier()
    t_step = e0.elapsed_time(e1) / 1e3 / args.steps
    # (B)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in layers] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        for i, l in enumerate(layers):
            split(l, evs[s][i])
    torch.cuda.synchronize()
    barrier()
    # (C) reading 256 MB first evicts what the previous kernel left (the GEMM's
    # dirty output would otherwise be written back while the quantizer streams)
    cold = torch.empty(64 << 20, dtype=torch.float32, device=layers[0]["x"].device)
    cold.zero_()
    cold.sum()                          # writes the zeros back: later reads leave clean lines
    qevs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in layers]
            for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s in range(args.steps):
        for i, l in enumerate(layers):
            p = l["p"]
            cold.sum()
            qevs[s][i][0].record()
            nv.nvfp4_quant_act(l["x"], p.m, p.k, p.k, l["gs_x"], None, 0, l["a_fp4"], l["a_sf"], stream)
            qevs[s][i][1].record()
    torch.cuda.synchronize()
    del cold
    nv.nvfp4_device_error()
    n = len(layers)
    return {
        "step": t_step,
        "quant": [sum(evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(args.steps)) / args.steps / 1e3
                  for i in range(n)],
        "gemm": [sum(evs[s][i][1].elapsed_time(evs[s][i][2]) for s in range(args.steps)) / args.steps / 1e3
                 for i in range(n)],
        "quant_cold": [sum(qevs[s][i][0].elapsed_time(qevs[s][i][1]) for s in range(args.steps)) / args.steps / 1e3
                       for i in range(n)],
    }


def per_layer_rows(layers, t):
    return [{"layer": l["p"].name, "m": l["p"].m, "k": l["p"].k, "n": l["p"].n,
             "quant_us": round(tq * 1e6, 2), "quant_us_in_pipeline": round(tqp * 1e6, 2),
             "gemm_us": round(tg * 1e6, 2), "gemm_tflops": round(l["p"].flops / tg / 1e12, 1),
             "quant_gbs": round(quant_bytes(l["p"].m, l["p"].k) / tq / 1e9, 1)}
            for l, tq, tqp, tg in zip(layers, t["quant_cold"], t["quant"], t["gemm"])]


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import nvfp4_quantized_linear_gb300 as nv

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nv.build()
    ok, why = nv.nvfp4_is_supported(local_rank)
    if not ok:
        raise RuntimeError(why)
    peaks, peak_src = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16                 # burst: a kernel timed alone
    fp4_peak_sustained = peaks["bf16_tflops_sustained"] * FP4_OVER_BF16

    def barrier():
        if world > 1:
            dist.barrier()

    def slowest(v: float) -> float:
        return max_over_ranks(v, dev)

    layers = setup_layers(layer_problems(args.workload, args.m, rank), dev)
    stream = torch.cuda.current_stream().cuda_stream
    flops_step = sum(l["p"].flops for l in layers)
    sampler = ClockSampler(local_rank)
    with sampler:
        t = measure_step(layers, args, stream, barrier)
    clocks = sampler.summary()

    t_step_max = slowest(t["step"])
    value = aggregate(flops_step, world, t_step_max) / 1e12
    gemm_tflops = flops_step / sum(t["gemm"]) / 1e12
    top = max(range(len(layers)), key=lambda i: t["gemm"][i])          # the dominant launch (gate_up)
    top_tflops = layers[top]["p"].flops / t["gemm"][top] / 1e12
    q_bytes = sum(quant_bytes(l["p"].m, l["p"].k) for l in layers)
    quant_gbs = q_bytes / sum(t["quant_cold"]) / 1e9
    quant_gbs_pipe = q_bytes / sum(t["quant"]) / 1e9
    traffic = recorded_traffic() if (args.workload, args.m) == (DEFAULT_WORKLOAD, WORKLOADS[DEFAULT_WORKLOAD][1]) \
        else None
    top_kernel = "gemm_nvf4_pair_kernel" if layers[top]["p"].m > 128 else "gemm_nvf4_kernel"

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step_max * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4",
        "data": "synthetic",
        "config": {"workload": workload_label(args.workload, args.m),
                   "m": args.m, "layers": [[l["p"].name, l["p"].k, l["p"].n] for l in layers],
                   "l2": f"inputs larger than L2 ({sum(l['x'].numel() * 2 for l in layers) / 1e9:.2f} GB of "
                         "activations per step)", "bias": False, "transform": None},
        "roofline": {"bound": "tensor", "kernel": f"{top_kernel} ({layers[top]['p'].name} launch)",
                     "achieved": round(top_tflops, 2), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(top_tflops / fp4_peak, 4),
                     "traffic": (round(traffic) if traffic else None),
                     "algorithmic_bytes": gemm_bytes(layers[top]["p"]),
                     "flops_per_launch": layers[top]["p"].flops,
                     "all_gemm_launches_achieved": round(gemm_tflops, 2),
                     "peak_note": (f"dense FP4 = burst bf16 {peaks.get('bf16_tflops')} x {FP4_OVER_BF16:g} from "
                                   f"{peak_src}: the kernel is timed by CUDA events in a sub-second region at the "
                                   "clocks in 'clocks'.  Sustained-based peak "
                                   f"{fp4_peak_sustained:.0f} (frac_of_sustained: the figure for a seconds-long "
                                   "loop; the Qwen gate_up GEMM back to back takes about 1223 us a launch for its "
                                   "first 20 launches and 1394 us after 80, at the power cap), nominal 13500"),
                     "frac_of_sustained": round(top_tflops / fp4_peak_sustained, 4),
                     "frac_of_nominal_13p5": round(top_tflops / 13500.0, 4)},
        "act_quant": {"bound": "hbm", "kernel": "quant_kernel", "achieved": round(quant_gbs, 1),
                      "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(quant_gbs / peaks["hbm_gbs"], 4),
                      "bytes_per_step": q_bytes,
                      "l2": "cold and clean: a 256 MB read before each launch",
                      "in_pipeline": {"achieved": round(quant_gbs_pipe, 1),
                                      "frac": round(quant_gbs_pipe / peaks["hbm_gbs"], 4),
                                      "note": "each launch right after the previous layer's GEMM, whose output "
                                              "is still being written back from L2"}},
        "per_layer": per_layer_rows(layers, t),
        "gpu_launches": 2 * len(layers) * args.steps,
        "clocks": clocks,
    }

    if not args.no_e2e:
        result["e2e"] = run_e2e(args, layers, flops_step, barrier, slowest, world, stream)
    del layers
    torch.cuda.empty_cache()
    if args.workload == DEFAULT_WORKLOAD and not args.no_sweep:
        # the Llama-3.1-8B-shaped step at M = 8192 (the smaller prefill workload)
        sec = setup_layers(layer_problems("llama", 8192, rank), dev)
        sampler2 = ClockSampler(local_rank)
        with sampler2:
            t2 = measure_step(sec, args, stream, barrier)
        f2 = sum(l["p"].flops for l in sec)
        top2 = max(range(len(sec)), key=lambda i: t2["gemm"][i])
        result["llama_m8192"] = {
            "workload": workload_label("llama", 8192),
            "value": round(aggregate(f2, world, slowest(t2["step"])) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(t2["step"] * 1e3, 4),
            "gate_up_gemm_tflops": round(sec[top2]["p"].flops / t2["gemm"][top2] / 1e12, 2),
            "gate_up_frac": round(sec[top2]["p"].flops / t2["gemm"][top2] / 1e12 / fp4_peak, 4),
            "per_layer": per_layer_rows(sec, t2), "clocks": sampler2.summary()}
        result["gpu_launches"] += 2 * len(sec) * args.steps
        del sec
        torch.cuda.empty_cache()
    if not args.no_sweep:
        result["m_sweep"] = run_sweep(args, rank, dev, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(layer_problems(args.workload, args.m, 0), CPU_SAMPLE_ROWS, CPU_SAMPLE_COLS)
        cores = host_cores()
        v, el, reps = time_oracle(sample, cores)
        result["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                  "sample": f"{CPU_SAMPLE_ROWS} rows x {CPU_SAMPLE_COLS} output columns of each of "
                                            f"the 4 linears (act quant + FP64 GEMM) per pass, one single-threaded "
                                            f"process per core, >= {reps} passes each in {el:.1f} s"}
    return result


def _cpu_list(text: str) -> set:
    """The CPUs of a sysfs list such as "0-3,8,10-11"."""
    cpus = set()
    for part in text.strip().split(","):
        if part:
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def gpu_local_cpus(torch, dev) -> set:
    """The CPUs on the GPU's own NUMA node (its PCI device's local_cpulist in
    sysfs) that this process may run on; empty when that cannot be read.
    Pinned host buffers are placed on the node of the thread that first
    touches them, and copies to and from a remote node cross the CPUs'
    interconnect too."""
    try:
        props = torch.cuda.get_device_properties(dev)
        bus = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            return _cpu_list(f.read()) & os.sched_getaffinity(0)
    except (AttributeError, OSError, ValueError, RuntimeError):
        return set()


def run_e2e(args, layers, flops_step, barrier, slowest, world, stream):
    """Through the public API with host buffers: every step copies every layer's
    activation in from pinned host memory, runs nvfp4_linear and copies its
    output back to pinned host memory, all inside the timed region.  As a
    serving pipeline runs it, the copies in, the linears and the copies out
    go on three streams ordered by events, with two device buffers per
    activation and output, so that one layer's (or step's) copies overlap
    another's compute; the link's two directions run concurrently."""
    import torch

    import nvfp4_quantized_linear_gb300 as nv
    steps = max(3, min(args.steps, 10))
    # the host side of the copies on the GPU's NUMA node, where the node can be read
    allowed = os.sched_getaffinity(0)
    local = gpu_local_cpus(torch, torch.cuda.current_device())
    if local and local != allowed:
        os.sched_setaffinity(0, local)
    host_cpus = (f"{len(local)} of {len(allowed)} usable CPUs, the GPU's NUMA node" if local
                 else f"{len(allowed)} usable CPUs (the GPU's NUMA node unknown)")
    hx = [l["x"].cpu().pin_memory() for l in layers]
    ho = [torch.empty(l["out"].shape, dtype=torch.bfloat16).pin_memory() for l in layers]
    h2d = sum(h.numel() * 2 for h in hx)
    d2h = sum(h.numel() * 2 for h in ho)
    xbuf = [[l["x"] for l in layers], [torch.empty_like(l["x"]) for l in layers]]          # [buffer][layer]
    obuf = [[l["out"] for l in layers], [torch.empty_like(l["out"]) for l in layers]]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    ev_in = [[ev() for _ in layers] for _ in range(2)]
    ev_cmp = [[None for _ in layers] for _ in range(2)]      # the linear that read xbuf[b][i] / wrote obuf[b][i]
    ev_out = [[None for _ in layers] for _ in range(2)]      # the copy that read obuf[b][i]

    def step(sidx):
        b = sidx & 1
        for i, l in enumerate(layers):
            p = l["p"]
            with torch.cuda.stream(s_in):
                if ev_cmp[b][i] is not None:
                    s_in.wait_event(ev_cmp[b][i])               # the linear two steps back has read xbuf[b][i]
                xbuf[b][i].copy_(hx[i], non_blocking=True)
                ev_in[b][i].record(s_in)
            s_cmp.wait_event(ev_in[b][i])
            if ev_out[b][i] is not None:
                s_cmp.wait_event(ev_out[b][i])                  # obuf[b][i] has been copied out
            nv.nvfp4_linear(xbuf[b][i], p.m, p.k, p.k, l["gs_x"], None, 0, l["w_fp4"], l["w_sf"], p.n, p.n,
                            l["alpha"], None, obuf[b][i], p.n, l["ws"], l["ws"].numel(), s_cmp.cuda_stream)
            e = ev()
            e.record(s_cmp)
            ev_cmp[b][i] = e
            with torch.cuda.stream(s_out):
                s_out.wait_event(e)
                ho[i].copy_(obuf[b][i], non_blocking=True)
                eo = ev()
                eo.record(s_out)
                ev_out[b][i] = eo

    def join():
        s_cmp.wait_stream(s_in)
        s_cmp.wait_stream(s_out)

    step(0)
    step(1)
    join()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_cmp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for sidx in range(steps):
        step(sidx)
    join()
    e1.record(s_cmp)
    torch.cuda.synchronize()
    barrier()
    t = slowest(e0.elapsed_time(e1) / 1e3 / steps)
    os.sched_setaffinity(0, allowed)
    return {"value": round(aggregate(flops_step, world, t) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(t * 1e3, 3),
            "pipeline": "copies in, nvfp4_linear and copies out on three streams, two device buffers per "
                        "activation and output",
            "host_cpus": host_cpus}


def run_sweep(args, rank, dev, stream):
    """Decode/prefill-size breakdown: the four Llama-3.1-8B-shaped linears at
    smaller M (not the headline value)."""
    import torch

    import nvfp4_quantized_linear_gb300 as nv
    from nvfp4_quantized_linear_gb300 import synthetic as syn
    out = []
    # a 256 MB read before each timed step evicts the previous step's lines
    # (clean ones: a write-based flush would leave write-backs to compete)
    flush = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
    for m in [1, 16, 128, 1024]:
        layers = []
        for p in layer_problems("llama", m, rank):
            L = syn.make_layer(p, device=dev)
            gs_x = torch.tensor([L.gs_x], dtype=torch.float32, device=dev)
            alpha = torch.tensor([L.alpha], dtype=torch.float32, device=dev)
            w_fp4, w_sf = nv.prepare_weight(L.w, torch.tensor([L.gs_w], dtype=torch.float32, device=dev))
            ws = torch.empty(nv.nvfp4_linear_workspace_bytes(p.m, p.k, p.n), dtype=torch.uint8, device=dev)
            o = torch.empty((p.m, p.n), dtype=torch.bfloat16, device=dev)
            layers.append((p, L.x, gs_x, alpha, w_fp4, w_sf, ws, o))

        def step(s):
            for p, x, gs_x, alpha, w_fp4, w_sf, ws, o in layers:
                nv.nvfp4_linear(x, p.m, p.k, p.k, gs_x, None, 0, w_fp4, w_sf, p.n, p.n, alpha, None, o, p.n,
                                ws, ws.numel(), s)

        for _ in range(3):
            step(stream)
        torch.cuda.synchronize()
        # The step as a serving engine runs it: captured once in a CUDA graph
        # and replayed (the CPU does not issue each launch).
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step(side.cuda_stream)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        # The four layers' weights (~116 MB of FP4 + scales) would stay in the
        # 129 MB L2 across back-to-back steps; a real decoder streams them from
        # HBM, so L2 is flushed before every timed step.
        iters = 30
        timings = {}
        for mode in ("graph", "eager"):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
            for e0, e1 in evs:
                flush.sum()
                e0.record()
                if mode == "graph":
                    graph.replay()
                else:
                    step(stream)
                e1.record()
            torch.cuda.synchronize()
            timings[mode] = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
        nv.nvfp4_device_error()
        t = timings["graph"]
        flops = sum(p.flops for p, *_ in layers)
        wbytes = sum(w.numel() + s.numel() for _, _, _, _, w, s, _, _ in layers)
        abytes = sum(quant_bytes(p.m, p.k) + 2 * p.m * p.n for p, *_ in layers)
        out.append({"workload": "llama3.1-8b", "m": m, "us_per_step": round(t * 1e6, 2),
                    "tflops": round(flops / t / 1e12, 2), "algorithmic_gbs": round((wbytes + abytes) / t / 1e9, 1),
                    "us_per_step_eager": round(timings["eager"] * 1e6, 2),
                    "launch": "CUDA graph replay of the 4-layer step (eager launches: us_per_step_eager)",
                    "l2": "256 MB read before each step"})
        del layers, graph
    return out


def _cold_timer(torch, dev, iters: int = 15, warm: int = 3):
    """Median CUDA-event time of fn() with a clean, cold L2 before every launch
    (a 256 MB read evicts what the previous launch left behind)."""
    cold = torch.zeros(64 << 20, dtype=torch.float32, device=dev)

    def timed(fn) -> float:
        for _ in range(warm):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        for e0, e1 in evs:
            cold.sum()
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
    return timed


def run_suite(args, dev):
    """Every layer problem of the workloads, timed kernel by kernel with a cold
    L2: the activation quantizer (with the block-diagonal transform where the
    workload has one), the GEMM on pre-quantized operands, and nvfp4_linear end
    to end; then the quantizer bandwidth sweep.  Yields one dict per row."""
    import torch

    import nvfp4_quantized_linear_gb300 as nv
    from nvfp4_quantized_linear_gb300 import synthetic as syn
    nv.build()
    peaks, _ = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16          # burst: each kernel is timed alone
    hbm = peaks["hbm_gbs"]
    stream = torch.cuda.current_stream().cuda_stream
    timed = _cold_timer(torch, dev)
    f32 = dict(dtype=torch.float32, device=dev)

    problems = syn.llama() + syn.qwen() + syn.padded() + syn.transform_fused()
    for p in problems:
        L = syn.make_layer(p, device=dev)
        gs_x, gs_w, alpha = (torch.tensor([v], **f32) for v in (L.gs_x, L.gs_w, L.alpha))
        w_fp4, w_sf = nv.prepare_weight(L.w, gs_w)
        L.w = None
        ws = torch.empty(nv.nvfp4_linear_workspace_bytes(p.m, p.k, p.n), dtype=torch.uint8, device=dev)
        kp = nv.padded_k(p.k)
        a_fp4 = ws[:p.m * kp // 2]
        a_sf = ws[(p.m * kp // 2 + 255) // 256 * 256:]
        out = torch.empty((p.m, p.n_keep), dtype=torch.bfloat16, device=dev)
        t, bs = L.t, p.bs

        def quant():
            nv.nvfp4_quant_act(L.x, p.m, p.k, p.k, gs_x, t, bs, a_fp4, a_sf, stream)

        def gemm():
            nv.nvfp4_gemm(a_fp4, a_sf, p.m, w_fp4, w_sf, p.n, p.n_keep, p.k, alpha, L.bias, out, p.n_keep, stream)

        def linear():
            nv.nvfp4_linear(L.x, p.m, p.k, p.k, gs_x, t, bs, w_fp4, w_sf, p.n, p.n_keep, alpha, L.bias, out,
                            p.n_keep, ws, ws.numel(), stream)

        tq, tg, tl = timed(quant), timed(gemm), timed(linear)
        nv.nvfp4_device_error()
        qb, gb = quant_bytes(p.m, p.k), gemm_bytes(p)
        yield {"suite": p.workload, "layer": p.name, "m": p.m, "k": p.k, "n": p.n_keep, "bs": bs,
               "bias": p.bias,
               "quant_us": round(tq * 1e6, 2), "quant_gbs": round(qb / tq / 1e9, 1),
               "quant_frac_hbm": round(qb / tq / 1e9 / hbm, 4),
               "gemm_us": round(tg * 1e6, 2), "gemm_tflops": round(p.flops / tg / 1e12, 1),
               "gemm_frac_fp4": round(p.flops / tg / 1e12 / fp4_peak, 4),
               "gemm_gbs": round(gb / tg / 1e9, 1), "gemm_frac_hbm": round(gb / tg / 1e9 / hbm, 4),
               "linear_us": round(tl * 1e6, 2), "linear_tflops": round(p.flops / tl / 1e12, 1)}
        del L, w_fp4, w_sf, ws, a_fp4, a_sf, out
        torch.cuda.empty_cache()

    # the transform quantizer at sizes far above L2 (steady state), and the
    # dynamic global scale: its amax pass alone and followed by the quantizer
    for m, bs in [(16384, 16), (16384, 128), (65536, 16), (65536, 128)]:
        x = syn.bf16_normal((m, 4096), 1.0, 4600 + bs, device=dev)
        t = syn.random_hadamard_transform(bs, seed=bs).to(dev)
        gs = torch.tensor([30.0], **f32)
        x_fp4, x_sf = nv.quant_act(x, gs, t, bs)
        tq = timed(lambda: nv.nvfp4_quant_act(x, m, 4096, 4096, gs, t, bs, x_fp4, x_sf, stream))
        nv.nvfp4_device_error()
        qb = quant_bytes(m, 4096)
        yield {"suite": "transform_sweep", "m": m, "k": 4096, "bs": bs, "quant_us": round(tq * 1e6, 2),
               "quant_gbs": round(qb / tq / 1e9, 1), "quant_frac_hbm": round(qb / tq / 1e9 / hbm, 4)}
        del x, x_fp4, x_sf
        torch.cuda.empty_cache()
    for m, k, bs in [(8192, 4096, 0), (8192, 14336, 0), (65536, 16384, 0), (4096, 4096, 128), (65536, 4096, 128)]:
        x = syn.bf16_normal((m, k), 1.0, 4700 + m % 1000 + bs, device=dev)
        t = syn.random_hadamard_transform(bs, seed=bs).to(dev) if bs else None
        gs = torch.empty(1, **f32)
        x_fp4, x_sf = nv.quant_act(x, torch.tensor([30.0], **f32), t, bs)

        def amax_pass():
            nv.nvfp4_act_global_scale(x, m, k, k, t, bs, None, gs, None, stream)

        def dynamic_quant():
            amax_pass()
            nv.nvfp4_quant_act(x, m, k, k, gs, t, bs, x_fp4, x_sf, stream)

        ta, td = timed(amax_pass), timed(dynamic_quant)
        nv.nvfp4_device_error()
        yield {"suite": "global_scale", "m": m, "k": k, "bs": bs, "amax_us": round(ta * 1e6, 2),
               "amax_read_gbs": round(2 * m * k / ta / 1e9, 1), "amax_frac_hbm": round(2 * m * k / ta / 1e9 / hbm, 4),
               "dynamic_quant_us": round(td * 1e6, 2),
               "note": "amax pass (read of x, memset and finalize launches included), then the quantizer"}
        del x, x_fp4, x_sf
        torch.cuda.empty_cache()

    # MXFP4 GEMM and linear on the largest layers of the Llama and Qwen
    # workloads (operands quantized by the MXFP4 quantizer, no alpha)
    for p in [q for q in syn.llama([8192]) + syn.qwen([16384]) if q.name in ("gate_up", "down")]:
        x = syn.make_activation(p, device=dev)
        w = syn.bf16_normal((p.n, p.k), 0.02, p.seed + 100_000, device=dev)
        a_fp4, a_sf = nv.quant_act_mx(x)
        w_fp4, w_sf = nv.quant_act_mx(w)
        del w
        out = torch.empty((p.m, p.n), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_mxfp4_linear_workspace_bytes(p.m, p.k, p.n), dtype=torch.uint8, device=dev)
        tg = timed(lambda: nv.nvfp4_mxfp4_gemm(a_fp4, a_sf, p.m, w_fp4, w_sf, p.n, p.n, p.k, None, out, p.n, stream))
        tl = timed(lambda: nv.nvfp4_mxfp4_linear(x, p.m, p.k, p.k, w_fp4, w_sf, p.n, p.n, None, out, p.n, ws,
                                                 ws.numel(), stream))
        nv.nvfp4_device_error()
        yield {"suite": "mxfp4_gemm", "workload": p.workload, "layer": p.name, "m": p.m, "k": p.k, "n": p.n,
               "gemm_us": round(tg * 1e6, 2), "gemm_tflops": round(p.flops / tg / 1e12, 1),
               "gemm_frac_fp4": round(p.flops / tg / 1e12 / fp4_peak, 4),
               "linear_us": round(tl * 1e6, 2), "linear_tflops": round(p.flops / tl / 1e12, 1)}
        del x, a_fp4, a_sf, w_fp4, w_sf, out, ws
        torch.cuda.empty_cache()

    # grouped (mixture-of-experts) GEMM: 8 experts, about 1000 tokens each
    # (a prefill batch routed top-2), K = 4096 -> N = 2 x 14336 / 8 per expert
    group_m = [1000, 1200, 880, 1024, 1111, 960, 1030, 990]
    gk, gn = 4096, 3584
    offs = [0]
    for gm in group_m:
        offs.append(offs[-1] + (gm + 127) // 128 * 128)
    rows = offs[-1]
    x = syn.bf16_normal((rows, gk), 1.0, 4900, device=dev)
    w = syn.bf16_normal((len(group_m) * gn, gk), 0.02, 4901, device=dev)
    a_fp4, a_sf = nv.quant_act(x, torch.tensor([30.0], **f32))
    w_fp4, w_sf = nv.prepare_weight(w, torch.tensor([syn.global_scale(w)], **f32))
    del w
    offsets = torch.tensor(offs, dtype=torch.int32, device=dev)
    alphas = torch.full((len(group_m),), 1e-3, **f32)
    out = torch.empty((rows, gn), dtype=torch.bfloat16, device=dev)
    tg = timed(lambda: nv.nvfp4_grouped_gemm(a_fp4, a_sf, rows, offsets, len(group_m), w_fp4, w_sf, gn, gk, alphas,
                                             None, out, gn, stream))
    nv.nvfp4_device_error()
    flops = 2 * sum(group_m) * gn * gk
    yield {"suite": "grouped_gemm", "groups": len(group_m), "tokens": sum(group_m), "rows_padded": rows, "k": gk,
           "n": gn, "gemm_us": round(tg * 1e6, 2), "tflops": round(flops / tg / 1e12, 1),
           "frac_fp4": round(flops / tg / 1e12 / fp4_peak, 4),
           "note": "FLOPs of the real tokens; the padding rows of each group's last band are computed too"}
    del x, a_fp4, a_sf, w_fp4, w_sf, out
    torch.cuda.empty_cache()

    # MXFP4 activation quantization (block 32, E8M0 scales, no global scale)
    for m, k in [(8192, 4096), (8192, 14336), (65536, 16384)]:
        x = syn.bf16_normal((m, k), 1.0, 4800 + m % 1000, device=dev)
        x_fp4, x_sf = nv.quant_act_mx(x)
        tq = timed(lambda: nv.nvfp4_mxfp4_quant_act(x, m, k, k, x_fp4, x_sf, stream))
        nv.nvfp4_device_error()
        qb = 2 * m * k + m * nv.padded_k(k) // 2 + nv.nvfp4_mxfp4_scale_bytes(m, k)
        yield {"suite": "mxfp4_quant", "m": m, "k": k, "quant_us": round(tq * 1e6, 2),
               "quant_gbs": round(qb / tq / 1e9, 1), "quant_frac_hbm": round(qb / tq / 1e9 / hbm, 4), "bytes": qb}
        del x, x_fp4, x_sf
        torch.cuda.empty_cache()

    for m, k, seed in syn.quant_sweep():
        x = syn.bf16_normal((m, k), 1.0, seed, device=dev)
        gs = torch.tensor([syn.global_scale(x)], **f32)
        x_fp4, x_sf = nv.quant_act(x, gs)
        tq = timed(lambda: nv.nvfp4_quant_act(x, m, k, k, gs, None, 0, x_fp4, x_sf, stream))
        nv.nvfp4_device_error()
        qb = quant_bytes(m, k)
        yield {"suite": "quant_sweep", "m": m, "k": k, "quant_us": round(tq * 1e6, 2),
               "quant_gbs": round(qb / tq / 1e9, 1), "quant_frac_hbm": round(qb / tq / 1e9 / hbm, 4),
               "bytes": qb}
        del x, x_fp4, x_sf
        torch.cuda.empty_cache()


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample of
    the same workload per step (rank 0 only)."""
    if rank != 0:
        return None
    sample = OracleSample(layer_problems(args.workload, args.m, 0), REF_STEP_ROWS, REF_STEP_COLS)
    cores = host_cores()
    value, el, _ = time_oracle(sample, cores, steps=args.steps, warmup=args.warmup)
    desc = (f"{REF_STEP_ROWS} rows x {REF_STEP_COLS} output columns of each of the 4 linears "
            f"(act quant + FP64 GEMM) per pass; a step is one pass in each of {cores} single-threaded "
            "processes, one per host core")
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_label(args.workload, args.m), "m": args.m, "sample": desc},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_case(args):
    """One kernel on a synthetic N(0, 1) activation [M, K] (transformed by a
    random bs x bs Hadamard block when --bs > 0) and an N(0, 0.02) weight
    [N, K], launched --steps times; or ('step') the workload's layers at --m
    through nvfp4_linear, --steps times.  Prints 'ok'."""
    import torch

    import nvfp4_quantized_linear_gb300 as nv
    from nvfp4_quantized_linear_gb300 import synthetic as syn
    nv.build()
    dev = torch.device("cuda", 0)
    if args.case == "step":
        layers = setup_layers(layer_problems(args.workload, args.m, 0), dev)
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(args.steps):
            for l in layers:
                p = l["p"]
                nv.nvfp4_linear(l["x"], p.m, p.k, p.k, l["gs_x"], None, 0, l["w_fp4"], l["w_sf"], p.n, p.n,
                                l["alpha"], None, l["out"], p.n, l["ws"], l["ws"].numel(), stream)
        torch.cuda.synchronize()
        nv.nvfp4_device_error()
        print("ok")
        return
    m, k, n, bs = args.m, args.k, args.n, args.bs
    x = syn.bf16_normal((m, k), 1.0, 3, device=dev)
    t = syn.random_hadamard_transform(bs, seed=bs).to(dev) if bs else None
    gs = torch.tensor([30.0], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    x_fp4, x_sf = nv.quant_act(x, gs, t, bs)
    if args.case != "quant":
        w = syn.bf16_normal((n, k), 0.02, 4, device=dev)
        w_fp4, w_sf = nv.prepare_weight(w, torch.tensor([syn.global_scale(w)], dtype=torch.float32, device=dev))
        alpha = torch.tensor([1e-3], dtype=torch.float32, device=dev)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_linear_workspace_bytes(m, k, n), dtype=torch.uint8, device=dev)
    for _ in range(args.steps):
        if args.case == "quant":
            nv.nvfp4_quant_act(x, m, k, k, gs, t, bs, x_fp4, x_sf, stream)
        elif args.case == "gemm":
            nv.nvfp4_gemm(x_fp4, x_sf, m, w_fp4, w_sf, n, n, k, alpha, None, out, n, stream)
        else:
            nv.nvfp4_linear(x, m, k, k, gs, t, bs, w_fp4, w_sf, n, n, alpha, None, out, n, ws, ws.numel(), stream)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    print("ok")


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if args.case:
        run_case(args)
        return
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.suite:
        import torch
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        sampler = ClockSampler(local_rank)
        with sampler:
            for row in run_suite(args, dev):
                print(json.dumps(row), flush=True)
        print(json.dumps({"suite": "clocks", **sampler.summary(), "l2": "256 MB read before every launch; "
                          "median of 15 launches after 3 warm-up"}), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
