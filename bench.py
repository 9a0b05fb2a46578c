"""Throughput of the fused GEMM hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one call of the hot path (one persistent-kernel launch through
the C ABI) over one batch of seeded synthetic input of the named workload
(default: 8192^3 bf16 GEMM + gelu_tanh writing D and PostAct, the shape the
70 % tensor-peak target is quoted on).  At N = 1 the same run also measures
the metric's other workloads (``per_config``: 256^3 bf16, 4096^3 bf16 + C +
GELU, 8192^3 and 16 x 2048^2 x 4096 fp16 ReLU, the varlen gather-A SiLU MoE
layer, 8192^3 fp8), each autotuned and timed on its own.
Inputs are resident in HBM; consecutive steps rotate over input sets whose
total size exceeds the 129 MB L2, so no step reads warm operands.  Device
time comes from CUDA events on the launching stream around exactly K steps,
bracketed by a barrier and a synchronize; rank 0 prints one JSON line.

Under torchrun (N > 1) each rank runs the same problem on its own GPU (the
problems are independent: weak scaling, no collective on the data path) and
the max time over ranks is used.

``--impl reference`` times the CPU oracle on the host cores on a bounded
sample of the same workload (the reference arm of this build).
"""

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from grouped_gemm_epilogues_gb300 import workloads as wl  # noqa: E402

METRIC = "TFLOP/s per GEMM shape and % of GB300 dense bf16/fp8 tensor peak (1 GPU)"
DEFAULT_WORKLOAD = "gemm_act_8192_bf16_gelu"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_PEAK = {"bf16": 2250.0, "f16": 2250.0, "e4m3": 4500.0, "e5m2": 4500.0}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, world_size, device=None):
    """The slowest rank's value (every rank gets it); no-op for one rank.
    Works on any process-group backend (a CUDA tensor for NCCL, CPU for gloo)."""
    if world_size <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step, world_size, ms_per_step):
    """Whole-job TFLOP/s: every rank runs its own problem per step (replicas,
    weak scaling), timed by the slowest rank."""
    return world_size * flops_per_step / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    """Hash of the device code (kernel headers and instantiation units, with
    // comments removed), so that recorded DRAM traffic is dropped as soon as the
    kernels change but survives edits of comments and of host-only code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "grouped_gemm_epilogues_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        device = name.endswith((".cuh", "params.h")) or name.startswith("gge_inst_")
        if not device:
            continue
        with open(os.path.join(csrc, name)) as f:
            lines = (line.split("//", 1)[0].rstrip() for line in f)
            code = "\n".join(line for line in lines if line)
        h.update(name.encode() + code.encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- our arm (GPU)

def _out_shape(w):
    if w.k_groups:
        return (w.k_groups, w.M, w.N)
    return (w.M, w.N) if w.groups else (w.L, w.M, w.N)


def _to_device(v, dev):
    """A device copy with the same strides (a transposed view stays transposed)."""
    d = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=dev)
    d.copy_(v)
    return d


def _rotate_rows(a, i):
    """Distinct values of the same distribution: roll the storage rows of A
    (the rows of its contiguous form; a transposed view is rolled underneath)."""
    t = a if a.is_contiguous() else a.transpose(-1, -2)
    r = torch.roll(t.view(torch.uint8), shifts=i, dims=-2).view(t.dtype).contiguous()
    return r if a.is_contiguous() else r.transpose(-1, -2)


def _device_sets(w, dev, n_sets, base=None):
    sets = []
    base = wl.make(w) if base is None else base
    for i in range(n_sets):
        s = {}
        for k, v in base.items():
            if isinstance(v, torch.Tensor):
                s[k] = _to_device(v, dev)
        if i > 0:
            s["A"] = _rotate_rows(s["A"], i)
        shape = _out_shape(w)
        if w.d_dtype:
            s["D"] = torch.empty(shape, dtype=wl.DT[w.d_dtype], device=dev)
        if w.p_dtype:
            s["P"] = torch.empty(shape, dtype=wl.DT[w.p_dtype], device=dev)
        sets.append(s)
    return base, sets


def _set_bytes(s):
    return sum(v.numel() * v.element_size() for v in s.values() if isinstance(v, torch.Tensor))


def _op_of(w):
    if w.k_groups:
        return "gather_k" if w.gather_rows else "varlen_k"
    if w.groups:
        return "gather_a" if w.gather_rows else "varlen_m"
    return "gemm"


def _step_fn(w, binding, config=None):
    def step(s):
        if w.k_groups and w.gather_rows:
            binding.gge_gemm_gather_k(s["A"], s["B"], s["a_idx"], s["cu_seqlens_k"],
                                      D=s.get("D"), PostAct=s.get("P"), act=w.act, C=s.get("C"),
                                      alpha=w.alpha, beta=w.beta, config=config)
        elif w.k_groups:
            binding.gge_gemm_varlen_k(s["A"], s["B"], s["cu_seqlens_k"], D=s.get("D"),
                                      PostAct=s.get("P"), act=w.act, C=s.get("C"),
                                      alpha=w.alpha, beta=w.beta, config=config)
        elif w.groups:
            if w.gather_rows:
                binding.gge_gemm_gather_a(s["A"], s["B"], s["a_idx"], s["cu_seqlens_m"],
                                          D=s.get("D"), PostAct=s.get("P"), act=w.act,
                                          C=s.get("C"), alpha=w.alpha, beta=w.beta, config=config)
            else:
                binding.gge_gemm_varlen_m(s["A"], s["B"], s["cu_seqlens_m"], D=s.get("D"),
                                          PostAct=s.get("P"), act=w.act, C=s.get("C"),
                                          alpha=w.alpha, beta=w.beta, config=config)
        elif w.act == "none" and "P" not in s:
            binding.gge_gemm(s["A"], s["B"], s["D"], C=s.get("C"), alpha=w.alpha, beta=w.beta, config=config)
        else:
            binding.gge_gemm_act(s["A"], s["B"], s["P"], w.act, D=s.get("D"), C=s.get("C"),
                                 alpha=w.alpha, beta=w.beta, config=config)
    return step


# The other workloads of the metric, measured in the same run (N = 1) next to the
# headline: (key, workload)
PER_CONFIG = [("c1", "gemm_256_bf16"), ("c2", "gemm_act_4096_bf16_gelu"),
              ("c3a", "gemm_8192_f16_relu"), ("c3b", "bgemm_2048x2048x4096x16_f16_relu"),
              ("c4", "varlen_gather_g64_m32768_silu"), ("c5", "gemm_8192_fp8")]


def _prepare(w, dev, binding, tune, fixed=None):
    """Rotating device input sets (their total above L2 where the problem allows),
    the launch configuration (autotuned unless tune is False) and the step."""
    base, probe = _device_sets(w, dev, 1)
    per_set = _set_bytes(probe[0])
    n_sets = max(2, int(np.ceil(2.5 * L2_BYTES / per_set)) + 1)
    n_sets = min(n_sets, 8)
    del probe
    _, sets = _device_sets(w, dev, n_sets, base)
    # launch shape: the autotuner's pick for this problem (tuning runs before the
    # warm-up and is not timed), or the planner's default
    tuned = None
    if tune:
        s0 = sets[0]
        tuned, _ = binding.gge_autotune(_op_of(w), s0["A"], s0["B"], idx=s0.get("a_idx"),
                                        cu=s0.get("cu_seqlens_k", s0.get("cu_seqlens_m")),
                                        C=s0.get("C"), D=s0.get("D"), PostAct=s0.get("P"),
                                        act=w.act, alpha=w.alpha, beta=w.beta, reps=5)
    if tuned is None and fixed:
        tuned = dict(fixed)
    step = _step_fn(w, binding, binding.make_config(**tuned) if tuned else None)
    l2 = (f"{n_sets} rotating input sets of {per_set / 2**20:.0f} MiB (> L2)"
          if n_sets * per_set > L2_BYTES else
          f"{n_sets} rotating input sets of {per_set / 2**20:.2f} MiB "
          "(whole working set < L2: L2-resident)")
    return base, sets, tuned, step, l2


def _graph_runner(step, sets, steps):
    """Exactly `steps` launches replayed from CUDA graphs (a graph of whole passes
    over the input sets, up to ~64 launches, then one for the remainder), without
    the per-call host cost of the Python binding in the way of small problems."""
    n_sets = len(sets)
    per_graph = n_sets * max(1, min(64 // n_sets, steps // n_sets))
    full, rem = divmod(steps, per_graph)
    graphs = []
    if full:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(per_graph):
                step(sets[i % n_sets])
        graphs += [g] * full
    if rem:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(rem):
                step(sets[i % n_sets])
        graphs.append(g)
    torch.cuda.synchronize()

    def run():
        for g in graphs:
            g.replay()
    run()  # warm the graphs once
    torch.cuda.synchronize()
    return run


def _settle(step, sets, seconds):
    """Extra untimed work so that clocks settle under load."""
    t_end = time.time() + seconds
    i = 0
    while time.time() < t_end:
        for _ in range(20):
            step(sets[i % len(sets)])
            i += 1
        torch.cuda.synchronize()


def _timed(step, sets, steps, stream, eager, barrier=lambda: None):
    """Device time (ms) of exactly `steps` steps, CUDA events on the launching
    stream, bracketed by a barrier and a synchronize on both sides."""
    runner = None if eager else _graph_runner(step, sets, steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    if runner is not None:
        runner()
    else:
        for i in range(steps):
            step(sets[i % len(sets)])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1)


def _peak_for(w, peaks, src):
    bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    is8 = w.ab_dtype in ("e4m3", "e5m2")
    return (bf16 * (2.0 if is8 else 1.0),
            f"{src} cuBLAS bf16 burst" + (" x2 (fp8/bf16 nominal ratio)" if is8 else ""))


def _sustained_frac(w, peaks, tflops):
    """Context beside `frac`: the same number against cuBLAS run back to back for
    seconds under the power cap (the timed region here follows 0.2-0.5 s of load)."""
    s = peaks.get("bf16_tflops_sustained")
    if not s:
        return None
    return round(tflops / (s * (2.0 if w.ab_dtype in ("e4m3", "e5m2") else 1.0)), 4)


def _fixed_shape(args):
    """A launch shape given on the command line (with --no-tune), or None."""
    d = json.loads(args.config_json) if args.config_json else {}
    d.update({k: v for k, v in (("cta_group", args.cta_group), ("tile_n", args.tile_n)) if v})
    d.pop("source", None)
    return d or None


def _shape_note(tuned, args):
    if tuned is None:
        return {"source": "planner default"}
    return dict(tuned, source="autotuned" if not args.no_tune else "command line")


def algorithmic_bytes(w, base):
    """Fewest HBM bytes one call must move: every operand read once and every
    output written once (varlen gather: the gathered rows, the B of each
    non-empty group and the indices)."""
    def nbytes(t):
        return t.numel() * t.element_size()
    out_el = (w.k_groups or 1) * w.M * w.N if w.k_groups else (w.M * w.N * (1 if w.groups else w.L))
    out = sum(out_el * wl.DT[d].itemsize for d in (w.d_dtype, w.p_dtype) if d)
    c = nbytes(base["C"]) if "C" in base else 0
    if w.groups:
        cu = base["cu_seqlens_m"].numpy()
        live = int((np.diff(cu) > 0).sum())
        b = nbytes(base["B"]) * live // w.groups
        a = w.M * w.K * base["A"].element_size()
        idx = nbytes(base["a_idx"]) if "a_idx" in base else 0
        return a + b + c + out + idx
    if w.k_groups and w.gather_rows:
        return w.K * w.M * base["A"].element_size() + nbytes(base["B"]) + c + out
    return nbytes(base["A"]) + nbytes(base["B"]) + c + out


def cublas_comparator(w, dev, local, steps):
    """torch.matmul (cuBLAS) on the same 16-bit plain problem, the product alone
    (no epilogue), as a context column, timed like our own runs: rotating input
    sets larger than L2, 0.5 s of untimed load first, then at least `steps`
    launches and ~0.3 s, clocks sampled meanwhile.  None for the other forms."""
    if w.groups or w.k_groups or w.ab_dtype not in ("bf16", "f16"):
        return None
    dt = wl.DT[w.ab_dtype]
    per_set = 2 * (w.L * w.M * w.K + w.L * w.K * w.N + w.L * w.M * w.N)
    n_sets = min(8, max(2, int(np.ceil(2.5 * L2_BYTES / per_set)) + 1))
    As = [torch.randn(w.L, w.M, w.K, device=dev).to(dt) for _ in range(n_sets)]
    Bs = [torch.randn(w.L, w.K, w.N, device=dev).to(dt) for _ in range(n_sets)]
    Ds = [torch.empty(w.L, w.M, w.N, device=dev, dtype=dt) for _ in range(n_sets)]

    def step(i):
        torch.matmul(As[i % n_sets], Bs[i % n_sets], out=Ds[i % n_sets])

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_end, i = time.time() + 0.5, 0
    while time.time() < t_end:
        for _ in range(20):
            step(i)
            i += 1
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for j in range(n_sets):
        step(j)
    e1.record()
    torch.cuda.synchronize()
    est = e0.elapsed_time(e1) / n_sets
    n = max(steps, int(np.ceil(300.0 / max(est, 1e-3))))
    e0.record()
    for j in range(n):
        step(j)
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / n
    del As, Bs, Ds
    torch.cuda.empty_cache()
    return {"value": round(w.flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 5), "steps": n, "clocks": clocks,
            "what": "torch.matmul of the same shape and dtype, no epilogue, timed like this "
                    "line (context only, not on the product path)"}


def measure_config(args, w, dev, binding, local, peaks, src):
    """One per-config line: autotuned shape, warm-up, then at least ~0.3 s of
    timed launches (at least --steps) with the clocks sampled meanwhile."""
    base, sets, tuned, step, l2 = _prepare(w, dev, binding, not args.no_tune)
    stream = torch.cuda.current_stream(dev)
    for i in range(max(args.warmup, len(sets))):
        step(sets[i % len(sets)])
    torch.cuda.synchronize()
    status = binding.gge_read_device_status(dev)
    if status[0] != "GGE_OK":
        raise RuntimeError(f"{w.name}: device status after warm-up: {status}")
    est = _timed(step, sets, len(sets), stream, True) / len(sets)
    steps = max(args.steps, int(np.ceil(300.0 / max(est, 1e-3))))
    sampler = ClockSampler(local)
    sampler.start()
    _settle(step, sets, 0.2)
    ms = _timed(step, sets, steps, stream, args.eager)
    clocks = sampler.stop()
    status = binding.gge_read_device_status(dev)
    if status[0] != "GGE_OK":
        raise RuntimeError(f"{w.name}: device status after the timed region: {status}")
    ms_per_step = ms / steps
    tflops = w.flops / (ms_per_step * 1e-3) / 1e12
    peak, peak_src = _peak_for(w, peaks, src)
    alg = algorithmic_bytes(w, base)
    hbm = alg / (ms_per_step * 1e-3) / 1e9
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out = {"workload": w.name, "value": round(tflops, 1), "unit": "TFLOP/s",
           "ms_per_step": round(ms_per_step, 5), "steps": steps,
           "frac": round(tflops / peak, 4), "peak": peak, "peak_source": peak_src,
           "frac_of_nominal_dense_peak": round(tflops / NOMINAL_PEAK[w.ab_dtype], 4),
           "frac_of_measured_sustained": _sustained_frac(w, peaks, tflops),
           "hbm": {"algorithmic_bytes": int(alg), "achieved_gbs": round(hbm, 1),
                   "peak_gbs": hbm_peak, "frac": round(hbm / hbm_peak, 4)},
           "traffic": profiled_traffic(w.name), "l2": l2, "clocks": clocks,
           "launch_shape": _shape_note(tuned, args)}
    del sets
    torch.cuda.empty_cache()
    out["cublas"] = cublas_comparator(w, dev, local, args.steps)
    return out


def run_ours(args, w):
    from grouped_gemm_epilogues_gb300 import binding

    ws_n, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    binding.load()

    base, sets, tuned, step, l2 = _prepare(w, dev, binding, not args.no_tune, _fixed_shape(args))
    n_sets = len(sets)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    sampler = ClockSampler(local)
    for i in range(args.warmup):
        step(sets[i % n_sets])
    torch.cuda.synchronize()
    status = binding.gge_read_device_status(dev)
    if status[0] != "GGE_OK":
        raise RuntimeError(f"device status after warm-up: {status}")

    sampler.start()
    _settle(step, sets, 0.5)
    ms = _timed(step, sets, args.steps, stream, args.eager, barrier)
    clocks = sampler.stop()
    status = binding.gge_read_device_status(dev)
    if status[0] != "GGE_OK":
        raise RuntimeError(f"device status after the timed region: {status}")
    ms_per_step = max_over_ranks(ms / args.steps, ws_n, dev)
    flops = w.flops
    value = job_throughput(flops, ws_n, ms_per_step)

    # end-to-end through the public API with host buffers
    e2e = run_e2e(args, w, base, dev, step)
    alg = algorithmic_bytes(w, base)

    peaks, src = measured_peaks()
    peak, peak_src = _peak_for(w, peaks, src)
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    roofline = {
        "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
        "frac": round(achieved / peak, 4), "traffic": profiled_traffic(w.name),
        "peak_source": peak_src,
        "frac_of_nominal_dense_peak": round(achieved / NOMINAL_PEAK[w.ab_dtype], 4),
        "frac_of_measured_sustained": _sustained_frac(w, peaks, achieved),
    }
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.ab_dtype if w.bdt == w.ab_dtype else f"{w.ab_dtype}x{w.bdt}",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "L": w.L,
                   "groups": w.groups, "gather_rows": w.gather_rows, "act": w.act,
                   **({"k_groups": w.k_groups, "a_major": w.a_major, "b_major": w.b_major}
                      if w.k_groups else {}),
                   "with_c": w.with_c, "alpha": w.alpha, "beta": w.beta,
                   "accumulate": "f32", "out": w.p_dtype or w.d_dtype,
                   "l2": l2,
                   "parallelism": f"replicas{ws_n}" if ws_n > 1 else "single",
                   "launch": "eager" if args.eager else "cuda_graph",
                   "launch_shape": _shape_note(tuned, args)},
        "roofline": roofline,
        "hbm": {"algorithmic_bytes": int(alg),
                "achieved_gbs": round(alg / (ms_per_step * 1e-3) / 1e9, 1)},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    del sets
    torch.cuda.empty_cache()
    if ws_n == 1:
        line["cublas"] = cublas_comparator(w, dev, local, args.steps)
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, base, budget_s=args.cpu_seconds)
    if ws_n == 1 and not args.no_per_config:
        line["per_config"] = {key: measure_config(args, wl.WORKLOADS[name], dev, binding, local,
                                                  peaks, src)
                              for key, name in PER_CONFIG}
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line, rank


def run_e2e(args, w, base, dev, step):
    """Same metric through the public API with host (pinned) buffers: every
    step copies its inputs host->device and its outputs device->host.  Steps
    are pipelined over two device buffer sets and three streams (inputs in,
    compute, results out), so the copies of one step overlap the GEMM of the
    next; the timed region spans the first input copy to the last result copy."""
    host_in = {}
    for k, v in base.items():
        if isinstance(v, torch.Tensor):   # pinned, in the same layout as the device copy
            h = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, pin_memory=True)
            host_in[k] = h.copy_(v)
    shape = _out_shape(w)
    bufs = []
    for _ in range(2):
        d = {k: torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=dev)
             for k, v in host_in.items()}
        if w.d_dtype:
            d["D"] = torch.empty(shape, dtype=wl.DT[w.d_dtype], device=dev)
        if w.p_dtype:
            d["P"] = torch.empty(shape, dtype=wl.DT[w.p_dtype], device=dev)
        bufs.append(d)
    out_keys = [k for k in ("D", "P") if k in bufs[0]]
    host_out = [{k: torch.empty(bufs[0][k].shape, dtype=bufs[0][k].dtype, pin_memory=True)
                 for k in out_keys} for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("in", "comp", "out")}
    used = [False, False]

    def one(i):
        b = i % 2
        d = bufs[b]
        if used[b]:   # buffer set b was last used two steps ago
            s_in.wait_event(ev["comp"][b])
        with torch.cuda.stream(s_in):
            for k, v in host_in.items():
                d[k].copy_(v, non_blocking=True)
            ev["in"][b].record(s_in)
        s_comp.wait_event(ev["in"][b])
        if used[b]:
            s_comp.wait_event(ev["out"][b])
        with torch.cuda.stream(s_comp):
            step(d)
            ev["comp"][b].record(s_comp)
        s_out.wait_event(ev["comp"][b])
        with torch.cuda.stream(s_out):
            for k in out_keys:
                host_out[b][k].copy_(d[k], non_blocking=True)
            ev["out"][b].record(s_out)
        used[b] = True

    n = max(3, min(args.steps, 50))
    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(3, 3 + n):
        one(i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"value": round(w.flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 4), "steps": n,
            "pipeline": "2 buffer sets, copy-in / compute / copy-out streams overlapped"}


# ------------------------------------------------------ the oracle (CPU)

def _oracle_rows(w, base, rows):
    """The oracle on a subset of output rows of the workload; returns the
    FLOPs that the sample covers."""
    from oracle import activations, formats, gemm as og

    def dec(t):
        t = t.contiguous()
        fmt = {torch.bfloat16: formats.BF16, torch.float16: formats.F16,
               torch.float8_e4m3fn: formats.E4M3, torch.float8_e5m2: formats.E5M2,
               torch.float32: formats.F32}[t.dtype]
        ity = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[fmt.nbytes]
        return formats.decode(t.view(ity).numpy(), fmt)

    fm = {"bf16": formats.BF16, "f16": formats.F16, "f32": formats.F32, None: None}
    kw = dict(alpha=w.alpha, beta=w.beta, act=w.act, d_fmt=fm[w.d_dtype], p_fmt=fm[w.p_dtype])
    if w.k_groups:
        # output rows m of every group: A's rows against all of B
        C = base["C"][:, rows] if "C" in base else None
        if w.gather_rows:
            og.gemm_gather_k(dec(base["A"][rows]), base["a_idx"].numpy(), dec(base["B"]),
                             base["cu_seqlens_k"].numpy(), None if C is None else dec(C), **kw)
        else:
            og.gemm_varlen_k(dec(base["A"][rows]), dec(base["B"]), base["cu_seqlens_k"].numpy(),
                             None if C is None else dec(C), **kw)
        cu = base["cu_seqlens_k"].numpy()
        return 2.0 * len(rows) * w.N * float(cu[-1] - cu[0])
    if w.groups:
        cu = base["cu_seqlens_m"].numpy()
        A = base["A"][base["a_idx"][rows].long()] if w.gather_rows else base["A"][rows]
        out_rows = 0
        B = base["B"]
        # rows of the sample grouped by their group
        g_of = np.searchsorted(cu, rows, side="right") - 1
        for g in np.unique(g_of):
            sel = np.nonzero(g_of == g)[0]
            og.gemm(dec(A[sel])[None], dec(B[g])[None], None, **kw)
            out_rows += len(sel)
        return 2.0 * out_rows * w.N * w.K
    A = base["A"][:, rows]
    C = base["C"][:, rows] if "C" in base else None
    og.gemm(dec(A), dec(base["B"]), None if C is None else dec(C), **kw)
    return 2.0 * len(rows) * w.N * w.K * w.L


def _rows_for_budget(w, base, budget_s):
    """Rows whose oracle run takes about budget_s: two probes separate the fixed
    cost (decoding B) from the per-row cost."""
    t0 = time.perf_counter()
    _oracle_rows(w, base, np.arange(min(w.M, 8)))
    t1 = time.perf_counter()
    _oracle_rows(w, base, np.arange(min(w.M, 72)))
    t2 = time.perf_counter()
    per_row = max((t2 - t1) - (t1 - t0), 1e-6) / max(1, min(w.M, 72) - min(w.M, 8))
    fixed = max((t1 - t0) - 8 * per_row, 0.0)
    return int(min(w.M, max(16, (budget_s - fixed) / per_row)))


def cpu_baseline(w, base, budget_s=15.0):
    """Time the oracle as it stands on the host cores over a bounded sample
    of the workload's output rows (about budget_s seconds of work)."""
    M = w.M
    n = _rows_for_budget(w, base, budget_s)
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(M, size=n, replace=False))
    t0 = time.perf_counter()
    f = _oracle_rows(w, base, rows)
    dt = time.perf_counter() - t0
    return {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} of {M} output rows (all N, K{', batches' if w.L > 1 else ''}), "
                      f"{f / 1e9:.1f} GFLOP in {dt:.1f} s, float64 numpy/BLAS"}


def run_reference(args, w):
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return None, rank
    base = wl.make(w)
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    n = _rows_for_budget(w, base, per_step)
    rng = np.random.default_rng(0)
    samples = [np.sort(rng.choice(w.M, size=n, replace=False))
               for _ in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        _oracle_rows(w, base, samples[i])
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(args.steps):
        flops += _oracle_rows(w, base, samples[args.warmup + i])
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    ms_per_step = dt * 1e3 / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "L": w.L},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"{n} of {w.M} output rows per step, float64 numpy/BLAS"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line, rank


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-tune", action="store_true",
                    help="use the planner's default launch shape instead of the autotuner's")
    ap.add_argument("--eager", action="store_true",
                    help="launch every timed step from Python instead of CUDA-graph replay")
    ap.add_argument("--cta-group", type=int, default=0,
                    help="with --no-tune: CTAs per tile (1, or 2 for a CTA pair)")
    ap.add_argument("--tile-n", type=int, default=0, help="with --no-tune: tile width")
    ap.add_argument("--config-json", default="",
                    help="with --no-tune: a whole launch configuration (gge_config fields as "
                         "JSON, e.g. a launch_shape this script printed)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-config lines (the other workloads of the metric)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        line, rank = run_reference(args, w)
    else:
        line, rank = run_ours(args, w)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
