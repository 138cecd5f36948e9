#!/usr/bin/env python
"""Benchmark of the FP8 linear-layer hot path on GB300.

One step = one training step of a linear layer with bias + tanh-GELU at
tokens m = 8192, in-features k = 4096, out-features n = 14336: five fp8 casts
(X and W rows e4m3, dY rows e5m2, dZ^T e5m2 and X^T e4m3 down the token axis),
the forward GEMM (bias + GELU, pre-activation kept), the data-gradient GEMM
(GELU derivative + bias-gradient column sums) and the accumulating fp32
weight-gradient GEMM.  Metric: FP8 GEMM TFLOPS = 3 * 2 m n k per step / step
time (casts included in the time).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs an
independent replica of the step on its own GPU (no collective on the data
path); the value is the work of all ranks over the slowest rank's time.
--impl reference times the CPU oracle (test infrastructure, fp64) on a
bounded slice of the same step on the host cores.
"""
import argparse
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

M_TOK, K_IN, N_OUT = 8192, 4096, 14336
SEED = 1002  # base seed of the training-step workload
WORKLOAD = "linear_train_step_m8192_k4096_n14336_bias_gelu"
METRIC = "FP8 GEMM TFLOPS (fprop/dgrad/wgrad) and % of GB300 dense-FP8 peak, 1 GPU"
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor-core ratio on this part
KERNEL_SOURCES = ("gemm_kernel.cuh", "ptx.cuh", "common.cuh", "cast_rule.cuh", "gemm_params.h", "gemm_fprop.cu", "gemm_dgrad.cu",
                  "gemm_wgrad.cu")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "gemm_fp8_kernel_m8192_k4096_n14336_traffic.md")
# the CTA-pair kernels share the epilogue sources of the 1x128 kernel
RECIPE_SOURCES = {"block128": KERNEL_SOURCES,
                  "mx": KERNEL_SOURCES[:5] + ("gemm_mx.cu",),
                  "tensor": KERNEL_SOURCES[:5] + ("gemm_tensor.cu",)}
RECIPE_TRAFFIC = {"mx": os.path.join(ROOT, "profiles", "gemm_mx_kernel_m8192_k4096_n14336_traffic.md"),
                  "tensor": os.path.join(ROOT, "profiles", "gemm_tensor_kernel_m8192_k4096_n14336_traffic.md")}


def kernel_source_digest(recipe="block128"):
    """sha256 over the recipe's GEMM kernel source files (a DRAM-traffic
    summary applies only to the build it was measured on)."""
    import hashlib
    h = hashlib.sha256()
    for name in RECIPE_SOURCES[recipe]:
        with open(os.path.join(ROOT, "fp8_linear_layer_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(recipe="block128"):
    """DRAM bytes per GEMM launch (dram__bytes_read.sum + dram__bytes_write.sum,
    averaged over the step's three launches) from the recipe's committed ncu
    summary, or None when its kernel sources changed since it was taken."""
    import re
    try:
        text = open(TRAFFIC_SUMMARY if recipe == "block128" else RECIPE_TRAFFIC[recipe]).read()
    except OSError:
        return None
    sha = re.search(r"sources_sha256:\s*([0-9a-f]{64})", text)
    val = re.search(r"bytes_per_launch:\s*([0-9]+)", text)
    if not sha or not val or sha.group(1) != kernel_source_digest(recipe):
        return None
    return int(val.group(1))


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--acc", choices=["full", "fast"], default="full")
    ap.add_argument("--recipe", choices=["block128", "mx", "tensor"], default="block128",
                    help="block128: one fp32 scale per 128 elements, promoted in software (the configured "
                         "workload); mx: MXFP8, one power-of-two scale per 32 elements applied by the tensor core; "
                         "tensor: one scale per tensor (delayed scaling), scaled once after the K loop")
    ap.add_argument("--bias-grad", choices=["cast", "dgrad", "operand"], default="cast",
                    help="1x128 step: db from the transposed cast of dZ (default), from the data-gradient GEMM's "
                         "epilogue, or reduced from the weight-gradient GEMM's fp8 operand dZ^T")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--nvtx", action="store_true",
                    help="name every launch of the step with an NVTX range (for an external profiler's "
                         "timeline; adds host work, so not for timed runs)")
    ap.add_argument("--e2e-copy-weights", action="store_true",
                    help="end-to-end leg: copy W and b from the host every step as well")
    ap.add_argument("--e2e-read-dw", action="store_true",
                    help="end-to-end leg: read the fp32 dW back every step as well (235 MB at the default size)")
    ap.add_argument("--m", type=int, default=M_TOK, help="tokens (default: the training-step workload)")
    ap.add_argument("--k", type=int, default=K_IN, help="in-features")
    ap.add_argument("--n", type=int, default=N_OUT, help="out-features")
    ap.add_argument("--study", choices=["long_k", "kernels", "fp8_peak", "wgrad_tables", "mx", "tensor", "casts",
                                        "input_grad"],
                    default=None,
                    help="long_k: forward GEMM M=N=16384 at long K with 1%% outlier rows, FULL vs FAST, "
                         "TFLOPS and max normalized error vs the oracle on sampled 256x256 tiles")
    ap.add_argument("--study-k", type=int, default=16384)
    ap.add_argument("--reps", type=int, default=10, help="timed launches per kernel in --study casts")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device=None):
    """The slowest rank's number (all ranks get it); the value itself at N = 1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tflops(world, flops_per_step, steps, ms):
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return world * flops_per_step * steps / (ms / 1e3) / 1e12


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]) * FP8_OVER_BF16, float(p["hbm_gbs"]), "of measured"
    except Exception:
        return 1900.0 * FP8_OVER_BF16, 6800.0, "of fallback"


def inputs(device, m=M_TOK, k=K_IN, n=N_OUT):
    import workloads
    X = workloads.normal_bf16((m, k), SEED, "X")
    W = workloads.normal_bf16((n, k), SEED, "W", std=0.02)
    b = workloads.normal_bf16((n,), SEED, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), SEED, "dY", std=1e-2)
    host = [t.pin_memory() for t in (X, W, b, dY)] if device.type == "cuda" else [X, W, b, dY]
    return host


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        # samples under load: power above the midpoint of the observed range
        if pw and len(pw) == len(rows):
            lo, hi = min(pw), max(pw)
            loaded = [num(r[1]) for r in rows if num(r[3]) >= lo + 0.5 * (hi - lo)]
        else:
            loaded = sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(num(r[2]) or 0 for r in rows), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def cpu_sample_inputs(tokens, feats):
    """bf16 bit patterns of a `tokens` x `feats` slice of the step's inputs."""
    import workloads
    X = workloads.normal_bf16((M_TOK, K_IN), SEED, "X")[:tokens]
    W = workloads.normal_bf16((N_OUT, K_IN), SEED, "W", std=0.02)[:feats]
    b = workloads.normal_bf16((N_OUT,), SEED, "b", std=0.02)[:feats]
    dY = workloads.normal_bf16((M_TOK, K_IN), SEED, "dY", std=1e-2)[:tokens]
    return tuple(workloads.bits(t) for t in (X, W, b, dY))


def cpu_step(xb, wb, bb, dyb):
    """The oracle, as it stands, through the same step: 5 casts, 3 fp64 GEMMs
    (with their sum|a b| side outputs) and the epilogues.  Returns seconds."""
    import oracle
    t0 = time.perf_counter()
    qx, sx = oracle.quantize(xb, oracle.E4M3)
    qw, sw = oracle.quantize(wb, oracle.E4M3)
    acc, _ = oracle.gemm(qx, sx, oracle.E4M3, qw, sw, oracle.E4M3)
    Z, Y = oracle.fprop_epilogue(acc, bb)
    zb = oracle.f64_to_bf16_array(Z)
    qdy, sdy = oracle.quantize(dyb, oracle.E5M2)
    acc2, _ = oracle.gemm(qdy, sdy, oracle.E5M2, qw, sw, oracle.E4M3)
    dZ = oracle.dgrad_epilogue(acc2, zb)
    dzb = oracle.f64_to_bf16_array(dZ)
    oracle.colsum(oracle.bf16_to_f64(dzb))  # db of the stored bf16 dZ, as the step takes it by default
    qdzt, sdzt = oracle.quantize(dzb, oracle.E5M2, transpose=True)
    qxt, sxt = oracle.quantize(xb, oracle.E4M3, transpose=True)
    oracle.gemm(qdzt, sdzt, oracle.E5M2, qxt, sxt, oracle.E4M3)
    return time.perf_counter() - t0


def sample_text(tokens, feats):
    flops = 3 * 2 * tokens * feats * K_IN
    return ("%d-token x %d-feature slice of the step (k=%d): 5 casts + 3 fp64 GEMMs with |a||b| sums + "
            "epilogues, %.1f GFLOP" % (tokens, feats, K_IN, flops / 1e9))


def cpu_baseline_sample(tokens=512, feats=N_OUT):
    """Oracle throughput on one slice of the step.  Returns (TFLOP/s, seconds, cores, sample text)."""
    import oracle
    ins = cpu_sample_inputs(tokens, feats)
    dt = cpu_step(*ins)
    flops = 3 * 2 * tokens * feats * K_IN
    return flops / dt / 1e12, dt, oracle.num_threads(), sample_text(tokens, feats)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    tokens, feats = 128, 1024
    ins = cpu_sample_inputs(tokens, feats)
    for _ in range(args.warmup):
        cpu_step(*ins)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_step(*ins)
    total = time.perf_counter() - t0
    cores, sample = oracle.num_threads(), sample_text(tokens, feats)
    flops = 3 * 2 * tokens * feats * K_IN
    value = flops * args.steps / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "reference": "CPU oracle (fp64, OpenMP)"},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def nvtx_named(name, fn):
    """fn wrapped in an NVTX range of that name."""
    import torch

    def wrapped():
        torch.cuda.nvtx.range_push(name)
        try:
            fn()
        finally:
            torch.cuda.nvtx.range_pop()
    return wrapped


def run_e2e(args, step, host, dev_in, stream, barrier, world, dev):
    """The same step through the public API with host buffers: each step copies
    its batch (X, dY) from pinned host memory and reads its result back, all
    inside the timed region.  The layer's parameters W and b stay on the device
    as in training, where the optimizer updates them there (--e2e-copy-weights
    copies them every step as well); the result read back is the bias gradient
    db (dW stays on the device for the optimizer; --e2e-read-dw reads the
    235 MB fp32 dW back every step as well).  The
    copies run on their own streams so that they overlap the neighbouring
    steps' kernels: inputs alternate between two device buffer sets (step i+1's
    inputs arrive while step i computes), and a dW read back goes through a
    device snapshot that is copied to the host while the next step computes
    (the next snapshot waits for that read-back)."""
    import torch
    hX, hW, hb, hdY = host
    flops_step = step.gemm_flops
    sets = [tuple(dev_in), tuple(torch.empty_like(t) for t in dev_in)]
    copy_w = args.e2e_copy_weights
    per_step = (0, 1, 2, 3) if copy_w else (0, 3)  # which of X, W, b, dY cross the link each step
    for t in range(4):
        if t not in per_step:
            sets[1][t].copy_(sets[0][t])  # resident parameters in both buffer sets
    plans = [step.launches(*s) for s in sets]
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    set_free = [torch.cuda.Event() for _ in range(2)]
    out_done = torch.cuda.Event()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    read_dw = args.e2e_read_dw
    h_dW = torch.empty(step.dW.shape, dtype=torch.float32).pin_memory() if read_dw else None
    h_db = torch.empty(step.db.shape, dtype=torch.float32).pin_memory()
    dW_snap = torch.empty_like(step.dW) if read_dw else None
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize()
    barrier()
    ev0.record(stream)
    copy_in.wait_event(ev0)
    copy_out.wait_event(ev0)
    for i in range(e2e_steps):
        s = i % 2
        with torch.cuda.stream(copy_in):
            if i >= 2:
                copy_in.wait_event(set_free[s])
            for t in per_step:
                sets[s][t].copy_((hX, hW, hb, hdY)[t], non_blocking=True)
            in_ready[s].record(copy_in)
        stream.wait_event(in_ready[s])
        for _, fn in plans[s]:
            fn()
        set_free[s].record(stream)
        # db (57 KB) is read back on the compute stream before the next step's
        # data-gradient GEMM rewrites it; dW (235 MB) goes to a device snapshot
        # (once the previous snapshot has been read back) and from there to the
        # host on the copy stream
        h_db.copy_(step.db, non_blocking=True)
        if read_dw:
            if i >= 1:
                stream.wait_event(out_done)
            dW_snap.copy_(step.dW)
            step_done = torch.cuda.Event()
            step_done.record(stream)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(step_done)
                h_dW.copy_(dW_snap, non_blocking=True)
                out_done.record(copy_out)
    if read_dw:
        stream.wait_event(out_done)
    ev1.record(stream)
    ev1.synchronize()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    h2d = sum((hX, hW, hb, hdY)[t].numel() * (hX, hW, hb, hdY)[t].element_size() for t in per_step)
    d2h = (h_dW.numel() * 4 if read_dw else 0) + h_db.numel() * 4
    e2e_value = tflops(world, flops_step, e2e_steps, e2e_ms)
    return {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": e2e_steps, "copied_in": "X, W, b, dY" if copy_w else "X, dY (W, b resident)",
            "result_read_back": "db and dW" if read_dw else "db (dW stays on the device)",
            "overlap": "copies on separate streams, two input buffer sets"
                       + (", dW read back from a device snapshot" if read_dw else "")}


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import fp8_linear_layer_gb300 as fp8
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    fp8.lib()
    acc_mode = fp8.ACC_FAST if args.acc == "fast" else fp8.ACC_FULL

    m, k, n = args.m, args.k, args.n
    default_size = (m, k, n) == (M_TOK, K_IN, N_OUT)
    hX, hW, hb, hdY = inputs(dev, m, k, n)
    X, W, b, dY = (t.to(dev, non_blocking=True) for t in (hX, hW, hb, hdY))
    if args.recipe == "mx":
        from fp8_linear_layer_gb300.linear import MxLinearTrainStep
        if args.bias_grad == "operand":
            raise SystemExit("--bias-grad operand reduces 1x128-scaled operands only")
        step = MxLinearTrainStep(m, k, n, dev, bias_grad=args.bias_grad)
    elif args.recipe == "tensor":
        from fp8_linear_layer_gb300.linear import TensorLinearTrainStep
        step = TensorLinearTrainStep(m, k, n, dev)
    else:
        step = LinearTrainStep(m, k, n, dev, acc_mode, bias_grad=args.bias_grad)
    launches = step.launches(X, W, b, dY)
    if args.nvtx:
        launches = [(kind, nvtx_named("%d:%s" % (j, kind), fn)) for j, (kind, fn) in enumerate(launches)]
    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        for _, fn in launches:
            fn()
    torch.cuda.synchronize()
    if fp8.device_status() != 0:
        raise RuntimeError("device status not ok after warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---------------------------------------------------------- timed region
    n_gemm = sum(1 for kind, _ in launches if kind == "gemm")
    gemm_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps * n_gemm)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    start.record(stream)
    gi = 0
    for _ in range(args.steps):
        for kind, fn in launches:
            if kind == "gemm":
                gemm_ev[gi][0].record(stream)
                fn()
                gemm_ev[gi][1].record(stream)
                gi += 1
            else:
                fn()
    end.record(stream)
    end.synchronize()
    clk = clocks.stop()
    barrier()
    ms = max_over_ranks(start.elapsed_time(end), world, dev)
    gemm_ms = [a.elapsed_time(b_) for a, b_ in gemm_ev]
    status = fp8.device_status()
    if status != 0:
        raise RuntimeError("device status %d after the timed region" % status)

    flops_step = step.gemm_flops
    value = tflops(world, flops_step, args.steps, ms)
    fp8_peak, hbm_peak, peak_src = peaks()
    per_gemm_flops = 2 * m * n * k
    avg_gemm_ms = sum(gemm_ms) / len(gemm_ms)
    achieved = per_gemm_flops / (avg_gemm_ms / 1e3) / 1e12

    # ------------------------------------------------ end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, step, (hX, hW, hb, hdY), (X, W, b, dY), stream, barrier, world, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and default_size and args.recipe == "block128":
        v, dt, cores, sample = cpu_baseline_sample()
        cpu = {"value": v, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8(e4m3/e5m2) x fp8 -> fp32 accumulate", "data": "synthetic",
            "config": {"workload": (WORKLOAD if default_size else "linear_train_step_m%d_k%d_n%d_bias_gelu" % (m, k, n))
                       + {"block128": "", "mx": "_mxfp8", "tensor": "_per_tensor_delayed"}[args.recipe]
                       + ({"cast": "", "dgrad": "_bgrad_in_dgrad_epilogue", "operand": "_bgrad_from_operand"}[
                           args.bias_grad]
                          if args.recipe in ("block128", "mx") else ""),
                       "m_tokens": m, "k_in": k, "n_out": n,
                       "acc_mode": args.acc if args.recipe == "block128" else None, "recipe": args.recipe,
                       "bias_grad": getattr(step, "bias_grad", "dgrad"),
                       # what the timed data-gradient GEMM's epilogue does (the per-GEMM
                       # figure of the bias-gradient epilogue is bench.py --study kernels')
                       "dgrad_epilogue": "dGELU + bias-gradient column sums"
                       if getattr(step, "bias_grad", "dgrad") == "dgrad"
                       else "dGELU only (db taken %s)" % {"cast": "in dZ's transposed cast",
                                                          "operand": "from dZ^T's fp8 codes"}[step.bias_grad],
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "working set ~1.3 GB per step >> 129 MB L2 (no flush needed)",
                       "pct_of_fp8_peak": 100.0 * value / world / fp8_peak},
            "roofline": {"bound": "tensor", "kernel": {"block128": "gemm_fp8_kernel", "mx": "gemm_mx_kernel",
                                                       "tensor": "gemm_tensor_kernel (CTA pairs)"}[args.recipe]
                         + " (fprop, dgrad, wgrad launches)",
                         "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                         "peak_source": "%s bf16 burst x %.0f (nominal fp8/bf16 ratio)" % (peak_src, FP8_OVER_BF16),
                         # the summaries were taken on the default step of each recipe
                         "traffic": measured_traffic(args.recipe)
                         if default_size and (args.recipe == "tensor" or args.bias_grad == "cast") else None,
                         "traffic_unit": "bytes",
                         "avg_gemm_ms": avg_gemm_ms},
            "e2e": e2e,
            "gpu_launches": step.KERNELS_PER_STEP * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_long_k_study(args):
    """Long-K accumulation study: Y = X W^T (bf16 out, no epilogue) with
    M = N = 16384, K = --study-k; X, W ~ N(0,1) with a seeded 1% of rows of each
    scaled by 64; e4m3 1x128 casts.  Both accumulation modes are timed (CUDA
    events) and compared with the oracle on sampled 256 x 256 output tiles
    (6 random, 2 through outlier rows, the last corner): the reported error is
    max |gpu - oracle| / sum_k |a b| over those tiles."""
    import numpy as np
    import torch
    import oracle
    import workloads
    import fp8_linear_layer_gb300 as fp8
    M = N = 16384
    K = args.study_k
    seed = 5000 + K // 1024
    x, xo = workloads.with_outlier_rows(workloads.normal_bf16((M, K), seed, "X"), seed, "X")
    w, wo = workloads.with_outlier_rows(workloads.normal_bf16((N, K), seed, "W"), seed, "W")
    X = fp8.quantize(x.cuda(), fp8.E4M3)
    W = fp8.quantize(w.cuda(), fp8.E4M3)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rng = np.random.default_rng(seed)
    tiles = [(int(rng.integers(0, M // 256)), int(rng.integers(0, N // 256))) for _ in range(6)]
    tiles += [(int(xo[0]) // 256, int(rng.integers(0, N // 256))), (int(rng.integers(0, M // 256)), int(wo[0]) // 256)]
    tiles += [(M // 256 - 1, N // 256 - 1)]
    # oracle: only the rows of X and W the tiles touch
    rows = sorted({256 * t[0] + i for t in tiles for i in range(256)})
    cols = sorted({256 * t[1] + i for t in tiles for i in range(256)})
    rpos = {r: i for i, r in enumerate(rows)}
    cpos = {c: i for i, c in enumerate(cols)}
    qa, sa = oracle.quantize(workloads.bits(x[torch.tensor(rows)]), oracle.E4M3)
    qb, sb = oracle.quantize(workloads.bits(w[torch.tensor(cols)]), oracle.E4M3)
    t0 = time.perf_counter()
    ref = []
    for (ti, tj) in tiles:
        ri = np.array([rpos[256 * ti + i] for i in range(256)])
        ci = np.array([cpos[256 * tj + i] for i in range(256)])
        ref.append(oracle.gemm(qa, sa, oracle.E4M3, qb, sb, oracle.E4M3, rows=ri, cols=ci))
    oracle_s = time.perf_counter() - t0
    out = {}
    for name, mode in (("full", fp8.ACC_FULL), ("fast", fp8.ACC_FAST)):
        for _ in range(2):
            fp8.gemm_fprop(X, W, None, fp8.EPI_NONE, mode, out=Y)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 3
        s.record()
        for _ in range(reps):
            fp8.gemm_fprop(X, W, None, fp8.EPI_NONE, mode, out=Y)
        e.record()
        e.synchronize()
        ms = s.elapsed_time(e) / reps
        err = 0.0
        for (ti, tj), (acc, S) in zip(tiles, ref):
            got = Y[256 * ti:256 * ti + 256, 256 * tj:256 * tj + 256].float().cpu().double().numpy()
            err = max(err, float(np.max(np.abs(got - acc) / S)))
        out[name] = {"tflops": 2.0 * M * N * K / (ms / 1e3) / 1e12, "ms": ms, "max_norm_err": err}
    if fp8.device_status() != 0:
        raise RuntimeError("device status not ok")
    line = {"study": "long_k_accumulation", "M": M, "N": N, "K": K, "outlier_rows": "1% of X and W rows x64",
            "tiles": "9 of 256x256 (6 random, 2 through outlier rows, last corner)",
            "note": "max_norm_err includes the bf16 rounding of Y (up to 2^-9 |y| / S)",
            "bound": {"full": 2e-3, "fast": 8e-3}, "full": out["full"], "fast": out["fast"],
            "oracle_seconds": round(oracle_s, 1), "oracle_cores": oracle.num_threads()}
    print(json.dumps(line), flush=True)
    return 0


def run_kernel_study(args):
    """Per-launch speed of every kernel of the training step (m, k, n from the
    command line) plus the dense weight-gradient table's largest shape and a
    long-K weight gradient: CUDA events around `reps` launches after 3 warm-ups;
    GEMMs in TFLOP/s (2 M N K per launch), casts in GB/s of algorithmic bytes
    (2 read + 1 written + 4/128 of scale per element)."""
    import torch
    import workloads
    import fp8_linear_layer_gb300 as fp8
    reps = 10
    m, k, n = args.m, args.k, args.n

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps

    def graph_timed(fn):
        # a kernel shorter than the host's per-call overhead: `reps` launches
        # replayed from one CUDA graph, so the device time is what is measured
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps

    out = {"study": "kernels", "reps": reps, "gemm_tflops": {}, "cast_gbs": {}}
    x = workloads.normal_bf16((m, k), SEED, "X").cuda()
    w = workloads.normal_bf16((n, k), SEED, "W", std=0.02).cuda()
    bias = workloads.normal_bf16((n,), SEED, "b", std=0.02).cuda()
    dy = workloads.normal_bf16((m, k), SEED, "dY", std=1e-2).cuda()
    X, W, DY = fp8.quantize(x, fp8.E4M3), fp8.quantize(w, fp8.E4M3), fp8.quantize(dy, fp8.E5M2)
    Y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    Z, dZ = torch.empty_like(Y), torch.empty_like(Y)
    f = 2.0 * m * n * k / 1e9
    out["gemm_tflops"]["fprop_bias_gelu_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.gemm_fprop(X, W, bias, fp8.EPI_BIAS_GELU, out=Y, aux=Z))
    out["gemm_tflops"]["dgrad_dgelu_bgrad_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.gemm_dgrad(DY, W, Z, fp8.EPI_DGELU_BGRAD, out=dZ))
    out["gemm_tflops"]["dgrad_dgelu_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.gemm_dgrad(DY, W, Z, fp8.EPI_DGELU, out=dZ))
    DZT, XT = fp8.quantize(dZ, fp8.E5M2, transpose=True), fp8.quantize(x, fp8.E4M3, transpose=True)
    # the bias gradient reduced from dZ^T's codes: K + 4 K/128 bytes read, 4 written per row
    db = torch.empty((n,), dtype=torch.float32, device="cuda")
    out["reduce_gbs"] = {"bgrad_from_operand_e5m2_%dx%d" % (n, m): n * (m + 4.0 * m / 128 + 4) / 1e6 / graph_timed(
        lambda: fp8.bgrad_from_operand(DZT, out=db))}
    # dZ's transposed cast alone and with the bias-gradient sums (+ their
    # finalize launch), as the step runs them; algorithmic bytes of the cast
    gbz = m * n * (3.0 + 4.0 / 128) / 1e6
    wsz = torch.empty((fp8.workspace_size(m, n) // 4,), dtype=torch.float32, device="cuda")
    out["cast_gbs"]["transposed_e5m2_%dx%d" % (m, n)] = gbz / graph_timed(
        lambda: fp8.quantize(dZ, fp8.E5M2, transpose=True, out=DZT))
    out["cast_gbs"]["transposed_dbias_e5m2_%dx%d" % (m, n)] = gbz / graph_timed(
        lambda: fp8.quantize_dbias(dZ, fp8.E5M2, out_t=DZT, dbias=db, workspace=wsz))
    dW = torch.zeros((n, k), device="cuda")
    out["gemm_tflops"]["wgrad_accumulate_m%d_n%d_k%d" % (n, k, m)] = f / timed(lambda: fp8.gemm_wgrad(DZT, XT, dW))
    for (M, N, K) in ((16384, 7168, 8192), (8192, 8192, 16384)):
        a = fp8.quantize(workloads.normal_bf16((M, K), SEED + 1, "A", std=0.02).cuda(), fp8.E4M3)
        bq = fp8.quantize(workloads.normal_bf16((N, K), SEED + 1, "B", std=0.02).cuda(), fp8.E4M3)
        o = torch.zeros((M, N), device="cuda")
        out["gemm_tflops"]["wgrad_accumulate_m%d_n%d_k%d" % (M, N, K)] = 2.0 * M * N * K / 1e9 / timed(
            lambda: fp8.gemm_wgrad(a, bq, o))
        del a, bq, o
    xb = workloads.normal_bf16((32768, 8192), SEED + 2, "C").cuda()
    gb = xb.numel() * (3.0 + 4.0 / 128) / 1e6
    for fmt, nm in ((fp8.E4M3, "e4m3"), (fp8.E5M2, "e5m2")):
        out["cast_gbs"]["rows_%s_32768x8192" % nm] = gb / timed(lambda: fp8.quantize(xb, fmt))
        out["cast_gbs"]["transposed_%s_32768x8192" % nm] = gb / timed(lambda: fp8.quantize(xb, fmt, transpose=True))
    # both orientations from one read: 2 bytes read, 2 x (1 + 4/128) written per element
    gb2 = xb.numel() * (2.0 + 2.0 * (1.0 + 4.0 / 128)) / 1e6
    qr, qt = fp8.empty_fp8(32768, 8192, fp8.E4M3), fp8.empty_fp8(8192, 32768, fp8.E4M3)
    out["cast_gbs"]["dual_e4m3_32768x8192"] = gb2 / timed(lambda: fp8.quantize_dual(xb, fp8.E4M3, out=qr, out_t=qt))
    out["hbm_peak_gbs"] = peaks()[1]
    out["status"] = fp8.device_status()
    print(json.dumps(out))


def run_cast_study(args):
    """The 1x128 casts on a 32768 x 8192 bf16 matrix, in a fixed order (rows
    e4m3, rows e5m2, transposed e4m3, transposed e5m2 with the bias-gradient
    column sums, both orientations e4m3), each launched once untimed and then
    --reps times between CUDA events; GB/s of algorithmic bytes: 2 read + 1 +
    4/128 written per element and orientation (+ 4 per column per 128 rows
    for the column-sum partials).  With --reps 1 every kernel launches twice,
    so a profiler can take the second launch of each."""
    import torch
    import workloads
    import fp8_linear_layer_gb300 as fp8
    reps = max(1, args.reps)
    R, C = 32768, 8192
    x = workloads.normal_bf16((R, C), SEED + 2, "C").cuda()
    n = x.numel()

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps

    one = n * (3.0 + 4.0 / 128) / 1e6
    qr, qt = fp8.empty_fp8(R, C, fp8.E4M3), fp8.empty_fp8(C, R, fp8.E4M3)
    db = torch.empty((C,), dtype=torch.float32, device="cuda")
    ws = torch.empty(((R // 128) * C,), dtype=torch.float32, device="cuda")
    out = {"study": "casts", "reps": reps, "shape": [R, C], "cast_gbs": {}}
    out["cast_gbs"]["rows_e4m3"] = one / timed(lambda: fp8.quantize(x, fp8.E4M3, out=qr))
    out["cast_gbs"]["rows_e5m2"] = one / timed(lambda: fp8.quantize(x, fp8.E5M2, out=qr))
    out["cast_gbs"]["transposed_e4m3"] = one / timed(lambda: fp8.quantize(x, fp8.E4M3, transpose=True, out=qt))
    out["cast_gbs"]["transposed_dbias_e5m2"] = (one + R // 128 * C * 4 / 1e6) / timed(
        lambda: fp8.quantize_dbias(x, fp8.E5M2, out_t=qt, dbias=db, workspace=ws))
    out["cast_gbs"]["dual_e4m3"] = n * (2.0 + 2.0 * (1.0 + 4.0 / 128)) / 1e6 / timed(
        lambda: fp8.quantize_dual(x, fp8.E4M3, out=qr, out_t=qt))
    out["hbm_peak_gbs"] = peaks()[1]
    out["frac_of_hbm"] = {k: v / out["hbm_peak_gbs"] for k, v in out["cast_gbs"].items()}
    out["status"] = fp8.device_status()
    print(json.dumps(out))


def run_input_grad_study(args):
    """The training step with the layer's input gradient (dX = dZ W, a fourth
    GEMM) where dZ's row cast for dX comes either from the transposed cast's
    read of dZ (dz_rows="cast") or from the data-gradient GEMM's epilogue
    (dz_rows="dgrad", fp8_gemm_dgrad_quant): CUDA events around --reps steps
    after 3 warm-ups, the two plans alternated over 5 rounds; plus the two
    launches that differ (the data-gradient GEMM with and without the cast,
    the transposed cast of dZ with and without the row codes)."""
    import torch
    import fp8_linear_layer_gb300 as fp8
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    m, k, n = args.m, args.k, args.n
    reps = max(1, args.reps)
    dev = torch.device("cuda")
    X, W, b, dY = (t.to(dev) for t in inputs(dev, m, k, n))
    steps = {mode: LinearTrainStep(m, k, n, dev, input_grad=True, dz_rows=mode) for mode in ("cast", "dgrad")}

    def run(st):
        for _, fn in st.launches(X, W, b, dY):
            fn()
        st.input_grad(W)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(reps):
            fn()
        e0.record()
        e0.synchronize()
        return s0.elapsed_time(e0) / reps

    res = {"study": "input_grad", "reps": reps, "m": m, "k": k, "n": n, "step_ms": {"cast": [], "dgrad": []}}
    for _ in range(5):
        for mode, st in steps.items():
            res["step_ms"][mode].append(timed(lambda: run(st)))
    f4 = 4 * 2.0 * m * n * k
    res["step_tflops_median"] = {mode: f4 / sorted(v)[len(v) // 2] / 1e9 for mode, v in res["step_ms"].items()}
    st = steps["dgrad"]
    f = 2.0 * m * n * k / 1e9
    res["dgrad_tflops"] = {
        "dgelu": f / timed(lambda: fp8.gemm_dgrad(st.dYq, st.Wq, st.Z, fp8.EPI_DGELU, out=st.dZ)),
        "dgelu_quant": f / timed(lambda: fp8.gemm_dgrad_quant(st.dYq, st.Wq, st.Z, out=st.dZ, q_out=st.dZq))}
    res["dz_cast_us"] = {
        "transposed_dbias": 1e3 * timed(lambda: fp8.quantize_dbias(st.dZ, fp8.E5M2, out_t=st.dZTq, dbias=st.db,
                                                                    workspace=st.ws)),
        "transposed_dbias_and_rows": 1e3 * timed(lambda: fp8.quantize_dbias(st.dZ, fp8.E5M2, out_t=st.dZTq, out=st.dZq,
                                                                             dbias=st.db, workspace=st.ws))}
    res["status"] = fp8.device_status()
    print(json.dumps(res))


def run_wgrad_tables(args):
    """The weight-gradient tables: the dense sweep (six (M, N) shapes x K in
    {4096, 8192}, fp32 out += A B^T) and the k-grouped MoE table (G experts,
    per-expert token counts drawn multinomially and rounded to multiples of 128,
    zero groups allowed), each timed with CUDA events around 10 launches after
    3 warm-ups.  Operands are random on the device (values do not change the
    timing); TFLOP/s = sum over groups of 2 M N K_g per launch."""
    import torch
    import workloads
    import fp8_linear_layer_gb300 as fp8
    reps = 10
    g = torch.Generator(device="cuda").manual_seed(SEED)

    def operand(rows, k):
        return fp8.quantize((torch.randn(rows, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16), fp8.E4M3)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps

    dense, grouped = {}, {}
    for K in workloads.DENSE_WGRAD_K:
        for (M, N) in workloads.DENSE_WGRAD_MN:
            A, Bq = operand(M, K), operand(N, K)
            out = torch.zeros((M, N), device="cuda")
            dense["m%d_n%d_k%d" % (M, N, K)] = 2.0 * M * N * K / 1e9 / timed(lambda: fp8.gemm_wgrad(A, Bq, out))
            del A, Bq, out
    for i, (G, M, N, per) in enumerate(workloads.GROUPED_WGRAD):
        ks = workloads.moe_group_sizes(G, G * per, SEED + i)
        tot = sum(ks)
        A, Bq = operand(M, tot), operand(N, tot)
        out = torch.zeros((G, M, N), device="cuda")
        grouped["g%d_m%d_n%d_tokens%d" % (G, M, N, tot)] = {
            "k_sizes": ks, "tflops": 2.0 * M * N * tot / 1e9 / timed(lambda: fp8.grouped_wgrad(A, Bq, ks, out))}
        del A, Bq, out
    # a skewed split of 16384 tokens (60%, none, 25%, 15%) over 4 experts, the
    # large expert first and last in turn: the host schedules groups longest first
    for ks in ([9856, 0, 4096, 2432], [2432, 0, 4096, 9856]):
        M, N, tot = 2048, 7168, sum(ks)
        A, Bq = operand(M, tot), operand(N, tot)
        out = torch.zeros((len(ks), M, N), device="cuda")
        grouped["skewed_g4_m%d_n%d_tokens%d_%s" % (M, N, tot, "_".join(map(str, ks)))] = {
            "k_sizes": ks, "tflops": 2.0 * M * N * tot / 1e9 / timed(lambda: fp8.grouped_wgrad(A, Bq, ks, out))}
        del A, Bq, out
    print(json.dumps({"study": "wgrad_tables", "reps": reps, "dense_tflops": dense, "grouped": grouped,
                      "status": fp8.device_status()}))


def run_mx_study(args):
    """The MXFP8 GEMMs (tensor-core block scaling, no software promotion) at the
    training-step shapes and on long K, next to the 1x128 GEMMs on the same
    bf16 data: CUDA events around 10 launches after 3 warm-ups, TFLOP/s;
    plus the MX casts in GB/s of algorithmic bytes (2 read + 1 + 1/32 written
    per element)."""
    import torch
    import workloads
    import fp8_linear_layer_gb300 as fp8
    reps = 10
    m, k, n = args.m, args.k, args.n

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps

    res = {"study": "mx", "reps": reps, "mx_tflops": {}, "block128_tflops": {}, "mx_cast_gbs": {}}
    x = workloads.normal_bf16((m, k), SEED, "X").cuda()
    w = workloads.normal_bf16((n, k), SEED, "W", std=0.02).cuda()
    bias = workloads.normal_bf16((n,), SEED, "b", std=0.02).cuda()
    dy = workloads.normal_bf16((m, k), SEED, "dY", std=1e-2).cuda()
    f = 2.0 * m * n * k / 1e9
    Y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    Z, dZ = torch.empty_like(Y), torch.empty_like(Y)
    X, W, DY = fp8.mx_quantize(x, fp8.E4M3), fp8.mx_quantize(w, fp8.E4M3), fp8.mx_quantize(dy, fp8.E5M2)
    res["mx_tflops"]["fprop_bias_gelu_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.mx_gemm_fprop(X, W, bias, fp8.EPI_BIAS_GELU, out=Y, aux=Z))
    res["mx_tflops"]["dgrad_dgelu_bgrad_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.mx_gemm_dgrad(DY, W, Z, fp8.EPI_DGELU_BGRAD, out=dZ))
    DZT, XT = fp8.mx_quantize(dZ, fp8.E5M2, transpose=True), fp8.mx_quantize(x, fp8.E4M3, transpose=True)
    dW = torch.zeros((n, k), device="cuda")
    res["mx_tflops"]["wgrad_accumulate_m%d_n%d_k%d" % (n, k, m)] = f / timed(lambda: fp8.mx_gemm_wgrad(DZT, XT, dW))
    del X, W, DY, DZT, XT
    a = workloads.normal_bf16((8192, 16384), SEED + 1, "A", std=0.02).cuda()
    bb = workloads.normal_bf16((8192, 16384), SEED + 1, "B", std=0.02).cuda()
    fl = 2.0 * 8192 * 8192 * 16384 / 1e9
    o = torch.zeros((8192, 8192), device="cuda")
    Am, Bm = fp8.mx_quantize(a, fp8.E4M3), fp8.mx_quantize(bb, fp8.E4M3)
    res["mx_tflops"]["wgrad_accumulate_m8192_n8192_k16384"] = fl / timed(lambda: fp8.mx_gemm_wgrad(Am, Bm, o))
    del Am, Bm
    Ab, Bb = fp8.quantize(a, fp8.E4M3), fp8.quantize(bb, fp8.E4M3)
    res["block128_tflops"]["wgrad_accumulate_m8192_n8192_k16384"] = fl / timed(lambda: fp8.gemm_wgrad(Ab, Bb, o))
    del Ab, Bb
    xb = workloads.normal_bf16((32768, 8192), SEED + 2, "C").cuda()
    gb = xb.numel() * (3.0 + 1.0 / 32) / 1e6
    out_r = fp8.empty_mx(32768, 8192, fp8.E4M3, xb.device)
    out_t = fp8.empty_mx(8192, 32768, fp8.E4M3, xb.device)
    res["mx_cast_gbs"]["rows_e4m3_32768x8192"] = gb / timed(lambda: fp8.mx_quantize(xb, fp8.E4M3, out=out_r))
    res["mx_cast_gbs"]["transposed_e4m3_32768x8192"] = gb / timed(
        lambda: fp8.mx_quantize(xb, fp8.E4M3, transpose=True, out=out_t))
    res["status"] = fp8.device_status()
    print(json.dumps(res))


def run_tensor_study(args):
    """The per-tensor scaled GEMMs (one scale per operand, scaled once after the
    K loop) at the training-step shapes and on long K, and the per-tensor amax
    and casts in GB/s of algorithmic bytes (amax: 2 read; rows: 2 read + 1
    written; both orientations: 2 read + 2 written per element).  CUDA events
    around 10 launches after 3 warm-ups."""
    import torch
    import workloads
    import fp8_linear_layer_gb300 as fp8
    reps = 10
    m, k, n = args.m, args.k, args.n

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        e.synchronize()
        return s.elapsed_time(e) / reps

    def cast(t, fmt, **kw):
        return fp8.tensor_quantize(t, fmt, fp8.tensor_amax(t), **kw)

    res = {"study": "tensor", "reps": reps, "tensor_tflops": {}, "cast_gbs": {}}
    x = workloads.normal_bf16((m, k), SEED, "X").cuda()
    w = workloads.normal_bf16((n, k), SEED, "W", std=0.02).cuda()
    bias = workloads.normal_bf16((n,), SEED, "b", std=0.02).cuda()
    dy = workloads.normal_bf16((m, k), SEED, "dY", std=1e-2).cuda()
    f = 2.0 * m * n * k / 1e9
    Y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    Z, dZ = torch.empty_like(Y), torch.empty_like(Y)
    (X, XT), (W, _), (DY, _) = cast(x, fp8.E4M3, cols=True), cast(w, fp8.E4M3), cast(dy, fp8.E5M2)
    res["tensor_tflops"]["fprop_bias_gelu_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.tensor_gemm_fprop(X, W, bias, fp8.EPI_BIAS_GELU, out=Y, aux=Z))
    res["tensor_tflops"]["dgrad_dgelu_bgrad_m%d_n%d_k%d" % (m, n, k)] = f / timed(
        lambda: fp8.tensor_gemm_dgrad(DY, W, Z, fp8.EPI_DGELU_BGRAD, out=dZ))
    _, DZT = cast(dZ, fp8.E5M2, rows=False, cols=True)
    dW = torch.zeros((n, k), device="cuda")
    res["tensor_tflops"]["wgrad_accumulate_m%d_n%d_k%d" % (n, k, m)] = f / timed(
        lambda: fp8.tensor_gemm_wgrad(DZT, XT, dW))
    del X, XT, W, DY, DZT
    a = workloads.normal_bf16((8192, 16384), SEED + 1, "A", std=0.02).cuda()
    bb = workloads.normal_bf16((8192, 16384), SEED + 1, "B", std=0.02).cuda()
    fl = 2.0 * 8192 * 8192 * 16384 / 1e9
    o = torch.zeros((8192, 8192), device="cuda")
    (At, _), (Bt, _) = cast(a, fp8.E4M3), cast(bb, fp8.E4M3)
    res["tensor_tflops"]["wgrad_accumulate_m8192_n8192_k16384"] = fl / timed(lambda: fp8.tensor_gemm_wgrad(At, Bt, o))
    del At, Bt, a, bb, o
    xb = workloads.normal_bf16((32768, 8192), SEED + 2, "C").cuda()
    e = xb.numel()
    am, seen = fp8.tensor_amax(xb), torch.empty(1, device="cuda")
    qr = fp8.empty_tensor_scaled(32768, 8192, fp8.E4M3, xb.device)
    qt = fp8.Fp8TensorScaled(torch.empty((8192, 32768), dtype=torch.uint8, device="cuda"), qr.scale, fp8.E4M3)
    res["cast_gbs"]["amax_32768x8192"] = e * 2.0 / 1e6 / timed(lambda: fp8.tensor_amax(xb, out=seen))
    res["cast_gbs"]["rows_e4m3_32768x8192"] = e * 3.0 / 1e6 / timed(
        lambda: fp8.tensor_quantize(xb, fp8.E4M3, am, out=qr, amax_out=seen))
    res["cast_gbs"]["transposed_e4m3_32768x8192"] = e * 3.0 / 1e6 / timed(
        lambda: fp8.tensor_quantize(xb, fp8.E4M3, am, rows=False, cols=True, out_t=qt, amax_out=seen))
    res["cast_gbs"]["both_e4m3_32768x8192"] = e * 4.0 / 1e6 / timed(
        lambda: fp8.tensor_quantize(xb, fp8.E4M3, am, cols=True, out=qr, out_t=qt, amax_out=seen))
    res["status"] = fp8.device_status()
    print(json.dumps(res))


def run_fp8_peak_probe(args):
    """Dense fp8 tensor-core throughput of the vendor library on this GPU, for
    context beside the roofline denominator (which stays the measured bf16
    burst x the nominal ratio): torch._scaled_mm, e4m3 x e4m3 -> bf16 with
    per-tensor scales, 8192^3, best of 10 (burst) and back to back for ~4 s
    (sustained).  A probe outside the measured path: none of this library's
    kernels run here."""
    import torch
    n = 8192
    g = torch.Generator(device="cuda").manual_seed(SEED)
    a = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device="cuda", generator=g).to(torch.float8_e4m3fn).t()  # column-major operand
    one = torch.ones((), device="cuda")

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        mm()
        e.record()
        e.synchronize()
        best = min(best, s.elapsed_time(e))
    flops = 2.0 * n ** 3
    clocks = ClockSampler(0)
    clocks.start()
    reps, t0 = 0, time.time()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    while time.time() - t0 < 4.0:
        for _ in range(20):
            mm()
        reps += 20
        torch.cuda.synchronize()
    e.record()
    e.synchronize()
    clk = clocks.stop()
    out = {"study": "fp8_peak", "op": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3",
           "burst_tflops": flops / best / 1e9, "sustained_tflops": flops * reps / s.elapsed_time(e) / 1e9,
           "sustained_seconds": round(time.time() - t0, 2), "clocks": clk,
           "bf16_measured_x2": peaks()[0]}
    print(json.dumps(out))


def main():
    args = parse_args()
    if args.study == "long_k":
        return run_long_k_study(args)
    if args.study == "kernels":
        return run_kernel_study(args)
    if args.study == "fp8_peak":
        return run_fp8_peak_probe(args)
    if args.study == "wgrad_tables":
        return run_wgrad_tables(args)
    if args.study == "mx":
        return run_mx_study(args)
    if args.study == "tensor":
        return run_tensor_study(args)
    if args.study == "casts":
        return run_cast_study(args)
    if args.study == "input_grad":
        return run_input_grad_study(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
