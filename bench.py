#!/usr/bin/env python
"""Quantize + GEMM benchmark of one transformer layer's 12 GEMMs on GB300.

Workload ("How to optimize Transformer-based models for low-precision
training", model configuration and training input): CodonFM-5B, hidden 4096,
intermediate 16384, micro-batch 31 x sequence 512 = 15,872 tokens; the 12 GEMMs
are QKV / attention-out / MLP-up / MLP-down x Fprop / Dgrad / Wgrad.  Inputs are
synthetic bf16 (activations ~N(0,1), weights ~N(0,0.02^2), gradients
~N(0,(1e-3)^2)), resident in HBM before the timed region.

One step = one layer: for each of the 12 GEMMs, quantize the two operand copies
it reads (autocast mode: "before every GEMM the inputs are quantized
dynamically", same page, autocast vs pre-quantize) and run the GEMM, all in
liblpq's CUDA kernels.  The headline recipe is NVFP4 (1D 16-blocks for
activations and gradients, 16x16 blocks for weights, random Hadamard transform
on the Wgrad inputs, stochastic rounding of gradients).  The other recipes and
the pre-quantize mode (GEMM only) are measured in the same run and reported
under "recipes".

Usage (the pages' CLI flags are accepted): python bench.py [--gpus N] [--steps K]
[--warmup W] [--impl lpq|reference] [--recipe nvfp4|mxfp8|mxfp8_e5m2|mxfp4|
fp8_current|fp8_delayed|bf16] [--pre-quantize] [--no-fp8] [--no-fp4] ...
(mxfp8_e5m2: MXFP8 with E5M2 gradients; mxfp4: E2M1 with E8M0 scales per 32.)
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

RECIPES = ["bf16", "fp8_delayed", "fp8_current", "mxfp8", "mxfp8_e5m2", "mxfp4", "nvfp4"]


def sweep_recipes(args):
    """Recipes of the sweep, less those --no-fp8 / --no-fp4 leave out."""
    skip = set()
    if args.no_fp8:
        skip |= {"mxfp8", "mxfp8_e5m2"}
    if args.no_fp4:
        skip |= {"nvfp4", "mxfp4"}
    return [r for r in RECIPES if r not in skip]


def parse():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["lpq", "reference"], default="lpq")
    p.add_argument("--recipe", choices=RECIPES, default="nvfp4")
    p.add_argument("--pre-quantize", dest="prequant", action="store_true")
    p.add_argument("--no-fp8", action="store_true", help="skip the MXFP8 recipes in the recipe sweep")
    p.add_argument("--no-fp4", action="store_true", help="skip NVFP4 and MXFP4 in the recipe sweep")
    p.add_argument("--no-sweep", action="store_true", help="time only the headline recipe")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--hidden_size", type=int, default=4096)
    p.add_argument("--intermediate_size", type=int, default=16384)
    p.add_argument("--num_attention_heads", type=int, default=32)
    p.add_argument("--num_hidden_layers", type=int, default=24)
    p.add_argument("--micro_batch_size", type=int, default=31)
    p.add_argument("--sequence_length", type=int, default=512)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("-o", "--output", default=None, help="write the per-GEMM table as JSON here")
    p.add_argument("--workload", choices=["layer", "ksweep", "drift", "report"], default="layer",
                   help="layer: the contract line; ksweep / drift: the K-sweep and the FP8 drift runs")
    p.add_argument("--mma-peaks", action="store_true",
                   help="only measure the dense tcgen05 rates (shared-memory-resident operands) and exit")
    p.add_argument("--parallel", choices=["replicas", "tokens"], default="replicas",
                   help="N > 1: replicas (each rank its own layer, no exchange) or tokens (data parallelism: "
                        "each rank its own micro-batch of tokens, all-reduce MAX of the amaxes and SUM of dW)")
    p.add_argument("--no-drift", action="store_true", help="skip the FP8 drift summary in the layer run")
    p.add_argument("--no-ksweep", action="store_true", help="skip the K-sweep summary in the layer run")
    p.add_argument("--no-quant-kinds", action="store_true", help="skip the per-kind quantizer roofline")
    return p.parse_args()


# ------------------------------------------------------------------ contract line
METRIC = "quantize+GEMM TFLOP/s & % of FP8/FP4 peak; ms/layer (CodonFM-5B shape)"
# Nominal dense per-GPU tensor rates of GB300 (without 2:4 sparsity), TFLOP/s.
DATASHEET_DENSE_TFLOPS = {"bf16": 2250.0, "fp8": 4500.0, "mxfp8": 4500.0, "nvfp4": 13500.0}


def contract_config(args, world, recipe, autocast):
    """The `config` object of the JSON line, identical for both arms."""
    M = args.micro_batch_size * args.sequence_length
    mode = "autocast" if autocast else "pre-quantize"
    par = ("token-sharded data parallel (all-reduce MAX of amaxes, SUM of dW)" if args.parallel == "tokens"
           else "replicas") + f" x{world}"
    return {"workload": f"CodonFM-5B layer, 12 GEMMs, {recipe} {mode} (M={M}, hidden {args.hidden_size}, "
                        f"intermediate {args.intermediate_size})",
            "global_batch": args.micro_batch_size * world, "seq_len": args.sequence_length, "parallelism": par,
            "l2": "inputs larger than L2 (working set > 4 GB)"}


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms; start()
    returns once the first sample has arrived, so the samples cover the
    region that follows."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx, self.proc, self.lines = gpu_index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
            self.lines.clear()  # samples taken before the caller's region starts
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ layer workload
class Layer:
    """Inputs, quantized buffers and outputs of one CodonFM-5B-shaped layer."""

    def __init__(self, args, device):
        import torch
        from precision_transformer_gemms_gb300 import lpq, synth
        self.lpq, self.torch = lpq, torch
        h, f = args.hidden_size, args.intermediate_size
        self.M = args.micro_batch_size * args.sequence_length
        self.shapes = lpq.layer_shapes(h, f, args.micro_batch_size, args.sequence_length,
                                       args.num_attention_heads, args.num_hidden_layers)
        self.linears = {"qkv": (h, 3 * h), "attn_out": (h, h), "mlp_up": (h, f), "mlp_down": (f, h)}
        self.flops = sum(2 * m * k * n for _, _, m, k, n in self.shapes)
        self.inp = {}
        base = args.seed
        for i, (name, (K, N)) in enumerate(self.linears.items()):
            self.inp[name] = {
                "X": synth.bf16_normal((self.M, K), synth.ACT_STD, base + 100 * i + synth.SEED_X, device),
                "W": synth.bf16_normal((N, K), synth.WEIGHT_STD, base + 100 * i + synth.SEED_W, device),
                "dY": synth.bf16_normal((self.M, N), synth.GRAD_STD, base + 100 * i + synth.SEED_DY, device),
            }
        self.out = {}
        for name, lay, m, k, n in self.shapes:
            self.out[name] = torch.empty((m, n), dtype=torch.bfloat16, device=device)
        self.bufs = {}
        self.states = {}
        self.device = device

    # quantizer settings per recipe and tensor role: (fmt, flags_extra, scaling)
    def qcfg(self, recipe, role):
        L = self.lpq
        if recipe in ("fp8_current", "fp8_delayed"):
            fmt = L.FP8_E5M2 if role == "dY" else L.FP8_E4M3
            return fmt, 0, L.SCALING_DELAYED if recipe == "fp8_delayed" else L.SCALING_CURRENT
        if recipe == "mxfp8":
            return L.MXFP8, 0, L.SCALING_CURRENT
        if recipe == "mxfp8_e5m2":  # E5M2 codes for the gradients, E4M3 for X and W
            return (L.MXFP8_E5M2 if role == "dY" else L.MXFP8), 0, L.SCALING_CURRENT
        if recipe == "mxfp4":
            return L.MXFP4, 0, L.SCALING_CURRENT
        if recipe == "nvfp4":
            if role == "W":
                return L.NVFP4_2D, 0, L.SCALING_CURRENT
            extra = L.STOCHASTIC if role == "dY" else 0
            return L.NVFP4, extra, L.SCALING_CURRENT
        raise ValueError(recipe)

    def buf(self, recipe, lin, role, colwise):
        key = (recipe, lin, role, colwise)
        if key not in self.bufs:
            L = self.lpq
            x = self.inp[lin][role]
            R, C = x.shape
            if recipe == "bf16":
                t = x.t().contiguous() if colwise else x
                self.bufs[key] = L.Copy.of_bf16(t, colwise)
            else:
                fmt, _, _ = self.qcfg(recipe, role)
                self.bufs[key] = L.Copy(fmt, C if colwise else R, R if colwise else C, colwise, L.SF_GEMM,
                                        self.device)
        return self.bufs[key]

    def state(self, lin, role):
        if (lin, role) not in self.states:
            self.states[(lin, role)] = self.lpq.DelayedState(16, self.device)
        return self.states[(lin, role)]

    def quantize(self, recipe, lin, role, colwise, seed):
        """One lpq_quantize of one operand copy into its persistent buffer."""
        L = self.lpq
        fmt, extra, scaling = self.qcfg(recipe, role)
        flags = (L.COLWISE if colwise else L.ROWWISE) | extra
        if recipe == "nvfp4" and colwise and role in ("X", "dY"):
            flags |= L.RHT_COLWISE  # Wgrad inputs
        copy = self.buf(recipe, lin, role, colwise)
        qt = L.QTensor(None if colwise else copy, copy if colwise else None)
        st = self.state(lin, role) if scaling == L.SCALING_DELAYED else None
        L.quantize(self.inp[lin][role], fmt, flags, scaling=scaling, seed=seed, rht_seed=1234, state=st, out=qt)
        if st is not None:
            L.scale_update(st, copy.amax, L.FMAX[fmt])
        return copy

    # operands of each pass: (a role, a colwise), (b role, b colwise)
    PASS = {0: (("X", False), ("W", False)), 1: (("dY", False), ("W", True)), 2: (("dY", True), ("X", True))}

    def gemm_list(self):
        return [(name, lay, name.rsplit("_", 1)[0]) for name, lay, *_ in self.shapes]

    def prequantize(self, recipe):
        for _, lay, lin in self.gemm_list():
            for role, col in self.PASS[lay]:
                if recipe == "bf16":
                    self.buf(recipe, lin, role, col)
                else:
                    self.quantize(recipe, lin, role, col, seed=0)

    def step(self, recipe, autocast, step_idx=0, events=None):
        """Enqueue one layer step; `events` (optional) gets (name, kind, ev0, ev1)."""
        L, torch = self.lpq, self.torch
        delayed = recipe == "fp8_delayed"
        for name, lay, lin in self.gemm_list():
            (ra, ca), (rb, cb) = self.PASS[lay]
            if recipe != "bf16" and (autocast or delayed):
                e0 = torch.cuda.Event(enable_timing=True) if events is not None else None
                if e0:
                    e0.record()
                a = self.quantize(recipe, lin, ra, ca, seed=step_idx * 64 + lay)
                b = self.quantize(recipe, lin, rb, cb, seed=step_idx * 64 + lay + 8)
                if e0:
                    e1 = torch.cuda.Event(enable_timing=True)
                    e1.record()
                    events.append((name, "quantize", e0, e1))
            else:
                a, b = self.buf(recipe, lin, ra, ca), self.buf(recipe, lin, rb, cb)
            e0 = torch.cuda.Event(enable_timing=True) if events is not None else None
            if e0:
                e0.record()
            L.gemm(lay, a, b, c=self.out[name])
            if e0:
                e1 = torch.cuda.Event(enable_timing=True)
                e1.record()
                events.append((name, "gemm", e0, e1))

    def fused_step(self, recipe, step_idx=0):
        """One layer with each tensor quantized once into both copies (one
        lpq_quantize per tensor and linear), then the linear's three GEMMs."""
        L = self.lpq
        for lin in self.linears:
            for role in ("X", "W", "dY"):
                fmt, extra, scaling = self.qcfg(recipe, role)
                flags = L.ROWWISE | L.COLWISE | extra
                if recipe == "nvfp4" and role in ("X", "dY"):
                    flags |= L.RHT_COLWISE
                qt = L.QTensor(self.buf(recipe, lin, role, False), self.buf(recipe, lin, role, True))
                st = self.state(lin, role) if scaling == L.SCALING_DELAYED else None
                L.quantize(self.inp[lin][role], fmt, flags, scaling=scaling, seed=step_idx * 64, rht_seed=1234,
                           state=st, out=qt)
                if st is not None:
                    L.scale_update(st, qt.row.amax, L.FMAX[fmt])
            for name, lay, lin2 in self.gemm_list():
                if lin2 != lin:
                    continue
                (ra, ca), (rb, cb) = self.PASS[lay]
                L.gemm(lay, self.buf(recipe, lin, ra, ca), self.buf(recipe, lin, rb, cb), c=self.out[name])

    def kernels_per_step(self, recipe, autocast):
        """Kernels of liblpq launched by one step (memsets are not kernels of ours)."""
        n = 12  # GEMMs
        if recipe == "bf16" or not (autocast or recipe == "fp8_delayed"):
            return n
        per_q = {"fp8_current": 2, "fp8_delayed": 2, "mxfp8": 1, "mxfp8_e5m2": 1, "mxfp4": 1, "nvfp4": 2}[recipe]  # (amax pass) + tile pass
        if recipe == "fp8_delayed":
            per_q = 2  # tile pass + scale update
        return n + 24 * per_q

    def step_io_bytes(self):
        """Bytes of the step's bf16 inputs (H2D) and outputs (D2H)."""
        i = sum(t.numel() * 2 for d in self.inp.values() for t in d.values())
        o = sum(t.numel() * 2 for t in self.out.values())
        return i, o


def time_steps(layer, recipe, autocast, steps, warmup, world, per_kernel=False):
    import torch
    for w in range(warmup):
        layer.step(recipe, autocast, w)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    events = [] if per_kernel else None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(steps):
        layer.step(recipe, autocast, warmup + s, events)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    return ms / steps, events


def time_fn(step_fn, steps, warmup, world):
    """ms per call of step_fn(s) over `steps` calls after `warmup`, CUDA
    events on the current stream, barrier + synchronize on both sides, the
    max over ranks."""
    import torch
    for w in range(warmup):
        step_fn(w)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(steps):
        step_fn(warmup + s)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1), world) / steps


def summarize_events(layer, events, steps):
    """Per GEMM: mean GEMM ms and quantize ms over the timed steps."""
    acc = {}
    for name, kind, a, b in events:
        acc.setdefault((name, kind), []).append(a.elapsed_time(b))
    table = {}
    shp = {n: (m, k, nn) for n, _, m, k, nn in layer.shapes}
    for name, _, _ in layer.gemm_list():
        m, k, n = shp[name]
        g = statistics.mean(acc[(name, "gemm")])
        q = statistics.mean(acc[(name, "quantize")]) if (name, "quantize") in acc else 0.0
        table[name] = {"m": m, "k": k, "n": n, "gemm_ms": g, "quant_ms": q,
                       "gemm_tflops": 2 * m * k * n / (g * 1e-3) / 1e12}
    return table


def profiled_traffic(kernel_file, recipe):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary
    (profiles/gemm_<recipe>_layer_traffic.md), or None when the kernel source
    changed after the counters were taken (its sha256 is recorded there)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"gemm_{recipe}_layer_traffic.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    src = hashlib.sha256(open(kernel_file, "rb").read()).hexdigest()
    if vals.get("kernel_source_sha256") != src:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle sample
def oracle_sample(layer_shapes, M, linears, rows=2, cols=128, slab=16, seed=0):
    """Times the oracle on a bounded sample of one layer step and projects the
    step: per GEMM, `rows` x `cols` outputs of the FP64 GEMM (from NVFP4
    operands) and the NVFP4 quantization of a `slab`-row slab of each operand,
    both scaled to the full sizes.  Returns (projected seconds per layer, info)."""
    import numpy as np
    import oracle as o
    from precision_transformer_gemms_gb300 import synth
    t_gemm = t_q = 0.0
    rng = np.random.default_rng(seed)
    for name, lay, m, k, n in layer_shapes:
        xa = synth.host_bits(synth.bf16_normal((rows, k), 1.0, seed + 1, "cpu"))
        xb = synth.host_bits(synth.bf16_normal((cols, k), 0.02, seed + 2, "cpu"))
        t0 = time.perf_counter()
        qa = o.nvfp4(xa, o.NV_ROW)
        qb = o.nvfp4(xb, o.NV_ROW | o.NV_2D) if cols % 16 == 0 else o.nvfp4(xb, o.NV_ROW)
        t1 = time.perf_counter()
        A = o.Operand(o.K_NVFP4, qa["row"], qa["row_sf"], qa["row_ts"])
        B = o.Operand(o.K_NVFP4, qb["row"], qb["row_sf"], qb["row_ts"])
        o.gemm(A, B, rows, cols, k)
        t2 = time.perf_counter()
        t_gemm += (t2 - t1) * (m * n) / (rows * cols)
        # two operand copies quantized per GEMM, each of m*k or n*k elements
        t_q += (t1 - t0) * ((m * k) + (n * k)) / (rows * k + cols * k)
    return t_gemm + t_q, {"gemm_s": t_gemm, "quant_s": t_q}


def run_reference(args, rank, world):
    """The oracle arm: each step is a bounded sample of the layer workload on
    the host cores, projected to one layer."""
    if rank != 0:
        return
    import oracle as o
    from precision_transformer_gemms_gb300 import synth  # noqa: F401
    h, f = args.hidden_size, args.intermediate_size
    M = args.micro_batch_size * args.sequence_length
    lins = [("qkv", h, 3 * h), ("attn_out", h, h), ("mlp_up", h, f), ("mlp_down", f, h)]
    shapes = []
    for lin, K, N in lins:
        shapes += [(f"{lin}_fprop", 0, M, K, N), (f"{lin}_dgrad", 1, M, N, K), (f"{lin}_wgrad", 2, N, M, K)]
    flops = sum(2 * m * k * n for _, _, m, k, n in shapes)
    for w in range(args.warmup):
        oracle_sample(shapes, M, lins, rows=1, cols=32, slab=16, seed=w)
    proj = []
    t0 = time.perf_counter()
    for s in range(args.steps):
        sec, _ = oracle_sample(shapes, M, lins, rows=2, cols=128, slab=16, seed=args.warmup + s)
        proj.append(sec)
    wall = time.perf_counter() - t0
    sec = statistics.mean(proj)
    value = flops / sec / 1e12
    # ms_per_step is the measured wall time of one step's bounded sample; the
    # value is the layer throughput that sample projects to (whole layer:
    # projected_ms_per_step)
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / args.steps * 1e3, "projected_ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": contract_config(args, world, "nvfp4", True),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": o.num_threads(), "kind": "oracle",
                             "sample": "per step: per GEMM 2x128 outputs of the FP64 oracle GEMM on NVFP4 operands "
                                       "and their NVFP4 quantization (a 2-row and a 128-row slab of the operands), "
                                       "projected to the full layer",
                             "wall_s": wall},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main arm
def check_device(stage):
    """The device error word must be clean after a timed region: a GEMM whose
    bounded wait gave up leaves early and only sets that word, so its step
    would otherwise count as complete work."""
    from precision_transformer_gemms_gb300 import lpq
    code = lpq.device_status()
    if code != 0:
        raise RuntimeError(f"device error word {code} after {stage}: a bounded device wait gave up; "
                           "the timed work is incomplete and no number is reported")
    return code


# Algorithmic bytes per input element of one quantize call that emits one
# copy (the amax pass, where the recipe needs one, reads the input once more).
QUANT_BYTES_PER_ELEM = {
    "nvfp4": 2 + 2 + 0.5 + 1 / 16,         # amax pass + read + E2M1 codes and E4M3 scales
    "fp8_current": 2 + 2 + 1,              # amax pass + read + codes
    "fp8_delayed": 2 + 1,                  # amax fused into the quantize pass
    "mxfp8": 2 + 1 + 1 / 32,               # read + codes + E8M0 scales
    "mxfp8_e5m2": 2 + 1 + 1 / 32,
    "mxfp4": 2 + 0.5 + 1 / 32,
    "bf16": 0.0,
}


def quant_bytes_per_layer(layer, recipe):
    """Per-GEMM autocast: every GEMM quantizes one copy of each operand."""
    per = QUANT_BYTES_PER_ELEM[recipe]
    return sum((m * k + n * k) * per for _, _, m, k, n in layer.shapes)


def time_quant_kinds(layer, hbm_gbs, reps=10):
    """Each quantizer kind of the NVFP4 recipe (and the plain FP8 / MXFP8
    paths) timed alone with CUDA events around each launch, L2 flushed (a
    256 MB write) before every timed call, on the layer's own tensors:
    X = the QKV input 15872 x 4096, dY = the QKV gradient 15872 x 12288,
    W = the MLP-up weight 16384 x 4096.  The quantize calls take the amax as
    given (LPQ_GIVEN_AMAX), so the amax pass is timed on its own.  Bytes are
    algorithmic: the bf16 read plus the codes and scales written."""
    import torch
    from precision_transformer_gemms_gb300 import lpq as L
    X, dY, W = layer.inp["qkv"]["X"], layer.inp["qkv"]["dY"], layer.inp["mlp_up"]["W"]
    dev = X.device
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    nv_w = 0.5 + 1 / 16

    def nv_buf(t, fmt, flags, rht):
        q = L.alloc(fmt, t.shape[0], t.shape[1], flags, L.SF_GEMM, dev)
        a, r = L.amax(t, rht=rht, rht_seed=1234)
        if q.row is not None:
            q.row.amax.copy_(a)
        if q.col is not None:
            q.col.amax.copy_(r if rht else a)
        return q

    kinds = []
    a_out = torch.empty(2, dtype=torch.float32, device=dev)
    kinds.append(("amax", X, lambda: L.amax(X, out=a_out[0:1]), 2.0))
    kinds.append(("amax_rht", X, lambda: L.amax(X, rht=True, rht_seed=1234, out=a_out[0:1], rht_out=a_out[1:2]), 2.0))
    for name, t, fmt, flags, rht in (
            ("nvfp4_row", X, L.NVFP4, L.ROWWISE, False),
            ("nvfp4_col_rht", X, L.NVFP4, L.COLWISE | L.RHT_COLWISE, True),
            ("nvfp4_row_sr", dY, L.NVFP4, L.ROWWISE | L.STOCHASTIC, False),
            ("nvfp4_col_rht_sr", dY, L.NVFP4, L.COLWISE | L.RHT_COLWISE | L.STOCHASTIC, True),
            ("nvfp4_2d_row", W, L.NVFP4_2D, L.ROWWISE, False),
            ("nvfp4_2d_col", W, L.NVFP4_2D, L.COLWISE, False),
            ("fp8_row", X, L.FP8_E4M3, L.ROWWISE, False),
            ("fp8_col", X, L.FP8_E4M3, L.COLWISE, False)):
        q = nv_buf(t, fmt, flags, rht)
        per = 2 + (nv_w if fmt in (L.NVFP4, L.NVFP4_2D) else 1.0)
        kinds.append((name, t, (lambda t=t, fmt=fmt, flags=flags, q=q:
                                L.quantize(t, fmt, flags | L.GIVEN_AMAX, seed=7, rht_seed=1234, out=q)), per))
    for name, flags in (("mxfp8_row", L.ROWWISE), ("mxfp8_col", L.COLWISE)):
        q = L.alloc(L.MXFP8, X.shape[0], X.shape[1], flags, L.SF_GEMM, dev)
        kinds.append((name, X, (lambda flags=flags, q=q: L.quantize(X, L.MXFP8, flags, out=q)), 2 + 1 + 1 / 32))
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, t, fn, per in kinds:
        fn()
        total = 0.0
        for _ in range(reps):
            flush.zero_()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
        us = total / reps * 1e3
        nbytes = t.numel() * per
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"shape": list(t.shape), "us": round(us, 2), "bytes_per_elem": round(per, 4),
                     "gbs": round(gbs, 1), "frac": round(gbs / hbm_gbs, 3)}
    # The delayed-scaling update (amax history of 16, scale from its maximum):
    # a single tiny kernel, latency-bound, reported in microseconds.  The flush
    # write ahead of it keeps the GPU busy while the host enqueues the call, so
    # the events time the kernel, not the host's submission.
    st = L.DelayedState(16, dev)
    a1 = torch.ones(1, dtype=torch.float32, device=dev)
    L.scale_update(st, a1, L.FMAX[L.FP8_E4M3])
    total = 0.0
    for _ in range(reps):
        flush.zero_()
        e0.record()
        L.scale_update(st, a1, L.FMAX[L.FP8_E4M3])
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    out["scale_update"] = {"us": round(total / reps * 1e3, 2), "bound": "latency", "history": 16}
    check_device("quantizer kinds")
    del flush
    return out


def make_dp_linears(layer, recipe, first_row=0, group=None):
    """The four linears of the layer as token-sharded data-parallel steps
    (precision_transformer_gemms_gb300.dp) on this rank's inputs."""
    from precision_transformer_gemms_gb300 import dp
    return [dp.TokenShardedLinear(recipe, d["X"], d["W"], d["dY"], first_row=first_row, group=group)
            for d in layer.inp.values()]


def dp_kernels_per_step(recipe):
    """liblpq kernels of one token-sharded layer step (4 linears)."""
    per_lin = {"nvfp4": 2 + 2 + 2 + 3, "fp8_current": 2 + 2 + 2 + 3, "fp8_delayed": 3 + 3 + 3,
               "mxfp8": 3 + 3, "mxfp8_e5m2": 3 + 3, "mxfp4": 3 + 3, "bf16": 3}[recipe]
    # nvfp4 / fp8_current: W (amax + tile), 2 amax passes, X and dY tile passes, 3 GEMMs
    return 4 * per_lin


def run_lpq(args, rank, world, local):
    import torch
    from precision_transformer_gemms_gb300 import lpq
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    lpq.lib()
    layer = Layer(args, device)
    recipe = args.recipe
    autocast = not args.prequant
    if recipe == "fp8_delayed":
        autocast = True  # delayed scaling needs the amax history: always dynamic
    tokens = args.parallel == "tokens" and world > 1
    layer.prequantize(recipe)  # buffers exist before the timed region (pre-quantize mode reads them)
    torch.cuda.synchronize()
    peaks = measured_peaks()
    hbm = peaks["hbm_gbs"] if peaks else 6800.0

    # headline: K steps with whole-step CUDA events (replicas: the per-GEMM
    # autocast layer step; tokens: the data-parallel step with its exchanges)
    clocks = ClockSampler(local)
    if tokens:
        lins = make_dp_linears(layer, recipe, first_row=rank * layer.M)
        clocks.start()
        ms_step = time_fn(lambda s: [lin.step(seed=s) for lin in lins], args.steps, args.warmup, world)
        clk = clocks.stop()
        launches = dp_kernels_per_step(recipe)
        del lins
    else:
        clocks.start()
        ms_step, _ = time_steps(layer, recipe, autocast, args.steps, args.warmup, world)
        clk = clocks.stop()
        launches = layer.kernels_per_step(recipe, autocast)
    status = check_device("the headline steps")
    # per-kernel durations (the layer step, events around each launch)
    _, events = time_steps(layer, recipe, autocast, max(3, args.steps // 2), 1, world, per_kernel=True)
    check_device("the per-kernel steps")
    table = summarize_events(layer, events, max(3, args.steps // 2))

    value = layer.flops * world / (ms_step * 1e-3) / 1e12
    gemm_ms = sum(r["gemm_ms"] for r in table.values())
    quant_ms = sum(r["quant_ms"] for r in table.values())
    gemm_achieved = layer.flops / (gemm_ms * 1e-3) / 1e12
    ratio = {"bf16": 1, "fp8_current": 2, "fp8_delayed": 2, "mxfp8": 2, "mxfp8_e5m2": 2, "mxfp4": 6,
             "nvfp4": 6}[recipe]
    # The timed region is well under a second at the maximum SM clock: the
    # burst bf16 figure x the format's nominal dense ratio is the denominator.
    if peaks:
        peak = peaks["bf16_tflops"] * ratio
        peak_src = f"of measured: bf16_tflops (burst) x {ratio} (nominal dense ratio of the format)"
    else:
        peak = 1900.0 * ratio
        peak_src = f"of fallback: 1.9 PFLOP/s bf16 burst x {ratio}"
    # the tensor-core ceiling of the MMA shape the kernel issues, measured now
    mma_kind = {"bf16": "bf16", "fp8_current": "fp8", "fp8_delayed": "fp8", "mxfp8": "mxfp8",
                "mxfp8_e5m2": "mxfp8", "mxfp4": "nvfp4", "nvfp4": "nvfp4"}[recipe]
    ceiling = lpq.mma_peak(mma_kind, iters=8000, with_scale_copies=6)
    check_device("the tensor-core rate probe")
    algo_bytes = 0
    for name, lay, m, k, n in layer.shapes:
        per = {"nvfp4": 0.5 + 1 / 16, "mxfp8": 1 + 1 / 32, "mxfp8_e5m2": 1 + 1 / 32, "mxfp4": 0.5 + 1 / 32,
               "fp8_current": 1, "fp8_delayed": 1, "bf16": 2}[recipe]
        algo_bytes += (m * k + n * k) * per + m * n * 2
    # the committed counters were taken on the default CodonFM-5B layer (M = 15872, hidden 4096,
    # intermediate 16384): other shapes get no traffic figure
    default_layer = (layer.M, args.hidden_size, args.intermediate_size) == (15872, 4096, 16384)
    traffic = (profiled_traffic(os.path.join(ROOT, "precision_transformer_gemms_gb300", "csrc", "gemm.cu"), recipe)
               if default_layer and autocast else None)
    roof = {"bound": "tensor", "achieved": gemm_achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": gemm_achieved / peak, "traffic": traffic, "kernel": f"gemm_pair_kernel ({recipe})",
            "peak_source": peak_src, "algorithmic_bytes_per_launch": algo_bytes / len(layer.shapes),
            "tcgen05_ceiling": {"value": ceiling, "unit": "TFLOP/s", "frac": gemm_achieved / ceiling,
                                "how": f"lpq_mma_peak {mma_kind}, CTA pairs (256 x 256 MMAs), operands in shared "
                                       "memory, measured in this run"},
            "datasheet": {"value": DATASHEET_DENSE_TFLOPS[mma_kind], "unit": "TFLOP/s",
                          "frac": gemm_achieved / DATASHEET_DENSE_TFLOPS[mma_kind],
                          "how": "nominal dense (no 2:4 sparsity) per-GPU rate of the format"}}
    if recipe != "bf16" and autocast:
        qb = quant_bytes_per_layer(layer, recipe)
        roof["quantize"] = {"bound": "hbm", "bytes_per_layer": qb, "ms_per_layer": quant_ms,
                            "achieved": qb / (quant_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                            "frac": qb / (quant_ms * 1e-3) / 1e9 / hbm,
                            "how": "per-GEMM autocast: every GEMM quantizes one copy of each operand; bytes per "
                                   f"element {QUANT_BYTES_PER_ELEM[recipe]:.4f} (amax pass where the recipe has one, "
                                   "bf16 read, codes and scales written); time = CUDA events around the quantize "
                                   "calls of the per-kernel steps"}
        if not args.no_quant_kinds:
            roof["quantize"]["kinds"] = time_quant_kinds(layer, hbm)

    # e2e (right after the headline, before the recipe sweep: after the sweep's tens of
    # seconds the host link was seen to run slower): every step copies its bf16 inputs
    # from pinned host memory and its
    # outputs back to pinned host memory.  Copies run on their own streams,
    # double-buffered (inputs of step s+1 and outputs of step s-1 move while
    # step s computes); events order each buffer's reuse.
    e2e = None
    if not args.no_e2e:
        host_in = {lin: {r: t.cpu().pin_memory() for r, t in d.items()} for lin, d in layer.inp.items()}
        host_out = [{n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in layer.out.items()}
                    for _ in range(2)]
        inp_sets = [layer.inp, {lin: {r: torch.empty_like(t) for r, t in d.items()} for lin, d in layer.inp.items()}]
        out_sets = [layer.out, {n: torch.empty_like(t) for n, t in layer.out.items()}]
        bi, bo = layer.step_io_bytes()
        steps = max(3, args.steps // 2)
        comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_comp, ev_out = [None, None], [None, None]
        in_list = [(lin, r) for lin, d in layer.inp.items() for r in d]
        out_list = list(layer.out)

        def e2e_step(s):
            k = s % 2
            with torch.cuda.stream(s_in):
                if ev_comp[k] is not None:
                    s_in.wait_event(ev_comp[k])  # step s-2 no longer reads input set k
                for lin, r in in_list:
                    inp_sets[k][lin][r].copy_(host_in[lin][r], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            comp.wait_event(ev_in)
            if ev_out[k] is not None:
                comp.wait_event(ev_out[k])  # outputs of step s-2 have left output set k
            layer.inp, layer.out = inp_sets[k], out_sets[k]
            layer.step(recipe, autocast, s)
            ev_comp[k] = torch.cuda.Event()
            ev_comp[k].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[k])
                for n in out_list:
                    host_out[k][n].copy_(out_sets[k][n], non_blocking=True)
                ev_out[k] = torch.cuda.Event()
                ev_out[k].record(s_out)

        # warm-up: every buffer of both sets touched, and the host link past its slow first
        # copies on a fresh box (seen to last more than half a second): at least max(3, W)
        # steps and at least three seconds of steps
        t_w = time.perf_counter()
        w = 0
        while w < max(3, args.warmup) or (time.perf_counter() - t_w < 3.0 and w < 200):
            e2e_step(w)
            w += 1
            if w >= max(3, args.warmup):
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for s in range(steps):
            e2e_step(100 + s)
        torch.cuda.synchronize()
        barrier(world)
        dt = max_over_ranks((time.perf_counter() - t0) / steps, world)
        check_device("the end-to-end steps")
        layer.inp, layer.out = inp_sets[0], out_sets[0]
        e2e = {"value": layer.flops * world / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": dt * 1e3,
               "copies": "pinned host <-> device, one copy stream per direction, double-buffered against the "
                         "compute stream"}
        del host_in, host_out, inp_sets, out_sets

    # the data-parallel step on this rank alone (exchanges are no-ops at N = 1):
    # each tensor quantized once into both copies, then the three GEMMs
    dp_step = None
    if not tokens and recipe != "bf16":
        lins = make_dp_linears(layer, recipe)
        k = max(3, args.steps // 4)
        ms = time_fn(lambda s: [lin.step(seed=s) for lin in lins], k, 2, 1)
        check_device("the data-parallel step")
        dp_step = {"ms_per_layer": ms, "tflops": layer.flops / (ms * 1e-3) / 1e12,
                   "what": "precision_transformer_gemms_gb300.dp.TokenShardedLinear x 4 on one rank: amax passes, "
                           "all-reduce MAX (a no-op on one rank), each tensor quantized once into both copies, "
                           "Fprop, Dgrad, FP32 Wgrad partial, all-reduce SUM (no-op); under torchrun with "
                           "--parallel tokens the same step runs with NCCL exchanges"}
        del lins
        torch.cuda.empty_cache()

    # recipe sweep (fewer steps each)
    recipes = {}
    if not args.no_sweep:
        sweep = sweep_recipes(args)
        k = max(3, args.steps // 4)
        for r in sweep:
            layer.prequantize(r)
            res = {}
            for mode in ("autocast", "prequant"):
                ac = mode == "autocast" or r == "fp8_delayed"
                if r == "bf16":
                    ac = False
                ms, _ = time_steps(layer, r, ac, k, 2, world)
                res[f"{mode}_ms_per_layer"] = ms
                res[f"{mode}_tflops"] = layer.flops / (ms * 1e-3) / 1e12
            if r != "bf16":
                res["fused_ms_per_layer"] = time_fn(lambda s_: layer.fused_step(r, s_), k, 2, 1)
                res["fused_tflops"] = layer.flops / (res["fused_ms_per_layer"] * 1e-3) / 1e12
            check_device(f"the {r} sweep")
            recipes[r] = res
            # free this recipe's buffers before the next one
            for key in [k_ for k_ in layer.bufs if k_[0] == r and r != recipe]:
                del layer.bufs[key]
            torch.cuda.empty_cache()
        if "bf16" in recipes:
            # BF16 does the same work in both modes: the faster run is the baseline
            b = min(recipes["bf16"]["prequant_ms_per_layer"], recipes["bf16"]["autocast_ms_per_layer"])
            recipes["bf16"]["baseline_ms_per_layer"] = b
            for r, res in recipes.items():
                for mode in ("autocast", "prequant", "fused"):
                    if f"{mode}_ms_per_layer" in res:
                        res[f"{mode}_speedup_vs_bf16"] = b / res[f"{mode}_ms_per_layer"]

    # the FP8 drift run and the K-sweep (the other configurations' workloads), on rank 0
    drift = ksweep = None
    if rank == 0 and not args.no_drift:
        d = drift_results(args)
        drift = {sc: {"mean_ms_per_step": round(v["mean_ms"], 4),
                      "saturated_per_step": [r["saturated"] for r in v["steps"]],
                      "x_amax_first_last": [v["steps"][0]["x_amax"], v["steps"][-1]["x_amax"]]}
                 for sc, v in d.items()}
        drift["workload"] = (f"per-tensor FP8 (E4M3 X/W, E5M2 dY), attention-out GEMMs M={layer.M}, "
                             f"K=N={args.hidden_size}, 20 steps, X std 1 -> 4, Fprop+Dgrad+Wgrad autocast")
    if rank == 0 and not args.no_ksweep:
        kres = ksweep_results(reps=5)
        ksweep = {"workload": "8192 x K x 8192 GEMMs, speed-up vs the bf16 tcgen05 GEMM",
                  "prequant_speedup": {K: {f: round(v[f]["prequant_speedup_vs_bf16"], 3) for f in v
                                           if isinstance(v[f], dict)} for K, v in kres.items()},
                  "autocast_speedup": {K: {f: round(v[f]["autocast_speedup_vs_bf16"], 3) for f in v
                                           if isinstance(v[f], dict)} for K, v in kres.items()},
                  "bf16_tflops": {K: round(v["bf16_tflops"], 1) for K, v in kres.items()},
                  "prequant_tflops": {K: {f: round(v[f]["prequant_tflops"], 1) for f in v
                                          if isinstance(v[f], dict)} for K, v in kres.items()}}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle as o
        lins = [(n, K, N) for n, (K, N) in layer.linears.items()]
        shapes = [(n, lay, m, k, nn) for n, lay, m, k, nn in layer.shapes]
        t0 = time.perf_counter()
        sec, info = oracle_sample(shapes, layer.M, lins, rows=32, cols=256, slab=16)
        wall = time.perf_counter() - t0
        cpu = {"value": layer.flops / sec / 1e12, "unit": "TFLOP/s", "cores": o.num_threads(), "kind": "oracle",
               "sample": "per GEMM 32x256 outputs of the FP64 oracle GEMM on NVFP4 operands plus the NVFP4 "
                         "quantization of those operand rows, projected to the full layer (quantize share %.2f%%)"
                         % (100 * info["quant_s"] / sec),
               "wall_s": wall}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"nvfp4": "e2m1", "mxfp8": "e4m3", "mxfp8_e5m2": "e4m3/e5m2", "mxfp4": "e2m1",
                      "fp8_current": "e4m3/e5m2", "fp8_delayed": "e4m3/e5m2", "bf16": "bf16"}[recipe],
            "data": "synthetic",
            "config": contract_config(args, world, recipe, autocast),
            "roofline": roof,
            "quantize": {"ms_per_layer": quant_ms, "gemm_ms_per_layer": gemm_ms},
            "device_status": status,
            "recipes": recipes,
            "dp_step": dp_step,
            "drift": drift,
            "ksweep": ksweep,
            "gemms": {n: {kk: (round(v, 4) if isinstance(v, float) else v) for kk, v in r.items()}
                      for n, r in table.items()},
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launches * args.steps,
            "hbm_peak_gbs": hbm,
        }
        if args.output:
            json.dump(line, open(args.output, "w"), indent=1)
        print(json.dumps(line), flush=True)


def run_mma_peaks(args):
    """Dense tcgen05 rates per kind, operands resident in shared memory."""
    import torch
    from precision_transformer_gemms_gb300 import lpq
    torch.cuda.set_device(0)
    clocks = ClockSampler(0)
    clocks.start()
    out = {}
    for kind in ("bf16", "fp8", "mxfp8", "nvfp4"):
        iters = 40000 if kind == "nvfp4" else 20000
        out[kind] = lpq.mma_peak(kind, iters=iters, with_scale_copies=False)
        if kind in ("mxfp8", "nvfp4"):
            out[kind + "_with_scale_copies"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=1)
        if kind == "nvfp4":
            out[kind + "_scale_copies_two_regions"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=2)
            out[kind + "_scale_copies_interleaved"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=3)
            out[kind + "_scales_stored_by_warps"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=4)
            out[kind + "_scale_copies_by_other_warp"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=5)
        # CTA pairs (cta_group::2, 256 x 256 MMAs): the shape the product GEMM issues
        out[kind + "_pair"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=6)
        out[kind + "_pair_n128_halves"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=8)
        if kind in ("mxfp8", "nvfp4"):
            out[kind + "_pair_scales_stored_by_warps"] = lpq.mma_peak(kind, iters=iters, with_scale_copies=7)
    out["clocks"] = clocks.stop()
    out["unit"] = "TFLOP/s"
    print(json.dumps(out), flush=True)


def _event_ms(fn, reps):
    import torch
    for _ in range(2):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def ksweep_results(reps=10, ks=(1024, 2048, 4096, 8192, 16384)):
    """Scaling-granularity K-sweep ("Faster training throughput in FP8 with
    NVIDIA NeMo", scaling up recipe granularity): 8192 x K x 8192 GEMMs
    (inputs ~N(0,1), 0.1% entries x100) under per-tensor FP8, MXFP8,
    sub-channel FP8 (1x128 act, 128x128 weight), NVFP4 (1D act, 2D weight),
    MXFP4 and bf16; pre-quantize (GEMM only) and autocast (quantize both
    operands + GEMM) times and speed-ups vs the bf16 tcgen05 GEMM of the same
    shape.  The device error word is checked after each K."""
    import torch
    from precision_transformer_gemms_gb300 import lpq, synth
    M = N = 8192
    fmts = {"fp8_current": (lpq.FP8_E4M3, lpq.FP8_E4M3), "mxfp8": (lpq.MXFP8, lpq.MXFP8),
            "fp8_subchannel": (lpq.FP8_BLOCK_1x128, lpq.FP8_BLOCK_128x128), "nvfp4": (lpq.NVFP4, lpq.NVFP4_2D),
            "mxfp4": (lpq.MXFP4, lpq.MXFP4)}
    out = {}
    for K in ks:
        A = synth.bf16_normal((M, K), 1.0, 50, "cuda", 0.001, 100.0)
        B = synth.bf16_normal((N, K), 1.0, 51, "cuda", 0.001, 100.0)
        C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        ca, cb = lpq.Copy.of_bf16(A), lpq.Copy.of_bf16(B)
        flops = 2 * M * N * K
        row = {"bf16_ms": _event_ms(lambda: lpq.gemm(lpq.FPROP, ca, cb, c=C), reps)}
        for name, (fa, fb) in fmts.items():
            qa, qb = lpq.alloc(fa, M, K, lpq.ROWWISE), lpq.alloc(fb, N, K, lpq.ROWWISE)

            def quant():
                lpq.quantize(A, fa, lpq.ROWWISE, out=qa)
                lpq.quantize(B, fb, lpq.ROWWISE, out=qb)

            quant()
            g = _event_ms(lambda: lpq.gemm(lpq.FPROP, qa.row, qb.row, c=C), reps)
            ac = _event_ms(lambda: (quant(), lpq.gemm(lpq.FPROP, qa.row, qb.row, c=C)), reps)
            row[name] = {"prequant_ms": g, "autocast_ms": ac, "prequant_tflops": flops / g / 1e9,
                         "prequant_speedup_vs_bf16": row["bf16_ms"] / g, "autocast_speedup_vs_bf16": row["bf16_ms"] / ac}
            del qa, qb
        row["bf16_tflops"] = flops / row["bf16_ms"] / 1e9
        check_device(f"K-sweep K={K}")
        out[K] = row
        del A, B, C
        torch.cuda.empty_cache()
    return out


def run_ksweep(args):
    import torch
    torch.cuda.set_device(0)
    out = ksweep_results()
    print(json.dumps({"workload": "K-sweep 8192 x K x 8192", "unit": "ms / TFLOP/s", "results": out}), flush=True)


def drift_results(args, steps=20):
    """Per-tensor FP8 current vs delayed scaling on the attention-output GEMMs
    (M = micro-batch x sequence tokens, hidden x hidden weight) over 20 steps
    whose activation std drifts 1 -> 4 (gradients std 1e-3); Fprop + Dgrad +
    Wgrad each step, autocast.  Per step: the ms, the amax, the scale in use
    and how many activations exceed the E4M3 range at that scale (a
    device-side count).  Every step's codes are compared with the oracle in
    the GPU tests."""
    import torch
    from precision_transformer_gemms_gb300 import lpq, synth
    M, K, N = args.micro_batch_size * args.sequence_length, args.hidden_size, args.hidden_size
    W = synth.bf16_normal((N, K), synth.WEIGHT_STD, 1, "cuda")
    both = lpq.ROWWISE | lpq.COLWISE
    res = {}
    for scaling in ("current", "delayed"):
        sc = lpq.SCALING_DELAYED if scaling == "delayed" else lpq.SCALING_CURRENT
        st = {r: lpq.DelayedState(16) for r in ("X", "W", "dY")}
        bufs = {"X": lpq.alloc(lpq.FP8_E4M3, M, K, both), "W": lpq.alloc(lpq.FP8_E4M3, N, K, both),
                "dY": lpq.alloc(lpq.FP8_E5M2, M, N, both)}
        outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
                torch.empty((M, K), dtype=torch.bfloat16, device="cuda"),
                torch.empty((N, K), dtype=torch.bfloat16, device="cuda")]
        recs = []
        for t in range(steps):
            X = synth.bf16_normal((M, K), synth.drift_std(t), 10 * t, "cuda")
            dY = synth.bf16_normal((M, N), synth.GRAD_STD, 10 * t + 2, "cuda")
            x_scale = st["X"].scale.clone() if sc else None  # the scale this step's X is quantized with
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for role, x, fmt in (("X", X, lpq.FP8_E4M3), ("W", W, lpq.FP8_E4M3), ("dY", dY, lpq.FP8_E5M2)):
                lpq.quantize(x, fmt, both, scaling=sc, state=st[role] if sc else None, out=bufs[role])
                if sc:
                    lpq.scale_update(st[role], bufs[role].row.amax, lpq.FMAX[fmt])
            lpq.gemm(lpq.FPROP, bufs["X"].row, bufs["W"].row, c=outs[0])
            lpq.gemm(lpq.DGRAD, bufs["dY"].row, bufs["W"].col, c=outs[1])
            lpq.gemm(lpq.WGRAD, bufs["dY"].col, bufs["X"].col, c=outs[2])
            e1.record()
            torch.cuda.synchronize()
            rec = {"ms": e0.elapsed_time(e1), "x_amax": float(bufs["X"].row.amax.item()),
                   "x_scale_inv": float(bufs["X"].row.tensor_scale.item())}
            # diagnostic (outside the timed region): |X * scale| > 448 in fp32, the scale being
            # 448 / amax (current) or the delayed state's scale before this step's update
            scale = x_scale if sc else 448.0 / bufs["X"].row.amax
            rec["saturated"] = int(((X.float() * scale).abs() > 448.0).sum().item())
            recs.append(rec)
        check_device(f"drift ({scaling})")
        res[scaling] = {"steps": recs, "mean_ms": statistics.mean(r["ms"] for r in recs[2:])}
        del bufs, outs
        torch.cuda.empty_cache()
    return res


def run_drift(args):
    import torch
    torch.cuda.set_device(0)
    res = drift_results(args)
    M, K = args.micro_batch_size * args.sequence_length, args.hidden_size
    print(json.dumps({"workload": f"FP8 drift, attention-out M={M} K=N={K}, 20 steps", "results": res}), flush=True)


# GEMM-only speed-up / step speed-up above which the overhead outside the GEMMs
# is read as consuming the gain (the pages contrast "about equal" with "much
# larger" and give no number).
OVERHEAD_RATIO = 1.25


def step_diagnostic(gemm_only, step):
    """The pages' reading of a GEMM-only (pre-quantized) speed-up against the
    step's (here: the autocast layer, quantization included), from [TE]
    "interpreting real-model results"."""
    if gemm_only < 1.0:
        return "below 1.0 even kernel-only: not faster on these shapes (or a silent fallback)"
    if gemm_only / step > OVERHEAD_RATIO:
        return ("GEMM-only speed-up well above the step's: work outside the GEMMs (quantization: amax pass, "
                "RHT, stochastic rounding, 2D weight scaling for NVFP4) consumes the gain")
    return "GEMM-only speed-up close to the step's: the GEMMs dominate, as expected"


def report_tables(per, shapes_list, linears, layers=None):
    """Tables of the speed-up analysis from per-GEMM times: per[recipe][mode][gemm] = ms.
    `layers` (the model's layer count) scales the per-layer times into the
    end-to-end projection."""
    shapes = {n: (m, k, nn) for n, _, m, k, nn in shapes_list}
    names = [n for n, *_ in shapes_list]
    # BF16 does the same work in both modes; the faster of its two runs is the
    # baseline (the run order can cost a few percent under the power cap).
    base = ({n: min(per["bf16"]["autocast"][n], per["bf16"]["prequant"][n]) for n in per["bf16"]["prequant"]}
            if "bf16" in per else None)
    out = {"workload": "speed-up analysis, CodonFM-5B layer (12 GEMMs)", "unit": "ms", "per_gemm": per}
    if base:
        out["speedup_vs_bf16"] = {r: {m: {n: base[n] / per[r][m][n] for n in names} for m in per[r]} for r in per}
        out["below_bf16"] = [f"{r}/{m}/{n}" for r in per for m in per[r] for n in names
                             if r != "bf16" and base[n] / per[r][m][n] < 1.0]
    if "nvfp4" in per and "mxfp8" in per:
        fprop = [n for n in names if n.endswith("_fprop")]
        ratios = {}
        for m in ("autocast", "prequant"):
            ratios[m] = {n: per["mxfp8"][m][n] / per["nvfp4"][m][n] for n in fprop}
            ratios[m]["blended_fprop"] = (sum(per["mxfp8"][m][n] for n in fprop) /
                                         sum(per["nvfp4"][m][n] for n in fprop))
        out["nvfp4_vs_mxfp8"] = ratios
    out["dgrad_vs_fprop"] = {r: {lin: per[r]["autocast"][f"{lin}_dgrad"] / per[r]["autocast"][f"{lin}_fprop"]
                                 for lin in linears} for r in per}
    if base:
        # End-to-end projection: the layer's 12 GEMMs (with their quantization in
        # autocast) times the layer count, and the diagnostic of the GEMM-only
        # (pre-quantized) speed-up against the step's (autocast).
        base_layer = sum(base[n] for n in names)
        proj = {}
        for r in per:
            lay = {m: sum(per[r][m][n] for n in names) for m in per[r]}
            g_only, step = base_layer / lay["prequant"], base_layer / lay["autocast"]
            proj[r] = {"layer_ms": lay, "gemm_only_speedup": g_only, "step_speedup": step,
                       "diagnostic": "the baseline" if r == "bf16" else step_diagnostic(g_only, step)}
            if layers:
                proj[r]["model_ms"] = {m: layers * v for m, v in lay.items()}
        out["projection"] = {"layers": layers, "recipes": proj}
    # human-readable tables
    lines = []
    for m in ("autocast", "prequant"):
        lines.append(f"== {m} (ms per GEMM; speed-up vs BF16 in parentheses)")
        lines.append(f"{'GEMM':16s} {'m x k x n':22s} " + " ".join(f"{r:>16s}" for r in per))
        for n in names:
            mm, kk, nn = shapes[n]
            cells = []
            for r in per:
                v = per[r][m][n]
                cells.append(f"{v:8.3f} ({base[n] / v:4.2f}x)" if base else f"{v:16.3f}")
            lines.append(f"{n:16s} {f'{mm}x{kk}x{nn}':22s} " + " ".join(f"{c:>16s}" for c in cells))
    if "nvfp4_vs_mxfp8" in out:
        for m, rr in out["nvfp4_vs_mxfp8"].items():
            lines.append(f"NVFP4 vs MXFP8 Fprop ({m}): " + ", ".join(f"{n} {v:.2f}x" for n, v in rr.items()))
    if base:
        for r, v in out["projection"]["recipes"].items():
            model = f", {layers} layers {v['model_ms']['autocast']:.1f} ms" if layers else ""
            lines.append(f"{r}: GEMM-only {v['gemm_only_speedup']:.2f}x, step {v['step_speedup']:.2f}x{model}: "
                         f"{v['diagnostic']}")
        lines.append("below BF16: " + (", ".join(out["below_bf16"]) or "none"))
    return out, lines


def run_report(args):
    """The speedup analysis of the pages' tool for the CodonFM-5B layer: every
    GEMM shape timed separately (Fprop, Dgrad and Wgrad alike) under every
    enabled precision, in autocast (quantization of the GEMM's two operand
    copies + GEMM) and pre-quantize (GEMM only) mode.  Prints per-shape tables
    and speed-ups vs BF16 on stderr, and one JSON line with the numbers:
    per-shape NVFP4 / MXFP8 Fprop ratios and their blend, Dgrad vs Fprop per
    linear, the shapes whose speed-up vs BF16 is below 1 (not faster, or
    a silent fallback, which lpq does not have), and the end-to-end projection
    to the model's layer count with the GEMM-only vs step diagnostic."""
    import torch
    torch.cuda.set_device(0)
    layer = Layer(args, "cuda:0")
    sweep = sweep_recipes(args)
    steps = max(3, args.steps // 4)
    per = {}  # recipe -> mode -> gemm name -> ms
    for r in sweep:
        layer.prequantize(r)
        per[r] = {}
        for mode in ("autocast", "prequant"):
            ac = (mode == "autocast" or r == "fp8_delayed") and r != "bf16"
            _, events = time_steps(layer, r, ac, steps, 2, 1, per_kernel=True)
            table = summarize_events(layer, events, steps)
            per[r][mode] = {n: row["gemm_ms"] + row["quant_ms"] for n, row in table.items()}
        for key in [k_ for k_ in layer.bufs if k_[0] == r]:
            del layer.bufs[key]
        torch.cuda.empty_cache()
    out, lines = report_tables(per, layer.shapes, layer.linears, args.num_hidden_layers)
    print("\n".join(lines), file=sys.stderr, flush=True)
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.mma_peaks:
        run_mma_peaks(args)
        return
    if args.workload == "ksweep":
        run_ksweep(args)
        return
    if args.workload == "drift":
        run_drift(args)
        return
    if args.workload == "report":
        run_report(args)
        return
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_lpq(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
