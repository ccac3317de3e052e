"""GEMM throughput on one GB300 (or N replicas), one JSON line on rank 0.

A step is one call of the hot path: gemm_run (or grouped_gemm_run) on the
workload's resident device inputs.  Default workload: the gate+up projection
of a Llama-3.3-70B layer in bf16 at 8192 tokens (X [8192, 8192] times
W [8192, 57344], beta 0), the largest single-GPU shape of the Llama linear
layers that are 89% of that model's runtime ("Generating State-of-the-Art
GEMMs with TorchInductor's CuteDSL backend", section 2).  The metric is
TFLOP/s = 2*M*N*K / time; the L2 is flushed (256 MiB write, then a 256 MiB
read that leaves it holding clean lines) between timed steps, outside the
per-step CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of GB300 dense tensor peak per shape (1 GPU)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
ROTATE_BYTES = 2 * (129 << 20)  # --flush rotate: the copies of the inputs fill twice the L2
KERNEL_SOURCES = ("gemm_kernel.cuh", "ptx.cuh", "gemm_params.h", "gemm15_api.cu")


# ------------------------------------------------------------------ workloads

def workloads():
    from dense_gemm_15_gb300 import inputs as I
    w = {
        "fp16_4096x4096x4096_relu": lambda: [I.config2()],
        "fp16_1024_uniform": lambda: [I.config1("b")],
        "fp16_1024_ones": lambda: [I.config1("a")],
        "fp16_grouped_32": lambda: I.config4(),
        # the same group shapes in fp8 with per-group scales (CuteDSL page, section 5.1)
        "e4m3_grouped_32": lambda: I.config4_e4m3(),
        "e4m3_8192": lambda: [I.config5b()],
        # the bias + ReLU epilogue example of the kwkr.cn blog, section 5.2
        "fp16_bias_relu_512x1024x768": lambda: [I.random_problem(512, 1024, 768, act="relu",
                                                                 bias=True)],
        # batch_count 16 of one shape, packed strides (kwkr.cn blog section 6.3)
        BATCHED_WORKLOAD: lambda: [I.random_problem(1024, 1024, 1024, seed=b) for b in range(16)],
        # block-scaled _scaled_mm formats (CuteDSL page, section 5.1)
        "mxfp8_e4m3_8192": lambda: [I.block_scaled_problem(8192, 8192, 8192, elem="e4m3")],
        "mxfp4_8192": lambda: [I.block_scaled_problem(8192, 8192, 8192, elem="e2m1")],
        "nvfp4_8192": lambda: [I.block_scaled_problem(8192, 8192, 8192, elem="e2m1", block=16,
                                                      scale="e4m3")],
    }
    for layer in I.LLAMA70B_LAYERS:
        for m in I.LLAMA70B_TOKENS:
            w["bf16_llama70b_%s_m%d" % (layer, m)] = (lambda m=m, layer=layer: [I.config3(m, layer)])
    for (M, N, K) in I.STREAMK_SHAPES:
        w["fp16_streamk_%dx%dx%d" % (M, N, K)] = (lambda M=M, N=N, K=K: [I.config5a(M, N, K)])
    return w


DEFAULT_WORKLOAD = "bf16_llama70b_gate_up_m8192"
BATCHED_WORKLOAD = "fp16_batched_16x1024x1024x1024"


def custom_workload(name):
    """custom_<f16|bf16|e4m3>_<M>x<N>x<K>[_b<beta>][_relu|_sigmoid|_tanh][_bias][_acol][_bcol]:
    seeded U[-1,1] (N(0,1) for e4m3) operands of any shape, for sweeps and ablations."""
    from dense_gemm_15_gb300 import inputs as I
    parts = name.split("_")
    dtype = parts[1]
    M, N, K = (int(x) for x in parts[2].split("x"))
    beta = 0.0
    relu = acol = bcol = bias = False
    act = None
    for q in parts[3:]:
        if q == "relu":
            relu = True
        elif q in ("sigmoid", "tanh"):
            act = q
        elif q == "bias":
            bias = True
        elif q == "acol":
            acol = True
        elif q == "bcol":
            bcol = True
        elif q.startswith("b"):
            beta = float(q[1:])
    p = I.random_problem(M, N, K, dtype=dtype, beta=beta, relu=relu, alpha=1.0,
                         a_col_major=acol, b_col_major=bcol, act=act, bias=bias)
    p.name = name
    return [p]


def get_workload(name):
    if name.startswith("custom_"):
        return custom_workload(name)
    return workloads()[name]()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# nominal dense tensor-core ratios to bf16 (2.25 / 4.5 / 13.5 PFLOP/s on GB300)
PEAK_RATIO = {"f16": 1.0, "bf16": 1.0, "e4m3": 2.0, "e5m2": 2.0, "e2m1": 6.0}


def tensor_peak(dtype, pk, sustained=False):
    bf16 = pk["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return bf16 * PEAK_RATIO[dtype]


def code_only(src: str) -> str:
    """C / C++ source without its comments, whitespace runs collapsed to one
    space: what the compiler sees, so that the hash below follows the code
    and not the comments (string and character literals are kept whole)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_hash():
    """Identity of the kernel sources' code (comments excluded), which a
    recorded DRAM traffic figure is tied to."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_gemm_15_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
            h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the main kernel from a committed ncu summary,
    or None when none exists or the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


def algorithmic_bytes(probs):
    tot = 0
    for p in probs:
        ea = {"e4m3": 1, "e5m2": 1, "e2m1": 0.5}.get(p.a_dtype, 2)
        tot += int(p.M * p.K * ea + p.K * p.N * ea) + p.M * p.N * 2
        scales = getattr(p, "block_scales", None)
        if scales is not None:  # one byte per block of A's rows and B's columns
            tot += (p.M + p.N) * (p.K // scales[3])
        if p.beta != 0.0:
            tot += p.M * p.N * 2
        if getattr(p, "bias", None) is not None:
            tot += p.N * 2
        if getattr(p, "aux", None) is not None:
            tot += p.M * p.N * 2
        if getattr(p, "pre", None) is not None:
            tot += p.M * p.N * 2
    return tot


def roofline_entry(flops, abytes, ms, dtype, pk, pk_kind, traffic):
    """The roofline object of the JSON line for one launch of `flops` FLOPs
    and `abytes` algorithmic bytes taking `ms` milliseconds.  The bound is the
    roof the shape's arithmetic intensity meets first: HBM below the ridge
    point (peak FLOP/s / HBM bytes/s), the tensor pipe above it."""
    peak = tensor_peak(dtype, pk)
    achieved = flops / (ms * 1e-3) / 1e12
    achieved_gbs = abytes / (ms * 1e-3) / 1e9
    ridge = peak * 1e12 / (pk["hbm_gbs"] * 1e9)
    if flops / abytes < ridge:
        return {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved_gbs / pk["hbm_gbs"], "traffic": traffic,
                "peak_source": "%s HBM copy" % pk_kind, "algorithmic_bytes": abytes,
                "achieved_tflops": achieved, "intensity_flop_per_byte": flops / abytes}
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": "%s bf16 burst%s" % (
                pk_kind, "" if PEAK_RATIO[dtype] == 1.0 else
                " x%g (%s, nominal dense ratio)" % (PEAK_RATIO[dtype], dtype)),
            "algorithmic_bytes": abytes, "achieved_gbs": achieved_gbs,
            "intensity_flop_per_byte": flops / abytes}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.proc or not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        loaded = [s for s in sm if s > 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline

def _column_sample(p, cols):
    """Views of the operands for columns 0..cols of D (B's first cols columns,
    C's and the bias's too): the oracle decodes only those columns of B."""
    from dense_gemm_15_gb300 import inputs as I
    b = I.bits(p.B)
    b = b[:cols, :] if p.b_col_major else b[:, :cols]
    c = I.bits(p.C)[:, :cols] if p.C is not None and p.beta != 0.0 else None
    bv = I.bits(p.bias)[:cols] if p.bias is not None else None
    sc = getattr(p, "block_scales", None)
    scales = (I.bits(sc[0]), I.bits(sc[1])[:, :cols], sc[2], sc[3]) if sc is not None else None
    return b, c, bv, scales


def cpu_oracle_sample(probs, budget_s=10.0, max_rows=None):
    """Times the oracle (as it stands) on a bounded sample of the workload:
    rows 0..r and columns 0..c of D (whole K), growing first c up to 2048,
    then r up to M, then c up to N, until one run takes about half the budget.
    Returns (flops/s, cores, description, seconds)."""
    import oracle
    from dense_gemm_15_gb300 import inputs as I
    p = max(probs, key=lambda q: q.flops)
    threads = oracle.default_threads()
    a = I.bits(p.A)

    def run(rows, cols):
        b, c, bv, scales = _column_sample(p, cols)
        t0 = time.perf_counter()
        oracle.gemm(a, p.a_dtype, b, p.b_dtype, c, p.c_dtype, alpha=p.alpha, beta=p.beta,
                    act=p.act, bias=bv, bias_dtype=p.d_dtype, scale_a=p.scale_a,
                    scale_b=p.scale_b, a_col_major=p.a_col_major, b_col_major=p.b_col_major,
                    rows=(0, rows), threads=threads, scales=scales)
        return time.perf_counter() - t0

    cols = min(p.N, 2048)
    rows = min(p.M, max(1, threads))
    dt = run(rows, cols)
    while dt < 0.5 * budget_s and (rows < p.M or cols < p.N):
        grow = min(8.0, 0.8 * budget_s / max(dt, 1e-3))
        if rows < p.M and not (max_rows and rows >= max_rows):
            rows = min(p.M, max(rows + 1, int(rows * grow)))
            if max_rows:
                rows = min(rows, max_rows)
        else:
            cols = min(p.N, max(cols + 1, int(cols * grow)))
        dt = run(rows, cols)
    flops = 2.0 * rows * cols * p.K
    desc = "rows 0..%d x columns 0..%d of %s (full K=%d)" % (rows, cols, p.name, p.K)
    return flops / dt, threads, desc, dt, rows, cols


# ------------------------------------------------------------------ distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def maybe_init_dist(ws, backend):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x, device=None):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x, device=None):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The oracle as it stands, timed on the host cores; each step is the same
    bounded row sample of the workload, sized so the whole run stays within
    about two minutes."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from dense_gemm_15_gb300 import inputs as I
    probs = get_workload(args.workload)
    per_step = min(args.cpu_budget, 120.0 / max(1, args.steps + args.warmup))
    _, cores, desc, _, rows, cols = cpu_oracle_sample(probs, budget_s=per_step)
    p = max(probs, key=lambda q: q.flops)
    a = I.bits(p.A)
    b, c, bv, scales = _column_sample(p, cols)

    def step():
        oracle.gemm(a, p.a_dtype, b, p.b_dtype, c, p.c_dtype, alpha=p.alpha, beta=p.beta,
                    act=p.act, bias=bv, bias_dtype=p.d_dtype, scale_a=p.scale_a,
                    scale_b=p.scale_b, a_col_major=p.a_col_major, b_col_major=p.b_col_major,
                    rows=(0, rows), threads=cores, scales=scales)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = (time.perf_counter() - t0) / max(1, args.steps)
    value = 2.0 * rows * cols * p.K / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": p.M, "N": p.N, "K": p.K},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main arm

def run_gpu(args):
    import torch
    from dense_gemm_15_gb300 import binding as g
    from dense_gemm_15_gb300 import inputs as I

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = maybe_init_dist(ws, "nccl")
    dev = torch.device("cuda", local)
    probs = get_workload(args.workload)
    batched = args.workload == BATCHED_WORKLOAD
    grouped = len(probs) > 1
    p0 = probs[0]
    flops = sum(p.flops for p in probs)

    scaled = getattr(p0, "block_scales", None) is not None
    plan = g.Plan(p0.a_dtype, p0.d_dtype, epilogue=p0.act,
                  layout_a=g.COL_MAJOR if p0.a_col_major else g.ROW_MAJOR,
                  layout_b=g.COL_MAJOR if (p0.b_col_major or scaled) else g.ROW_MAJOR)
    for opt in args.opt or []:
        k, v = opt.split("=")
        plan.set(getattr(g, "OPT_" + k.upper()), int(v))
    dv = []
    if scaled:  # TN storage, packed fp4, scale atoms (inputs.block_scaled_storage)
        st_arrays = [torch.from_numpy(x).to(dev) for x in I.block_scaled_storage(p0)]
        scaled_kind = g.SCALE_NV if p0.block_scales[2] == "e4m3" else g.SCALE_MX
    for p in probs:
        if scaled:
            dv.append((st_arrays[0], st_arrays[1], None,
                       torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev)))
            continue
        A, B = p.A.to(dev), p.B.to(dev)
        C = p.C.to(dev) if p.C is not None else None
        D = torch.empty(p.M, p.N, dtype=I.TORCH_DTYPE[p.d_dtype], device=dev)
        dv.append((A, B, C, D))
    bias_dev = p0.bias.to(dev) if p0.bias is not None else None
    scales = None
    if p0.a_dtype == "e4m3":
        scales = (torch.tensor([p0.scale_a], device=dev), torch.tensor([p0.scale_b], device=dev))
    stream = torch.cuda.current_stream(dev)
    # "rotate": the dense and block-scaled workloads cycle through copies of
    # their inputs whose total is at least twice the L2, so that no step finds
    # its inputs cached and no flush kernel runs between steps
    rotate = args.flush == "rotate" and not grouped and not batched
    copies = 1
    if rotate:
        in_bytes = sum(t.numel() * t.element_size() for t in dv[0][:3] if t is not None)
        if scaled:
            in_bytes += sum(t.numel() * t.element_size() for t in st_arrays[2:])
        copies = max(2, min(64, -(-ROTATE_BYTES // max(in_bytes, 1))))
        if scaled:
            rot = [tuple(st_arrays)] + [tuple(t.clone() for t in st_arrays) for _ in range(copies - 1)]
        else:
            A0, B0, C0, D0 = dv[0]
            rot = [(A0, B0, C0)] + [(A0.clone(), B0.clone(), C0.clone() if C0 is not None else None)
                                    for _ in range(copies - 1)]
    rot_i = [0]
    flush = torch.empty(L2_FLUSH_BYTES // 4 if not rotate else 1, dtype=torch.float32, device=dev)
    flush_rd = (torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
                if args.flush == "write+read" else None)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def l2_flush():
        if rotate:
            return
        flush.zero_()
        if flush_rd is not None:
            # leave the L2 holding clean lines: the written ones are evicted here
            torch.sum(flush_rd, dim=0, out=flush_sink)
    table = [dict(M=p.M, N=p.N, K=p.K, A=A, B=B, C=C, D=D) for p, (A, B, C, D) in zip(probs, dv)]
    if grouped and p0.a_dtype == "e4m3":  # per-group fp8 scales
        for t, p in zip(table, probs):
            t["scale_a"] = torch.tensor([p.scale_a], dtype=torch.float32, device=dev)
            t["scale_b"] = torch.tensor([p.scale_b], dtype=torch.float32, device=dev)
    if batched:
        # one buffer per operand, entries at packed strides
        bA = torch.stack([A for A, _, _, _ in dv])
        bB = torch.stack([B for _, B, _, _ in dv])
        bD = torch.empty(len(probs), p0.M, p0.N, dtype=I.TORCH_DTYPE[p0.d_dtype], device=dev)
        del dv[1:]

    def step():
        r = rot_i[0] % copies
        rot_i[0] += 1
        if scaled:
            A, B, _, D = dv[0]
            sfa, sfb = st_arrays[2], st_arrays[3]
            if rotate:
                A, B, sfa, sfb = rot[r]
            st = g.gemm_run_block_scaled(plan.handle, A, B, sfa, sfb, D,
                                         p0.M, p0.N, p0.K, scale_kind=scaled_kind,
                                         alpha=p0.alpha, stream=stream)
            if st != g.OK:
                raise RuntimeError("gemm_run_block_scaled: " + g.status_string(st))
        elif batched:
            plan.batched(bA, bB, None, bD, p0.M, p0.N, p0.K, len(probs), p0.M * p0.K,
                         p0.K * p0.N, 0, p0.M * p0.N, alpha=p0.alpha, beta=p0.beta,
                         stream=stream)
        elif grouped:
            plan.grouped(table, alpha=p0.alpha, beta=p0.beta, stream=stream)
        else:
            A, B, C, D = dv[0]
            if rotate:
                A, B, C = rot[r]
            plan.run(A, B, C, D, p0.M, p0.N, p0.K, alpha=p0.alpha, beta=p0.beta,
                     scale_a=scales[0] if scales else None,
                     scale_b=scales[1] if scales else None, stream=stream, bias=bias_dev)

    tuned = None
    if args.autotune and not grouped and not scaled:
        A, B, C, D = dv[0]
        res = plan.autotune(A, B, C, D, p0.M, p0.N, p0.K, alpha=p0.alpha, beta=p0.beta,
                            bias=bias_dev, scale_a=scales[0] if scales else None,
                            scale_b=scales[1] if scales else None, iterations=5, stream=stream)
        tuned = {"candidates": len(res), "best_us": res[0]["us"], "worst_us": res[-1]["us"]}
    for _ in range(args.warmup):
        l2_flush()
        step()
    torch.cuda.synchronize(dev)
    st = plan.query_error()
    if st != g.OK:
        raise RuntimeError("device status after warm-up: " + g.status_string(st))
    cfg = plan.last_config()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        # give the host a head start so that no step waits for its launch:
        # every timed step then starts right after the preceding flush
        torch.cuda._sleep(int(2e6))
        host = 0.0
        if rotate:
            # no flush between steps: the K steps run back to back between one
            # pair of events (per-step events would add their own ~2 us)
            starts[0].record(stream)
            for i in range(args.steps):
                h0 = time.perf_counter()
                step()
                host += time.perf_counter() - h0
            ends[0].record(stream)
        else:
            for i in range(args.steps):
                l2_flush()
                starts[i].record(stream)
                h0 = time.perf_counter()
                step()
                host += time.perf_counter() - h0
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
    barrier(dist)
    st = plan.query_error()
    if st != g.OK:
        raise RuntimeError("device status after timed steps: " + g.status_string(st))
    if args.trace:
        # one extra, untimed step with the per-CTA timeline on
        import numpy as np
        plan.set(g.OPT_TRACE_ITEMS, 64)
        l2_flush()
        step()
        torch.cuda.synchronize(dev)
        np.save(args.trace, g.gemm_plan_trace(plan.handle))
        plan.set(g.OPT_TRACE_ITEMS, 0)
    ms = ([starts[0].elapsed_time(ends[0]) / args.steps] if rotate else
          [s.elapsed_time(e) for s, e in zip(starts, ends)])
    ms_step = sum(ms) / len(ms)
    ms_step_max = max_over_ranks(dist, ms_step, dev)
    total_flops = sum_over_ranks(dist, flops, dev)
    value = total_flops / (ms_step_max * 1e-3) / 1e12

    # host cost of one call at the C boundary: gemm_run_ex through ctypes with
    # the arguments already converted (the launch parameters come from the
    # plan's cache after the first call), timed on the host; the launches are
    # real and drained afterwards, untimed
    host_c_us = None
    if not grouped and not scaled and p0.bias is None and not args.no_e2e:
        lib = g.load()
        A, B, C, D = dv[0]
        lda = p0.M if p0.a_col_major else p0.K
        ldb = p0.K if p0.b_col_major else p0.N
        cargs = (plan.handle, A.data_ptr(), lda, B.data_ptr(), ldb,
                 C.data_ptr() if C is not None else None, p0.N, D.data_ptr(), p0.N, p0.M, p0.N,
                 p0.K, p0.alpha, p0.beta, scales[0].data_ptr() if scales else None,
                 scales[1].data_ptr() if scales else None, stream.cuda_stream)
        n_calls = 50
        torch.cuda._sleep(int(2e7))  # keep the GPU busy so that launches only queue
        t0 = time.perf_counter()
        for _ in range(n_calls):
            lib.gemm_run_ex(*cargs)
        host_c_us = 1e6 * (time.perf_counter() - t0) / n_calls
        torch.cuda.synchronize(dev)

    # end to end through the C ABI with pinned host buffers (single problems)
    e2e = None
    if not grouped and not scaled and not args.no_e2e:
        hA, hB = p0.A.pin_memory(), p0.B.pin_memory()
        hC = p0.C.pin_memory() if p0.C is not None else None
        hD = torch.empty(p0.M, p0.N, dtype=I.TORCH_DTYPE[p0.d_dtype]).pin_memory()
        e2e_steps = max(3, min(args.steps, 50))
        for _ in range(2):
            g.gemm_run_host(plan.handle, hA, hB, hC, hD, p0.M, p0.N, p0.K, p0.alpha, p0.beta,
                            p0.scale_a, p0.scale_b, stream)
        barrier(dist)
        per_call = []
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            t1 = time.perf_counter()
            s = g.gemm_run_host(plan.handle, hA, hB, hC, hD, p0.M, p0.N, p0.K, p0.alpha,
                                p0.beta, p0.scale_a, p0.scale_b, stream)
            per_call.append(time.perf_counter() - t1)
            if s != g.OK:
                raise RuntimeError("gemm_run_host: " + g.status_string(s))
        t_e2e = (time.perf_counter() - t0) / e2e_steps
        t_e2e = max_over_ranks(dist, t_e2e, dev)
        h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
        if hC is not None and p0.beta != 0.0:
            h2d += hC.numel() * hC.element_size()
        # value: total work / total time of the calls; the median call shows the
        # steady state apart from the occasional host stall of a shared machine
        e2e = {"value": total_flops / t_e2e / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hD.numel() * hD.element_size(),
               "ms_per_call": 1e3 * t_e2e, "ms_per_call_median": 1e3 * statistics.median(per_call),
               "ms_per_call_max": 1e3 * max(per_call), "calls": e2e_steps}

    pk, pk_kind = peaks()
    peak = tensor_peak(p0.a_dtype, pk)
    achieved = flops / (ms_step * 1e-3) / 1e12
    roofline = roofline_entry(flops, algorithmic_bytes(probs), ms_step, p0.a_dtype, pk, pk_kind,
                              recorded_traffic(args.workload))

    clocks = clk.summary()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        fl_s, cores, desc, secs, _, _ = cpu_oracle_sample(probs, budget_s=args.cpu_budget)
        cpu = {"value": fl_s / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc, "seconds": secs}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": p0.a_dtype,
            "data": "synthetic",
            "config": {"workload": args.workload, "M": p0.M if not grouped else [p.M for p in probs],
                       "N": p0.N, "K": p0.K, "alpha": p0.alpha, "beta": p0.beta,
                       "relu": p0.relu, "epilogue": p0.act,
                       "bias": p0.bias is not None,
                       "layout": ("A row-major, B column-major (TN), D row-major; %s block %d"
                                  % (p0.block_scales[2], p0.block_scales[3]) if scaled
                                  else "row-major A, B, C, D"),
                       "l2": (("inputs larger than L2: %d copies of the inputs (%.0f MB in all) "
                               "used in turn, no flush between steps; the steps run back to "
                               "back between one pair of events" % (copies, copies * in_bytes / 1e6))
                              if rotate else
                              "flushed between steps (256 MiB write%s, outside the step events)"
                              % (" then 256 MiB read" if args.flush == "write+read" else "")),
                       "parallelism": "replicas" if ws > 1 else "single",
                       "kernel": cfg, "autotuned": tuned},
            "pct_of_peak": 100.0 * achieved / peak,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * int(cfg.get("launches", 1)),
            "clocks": clocks,
            # time scaled to the maximum SM clock (median clock under load):
            # separates clock (power cap) effects from kernel changes
            "ms_per_step_at_max_clock": (ms_step * clocks["sm_mhz"] / clocks["sm_max_mhz"]
                                         if clocks.get("sm_mhz") and clocks.get("sm_max_mhz")
                                         else None),
            "frac_of_sustained_peak": achieved / tensor_peak(p0.a_dtype, pk, sustained=True),
            "wall_s_timed_region": wall,
            "host_us_per_call": 1e6 * host / args.steps,
            "host_us_per_call_c": host_c_us,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--opt", action="append", help="plan option NAME=VALUE (e.g. schedule=1)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer and host-overhead measurements (short launch "
                         "lists for profiling)")
    ap.add_argument("--list", action="store_true")
    ap.add_argument("--autotune", action="store_true",
                    help="time every kernel configuration first and keep the fastest")
    ap.add_argument("--trace", help="after timing, save one step's per-CTA timeline (.npy)")
    ap.add_argument("--flush", choices=["write", "write+read", "rotate"], default="write+read",
                    help="L2 between timed steps: a 256 MiB write, then (default) a "
                         "256 MiB read so that the L2 holds clean lines: after the write "
                         "alone the next kernel first pays for writing back ~L2-size dirty "
                         "lines (~19 us at HBM speed), a cost of the flush, not of the GEMM; "
                         "or 'rotate': no flush, the steps use copies of the inputs in turn "
                         "(twice the L2 in all), so the inputs are never cached but the "
                         "kernel's code stays in L2 as it does when one GEMM follows another; "
                         "the steps then run back to back, timed by one pair of events")
    args = ap.parse_args(argv)
    if args.list:
        print("\n".join(workloads()))
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload not in workloads() and not args.workload.startswith("custom_"):
        ap.error("unknown workload %s (see --list)" % args.workload)
    ws = dist_env()[0]
    if args.gpus != ws:
        ap.error("--gpus %d but %d process(es) were launched: run N replicas with "
                 "python -m torch.distributed.run --nproc-per-node N bench.py --gpus N"
                 % (args.gpus, ws))
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
