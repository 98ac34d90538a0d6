"""Throughput of the elementwise / row-op library on one GB300.

One step is one pass of the ops that the Llama-3-8B prefill workload names
(T = 8192 tokens, bf16 storage, f32 math), in a layer's order: embedding
gather (table [128256, 4096]), fused residual add + RMSNorm [8192, 4096],
RoPE half layout on q [8192, 32, 128] and k [8192, 8, 128] in one launch,
SiLU-mul [8192, 14336].  Every op reads its inputs from HBM once and writes
its outputs once; a step moves ~1.28 GB through distinct buffers, far more
than the 129 MB L2.

The metric is achieved HBM GB/s: the algorithmic bytes (what the ops must
read plus what they must write) over the measured time, with rows/s beside
it.  The line also carries `per_config`: every op of every large workload
-- the prefill ops beyond the step (interleaved RoPE, residual add, RMSNorm,
argmax over [8192, 128256] logits), the f32 in-place RoPE variants, the
wide f32 argmax and RMSNorm -- and the decode ops, each timed alone, back to
back over rotating copies of its buffers (more than four times the L2
together), from a CUDA graph and from the stream.  Printed as one JSON line
(rank 0).  `--impl reference` times the CPU oracle instead, on a bounded
sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       (N > 1: one process per GPU under torch.distributed.run; each rank runs
       its own replica of the step, no collective on the data path)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 peak per op; rows/sec at Llama-8B shapes"
WORKLOAD = "llama3-8b-prefill-T8192-bf16"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# op name -> the workload cases it runs on, in step order: the ops the
# prefill workload names
STEP = [
    ("embedding", ("embedding",)),
    ("add_rmsnorm", ("add_rmsnorm",)),
    ("rope_qk_half", ("rope_q", "rope_k")),
    ("silu_mul", ("silu_mul",)),
]
# the other Llama-3-8B prefill ops of the library, at the same shapes (timed
# alone for per_config)
PREFILL_MORE = [
    ("rope_qk_interleaved", ("rope_q_interleaved", "rope_k_interleaved")),
    ("add", ("add",)),
    ("rmsnorm", ("rmsnorm",)),
    ("argmax", ("argmax",)),
]
ALL_PREFILL = STEP + PREFILL_MORE
KERNEL_OF = {  # op -> the kernel it launches (names as ncu lists them)
    "embedding": "embedding_rows", "add_rmsnorm": "rmsnorm_rows", "rope_qk_half": "rope_vec",
    "rope_qk_interleaved": "rope_vec", "silu_mul": "pointwise_vec", "add": "pointwise_vec",
    "rmsnorm": "rmsnorm_rows", "argmax": "argmax_rows1",
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---- algorithmic bytes ------------------------------------------------------------

def op_bytes(op: str, arrays: dict, params: dict) -> tuple[int, int]:
    """(bytes the op must read + write, rows it processes)."""
    nb = lambda a: int(a.nbytes)
    if op == "embedding":
        n, d = params["n"], params["d"]
        es = arrays["table"].itemsize
        return 2 * n * d * es + nb(arrays["ids"]), n
    if op == "add_rmsnorm":
        return 4 * nb(arrays["x"]) + nb(arrays["w"]), params["rows"]
    if op == "qk_norm_rope":
        return (2 * (nb(arrays["q"]) + nb(arrays["k"])) + nb(arrays["gq"]) + nb(arrays["gk"]) + nb(arrays["pos"])
                + 4 * (params["r"] // 2)), params["T"]
    if op == "layernorm":
        return 2 * nb(arrays["x"]) + nb(arrays["g"]) + nb(arrays["b"]), params["rows"]
    if op == "rope_multi":
        return 2 * nb(arrays["x"]) + nb(arrays["pos"]) + nb(arrays["inv_freq"]), params["T"]
    if op == "rope_pair_inplace":  # q and k in place, each over its own rotated width
        moved = sum(arrays[k].shape[0] * arrays[k].shape[1] * params[k][0] * arrays[k].itemsize for k in ("q", "k"))
        return 2 * moved + nb(arrays["pos"]) + nb(arrays["fq"]) + nb(arrays["fk"]), params["T"]
    if op == "rope_qk_half_cached":
        T, r = params["T"], params["r"]
        return 2 * (nb(arrays["q"]) + nb(arrays["k"])) + nb(arrays["pos"]) + T * (r // 2) * 8, T
    if op.startswith("rope"):
        T, D, r = params["T"], params["D"], params["r"]
        moved = 0
        for key in ("q", "k", "x"):
            if key in arrays:
                x = arrays[key]
                H = x.shape[1]
                moved += x.nbytes if r == D or not params.get("in_place") else T * H * r * x.itemsize
        return 2 * moved + nb(arrays["pos"]) + 4 * (r // 2), T
    if op in ("silu_mul", "add"):
        k = "gate" if op == "silu_mul" else "a"
        a = arrays[k]
        return 3 * nb(a), a.shape[0]
    if op == "rmsnorm":
        return 2 * nb(arrays["x"]) + nb(arrays["w"]), params["rows"]
    if op == "argmax":
        return nb(arrays["x"]) + 4 * params["rows"], params["rows"]
    if op.startswith("sample_"):
        return nb(arrays["x"]) + nb(arrays["u"]) + 4 * params["rows"], params["rows"]
    raise KeyError(op)


# ---- clocks sampled during the timed region -------------------------------------

class Clocks:
    """nvidia-smi sampling every 50 ms in the background; only the samples
    whose timestamps fall inside the timed region are kept."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.window = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(1.0)  # let the sampler start before the timed region
        except Exception:
            self.proc = None

    def mark(self, t_begin: float, t_end: float):
        self.window = (t_begin, t_end)

    def stop(self):
        if self.proc is None:
            return None
        import datetime
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                rows.append((ts, parts))
        os.unlink(self.path)
        if self.window:
            inside = [r for t, r in rows if self.window[0] - 0.05 <= t <= self.window[1] + 0.05]
        else:
            inside = [r for _, r in rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        mx = [num(r[3]) for r in inside if num(r[3]) is not None]
        pw = [num(r[4]) for r in inside if num(r[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(inside)}


# ---- our arm: the CUDA library ------------------------------------------------------

def combine(op: str, parts):
    """Inputs of one step op from its workload cases (q and k for the fused RoPE)."""
    if op.startswith("rope_qk"):
        (aq, pq), (ak, _) = parts
        return {"q": aq["x"], "k": ak["x"], "pos": aq["pos"], "inv_freq": aq["inv_freq"]}, pq
    return parts[0]


EXTRA = ("qk_norm_rope", "rope_qk_half_cached", "layernorm", "rope_multi", "sample_temperature", "sample_top_k",
         "sample_top_p", "sample_min_p")
MULTI_DIMS = (32, 48, 48)  # multi-axis RoPE: (t, h, w) slices of head_dim 128
SAMPLING = {"sample_temperature": ("temperature", dict(temperature=0.7)),
            "sample_top_k": ("top_k", dict(temperature=0.7, top_k=50)),
            "sample_top_p": ("top_p", dict(temperature=0.7, p=0.9)),
            "sample_min_p": ("min_p", dict(temperature=0.7, p=0.05))}


def build_extra_inputs(tokens: int = 8192, ops=None):
    """Inputs of the ops beyond the step, at the same prefill shapes: QK-norm
    then RoPE on q [T, 32, 128] and k [T, 8, 128] (gains U(0.5, 1.5)); RoPE of
    q and k driven by a cos/sin table of 8192 positions; LayerNorm of
    [T, 4096] with gain and bias; multi-axis RoPE of x [T, 24, 128] bf16 in
    (t, h, w) slices of 32, 48, 48 (positions below 64, 256, 256, base
    10000 per axis); one draw per row of the logits
    [T, 128256] by each sampling method at a uniform u per row."""
    import synth
    from synth import workloads as W
    cases = W.cases(W.PREFILL)
    rows = None if tokens >= 8192 else (0, tokens)
    seed = W.SEEDS[W.PREFILL]
    (aq, pq), (ak, _) = cases["rope_q"](rows=rows), cases["rope_k"](rows=rows)
    gq = synth.uniform_bf16(seed, "qk_norm.gq", (128,), 0.5, 1.5)
    gk = synth.uniform_bf16(seed, "qk_norm.gk", (128,), 0.5, 1.5)
    qk = {"q": aq["x"], "k": ak["x"], "pos": aq["pos"], "inv_freq": aq["inv_freq"]}
    ax, px = cases["rmsnorm"](rows=rows)
    lb = synth.normal_bf16(seed, "layernorm.b", (ax["x"].shape[1],), 0.0, 0.2)
    T = ax["x"].shape[0]
    xm = synth.normal_bf16(seed, "rope_multi.x", (T, 24, 128), 0.0, 1.0)
    pm = np.stack([synth.randint(seed, f"rope_multi.pos{a}", (T,), 0, hi)
                   for a, hi in enumerate((64, 256, 256))], axis=1).astype(np.int32)
    fm = np.concatenate([(10000.0 ** (-2.0 * np.arange(d // 2) / d)).astype(np.float32) for d in MULTI_DIMS])
    sampling = {}
    if ops is None or any(op in SAMPLING for op in ops):  # the logits are 2.1 GB: only when asked for
        al, pl = cases["argmax"](rows=rows)
        u = synth.units(seed, "sample.u", al["x"].shape[0]).astype(np.float32)
        sampling = {op: ({"x": al["x"], "u": u}, dict(pl, method=m, kw=kw)) for op, (m, kw) in SAMPLING.items()}
    out = {
        "qk_norm_rope": (dict(qk, gq=gq, gk=gk), dict(pq, eps=1e-6)),
        "rope_qk_half_cached": (dict(qk), dict(pq, cache_len=8192)),
        "layernorm": ({"x": ax["x"], "g": ax["w"], "b": lb}, px),
        "rope_multi": ({"x": xm, "pos": pm, "inv_freq": fm}, {"T": T, "dims": MULTI_DIMS, "mu": 1.0, "layout": 0}),
        **sampling,
    }
    return out if ops is None else {op: v for op, v in out.items() if op in ops}


def build_workload_inputs(workload: str):
    """Per-op inputs of the other workloads, for --isolated: the f32 RoPE
    variants (each operand rotated in place), the wide f32 argmax and
    RMSNorm, and the decode step's ops (T = 64, launch-latency bound) with
    one draw per row of its logits by each sampling method."""
    from synth import workloads as W
    cases = W.cases(workload)
    if workload == W.ROPE_VARIANTS:
        (aq, pq), (ak, pk) = cases["rope_q"](), cases["rope_k"]()
        pair = ({"q": aq["x"], "k": ak["x"], "pos": aq["pos"], "fq": aq["inv_freq"], "fk": ak["inv_freq"]},
                {"T": pq["T"], "q": (pq["r"], pq["mu"], pq["layout"]), "k": (pk["r"], pk["mu"], pk["layout"])})
        return {"rope_q_inplace": (aq, pq), "rope_k_inplace": (ak, pk), "rope_pair_inplace": pair}
    if workload == W.WIDE:
        return {"argmax": cases["argmax"](), "rmsnorm": cases["rmsnorm"]()}
    if workload == W.DECODE:
        import synth
        rope = combine("rope_qk_half", [cases["rope_q"](), cases["rope_k"]()])
        al, pl = cases["argmax"]()
        u = synth.units(W.SEEDS[W.DECODE], "sample.u", al["x"].shape[0]).astype(np.float32)
        sampling = {op: ({"x": al["x"], "u": u}, dict(pl, method=m, kw=kw)) for op, (m, kw) in SAMPLING.items()}
        return {"add_rmsnorm": cases["add_rmsnorm"](), "rope_qk_half": rope, "silu_mul": cases["silu_mul"](),
                "argmax": (al, pl), **sampling}
    raise KeyError(workload)


def build_inputs(tokens: int = 8192, ops=None):
    """Inputs of the prefill ops (the step's by default); `tokens` < 8192
    takes the first rows of every op (a smaller case of the same kernels,
    for profiling)."""
    from synth import workloads as W
    cases = W.cases(W.PREFILL)
    rows = None if tokens >= 8192 else (0, tokens)
    return {op: combine(op, [cases[c](rows=rows) for c in names]) for op, names in (ops or STEP)}


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of the ranks' values (each rank passes its own): the
    job's elapsed time is that of its slowest replica."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(step_bytes: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every replica moves step_bytes per step."""
    return step_bytes * steps * world / (elapsed_ms * 1e-3) / 1e9


def run_ours(args):
    import torch
    import torch.distributed as dist

    import elementwise_row_rmsnorm_gb300 as gbe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gbe.lib()

    data = build_inputs(args.tokens)

    # device buffers: inputs (a separate copy per op), outputs
    bufs = {op: {k: to_device(torch, dev, v) for k, v in arrays.items()} for op, (arrays, params) in data.items()}
    out = {op: make_outputs(torch, dev, op, b) for op, b in bufs.items()}

    def call(op):
        run_op(gbe, op, data[op][1], bufs[op], out[op])

    nbytes = {op: op_bytes(op, *data[op]) for op in data}
    step_bytes = sum(b for b, _ in nbytes.values())

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for op, _names in STEP:
            call(op)
    barrier()

    clocks = Clocks(local)
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # timed region 1: the steps back to back, as a user runs them (consecutive
    # launches overlap through programmatic dependent launch)
    barrier()
    host_t0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        for op, _names in STEP:
            call(op)
    t1.record(stream)
    barrier()
    clocks.mark(host_t0, time.time())
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # timed region 2: the same steps with an event pair around every launch
    # (an event between two launches stops them overlapping, so these per-op
    # times include each launch's full ramp)
    ev = {op: [] for op, _ in STEP}
    op_steps = min(args.steps, 200)
    barrier()
    for _ in range(op_steps):
        for op, _names in STEP:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(op)
            b.record(stream)
            ev[op].append((a, b))
    barrier()
    per_op = {}
    for op, _ in STEP:
        ms = [a.elapsed_time(b) for a, b in ev[op]]
        mean = sum(ms) / len(ms)
        bts, rows = nbytes[op]
        per_op[op] = {"bytes": bts, "ms": round(mean, 5), "ms_min": round(min(ms), 5),
                      "gbs": round(bts / (mean * 1e-3) / 1e9, 1), "rows_per_s": round(rows / (mean * 1e-3), 1)}

    # e2e: the same step from pinned host buffers, copies inside the timed region
    e2e = run_e2e(args, gbe, torch, dev, data, bufs, out, call, nbytes, step_bytes) if not args.no_e2e else None
    # every op of every large workload, each alone (rank 0 of a single-GPU run)
    configs = per_config(torch, gbe, dev) if (world == 1 and not args.no_configs) else None

    peak, peak_kind = peaks()
    for op in per_op:
        per_op[op]["frac_of_peak"] = round(per_op[op]["gbs"] / peak, 4)
        per_op[op]["frac_of_8tbs"] = round(per_op[op]["gbs"] / NOMINAL_HBM_GBS, 4)
    # dominant kernel: the op with the largest share of the step's time
    dom = max(per_op, key=lambda o: per_op[o]["ms"])
    traffic = dram_traffic(dom)
    value = aggregate_gbs(step_bytes, args.steps, world, elapsed_ms)

    result = None
    if rank == 0:
        cpu = cpu_baseline(data) if (world == 1 and not args.no_cpu) else None
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded splitmix64; Llama-3-8B shapes)",
            "config": {"workload": WORKLOAD if args.tokens >= 8192 else f"{WORKLOAD} (first {args.tokens} tokens)",
                       "storage": "bf16", "tokens": min(args.tokens, 8192), "hidden": 4096,
                       "ffn": 14336, "heads_q": 32, "heads_kv": 8, "head_dim": 128, "vocab": 128256,
                       "step_ops": [op for op, _ in STEP], "bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2 (each step moves ~1.28 GB through distinct buffers)",
                       "parallelism": f"replicas{world}"},
            "roofline": {"bound": "hbm", "kernel": KERNEL_OF[dom], "op": dom,
                         "achieved": per_op[dom]["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": round(per_op[dom]["gbs"] / peak, 4), "peak_source": peak_kind,
                         "traffic": traffic},
            "per_op": per_op,
            "per_op_timing": f"{op_steps} further steps with a CUDA event pair around every launch (each op "
                             "also pays the write-back of the previous op's dirty L2 lines)",
            "per_config": configs,
            "per_config_timing": "each op alone, back to back over rotating copies of its buffers (> 4x L2); "
                                 "us/gbs from CUDA graph replays, *_stream from launches on the stream",
            "e2e": e2e,
            "gpu_launches": len(STEP) * args.steps,
            "launch": "programmatic dependent launch (each kernel overlaps the previous one's tail)",
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def batch_sweep(data):
    """Each row op of `data` on its first b rows, b = 1, 2, 4, ... up to all
    of them (keys "op@b"): the batch sweep of the row ops."""
    out = {}
    for op, (arrays, params) in data.items():
        rows = params.get("rows")
        if not rows:
            continue
        bs = sorted({min(rows, 1 << i) for i in range(0, 31) if (1 << i) <= 2 * rows})
        for b in bs:
            sl = {k: (v[:b] if getattr(v, "ndim", 0) >= 1 and v.shape[0] == rows else v) for k, v in arrays.items()}
            out[f"{op}@{b}"] = (sl, dict(params, rows=b))
    return out


def time_isolated(torch, gbe, dev, data: dict, graph: bool) -> dict:
    """Each op of `data` alone, launched back to back over rotating copies of
    its inputs and outputs (together more than four times the L2, so every
    launch reads from HBM), timed with one CUDA event pair around the loop:
    the op's sustained rate.  With `graph` the launches are captured once in
    a CUDA graph and timed over its replays (no per-call host cost)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, _kind = peaks()
    res = {}
    for key in list(data):
        op = key.split("@")[0]  # "op@b": the op on the first b rows
        arrays, params = data[key]
        nb, rows = op_bytes(op, arrays, params)
        sets = int(min(12, max(2, -(-4 * l2 // nb) + 1)))
        base = {k: to_device(torch, dev, v) for k, v in arrays.items()}
        shared = ("table", "w", "g", "gq", "gk", "inv_freq", "fq", "fk", "pos", "ids", "cos_sin", "u")
        if op == "rope_qk_half_cached":
            base["cos_sin"] = gbe.rope_cos_sin(base["inv_freq"], params["r"], params["cache_len"])
        rings = []
        for _ in range(sets):
            b = {k: (v if k in shared else v.clone()) for k, v in base.items()}
            rings.append((b, make_outputs(torch, dev, op, b)))

        def go(i, p=params, op=op):
            run_op(gbe, op, p, *rings[i % sets])
        for i in range(3 * sets):
            go(i)
        torch.cuda.synchronize()
        n = max(50, 4 * sets)
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        if graph:
            side = torch.cuda.Stream(dev)
            side.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(n):
                    go(i)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            reps = 10
            a.record()
            for _ in range(reps):
                g.replay()
            e.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(e) / (n * reps)
            del g
        else:
            a.record()
            for i in range(n):
                go(i)
            e.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(e) / n
        gbs = nb / ms / 1e6
        res[key] = {"bytes": nb, "us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "rows_per_s": round(rows / ms * 1e3, 1),
                    "frac_of_peak": round(gbs / peak, 4), "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                    "copies": sets}
        del rings, base
        torch.cuda.empty_cache()
    return res


def workload_ops(workload: str, tokens: int = 8192, extra: bool = False, keep=None):
    """The per-op inputs of a workload for the isolated timings (with
    `extra`, also the prefill-shaped ops beyond the workload's list, or those
    of them in `keep`)."""
    from synth import workloads as W
    if workload == W.PREFILL:
        data = build_inputs(tokens, ALL_PREFILL)
        if extra:
            data.update(build_extra_inputs(tokens, ops=keep or None))
        return data
    return build_workload_inputs(workload)


def per_config(torch, gbe, dev) -> dict:
    """Every op of every large workload (and the decode ops), timed alone
    from a CUDA graph and from the stream.  The headline figure of each op
    is the graph one; the stream one adds the per-call host cost of the
    Python binding and the C checks, which the small ops cannot hide."""
    from synth import workloads as W
    out = {}
    for wl, note in ((W.PREFILL, "the step's ops and the other prefill ops at the same shapes"),
                     (W.ROPE_VARIANTS, "f32 RoPE in place: q interleaved r=64, k half r=128 mu=1.2, each alone "
                                       "and both in one launch (gbe_rope_pair)"),
                     (W.WIDE, "f32 argmax [1024,152064] (5% tied rows, 1% NaN) and RMSNorm [1024,16384]"),
                     (W.DECODE, "T=64, L2-resident and launch-bound: reported, not held to the bar")):
        data = workload_ops(wl)
        g = time_isolated(torch, gbe, dev, data, graph=True)
        st = time_isolated(torch, gbe, dev, data, graph=False)
        ops = {}
        for op in g:
            ops[op] = dict(g[op], us_stream=st[op]["us"], gbs_stream=st[op]["gbs"],
                           frac_of_peak_stream=st[op]["frac_of_peak"])
        out[wl] = {"note": note, "ops": ops}
        del data
    return out


def run_isolated(args):
    """`--isolated`: each op of one workload alone (see time_isolated), one
    JSON line."""
    import torch

    import elementwise_row_rmsnorm_gb300 as gbe
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    gbe.lib()
    workload = args.workload or WORKLOAD
    data = workload_ops(workload, args.tokens, extra=args.extra or bool(args.keep and args.keep & set(EXTRA)),
                        keep=args.keep)
    if args.keep:
        data = {op: v for op, v in data.items() if op in args.keep}
    if args.sweep:
        data = batch_sweep(data)
    res = time_isolated(torch, gbe, dev, data, graph=args.graph)
    peak, kind = peaks()
    name = workload if workload != WORKLOAD or args.tokens >= 8192 else f"{WORKLOAD} (first {args.tokens} tokens)"
    line = {"mode": "isolated" + (" (CUDA graph)" if args.graph else ""), "workload": name,
            "unit": "GB/s", "peak": peak, "peak_source": kind, "per_op": res}
    print(json.dumps(line), flush=True)
    return line


def to_device(torch, dev, a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def make_outputs(torch, dev, op, b):
    if op == "embedding":
        return torch.empty((b["ids"].numel(), b["table"].shape[1]), dtype=b["table"].dtype, device=dev)
    if op == "add_rmsnorm":
        return (torch.empty_like(b["x"]), torch.empty_like(b["x"]))
    if op.startswith("rope_qk") or op == "qk_norm_rope":
        return (torch.empty_like(b["q"]), torch.empty_like(b["k"]))
    if op == "rope_pair_inplace":
        return None
    if op.endswith("_inplace"):
        return b["x"]
    if op == "argmax" or op.startswith("sample_"):
        return torch.empty((b["x"].shape[0],), dtype=torch.int32, device=dev)
    return torch.empty_like(b["x"] if "x" in b else (b["gate"] if "gate" in b else b["a"]))


def run_op(gbe, op, p, b, o):
    if op == "embedding":
        gbe.gbe_embedding(b["table"], b["ids"], o)
    elif op == "add_rmsnorm":
        gbe.gbe_add_rmsnorm(b["x"], b["residual"], b["w"], o[0], o[1], p["eps"])
    elif op == "rope_qk_half_cached":
        gbe.gbe_rope_qk(b["q"], o[0], b["k"], o[1], b["pos"], b["inv_freq"], p["r"], p["mu"], p["layout"],
                        cos_sin=b["cos_sin"])
    elif op.startswith("rope_qk"):
        gbe.gbe_rope_qk(b["q"], o[0], b["k"], o[1], b["pos"], b["inv_freq"], p["r"], p["mu"], p["layout"])
    elif op == "qk_norm_rope":
        gbe.gbe_qk_norm_rope(b["q"], o[0], b["gq"], b["k"], o[1], b["gk"], p["eps"], b["pos"], b["inv_freq"], p["r"],
                             p["mu"], p["layout"])
    elif op == "silu_mul":
        gbe.gbe_silu_mul(b["gate"], b["up"], o)
    elif op == "add":
        gbe.gbe_add(b["a"], b["b"], o)
    elif op == "rmsnorm":
        gbe.gbe_rmsnorm(b["x"], b["w"], o, p["eps"])
    elif op == "layernorm":
        gbe.gbe_layernorm(b["x"], b["g"], b["b"], o, p["eps"])
    elif op == "rope_pair_inplace":
        gbe.gbe_rope_pair((b["q"], b["q"], b["fq"], *p["q"]), (b["k"], b["k"], b["fk"], *p["k"]), b["pos"])
    elif op.startswith("rope") and op.endswith("_inplace"):
        gbe.gbe_rope(b["x"], b["x"], b["pos"], b["inv_freq"], p["r"], p["mu"], p["layout"])
    elif op == "rope_multi":
        gbe.gbe_rope_multi(b["x"], o, b["pos"], p["dims"], b["inv_freq"], p["mu"], p["layout"])
    elif op == "argmax":
        gbe.gbe_argmax(b["x"], o)
    elif op.startswith("sample_"):
        gbe.gbe_sample(b["x"], b["u"], o, p["method"], **p["kw"])


def run_e2e(args, gbe, torch, dev, data, bufs, out, call, nbytes, step_bytes):
    """The step from pinned host buffers: every op's per-step inputs copied
    host->device and every result copied back, inside the timed region
    (weights -- the embedding table, RMSNorm gains, RoPE frequencies -- stay
    resident).  Three streams overlap the work: host->device copies, the
    kernels, device->host copies; events order each op's copy-in before its
    kernel and its kernel before its copy-out, and keep the next step from
    overwriting a device buffer that is still being read."""
    weights = {("embedding", "table"), ("add_rmsnorm", "w"), ("rmsnorm", "w")}
    weights |= {(op, "inv_freq") for op in bufs if op.startswith("rope")}
    host_in, h2d = {op: [] for op in bufs}, 0
    for op, b in bufs.items():
        for k, t in b.items():
            if (op, k) in weights:
                continue
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            host_in[op].append((k, h))
            h2d += t.numel() * t.element_size()
    host_out, d2h = {op: [] for op in out}, 0
    for op, o in out.items():
        for i, t in enumerate(o if isinstance(o, tuple) else (o,)):
            host_out[op].append((i, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)))
            d2h += t.numel() * t.element_size()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ops = [op for op, _ in STEP]
    done_prev = {op: None for op in ops}   # kernel of the previous step finished (inputs free)
    out_prev = {op: None for op in ops}    # copy-out of the previous step finished (outputs free)

    def one():
        for op in ops:
            with torch.cuda.stream(s_in):
                if done_prev[op] is not None:
                    s_in.wait_event(done_prev[op])
                for k, h in host_in[op]:
                    bufs[op][k].copy_(h, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            comp.wait_event(ev_in)
            if out_prev[op] is not None:
                comp.wait_event(out_prev[op])
            call(op)
            ev_done = torch.cuda.Event()
            ev_done.record(comp)
            done_prev[op] = ev_done
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done)
                o = out[op]
                for i, h in host_out[op]:
                    h.copy_((o if isinstance(o, tuple) else (o,))[i], non_blocking=True)
                ev_out = torch.cuda.Event()
                ev_out.record(s_out)
            out_prev[op] = ev_out

    one()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 10))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    s_in.wait_stream(comp)
    s_out.wait_stream(comp)
    for _ in range(steps):
        one()
    comp.wait_stream(s_out)
    comp.wait_stream(s_in)
    b.record(comp)
    torch.cuda.synchronize()
    ms_copy = a.elapsed_time(b) / steps

    # the same step with no copies at all: the kernels read each op's inputs
    # from the pinned host buffers and write its results to pinned host
    # buffers, through the C ABI (pinned host memory is mapped at the same
    # address on the device, and NVLink-C2C carries the traffic)
    host_bufs = {op: dict(bufs[op]) for op in bufs}
    for op in host_bufs:
        for k, h in host_in[op]:
            host_bufs[op][k] = h
    host_outs = {op: (tuple(h for _, h in host_out[op]) if isinstance(out[op], tuple) else host_out[op][0][1])
                 for op in out}

    def one_zero_copy():
        for op in ops:
            run_op(gbe, op, data[op][1], host_bufs[op], host_outs[op])

    one_zero_copy()
    torch.cuda.synchronize()
    a.record(comp)
    for _ in range(steps):
        one_zero_copy()
    b.record(comp)
    torch.cuda.synchronize()
    ms_zero = a.elapsed_time(b) / steps
    copy_leg = {"value": round(step_bytes / (ms_copy * 1e-3) / 1e9, 1), "ms_per_step": round(ms_copy, 3),
                "method": "cudaMemcpyAsync in and out on their own streams, overlapped with the kernels"}
    zero_leg = {"value": round(step_bytes / (ms_zero * 1e-3) / 1e9, 1), "ms_per_step": round(ms_zero, 3),
                "method": "kernels read inputs from and write results to pinned host memory (zero-copy)"}
    best, other = (zero_leg, copy_leg) if ms_zero < ms_copy else (copy_leg, zero_leg)
    return {"value": best["value"], "unit": "GB/s", "ms_per_step": best["ms_per_step"], "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "method": best["method"],
            "alternative": other}


def dram_traffic(op: str):
    """DRAM bytes per launch of the op's kernel from the committed ncu summary,
    or None when there is none or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    if op not in SOURCE_OF:
        return None
    want = sources_hash(op)
    for line in open(path):
        parts = line.split()
        if len(parts) == 3 and not line.startswith("#") and parts[0] == op and parts[2] == want:
            return int(parts[1])
    return None


SOURCE_OF = {  # op -> the source file of its kernel and launcher
    "embedding": "embedding.cu", "add_rmsnorm": "rmsnorm.cu", "rope_qk_half": "rope.cu",
    "rope_qk_interleaved": "rope.cu", "silu_mul": "pointwise.cu", "add": "pointwise.cu",
    "rmsnorm": "rmsnorm.cu", "argmax": "argmax.cu",
}


def sources_hash(op: str) -> str:
    """Hash of the sources that decide an op's kernel: its own file and the
    shared device helpers."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "elementwise_row_rmsnorm_gb300", "csrc")
    for name in ("common.cuh", SOURCE_OF[op]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ---- the oracle on the host cores -------------------------------------------------------

SAMPLE_FRACTION = 4  # the CPU runs the first quarter of each op's rows
CPU_SECONDS = 10.0   # and repeats that sample for about this long

ROW_KEYS = ("x", "residual", "ids", "gate", "up", "a", "b", "pos", "q", "k")


def slice_rows(arrays: dict, params: dict, rows: int):
    """The first `rows` rows (tokens, ids, logits rows) of an op case."""
    out = {k: (v[:rows] if k in ROW_KEYS else v) for k, v in arrays.items()}
    p = dict(params)
    for k in ("rows", "T"):
        if k in p:
            p[k] = rows
    if "n" in p:
        lead = out.get("ids", out.get("gate", out.get("a", out.get("x"))))
        p["n"] = int(lead.shape[0]) if "ids" in out else int(lead.size)
    return out, p


def oracle_sample(data=None, fraction=SAMPLE_FRACTION):
    """A bounded sample of the step: the first 1/fraction of the rows of every
    op (from the full inputs when given, else drawn from the same streams),
    widened to the f32 the oracle reads."""
    from synth import workloads as W
    import oracle
    o = oracle.get()
    cases = W.cases(W.PREFILL)
    sample = []
    rows = max(1, 8192 // fraction)
    for op, names in STEP:
        if data is not None:
            arrays, params = slice_rows(*data[op], rows)
        else:
            arrays, params = combine(op, [cases[c](rows=(0, rows)) for c in names])
        bts, _ = op_bytes(op, arrays, params)
        f32 = {k: (o.bf16_widen(v) if v.dtype == np.uint16 else np.ascontiguousarray(v))
               for k, v in arrays.items()}
        sample.append((op, f32, params, bts, rows))
    return sample


def oracle_step(sample, times=None):
    """One pass of the oracle over the sample; with `times`, each op's
    elapsed seconds are added to times[op]."""
    import oracle
    o = oracle.get()
    for op, a, p, _b, _r in sample:
        t0 = time.perf_counter()
        oracle_op(o, op, a, p)
        if times is not None:
            times[op] = times.get(op, 0.0) + time.perf_counter() - t0


def oracle_op(o, op, a, p):
    if op == "embedding":
        o.embedding(a["table"], a["ids"])
    elif op == "add_rmsnorm":
        o.add_rmsnorm(a["x"], a["residual"], a["w"], p["eps"], h_bf16=True)
    elif op.startswith("rope_qk"):
        o.rope(a["q"], a["pos"], a["inv_freq"], p["r"], p["mu"], p["layout"])
        o.rope(a["k"], a["pos"], a["inv_freq"], p["r"], p["mu"], p["layout"])
    elif op == "silu_mul":
        o.silu_mul(a["gate"], a["up"])
    elif op == "add":
        o.add(a["a"], a["b"])
    elif op == "rmsnorm":
        o.rmsnorm(a["x"], a["w"], p["eps"])
    elif op == "argmax":
        o.argmax(a["x"])


def cpu_baseline(data=None):
    """The oracle, as it stands, on the host: one thread, the sample repeated
    for about CPU_SECONDS."""
    import platform
    sample = oracle_sample(data)
    bts = sum(s[3] for s in sample)
    times = {}
    reps, t = 0, time.perf_counter()
    while True:
        oracle_step(sample, times)
        reps += 1
        dt = time.perf_counter() - t
        if dt >= CPU_SECONDS:
            break
    per_op = {op: {"gbs": round(b * reps / times[op] / 1e9, 3), "rows_per_s": round(r * reps / times[op], 1)}
              for op, _a, _p, b, r in sample}
    return {"value": round(bts * reps / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 2), "repeats": reps, "per_op": per_op,
            "host": {"machine": platform.machine(), "cpus": os.cpu_count()},
            "sample": f"first 1/{SAMPLE_FRACTION} of the rows of every op of the step "
                      f"({bts / 1e6:.0f} MB algorithmic), single-threaded C in f32, repeated for "
                      f"{dt:.1f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    sample = oracle_sample()
    bts = sum(s[3] for s in sample)
    for _ in range(args.warmup):
        oracle_step(sample)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample)
    dt = time.perf_counter() - t
    value = bts * args.steps / dt / 1e9
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded splitmix64; Llama-3-8B shapes)",
        "config": {"workload": WORKLOAD, "storage": "bf16", "sample_fraction": SAMPLE_FRACTION,
                   "bytes_per_step": bts, "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first 1/{SAMPLE_FRACTION} of the rows of every op per step"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--ops", default="",
                    help="comma list: run only these ops of the step (for profiling one kernel)")
    ap.add_argument("--tokens", type=int, default=8192,
                    help="take the first T tokens of every op (a smaller case, for profiling)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="leave out the per_config timings")
    ap.add_argument("--isolated", action="store_true",
                    help="time each op alone, back to back over rotating buffers, and print that instead")
    ap.add_argument("--sweep", action="store_true",
                    help="with --isolated: each row op on its first b rows, b = 1, 2, 4, ... (batch sweep)")
    ap.add_argument("--graph", action="store_true",
                    help="with --isolated: capture each op's launches in a CUDA graph and time its replays")
    ap.add_argument("--workload", default="",
                    help="with --isolated: another workload's ops (rope-variants-T4096-f32, wide-argmax-rmsnorm-f32, "
                         "llama3-8b-decode-T64-bf16)")
    ap.add_argument("--extra", action="store_true",
                    help="with --isolated: also time the ops beyond the step (QK-norm+RoPE, table-driven RoPE, "
                         "LayerNorm, multi-axis RoPE, sampling)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    keep = None
    if args.ops:
        keep = set(args.ops.split(","))
        unknown = keep - {op for op, _ in ALL_PREFILL} - set(EXTRA) - {"rope_q_inplace", "rope_k_inplace",
                                                                         "rope_pair_inplace"}
        if unknown:
            ap.error(f"unknown ops {sorted(unknown)}")
        if keep & set(EXTRA) and not args.isolated:
            ap.error("the ops beyond the prefill list run with --isolated only")
        STEP[:] = [(op, c) for op, c in ALL_PREFILL if op in keep]
    args.keep = keep
    if args.impl == "reference":
        return run_reference(args)
    if args.isolated:
        return run_isolated(args)
    return run_ours(args)


if __name__ == "__main__":
    main()
