"""Benchmark of the routed-MoE hot path on GB300.

Default workload: the 48-layer decode stack (hidden 2048, 512 experts, top-10, expert
intermediate 512; 24,576 quantized experts = 19.93 GB resident in HBM; per step 256
sequential tokens, each token one CUDA graph replay of 48 x (router -> experts -> ordered
sum + residual), x <- x + MoE(RMSNorm(x))).  Each token reads 590.6 MB of weights, more than
L2 (129 MB), so no L2 flush is needed between tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_stack|decode_layer] [--no-prefill] [--no-bounded]

Besides the decode line it reports, at N=1, the 512-token prefill chunk ("prefill": tokens/s,
tensor-core TFLOP/s and weight GB/s of moe_prefill_chunk) and the 48-layer, 2048-token chunk
with bounded residency ("prefill_bounded": tokens/s with and without the host fills).

Prints ONE JSON line (rank 0).  Multi-GPU: one process per GPU (torchrun); every rank decodes
its own tokens (no collective on the data path, weak scaling); the line reports the whole-job
tokens/s over the max time across ranks.
--impl reference times the CPU oracle (the method's plain definition) on this host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed-MoE tokens/s (decode, prefill) and achieved HBM GB/s vs GB300 peak"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Dense 16-bit tensor-core peak in TFLOP/s (f16 and bf16 run at the same dense rate): the
    measured bf16 burst figure (the chunk's GEMMs are
    timed alone), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["bf16_tflops"]), "measured bf16_tflops"
    except Exception:
        return 1900.0, "fallback bf16_tflops"


# The translation unit that holds each profiled kernel: its recorded DRAM traffic stays valid
# while the code of that file and of every header it includes is unchanged.
_KERNEL_TU = {"moe_decode_stack": "stack.cu", "moe_decode_layer": "stack.cu", "moe_decode": "decode.cu",
              "tc_gemm": "prefill_tc.cu"}


def _src_digest(kernel: str, root: str = ROOT) -> str:
    """Digest of the code of `kernel`'s translation unit (the .cu file and, transitively, the
    quoted includes found in csrc/ or include/): comments and blank space are left out, so that
    a change of comments alone keeps the recorded DRAM traffic valid."""
    import re
    dirs = [os.path.join(root, "quantized_moe_expert_rl_gb300", "csrc"), os.path.join(root, "include")]
    h, seen, todo = hashlib.sha256(), set(), [_KERNEL_TU[kernel]]
    while todo:
        name = todo.pop(0)
        if name in seen:
            continue
        seen.add(name)
        path = next((os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name))), None)
        if path is None:
            raise FileNotFoundError(name)
        src = open(path, encoding="utf-8").read()
        todo += re.findall(r'^\s*#\s*include\s+"([^"]+)"', src, flags=re.M)
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(name.encode() + b"\0" + " ".join(src.split()).encode())
    return h.hexdigest()[:16]


def _traffic(kernel: str, units: float):
    """DRAM bytes per launch of `kernel` from the committed ncu capture summary, scaled to
    the launch's work; None when absent or when the kernel's translation unit changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        e = d[kernel]
        if e.get("src_digest") != _src_digest(kernel):
            return None
        return float(e["dram_bytes_per_unit"]) * units
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc, self.lines = gpu, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def token_shard(rank: int, T: int) -> tuple[int, int]:
    """Weak scaling with no exchange: rank r runs its own T tokens, numbers r*T .. r*T+T-1 of
    the workload's seeded token stream, so the ranks' shards are disjoint."""
    return rank * T, T


def reduce_max(v: float, dev, ws: int) -> float:
    """The maximum of v over the ranks (the job time is the slowest rank's)."""
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(ws: int, T: int, steps: int, ms_max: float) -> float:
    """Whole-job tokens/s: the tokens of every rank over the slowest rank's time."""
    return ws * T * steps / (ms_max / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------------------------------
# CPU oracle legs (reference arm and cpu_baseline)
# ------------------------------------------------------------------------------------------
def _oracle_token_layers(args):
    """Worker: run the oracle on (token, layer) pairs of the decode workload; returns count."""
    wname, pairs = args
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    import oracle
    import synth
    w = synth.WORKLOADS[wname]
    grid = synth.grid(w.seed)
    stacked = w.n_layers > 1
    for t, l in pairs:
        x = synth.tokens(w, t, 1).astype(np.float64)
        table = np.arange(1, w.n_experts + 1, dtype=np.uint64) * np.uint64(1 << 20)
        recs = {}

        def rec(slot, l=l):
            e = int(slot >> np.uint64(20)) - 1
            if e not in recs:
                recs[e] = synth.expert_records(w, l, e, 1, nthreads=1)[0]
            return recs[e]
        xn = oracle.rmsnorm(x) if stacked else x
        r = oracle.route(xn, synth.router(w, l), None, table, w.top_k, l)
        oracle.moe_experts(xn, r.ids, r.weights, r.slots, rec, w.hidden, w.inter, grid)
    return len(pairs)


def oracle_rate(wname: str, budget_s: float = 20.0, cores: int | None = None):
    """Oracle throughput on a bounded sample: (token, layer) units spread over a spawn pool
    of `cores` processes, each single-threaded; stops adding rounds after `budget_s`."""
    import multiprocessing as mp
    import synth
    w = synth.WORKLOADS[wname]
    cores = cores or max(1, len(os.sched_getaffinity(0)))
    ctx = mp.get_context("spawn")
    done, t0, rnd = 0, None, 0
    with ctx.Pool(cores) as pool:
        pool.map(_oracle_token_layers, [(wname, [])] * cores)      # start the workers
        t0 = time.perf_counter()
        while True:
            jobs = [(wname, [((rnd * cores + c) % w.tokens, (rnd * cores + c) % w.n_layers)])
                    for c in range(cores)]
            done += sum(pool.map(_oracle_token_layers, jobs))
            rnd += 1
            if time.perf_counter() - t0 >= budget_s:
                break
    wall = time.perf_counter() - t0
    tokens = done / w.n_layers
    return tokens / wall, cores, f"{done} (token, layer) units of {wname} ({rnd} rounds x {cores} processes, " \
                                 f"each unit = router + top-{w.top_k} experts of one token in one layer), {wall:.1f} s"


def run_reference(a):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import synth
    w = synth.WORKLOADS[a.workload]
    per_step = []
    cores = max(1, len(os.sched_getaffinity(0)))
    for i in range(a.warmup + a.steps):
        rate, cores, sample = oracle_rate(a.workload, budget_s=a.ref_step_s, cores=cores)
        if i >= a.warmup:
            per_step.append(rate)
    value = sum(per_step) / len(per_step)
    rate1, _, sample1 = oracle_rate(a.workload, budget_s=a.ref_step_s, cores=1)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000.0 * w.tokens / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, a),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: {sample}; ms_per_step is the time a whole step of "
                                       f"{w.tokens} tokens takes at that rate",
                             "single_thread": {"value": rate1, "unit": "tokens/s", "cores": 1, "sample": sample1}},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config(w, a):
    nl = getattr(a, "layers", None) or w.n_layers
    c = {"workload": w.name if nl == w.n_layers else f"{w.name} (first {nl} layers)", "hidden": w.hidden,
         "n_experts": w.n_experts, "top_k": w.top_k, "inter": w.inter, "n_layers": nl, "tokens_per_step": w.tokens,
         "record_bytes": w.record_bytes, "resident_bytes": nl * w.n_experts * w.record_bytes,
            "l2": "inputs larger than L2 (590.6 MB of weights per token)" if w.n_layers > 1 else
                  "per-token working set 12.3 MB (router stays L2-resident across tokens)",
            "parallelism": f"replicas x{a.gpus}", "seed": w.seed}
    c["decode_path"] = getattr(a, "decode_path", "fused")
    return c


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------
def run_ours(a):
    import numpy as np
    import torch
    import torch.distributed as dist

    import synth
    from quantized_moe_expert_rl_gb300 import _lib as L
    from quantized_moe_expert_rl_gb300 import build as cbuild
    from quantized_moe_expert_rl_gb300 import engine

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cbuild.build()
    w = synth.WORKLOADS[a.workload]
    stacked = w.n_layers > 1
    T = w.tokens
    model = engine.Model(w, device=dev, layers=a.layers)
    b = engine.DecodeBuffers.make(model)
    # this rank's tokens (weak scaling: every rank decodes its own 256 / 1000 tokens)
    t0, _ = token_shard(rank, T)
    x_host = torch.from_numpy(synth.tokens(w, t0, T)).pin_memory()
    x_in = x_host.to(dev)
    y_out = torch.zeros_like(x_in)
    y_host = torch.empty_like(x_host).pin_memory()
    stream = torch.cuda.Stream(device=dev)
    fused = a.decode_path == "fused"

    if fused:
        # one launch per token: moe_decode_stack runs all layers (plus the copy of x into y);
        # for one layer without residual, moe_decode_layer runs the router and the experts
        def token(t):
            if stacked:
                engine.enqueue_decode_token_fused(model, b, x_in[t], y_out[t], pregate=a.pregate)
            else:
                engine.enqueue_decode_layer_fused(model, b, x_in[t], y_out[t])
        launches_per_token = 1

        def step():
            for t in range(T):
                token(t)
    else:
        # per-token CUDA graphs of the per-layer chain: rl_route (1 kernel) + moe_decode (2)
        with torch.cuda.stream(stream):
            engine.enqueue_decode_token(model, b, x_in[0], y_out[0], stacked)
        stream.synchronize()
        graphs = []
        for t in range(T):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                engine.enqueue_decode_token(model, b, x_in[t], y_out[t], stacked)
            graphs.append(g)
        launches_per_token = model.L * 3

        def step():
            for g in graphs:
                g.replay()

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            step()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk, torch.cuda.stream(stream):
        barrier()
        ev0.record(stream)
        for _ in range(a.steps):
            step()
        ev1.record(stream)
        barrier()
    ms = ev0.elapsed_time(ev1)
    ctrl = b.ctrl.cpu().tolist()
    assert ctrl[0] == L.RL_NO_EARLY_OUT and ctrl[1] == 0, f"device control block {ctrl}"
    ms_max = reduce_max(ms, dev, ws)
    value = weak_value(ws, T, a.steps, ms_max)

    # ---- end to end: pinned host x -> device, the tokens, device -> pinned host y ----
    h2d = x_host.numel() * 4
    d2h = y_host.numel() * 4
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(a.steps):
            x_in.copy_(x_host, non_blocking=True)
            step()
            y_host.copy_(y_out, non_blocking=True)
        e1.record(stream)
    barrier()
    e2e_value = weak_value(ws, T, a.steps, reduce_max(e0.elapsed_time(e1), dev, ws))

    peak, peak_kind = _peaks()
    per_layer_bytes = w.top_k * w.record_bytes + w.n_experts * w.hidden * 4 + 2 * w.hidden * 4
    kt_tokens = min(T, 16)
    if fused and not stacked:
        # ---- dominant kernel: moe_decode_layer, one launch = router + experts of one token ----
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(kt_tokens)]
        ybuf = torch.zeros(w.hidden, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            for rep in range(2):                  # first pass warms the code path
                for t in range(kt_tokens):
                    s_, e_ = evs[t]
                    s_.record(stream)
                    engine.enqueue_decode_layer_fused(model, b, x_in[t], ybuf)
                    e_.record(stream)
        stream.synchronize()
        t_launch = float(np.mean([s_.elapsed_time(e_) for s_, e_ in evs])) * 1e-3
        achieved = per_layer_bytes / t_launch / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": _traffic("moe_decode_layer", 1.0),
                    "kernel": "moe_decode_layer (router + experts of one token per launch)",
                    "bytes_per_launch": per_layer_bytes, "launch_us": t_launch * 1e6,
                    "peak_source": f"{peak_kind} hbm_gbs"}
    elif fused:
        # ---- dominant kernel: moe_decode_stack, one launch = one token through every layer ----
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(kt_tokens)]
        ybuf = torch.zeros(w.hidden, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            for rep in range(2):                  # first pass warms the code path
                for t in range(kt_tokens):
                    ybuf.copy_(x_in[t])
                    s_, e_ = evs[t]
                    s_.record(stream)
                    L.moe_decode_stack(model.shape, 0, model.L, ybuf, engine.EPS, model.routers, model.bias,
                                       model.table, model.codebook, b.ids, b.weights, b.slots, b.miss, b.ctrl,
                                       None, None, a.pregate, None, b.stack_ws, b.stack_ws.numel(), stream)
                    e_.record(stream)
        stream.synchronize()
        durs = np.array([s_.elapsed_time(e_) for s_, e_ in evs]) * 1e-3
        t_launch = float(np.mean(durs))
        bytes_per_launch = model.L * per_layer_bytes
        achieved = bytes_per_launch / t_launch / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": _traffic("moe_decode_stack", 1.0),
                    "kernel": f"moe_decode_stack ({model.L} layers of router + experts per launch)",
                    "bytes_per_launch": bytes_per_launch, "launch_us": t_launch * 1e6,
                    "us_per_layer": t_launch * 1e6 / model.L, "peak_source": f"{peak_kind} hbm_gbs"}
    else:
        # ---- dominant call: moe_decode (expert gate/up GEMV + down GEMV with ordered combine) ----
        roofline = moe_decode_roofline(model, b, x_in, stacked, kt_tokens, stream, dev)

    line = None
    if rank == 0:
        cpu = None
        if ws == 1 and not a.no_cpu_baseline:
            rate, cores, sample = oracle_rate(a.workload, budget_s=a.cpu_budget_s)
            cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
            rate1, _, sample1 = oracle_rate(a.workload, budget_s=a.cpu_budget_s / 2, cores=1)
            cpu["single_thread"] = {"value": rate1, "unit": "tokens/s", "cores": 1, "sample": sample1}
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": a.steps,
                "warmup": a.warmup, "ms_per_step": ms_max / a.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": _config(w, a), "clocks": clk.summary(), "roofline": roofline,
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": launches_per_token * T * a.steps,
                "us_per_token": ms_max * 1e3 / (T * a.steps)}
        if ws == 1 and not a.no_prefill:
            del model
            torch.cuda.empty_cache()
            if a.workload == "decode_stack":
                line["decode_layer"] = decode_layer_leg(dev, max(1, a.steps // 3), 3)
                torch.cuda.empty_cache()
                if not a.no_bounded:
                    line["decode_bounded"] = bounded_decode_leg(dev)
                    torch.cuda.empty_cache()
            line["prefill"] = prefill_leg(dev, a.steps, a.warmup)
            if not a.no_bounded:
                torch.cuda.empty_cache()
                line["prefill_bounded"] = bounded_leg(dev, max(1, a.steps // 3), 1)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def moe_decode_roofline(model, b, x_in, stacked: bool, kt_tokens: int, stream, dev) -> dict:
    """moe_decode (expert gate/up GEMV + down GEMV with ordered combine) timed alone per call
    with events on its stream, over kt_tokens sampled tokens x all layers; the slots, weights
    and layer inputs of each (token, layer) are recorded first from the real chain."""
    import numpy as np
    import torch

    from quantized_moe_expert_rl_gb300 import _lib as L
    from quantized_moe_expert_rl_gb300 import engine
    w = model.w
    slots_rec = torch.zeros((kt_tokens, model.L, w.top_k), dtype=torch.int64, device=dev)
    w_rec = torch.zeros((kt_tokens, model.L, w.top_k), dtype=torch.float32, device=dev)
    xs_rec = torch.zeros((kt_tokens, model.L, w.hidden), dtype=torch.float32, device=dev)
    yscr = torch.zeros(w.hidden, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        for t in range(kt_tokens):
            engine.enqueue_decode_token(model, b, x_in[t], yscr, stacked, x_hist=xs_rec[t] if stacked else None)
            slots_rec[t].copy_(b.slots)
            w_rec[t].copy_(b.weights)
            if not stacked:
                xs_rec[t, 0].copy_(x_in[t])
    stream.synchronize()
    ybuf = torch.zeros(w.hidden, dtype=torch.float32, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(kt_tokens * model.L)]
    eps = engine.EPS if stacked else -1.0
    with torch.cuda.stream(stream):
        for rep in range(2):                      # first pass warms the code path
            i = 0
            for t in range(kt_tokens):
                for l in range(model.L):
                    s_, e_ = evs[i]
                    s_.record(stream)
                    L.moe_decode(model.shape, l, xs_rec[t, l], eps, slots_rec[t, l], w_rec[t, l],
                                 model.codebook, ybuf, 0, b.ctrl, b.dec_ws, b.dec_ws.numel(), stream)
                    e_.record(stream)
                    i += 1
    stream.synchronize()
    durs = np.array([s_.elapsed_time(e_) for s_, e_ in evs]) * 1e-3      # seconds
    t_launch = float(np.mean(durs))
    bytes_per_launch = (w.top_k * w.record_bytes + 2 * w.hidden * 4 + 2 * w.top_k * w.inter * 4)
    achieved = bytes_per_launch / t_launch / 1e9
    peak, peak_kind = _peaks()
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": _traffic("moe_decode", 1.0), "kernel": "moe_decode (gate/up + down GEMVs)",
            "bytes_per_launch": bytes_per_launch, "launch_us": t_launch * 1e6,
            "peak_source": f"{peak_kind} hbm_gbs"}


def decode_layer_leg(dev, steps: int, warmup: int) -> dict:
    """Single-token decode of one layer (hidden 2048, 512 experts, top-10, inter 512): 1000
    seeded tokens, one at a time, each one CUDA graph of rl_route + moe_decode (y = MoE(x), no
    norm, no residual); moe_decode also timed alone per call against the HBM roofline."""
    import torch

    import synth
    from quantized_moe_expert_rl_gb300 import engine
    w = synth.WORKLOADS["decode_layer"]
    model = engine.Model(w, device=dev)
    b = engine.DecodeBuffers.make(model)
    T = w.tokens
    x = torch.from_numpy(synth.tokens(w, 0, T)).to(dev)
    y = torch.zeros_like(x)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        engine.enqueue_decode_token(model, b, x[0], y[0], False)
    stream.synchronize()
    graphs = []
    for t in range(T):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            engine.enqueue_decode_token(model, b, x[t], y[t], False)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for g in graphs:
                g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            for g in graphs:
                g.replay()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / steps
    roof = moe_decode_roofline(model, b, x, False, 16, stream, dev)
    ctrl = b.ctrl.cpu().tolist()
    assert ctrl == [0x7FFFFFFF, 0], ctrl
    # the same tokens through moe_decode_layer: router and experts of a token in one launch,
    # held in one CUDA graph per token like the chain above, so that the host's argument checks
    # and launch calls (tens of microseconds on the host, more than the kernel) stay out of the
    # timing; direct launches if the driver refuses to capture the cooperative launch
    bf = engine.DecodeBuffers.make(model)
    yf = torch.zeros_like(x)
    with torch.cuda.stream(stream):
        for t in range(T):                            # first-use setup outside any capture
            engine.enqueue_decode_layer_fused(model, bf, x[t], yf[t])
    stream.synchronize()
    fgraphs, fpath = [], "one CUDA graph per token holding its moe_decode_layer launch (router + experts)"
    try:
        for t in range(T):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                engine.enqueue_decode_layer_fused(model, bf, x[t], yf[t])
            fgraphs.append(g)
    except RuntimeError as ex:
        torch.cuda.synchronize(dev)
        fgraphs = []
        fpath = f"one moe_decode_layer launch per token from the host (graph capture refused: {str(ex)[:120]})"

    def run_fused(t):
        if fgraphs:
            fgraphs[t].replay()
        else:
            engine.enqueue_decode_layer_fused(model, bf, x[t], yf[t])
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(T)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for t in range(T):
                run_fused(t)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(steps):
            for t in range(T):
                run_fused(t)
        f1.record(stream)
        for t in range(T):                            # each launch alone, for the roofline
            evs[t][0].record(stream)
            run_fused(t)
            evs[t][1].record(stream)
    stream.synchronize()
    assert bf.ctrl.cpu().tolist() == [0x7FFFFFFF, 0]
    msf = f0.elapsed_time(f1) / steps
    t_launch = sum(a_.elapsed_time(b_) for a_, b_ in evs) / T * 1e-3
    bytes_launch = w.top_k * w.record_bytes + w.n_experts * w.hidden * 4 + 2 * w.hidden * 4
    peak, peak_kind = _peaks()
    froof = {"bound": "hbm", "achieved": bytes_launch / t_launch / 1e9, "peak": peak, "unit": "GB/s",
             "frac": bytes_launch / t_launch / 1e9 / peak, "traffic": _traffic("moe_decode_layer", 1.0),
             "kernel": "moe_decode_layer (router + experts of one token, one launch)",
             "bytes_per_launch": bytes_launch, "launch_us": t_launch * 1e6, "peak_source": f"{peak_kind} hbm_gbs"}
    return {"workload": "decode_layer (1 layer, 1000 tokens one at a time)",
            "path": fpath,
            "tokens_per_s": T / (msf * 1e-3), "us_per_token": msf * 1e3 / T, "roofline": froof,
            "chain": {"path": "per-token CUDA graph: rl_route + moe_decode (3 kernels)",
                      "tokens_per_s": T / (ms * 1e-3), "us_per_token": ms * 1e3 / T, "roofline": roof},
            "target": "expert GEMVs at >= 70% of HBM peak"}


def bounded_decode_leg(dev, n_tokens: int = 16) -> dict:
    """The decode stack with bounded residency at full shape: 48 layers x 512 experts, 435 of
    them resident per layer (seeded), the first n_tokens seeded tokens from that residency.
    Device path: one moe_decode_stack_fill launch per token (absent experts copied by the GPU
    from the pinned backing store inside the launch); host path: the stack stops at each layer
    that selects an absent expert, the host fills and the stack resumes."""
    import time
    from dataclasses import replace

    import torch

    import synth
    from quantized_moe_expert_rl_gb300 import engine
    w = replace(synth.WORKLOADS["decode_stack"], n_resident=435)
    model = engine.Model(w, device=dev)
    b = engine.DecodeBuffers.make(model)
    x = torch.from_numpy(synth.tokens(w, 0, n_tokens)).to(dev)
    y = torch.zeros_like(x)
    pass_stats = {}

    def one_pass(mode, filled):
        stops = fills = misses = 0
        for t in range(n_tokens):
            b.miss.zero_()
            if mode == "device":
                engine.run_bounded_decode_token_device(model, b, x[t], y[t], filled)
            else:
                st = engine.run_bounded_decode_token(model, b, x[t], y[t])
                stops += len(st.early_outs)
                fills += len(st.filled)
            misses += int(b.miss.sum().item())
        pass_stats.update(stops=stops, fills=fills, misses=misses)

    res = {}
    for mode in ("device", "host"):
        # one untimed pass over the same tokens first (first use of the mapped backing store,
        # the fill tables, the code), then the timed pass from the seeded residency again
        for timed in (False, True):
            model.reset_residency()
            filled = torch.zeros(1, dtype=torch.int32, device=dev)
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            one_pass(mode, filled)
            if timed:
                break
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        fills = int(filled.item()) if mode == "device" else pass_stats["fills"]
        stops, misses = pass_stats["stops"], pass_stats["misses"]
        assert b.ctrl.cpu().tolist() == [0x7FFFFFFF, 0]
        res[mode] = {"tokens_per_s": n_tokens / wall, "ms_per_token": wall * 1e3 / n_tokens,
                     "experts_filled": fills, "misses": misses}
        if mode == "host":
            res[mode]["stops"] = stops
    return {"workload": f"decode_stack with 435/512 experts resident per layer, first {n_tokens} tokens "
                        f"from the seeded residency", **res}


def prefill_leg(dev, steps: int, warmup: int, path: str = "tc"):
    """The 512-token prefill chunk (one layer, 512 experts, 5120 pairs): routing, pair build,
    grouped expert GEMMs and the ordered combine, timed with events on the launching stream."""
    import torch

    import synth
    from quantized_moe_expert_rl_gb300 import _lib as L
    from quantized_moe_expert_rl_gb300 import engine
    w = synth.WORKLOADS["prefill_chunk"]
    model = engine.Model(w, device=dev)
    T = w.tokens
    b = engine.PrefillBuffers.make(model, T)
    x = torch.from_numpy(synth.tokens(w)).to(dev)
    y = torch.zeros_like(x)
    stream = torch.cuda.Stream(device=dev)
    fn = engine._experts_fn(path)

    def full():
        engine.enqueue_prefill_route(model, b, 0, x, stacked=False)
        engine.enqueue_prefill_experts(model, b, 0, x, y, stacked=False, path=path)

    def experts_only():
        fn(model.shape, 0, T, x, b.offs, b.pair_tok, b.pair_k, b.slots, b.weights, model.codebook, y, 0, b.ctrl,
           b.ws, b.ws.numel(), stream)

    res = {}
    with torch.cuda.stream(stream):
        for name, f in (("path", full), ("experts", experts_only)):
            for _ in range(warmup):
                f()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                f()
            e1.record(stream)
            stream.synchronize()
            res[name] = e0.elapsed_time(e1) / steps
    assert b.ctrl.tolist() == [L.RL_NO_EARLY_OUT, 0], b.ctrl.tolist()
    union = int((b.offs[1:] - b.offs[:-1] > 0).sum().item())
    P = T * w.top_k
    flops = 2.0 * P * 3 * w.hidden * w.inter
    bytes_ = union * w.record_bytes
    t_ex = res["experts"] * 1e-3
    hbm, hbm_kind = _peaks()
    tf, tf_kind = _tensor_peak()
    t_hbm, t_tc = bytes_ / (hbm * 1e9), flops / (tf * 1e12)
    roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor", "kernel": "moe_prefill_chunk (tc_gemm gate/up + down)",
            "achieved_gbs": bytes_ / t_ex / 1e9, "peak_gbs": hbm, "frac_hbm": t_hbm / t_ex,
            "achieved_tflops": flops / t_ex / 1e12, "peak_tflops": tf, "frac_tensor": t_tc / t_ex,
            "traffic": _traffic("tc_gemm", 1.0), "peak_source": f"{hbm_kind} hbm_gbs, {tf_kind}"}
    return {"workload": "prefill_chunk (1 layer, 512 tokens, 5120 pairs)", "operands": "f16" if path == "tc" else "f32",
            "roofline": roof,
            "tokens_per_s": T / (res["path"] * 1e-3), "ms_per_chunk": res["path"],
            "experts_ms_per_chunk": res["experts"], "experts_tokens_per_s": T / t_ex,
            "experts_tflops": flops / t_ex / 1e12, "experts_hbm_gbs": bytes_ / t_ex / 1e9,
            "union_experts": union, "flop_per_chunk": flops, "weight_bytes_per_chunk": bytes_}


def bounded_leg(dev, steps: int, warmup: int, path: str = "tc"):
    """48 layers x 2048 tokens with Zipf router bias and 85% residency: every step runs the
    chunk from the seeded residency (fills from pinned host memory on each early-out)."""
    import time

    import numpy as np
    import torch

    import synth
    from quantized_moe_expert_rl_gb300 import engine
    w = synth.WORKLOADS["prefill_bounded"]
    model = engine.Model(w, device=dev)
    b = engine.PrefillBuffers.make(model, w.tokens)
    x0 = torch.from_numpy(synth.tokens(w)).to(dev)
    x = torch.empty_like(x0)
    walls, fills, last = [], [], None
    for i in range(warmup + steps):
        model.reset_residency()
        x.copy_(x0)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        st = engine.run_bounded_chunk(model, b, x, path=path)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        if i >= warmup:
            walls.append(wall)
            fills.append(st.fill_seconds)
            last = st
    wall = sum(walls) / len(walls)
    fill = sum(fills) / len(fills)
    # the same chunks with every fill done by the device (rl_fill_missing): one host sync
    dwalls, dlast = [], None
    for i in range(warmup + steps):
        model.reset_residency()
        x.copy_(x0)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        dst = engine.run_bounded_chunk_device(model, b, x, path=path)
        torch.cuda.synchronize(dev)
        if i >= warmup:
            dwalls.append(time.perf_counter() - t0)
            dlast = dst
    dwall = sum(dwalls) / len(dwalls)
    # one more device-filled chunk with every stage timed by events, the routing of every
    # layer kept to count the distinct experts each layer runs
    model.reset_residency()
    x.copy_(x0)
    ids_hist = torch.zeros((model.L, w.tokens, w.top_k), dtype=torch.int32, device=dev)
    split = {}
    engine.run_bounded_chunk_device(model, b, x, path=path, hist={"ids": ids_hist}, timing=split)
    ids_np = ids_hist.cpu().numpy()
    union = sum(len(np.unique(ids_np[l])) for l in range(model.L))
    P = w.tokens * w.top_k
    flops = model.L * 2.0 * P * 3 * w.hidden * w.inter
    wbytes = union * w.record_bytes
    t_ex = split["experts"] * 1e-3
    hbm, hbm_kind = _peaks()
    tf, tf_kind = _tensor_peak()
    t_hbm, t_tc = wbytes / (hbm * 1e9), flops / (tf * 1e12)
    roof = {"bound": "hbm" if t_hbm >= t_tc else "tensor",
            "kernel": f"moe_prefill_chunk over the {model.L} layers (pair build + grouped tc_gemm)",
            "achieved_tflops": flops / t_ex / 1e12, "peak_tflops": tf, "frac_tensor": t_tc / t_ex,
            "achieved_gbs": wbytes / t_ex / 1e9, "peak_gbs": hbm, "frac_hbm": t_hbm / t_ex,
            "flop_per_chunk": flops, "weight_bytes_per_chunk": wbytes, "union_experts": union,
            "peak_source": f"{hbm_kind} hbm_gbs, {tf_kind}"}
    return {"workload": "prefill_bounded (48 layers x 2048 tokens, Zipf 1.1, 435/512 resident)",
            "tokens_per_s_excl_fill": w.tokens / (wall - fill), "tokens_per_s_incl_fill": w.tokens / wall,
            "s_per_chunk": wall, "fill_s_per_chunk": fill, "early_outs": len(last.early_outs),
            "first_early_out": last.first_early_out, "misses_total": sum(last.miss),
            "experts_filled": len(last.filled), "fill_bytes": last.fill_bytes, "host_syncs": last.syncs,
            "device_fill": {"tokens_per_s": w.tokens / dwall, "s_per_chunk": dwall,
                            "experts_filled": len(dlast.filled), "misses_total": sum(dlast.miss),
                            "host_syncs": dlast.syncs,
                            "split_ms": {k: round(v, 3) for k, v in split.items()},
                            "roofline": roof}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode_stack", "decode_layer"], default="decode_stack")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--ref-step-s", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-bounded", action="store_true")
    ap.add_argument("--decode-path", choices=["fused", "chain"], default="fused",
                    help="one fused launch per token (moe_decode_stack through every layer; moe_decode_layer "
                         "for the single-layer workload), or per-token graphs of the per-layer rl_route + "
                         "moe_decode chain")
    ap.add_argument("--pregate", type=int, default=0,
                    help="fused decode: experts of the next layer prefetched into L2 on the pre-gated "
                         "prediction (0 = off)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers of the stacked workload (profiling of smaller cases)")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
