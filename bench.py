"""Benchmark: one MoE layer forward + backward per step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one pass of the whole path over one batch of synthetic input:
router logits, top-k gate, dispatch, permute, expert FFN, combine, and the
backward of each (all dispatch chunks of the workload).  Inputs are resident
in HBM before the timed region; L2 is flushed (a 256 MiB write) between
steps, outside the per-step CUDA-event brackets.  Prints ONE JSON line on
rank 0.

Multi-GPU: the layer does not shard (one GPU per layer pass, no collective in
the data path), so N ranks run N independent replicas; the timed region is
bracketed by a barrier and the slowest rank's time is taken ("scaling":
"weak").

--impl reference times the CPU oracle (the plain definition of the layer, in
double precision) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mixture_experts_layer_11_gb300 import synth  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s and TFLOP/s on 1 GB300; % of bf16 peak and HBM roofline"
DEFAULT_CONFIG = "moe_s_bf16"
L2_FLUSH_BYTES = 256 << 20

def launches_per_chunk(cfg) -> int:
    """Library kernels one dispatch chunk of a step launches.
    Route: bf16 with d_model % 64 == 0 runs the logits GEMM, the gate, the
    scan and the rank (4); otherwise logits + gate fused for E <= 32 (3) or
    separate (4).  Permute (1); two expert GEMMs (2); combine (1); combine
    backward (1).  Expert backward: bf16 has the dH GEMM + its db1 reduction,
    the dX GEMM and two weight-gradient GEMMs (db2 inside the dW2 one) = 5;
    fp32 has four GEMMs and two column sums of two kernels each = 8.  Router
    backward: with renorm, dx with the permute backward fused in and dWg (2
    kernels) = 3; without (dense gate Jacobian), dL, the tiled dx product
    with the permute backward, and dWg (2 kernels) = 4."""
    bf16_tc = cfg.dtype == "bf16" and cfg.d % 64 == 0
    route = 4 if (bf16_tc or cfg.E > 32) else 3
    ffn_bwd = 5 if cfg.dtype == "bf16" else 8
    route_bwd = 3 if cfg.renorm else 4
    return route + 1 + 2 + 1 + 1 + ffn_bwd + route_bwd


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the six expert
# GEMM launches of one step, from one ncu capture (profiles/gemm_tc_moe_s_bf16.md),
# valid only for the grouped-GEMM source it was taken on (first 16 hex digits of
# its SHA-256); any other source or workload reports null.
GEMM_TRAFFIC = {"moe_s_bf16": (1087.1e6, "14e8d341c1309f45")}


def gemm_traffic(cfg):
    entry = GEMM_TRAFFIC.get(cfg.name)
    if entry is None:
        return None
    import hashlib
    src = os.path.join(ROOT, "mixture_experts_layer_11_gb300", "csrc", "gemm_tc.cu")
    try:
        with open(src, "rb") as fh:
            digest = hashlib.sha256(fh.read()).hexdigest()[:16]
    except OSError:
        return None
    return entry[0] if digest == entry[1] else None


def workload_desc(cfg) -> str:
    s = (f"{cfg.name}: T={cfg.T} d_model={cfg.d} d_ffn={cfg.f} E={cfg.E} top-{cfg.k}"
         f"{' renorm' if cfg.renorm else ''} {cfg.dtype}")
    if cfg.zipf_s:
        s += f" zipf_s={cfg.zipf_s} logit shift"
    if cfg.chunk:
        s += f" dispatch chunks of {cfg.chunk}"
    return s


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---- clocks sampled during the timed region ------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.proc = None
        self.dev = dev_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = max(smax, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- CPU oracle timing ------------------------------------------------------------------

def oracle_tokens_per_s(cfg, budget_s: float = 15.0, seed: int = 0):
    """Time the oracle's full forward + backward on growing token samples of
    the workload (same sizes d, f, E, k) until one run takes a few seconds or
    the cumulative budget is spent.  Returns (tokens/s, sample description,
    cores)."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    oracle.build()
    Ts, spent, best = 64, 0.0, None
    while True:
        Ts = min(Ts, cfg.T)
        sub = cfg.scaled(T=Ts, chunk=None)
        inp = synth.make_inputs(sub, seed=seed)
        t0 = time.perf_counter()
        oracle.layer(inp, sub.k, sub.renorm, sub.dtype == "bf16")
        dt = time.perf_counter() - t0
        spent += dt
        best = (Ts / dt, Ts, dt)
        if dt > budget_s / 4 or Ts >= cfg.T or spent + 4 * dt > budget_s:
            break
        Ts *= 2
    tps, Ts, dt = best
    desc = (f"oracle fwd+bwd on the first {Ts} of {cfg.T} tokens (same d_model, d_ffn, E, k, "
            f"weights drawn with the same recipe) took {dt:.2f} s; tokens/s scales linearly")
    return tps, desc, cores


# ---- reference arm: the oracle as the baseline implementation --------------------------

def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    vals, desc, cores = [], "", 1
    budget = max(5.0, 120.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        tps, desc, cores = oracle_tokens_per_s(cfg, budget_s=budget, seed=i)
        if i >= args.warmup:
            vals.append(tps)
    v = statistics.median(vals)
    flops_per_token = (cfg.expert_flops() + cfg.router_flops()) / cfg.T
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": cfg.T / v * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "tflops": v * flops_per_token / 1e12,
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "d_model": cfg.d,
                   "d_ffn": cfg.f, "E": cfg.E, "k": cfg.k},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- replicas: the slowest rank's times and the whole job's rate ---------------------------

def max_over_ranks(values, dist, device):
    """Element-wise maximum of a list of times over all ranks (the values
    unchanged with one process).  dist: torch.distributed or None."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(tokens_per_rank_step: int, steps: int, world: int, ms: float) -> float:
    """Tokens per second of all replicas together: every rank processed
    tokens_per_rank_step tokens per step, over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / (ms / 1e3)


# ---- our arm -----------------------------------------------------------------------------

def run_ours(args, cfg):
    from mixture_experts_layer_11_gb300 import ops
    from mixture_experts_layer_11_gb300.layer import LayerPass

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ops.lib()  # fail loudly if the library is missing

    inp = synth.make_inputs(cfg, seed=rank, device=str(dev))
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=dev, recompute=args.recompute)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ev = lambda **kw: torch.cuda.Event(enable_timing=True, **kw)  # noqa: E731
    x_buf, dy_buf = inp["x"], inp["dy"]   # fixed input buffers (the graph reads these)

    # events around the expert-FFN calls (the grouped GEMM launches), recorded
    # on the launching stream; inside a captured graph they are graph nodes
    ffn_events = []
    orig_fwd, orig_bwd = ops.moe_expert_ffn_fwd, ops.moe_expert_ffn_bwd
    state = {"record": False, "external": False}

    def timed(fn, kind):
        def wrapper(*a, **kw):
            if not state["record"]:
                return fn(*a, **kw)
            e0, e1 = ev(external=state["external"]), ev(external=state["external"])
            e0.record()
            r = fn(*a, **kw)
            e1.record()
            ffn_events.append((kind, e0, e1))
            return r
        return wrapper

    import mixture_experts_layer_11_gb300.layer as layer_mod
    layer_mod.ops.moe_expert_ffn_fwd = timed(orig_fwd, "fwd")
    layer_mod.ops.moe_expert_ffn_bwd = timed(orig_bwd, "bwd")

    def step():
        lp.forward(x_buf, inp["Wg"], inp["W1"], inp["b1"], inp["W2"], inp["b2"], inp["beta"])
        lp.backward(dy_buf, x_buf, inp["Wg"], inp["W1"], inp["W2"])

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    lp.check_status()

    graph = None
    if not args.no_graph:
        # one whole step (every chunk, forward and backward) as one CUDA graph
        graph = torch.cuda.CUDAGraph()
        state.update(record=True, external=True)
        with torch.cuda.graph(graph):
            step()
        state.update(record=False, external=False)
        graph_ffn = list(ffn_events)
        ffn_events.clear()
        graph.replay()
        torch.cuda.synchronize()
        lp.check_status()

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    st = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = []
    ffn_ms = {"fwd": 0.0, "bwd": 0.0}
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.fill_(1)
        e0, e1 = ev(), ev()
        if graph is None:
            state["record"] = True
        e0.record(st)
        run_step()
        e1.record(st)
        state["record"] = False
        torch.cuda.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        marks = graph_ffn if graph is not None else ffn_events
        for kind, a, b in marks:
            ffn_ms[kind] += a.elapsed_time(b)
        ffn_events.clear()
    wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    lp.check_status()
    total_ms = sum(step_ms)
    layer_mod.ops.moe_expert_ffn_fwd, layer_mod.ops.moe_expert_ffn_bwd = orig_fwd, orig_bwd

    # ---- end to end through the public API with host buffers ----
    # A training loop's input pipeline: two device sets of inputs (x, dy) and
    # outputs (y, dx), one CUDA graph per set.  Pinned host inputs are copied
    # (H2D stream) into one set while the other set's step computes; a step's
    # y and dx are read back (D2H stream) while the next step computes.
    # Events order every reuse.  The timed span runs from the compute stream reaching the first
    # timed step (whose inputs were copied during the step before, like every
    # later step's) to the end of the last step's D2H (the drain included, as
    # is the L2 flush before every step on the compute stream).
    x_h = inp["x"].cpu().pin_memory()
    dy_h = inp["dy"].cpu().pin_memory()
    in_bufs = [(x_buf, dy_buf), (torch.empty_like(x_buf), torch.empty_like(dy_buf))]
    out_bufs = [(lp.y, lp.dx), (torch.empty_like(lp.y), torch.empty_like(lp.dx))]
    out_h = [(torch.empty(x_h.shape, dtype=x_h.dtype, pin_memory=True),
              torch.empty(x_h.shape, dtype=x_h.dtype, pin_memory=True)) for _ in range(2)]

    def step_on(b):
        xb, dyb = in_bufs[b]
        lp.y, lp.dx = out_bufs[b]
        lp.forward(xb, inp["Wg"], inp["W1"], inp["b1"], inp["W2"], inp["b2"], inp["beta"])
        lp.backward(dyb, xb, inp["Wg"], inp["W1"], inp["W2"])

    graphs = [graph, None]
    if graph is not None:
        graphs[1] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[1]):
            step_on(1)
        lp.y, lp.dx = out_bufs[0]
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set b copied
    ev_done = [torch.cuda.Event() for _ in range(2)]   # step on set b done
    ev_read = [torch.cuda.Event() for _ in range(2)]   # outputs of set b read back
    t_start, t_end = ev(), ev()
    n = args.warmup + args.steps
    torch.cuda.synchronize()

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(cs_in):
            if i >= 2:
                cs_in.wait_event(ev_done[b])    # step i-2 has consumed set b
            in_bufs[b][0].copy_(x_h, non_blocking=True)
            in_bufs[b][1].copy_(dy_h, non_blocking=True)
            ev_in[b].record(cs_in)

    h2d(0)
    for i in range(n):
        b = i % 2
        if i == args.warmup:
            t_start.record(st)
        st.wait_event(ev_in[b])
        if i >= 2:
            st.wait_event(ev_read[b])           # outputs of set b read back
        flush.fill_(1)
        if graphs[b] is not None:
            graphs[b].replay()
        else:
            step_on(b)
        ev_done[b].record(st)
        if i + 1 < n:
            h2d(i + 1)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(ev_done[b])
            out_h[b][0].copy_(out_bufs[b][0], non_blocking=True)
            out_h[b][1].copy_(out_bufs[b][1], non_blocking=True)
            ev_read[b].record(cs_out)
            if i == n - 1:
                t_end.record(cs_out)
    torch.cuda.synchronize()
    lp.check_status()
    e2e_ms = t_start.elapsed_time(t_end)
    # the device path of the same workload must have given the same outputs
    lp.y, lp.dx = out_bufs[0]
    if not torch.equal(out_h[(n - 1) % 2][0], out_bufs[(n - 1) % 2][0].cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident step")

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    tokens = cfg.T * args.steps * world
    value = whole_job_rate(cfg.T, args.steps, world, total_ms)
    flops = cfg.expert_flops() + cfg.router_flops()
    pk, pk_kind = peaks()
    gemm_flops = cfg.expert_flops() * args.steps
    gemm_ms = ffn_ms["fwd"] + ffn_ms["bwd"]
    achieved = gemm_flops / (gemm_ms / 1e3) / 1e12
    peak = pk.get("bf16_tflops_sustained", pk.get("bf16_tflops"))
    chunks = len(lp.chunks)
    # recompute: the backward re-runs each chunk's permute and two expert GEMMs
    launches = (launches_per_chunk(cfg) + (3 if args.recompute else 0)) * chunks * args.steps
    elem = 2 if cfg.dtype == "bf16" else 4
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic (seeded N(0,1) inputs, N(0,1/fan_in) weights)",
        "tflops": flops * args.steps * world / (total_ms / 1e3) / 1e12,
        "device_memory_gib": torch.cuda.max_memory_allocated(dev) / 2**30,
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "d_model": cfg.d,
                   "d_ffn": cfg.f, "E": cfg.E, "k": cfg.k,
                   "l2": "flushed between steps (256 MiB write, outside the step timing)",
                   "launch": "one CUDA graph per step" if graph is not None else "eager",
                   "activations": ("recomputed in the backward (routing kept)" if args.recompute
                                   else "kept from the forward for the backward"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {
            "bound": "tensor", "kernel": "grouped expert GEMM (tcgen05), all expert FFN calls",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_kind": f"bf16 dense cuBLAS, sustained ({pk_kind})",
            "traffic": gemm_traffic(cfg),
            "traffic_unit": "bytes per step (the six expert GEMM launches)",
            "algorithmic_flops_per_step": cfg.expert_flops(),
            "ffn_ms_per_step": {k: v / args.steps for k, v in ffn_ms.items()},
        },
        "gpu_launches": launches,
        "e2e": {"value": whole_job_rate(cfg.T, args.steps, world, e2e_ms), "unit": "tokens/s",
                "pipeline": "H2D of step i+1 and D2H of step i on copy streams, overlapping step i",
                "h2d_bytes_per_step": 2 * cfg.T * cfg.d * elem,
                "d2h_bytes_per_step": 2 * cfg.T * cfg.d * elem},
        "wall_s_timed_region": wall,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        tps, desc, cores = oracle_tokens_per_s(cfg)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--recompute", action="store_true",
                    help="keep only the routing between forward and backward; the backward "
                         "re-runs each chunk's permute and expert forward")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels one by one instead of as one CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
