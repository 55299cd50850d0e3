"""Benchmark: one MoE layer forward + backward per step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-sub-configs]

A step is one pass of the whole path over one batch of synthetic input:
router logits, top-k gate, dispatch, permute, expert FFN, combine, and the
backward of each (all dispatch chunks of the workload).  Inputs are resident
in HBM before the timed region; L2 is flushed (a 256 MiB write) between
steps, outside the per-step CUDA-event brackets.  Prints ONE JSON line on
rank 0.

The headline workload is the long-context one (T = 262144 in dispatch chunks
of 32768, d_model 4096, d_ffn 1024, E 128, top-8): the largest of the
layer's workloads that one GPU holds.  The line also carries, per other
workload, its device-timed rate, the grouped GEMM's fraction of the bf16
tensor peak and the dispatch kernels' fraction of HBM bandwidth.

Multi-GPU: the layer does not shard (one GPU per layer pass, no collective in
the data path), so N ranks run N independent replicas; the timed region is
bracketed by a barrier and the slowest rank's time is taken ("scaling":
"weak").

--impl reference times the CPU oracle (the plain definition of the layer, in
double precision) on the host cores, on a bounded token sample of the same
workload (every step runs that sample).
"""
from __future__ import annotations

import argparse
import json
import re
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
DEFAULT_CONFIG = "longctx128_bf16"
L2_FLUSH_BYTES = 256 << 20
ROUTER_TC_ENV = "MOE_ROUTER_TENSOR_CORES"


# weight-gradient GEMM calls over more rows than this (or over several chunks)
# take the segment-walking kernel, which adds a split-reduction kernel
VARK_LEAN_MAX_ROWS = 512 * 64


def launches_per_step(cfg, nchunks: int, router_tc: bool, recompute: bool, defer: bool,
                      gather: bool = False) -> int:
    """Library kernels one step launches.
    Per dispatch chunk.  Route: the tensor-core logits (bf16, d_model % 64 ==
    0, opt-in) or the CUDA-core logits kernel, then the gate, the scan and the
    rank (4); the CUDA-core router fuses logits and gate for E <= 32 (3).
    Permute (1; none when fused into the GEMM loads); two expert GEMMs (2);
    combine (1); combine backward (1).  Expert backward, bf16: the dH GEMM +
    its db1 reduction and the dX GEMM (3), and unless the weight gradients are
    deferred, the two weight-gradient GEMMs (db2 inside the dW2 one) (2), each
    with its split reduction when it walks more than VARK_LEAN_MAX_ROWS rows
    (+2); fp32: dH and dX GEMMs and db1's column sum of two kernels (4), plus
    two weight-gradient GEMMs and db2's column sum (4).  Router backward: with
    renorm, dx with the permute backward fused in and dWg (2 kernels) = 3;
    without (dense gate Jacobian), dL, the tiled dx product with the permute
    backward, and dWg (2 kernels) = 4.  Recompute re-runs the permute (unless
    fused) and the two forward GEMMs.  Deferred weight gradients: once per
    step, the two weight-gradient GEMMs and their split reductions (bf16), or
    per chunk two GEMMs and db2's column sum (fp32)."""
    bf = cfg.dtype == "bf16"
    tc = router_tc and bf and cfg.d % 64 == 0
    route = 4 if (tc or cfg.E > 32) else 3
    if not tc and cfg.E > 32:
        # CUDA-core logits in 128-row tiles of 64 (E <= 64) or 128 experts, two or
        # three blocks per SM; a stream-K split (and its fix-up kernel) when the
        # tiles do not fill whole waves
        Tc = min(cfg.T, cfg.chunk or cfg.T)
        bn = 64 if cfg.E <= 64 else 128
        tiles = -(-Tc // 128) * -(-cfg.E // bn)
        sms = torch.cuda.get_device_properties(0).multi_processor_count \
            if torch.cuda.is_available() else 152
        route += 1 if tiles % (sms * (3 if bn == 64 else 2)) else 0
    permute = 0 if gather else 1
    data = 3 if bf else 4
    chunk_rows = min(cfg.T, cfg.chunk or cfg.T) * cfg.k
    wgrad = (2 + (2 if chunk_rows > VARK_LEAN_MAX_ROWS else 0)) if bf else 4
    route_bwd = 3 if cfg.renorm else 4
    per_chunk = route + permute + 2 + 1 + 1 + data + (0 if defer else wgrad) + route_bwd
    per_chunk += (permute + 2) if recompute else 0
    multi = nchunks > 1 or cfg.T * cfg.k > VARK_LEAN_MAX_ROWS
    per_step = ((4 if multi else 2) if bf else 4 * nchunks) if defer else 0
    return per_chunk * nchunks + per_step


def gemm_traffic(cfg):
    """DRAM bytes per step of all expert GEMM launches, from the committed ncu
    summary of this workload, while the GEMM source is the one it was taken
    on; else None."""
    path = os.path.join(ROOT, "profiles", f"dram_gemm_{cfg.name}.md")
    src = os.path.join(ROOT, "mixture_experts_layer_11_gb300", "csrc", "gemm_tc.cu")
    try:
        import hashlib
        text = open(path).read()
        want = re.search(r"gemm_tc\.cu sha256: ([0-9a-f]{64})", text).group(1)
        n = int(re.search(r"traffic_bytes_per_step: (\d+)", text).group(1))
        # hash of the source without whitespace (layout changes keep the kernel)
        have = hashlib.sha256(re.sub(rb"\s+", b"", open(src, "rb").read())).hexdigest()
    except Exception:
        return None, "no DRAM counter capture of this workload's GEMMs"
    if have != want:
        return None, "the GEMM source changed since its DRAM counters were taken"
    return n, ("dram__bytes_read.sum + dram__bytes_write.sum of one step's expert GEMM launches "
               "(bytes per step, from one ncu pass over the step's launches)")


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


def elem_bytes(cfg) -> int:
    return 2 if cfg.dtype == "bf16" else 4


def dispatch_bytes(cfg, kind: str, T: int) -> float:
    """Algorithmic DRAM bytes of one call on T tokens (b bytes per element,
    P = T k rows): every row read or written once, plus the index / weight
    vectors.  route_bwd is the permute backward (dX_perm gathered, dx written)
    with the router's dWg = dL^T x (x read per selected expert)."""
    b, d, k = elem_bytes(cfg), cfg.d, cfg.k
    P = T * k
    if kind == "permute":          # x read, X_perm written, pos read
        return b * d * (T + P) + 4 * P
    if kind == "combine":          # Y_perm read, y written, pos and w read
        return b * d * (P + T) + 8 * P
    if kind == "combine_bwd":      # dy and Y_perm read, dY_perm written; pos, w, dw
        return b * d * (T + 2 * P) + 12 * P
    if kind == "route_bwd":        # dX_perm and x rows read, dx written
        return b * d * (2 * P + T) + 16 * P
    raise ValueError(kind)


# ---- clocks sampled during the timed region ------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int, period_ms: int = 100):
        self.proc = None
        self.dev = dev_index
        self.period = period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
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
        sm, power, smax, reasons = [], [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = max(smax, float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        # samples under load: power well above idle
        loaded = [s for s, p in zip(sm, power) if p > 0.4 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded),
                "period_ms": self.period, "power_w_max": max(power) if power else None}


# ---- the oracle on bounded token samples -----------------------------------------------

SAMPLE_TOKENS = {"tiny_f32": 128, "moe_s_bf16": 1024, "skewed64_bf16": 1024,
                 "moe_l_bf16": 128, "longctx128_bf16": 64}


class OracleSample:
    """The oracle's forward + backward on the first S tokens of a workload of
    the same family (same d_model, d_ffn, E, k, distributions and logit
    shift; one dispatch chunk).  Inputs are handed to the oracle in its own
    float64 format, converted once per sample size before any timing."""

    def __init__(self, cfg, seed=0):
        import oracle
        self.oracle = oracle
        self.cfg = cfg
        self.seed = seed
        self.cores = len(os.sched_getaffinity(0))
        os.environ.setdefault("OMP_NUM_THREADS", str(self.cores))
        oracle.build()
        self._inp = {}

    def run(self, S: int) -> float:
        if S not in self._inp:
            sub = self.cfg.scaled(T=S, chunk=None)
            inp = synth.make_inputs(sub, seed=self.seed)
            self._inp = {S: {n: (None if v is None else self.oracle._f64(v))
                             for n, v in inp.items()}}
        c = self.cfg
        t0 = time.perf_counter()
        self.oracle.layer(self._inp[S], c.k, c.renorm, c.dtype == "bf16")
        return time.perf_counter() - t0


def oracle_rate(cfg, budget_s: float, max_runs: int, seed: int = 0) -> dict:
    """The oracle's rate on this workload, from timed runs on two token
    samples S_a and S_b = 2 S_a (one untimed run first).  Every oracle call
    has a fixed cost that does not depend on the tokens (allocating and
    zeroing the float64 weight gradients of all E experts: 8.6 GB at the
    long-context size), which a full-size run spreads over every token; the
    rate is therefore the marginal one, (S_b - S_a) / (t_b - t_a), with the
    fixed cost t_a - S_a (t_b - t_a) / (S_b - S_a) reported beside it.  Runs
    alternate between the two sizes until ``max_runs`` runs or ``budget_s``
    seconds."""
    smp = OracleSample(cfg, seed=seed)
    Sa = min(cfg.T, SAMPLE_TOKENS.get(cfg.name, 256))
    Sb = min(cfg.T, 2 * Sa)
    if Sb == Sa:
        Sa = max(1, Sb // 2)
    smp.run(Sa)
    ta, tb = [], []
    t0 = time.perf_counter()
    while len(ta) + len(tb) + 2 <= max(2, max_runs) and (not ta or
                                                         time.perf_counter() - t0 < budget_s):
        ta.append(smp.run(Sa))
        tb.append(smp.run(Sb))
    a, b = statistics.median(ta), statistics.median(tb)
    per_tok = (b - a) / (Sb - Sa) if b > a else b / Sb
    fixed = max(0.0, a - Sa * per_tok)
    runs = ta + tb
    return {"value": 1.0 / per_tok, "cores": smp.cores, "runs": len(runs),
            "mean_run_s": sum(runs) / len(runs), "fixed_s": fixed, "Sa": Sa, "Sb": Sb,
            "sample": (f"oracle fwd+bwd (double precision, {smp.cores} host threads) on the first "
                       f"{Sa} and {Sb} of {cfg.T} tokens of the workload (same d_model, d_ffn, E, "
                       f"k, distributions; one dispatch chunk): median {a:.2f} s and {b:.2f} s "
                       f"over {len(ta)} runs each; marginal rate {1.0 / per_tok:.4g} tokens/s "
                       f"with a fixed {fixed:.2f} s per call removed; extrapolated to the "
                       f"whole workload")}


def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wall0 = time.perf_counter()
    r = oracle_rate(cfg, budget_s=120.0, max_runs=2 * args.steps)
    wall = time.perf_counter() - wall0
    v = r["value"]
    flops_per_token = (cfg.expert_flops() + cfg.router_flops()) / cfg.T
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": r["runs"], "warmup": 1,
        "ms_per_step": r["mean_run_s"] * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "extrapolated": True, "sample_tokens": [r["Sa"], r["Sb"]], "workload_tokens": cfg.T,
        "step": "one oracle run on a token sample; steps = the timed runs (the requested "
                f"--steps {args.steps} --warmup {args.warmup} bounded by a 120 s budget)",
        "tflops": v * flops_per_token / 1e12, "wall_s": wall,
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "d_model": cfg.d,
                   "d_ffn": cfg.f, "E": cfg.E, "k": cfg.k},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": r["cores"], "kind": "oracle",
                         "sample": r["sample"]},
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


# ---- device timing of one workload ---------------------------------------------------------

CALLS = ("moe_route", "moe_permute", "moe_expert_ffn_fwd", "moe_expert_ffn_fwd_gather",
         "moe_combine_fwd", "moe_combine_bwd", "moe_expert_ffn_bwd", "moe_expert_ffn_bwd_data",
         "moe_expert_ffn_bwd_weights", "moe_expert_ffn_bwd_weights_gather", "moe_route_bwd")
GEMM_CALLS = ("moe_expert_ffn_fwd", "moe_expert_ffn_fwd_gather", "moe_expert_ffn_bwd",
              "moe_expert_ffn_bwd_data", "moe_expert_ffn_bwd_weights",
              "moe_expert_ffn_bwd_weights_gather")


class CallTimer:
    """CUDA events around the library calls that ``layer.LayerPass`` makes,
    recorded on the stream each call is launched on (the current stream at
    the call); inside a CUDA-graph capture they become graph nodes."""

    def __init__(self):
        from mixture_experts_layer_11_gb300 import ops
        self.ops = ops
        self.orig = {n: getattr(ops, n) for n in CALLS}
        self.record = False
        self.external = False
        self.marks = []          # (call, shape T, start event, end event)

    def __enter__(self):
        for n in CALLS:
            setattr(self.ops, n, self._wrap(n, self.orig[n]))
        return self

    def __exit__(self, *exc):
        for n, f in self.orig.items():
            setattr(self.ops, n, f)

    def _wrap(self, name, fn):
        def wrapper(s, *a, **kw):
            if not self.record:
                return fn(s, *a, **kw)
            e0 = torch.cuda.Event(enable_timing=True, external=self.external)
            e1 = torch.cuda.Event(enable_timing=True, external=self.external)
            e0.record()
            r = fn(s, *a, **kw)
            e1.record()
            self.marks.append((name, int(s.T), e0, e1))
            return r
        return wrapper

    def take(self):
        m, self.marks = self.marks, []
        return m


def _sum_ms(marks):
    out = {}
    for name, T, a, b in marks:
        ms, tok = out.get(name, (0.0, 0))
        out[name] = (ms + a.elapsed_time(b), tok + T)
    return out


def measure(cfg, dev, steps, warmup, *, pipeline=True, graph=True, router_tc=False,
            recompute=False, defer_wgrad=None, sampler=None, e2e=False, dist=None, seed=0,
            gather=False, gemm_units=None):
    """Times `steps` layer steps of one workload.  Returns a dict of measured
    values; with e2e also the end-to-end rate through host buffers."""
    from mixture_experts_layer_11_gb300.layer import LayerPass
    prev = os.environ.get(ROUTER_TC_ENV)
    if router_tc:
        os.environ[ROUTER_TC_ENV] = "1"
    else:
        os.environ.pop(ROUTER_TC_ENV, None)
    try:
        return _measure(cfg, dev, steps, warmup, pipeline, graph, router_tc, recompute,
                        defer_wgrad, sampler, e2e, dist, seed, LayerPass, gather, gemm_units)
    finally:
        if prev is None:
            os.environ.pop(ROUTER_TC_ENV, None)
        else:
            os.environ[ROUTER_TC_ENV] = prev


def _measure(cfg, dev, steps, warmup, pipeline, graph_on, router_tc, recompute, defer_wgrad,
             sampler, e2e, dist, seed, LayerPass, gather, gemm_units):
    torch.cuda.reset_peak_memory_stats(dev)
    inp = synth.make_inputs(cfg, seed=seed, device=str(dev))
    lp = LayerPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                   chunk=cfg.chunk, device=dev, pipeline=pipeline, recompute=recompute,
                   defer_wgrad=defer_wgrad, gather=gather, gemm_units=gemm_units)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    x_buf, dy_buf = inp["x"], inp["dy"]

    def step():
        lp.forward(x_buf, inp["Wg"], inp["W1"], inp["b1"], inp["W2"], inp["b2"], inp["beta"])
        lp.backward(dy_buf, x_buf, inp["Wg"], inp["W1"], inp["W2"])

    res = {}
    with CallTimer() as tm:
        for _ in range(warmup):
            flush.fill_(1)
            step()
        torch.cuda.synchronize()
        lp.check_status()
        graph = None
        graph_marks = []
        if graph_on:
            graph = torch.cuda.CUDAGraph()
            tm.record, tm.external = True, True
            with torch.cuda.graph(graph):
                step()
            tm.record, tm.external = False, False
            graph_marks = tm.take()
            graph.replay()
            torch.cuda.synchronize()
            lp.check_status()
        st = torch.cuda.current_stream()
        if sampler:
            sampler.start()
            time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        step_ms, calls = [], {}
        wall0 = time.perf_counter()
        for _ in range(steps):
            flush.fill_(1)
            e0, e1 = ev(), ev()
            if graph is None:
                tm.record = True
            e0.record(st)
            if graph is not None:
                graph.replay()
            else:
                step()
            e1.record(st)
            tm.record = False
            torch.cuda.synchronize()
            step_ms.append(e0.elapsed_time(e1))
            marks = graph_marks if graph is not None else tm.take()
            for name, (ms, tok) in _sum_ms(marks).items():
                a, b = calls.get(name, (0.0, 0))
                calls[name] = (a + ms, b + tok)
        wall = time.perf_counter() - wall0
        if dist:
            dist.barrier()
        if sampler:
            res["clocks"] = sampler.stop()
        lp.check_status()
    res.update(total_ms=sum(step_ms), steps=steps, wall_s=wall, chunks=len(lp.chunks),
               calls={n: (ms / steps, tok // steps) for n, (ms, tok) in calls.items()},
               device_memory_gib=torch.cuda.max_memory_allocated(dev) / 2**30,
               pipelined=lp.pipeline, defer_wgrad=lp.defer_wgrad, gather=lp.gather,
               gemm_units=lp.gemm_units,
               launches=launches_per_step(cfg, len(lp.chunks), router_tc, recompute,
                                          lp.defer_wgrad, lp.gather) * steps)
    if e2e:
        res["e2e_ms"], res["e2e_steps"] = _end_to_end(cfg, lp, inp, graph, flush, steps, warmup,
                                                      dev)
    del lp, graph, inp
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def measure_streaming(cfg, dev, steps, warmup, group, sampler=None, seed=0):
    """Times `steps` layer steps with the expert weights in pinned host memory,
    streamed one group of experts at a time (eager launches: the host copies
    run on their own stream)."""
    from mixture_experts_layer_11_gb300.streaming import ExpertStreamingPass
    torch.cuda.reset_peak_memory_stats(dev)
    inp = synth.make_inputs(cfg, seed=seed, device=str(dev))
    host = {n: inp.pop(n).cpu().pin_memory() for n in ("W1", "b1", "W2", "b2")}
    sp = ExpertStreamingPass(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.torch_dtype, cfg.renorm,
                             chunk=cfg.chunk, group=group, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        sp.forward(inp["x"], inp["Wg"], host["W1"], host["b1"], host["W2"], host["b2"],
                   inp["beta"])
        sp.backward(inp["dy"], inp["x"], inp["Wg"], host["W1"], host["W2"])

    for _ in range(warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    sp.check_status()
    st = torch.cuda.current_stream()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    ms = []
    for _ in range(steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        step()
        e1.record(st)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    clocks = sampler.stop() if sampler else None
    sp.check_status()
    esize = elem_bytes(cfg)
    wbytes = 2 * cfg.E * cfg.d * cfg.f * esize
    res = {"total_ms": sum(ms), "steps": steps, "group": group, "groups": len(sp.groups),
           "device_memory_gib": torch.cuda.max_memory_allocated(dev) / 2**30,
           "h2d_weight_bytes_per_step": 2 * wbytes + cfg.E * (cfg.d + cfg.f) * esize,
           "d2h_grad_bytes_per_step": 2 * cfg.E * cfg.d * cfg.f * 4, "clocks": clocks}
    del sp, host, inp
    torch.cuda.empty_cache()
    return res


def _end_to_end(cfg, lp, inp, graph, flush, steps, warmup, dev):
    """A training loop's input pipeline through the public API: two device
    sets of inputs (x, dy) and outputs (y, dx), one CUDA graph per set.  The
    pinned host inputs of step i+1 are copied (H2D stream) while step i
    computes; a step's y and dx are read back (D2H stream) while the next step
    computes.  Events order every reuse.  The timed span runs from the compute
    stream reaching the first timed step to the end of the last step's D2H (the
    L2 flush before every step on the compute stream included)."""
    x_buf, dy_buf = inp["x"], inp["dy"]
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
    st = torch.cuda.current_stream()
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    n = warmup + steps
    torch.cuda.synchronize()

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(cs_in):
            if i >= 2:
                cs_in.wait_event(ev_done[b])
            in_bufs[b][0].copy_(x_h, non_blocking=True)
            in_bufs[b][1].copy_(dy_h, non_blocking=True)
            ev_in[b].record(cs_in)

    h2d(0)
    for i in range(n):
        b = i % 2
        if i == warmup:
            t_start.record(st)
        st.wait_event(ev_in[b])
        if i >= 2:
            st.wait_event(ev_read[b])
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
    last = (n - 1) % 2
    if not torch.equal(out_h[last][0], out_bufs[last][0].cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident step")
    lp.y, lp.dx = out_bufs[0]
    return e2e_ms, steps


def summarize(cfg, res, pk):
    """Per-workload figures: rate, layer TFLOP/s, the grouped GEMM's fraction
    of the bf16 tensor peak, and the dispatch kernels' fraction of HBM."""
    steps = res["steps"]
    ms = res["total_ms"] / steps
    out = {"tokens_per_s": cfg.T / (ms / 1e3), "ms_per_step": ms,
           "tflops": (cfg.expert_flops() + cfg.router_flops()) / (ms / 1e3) / 1e12,
           "device_memory_gib": res["device_memory_gib"]}
    calls = res["calls"]
    gemm_ms = sum(calls.get(n, (0.0, 0))[0] for n in GEMM_CALLS)
    if gemm_ms > 0:
        ach = cfg.expert_flops() / (gemm_ms / 1e3) / 1e12
        out["gemm"] = {"ms_per_step": gemm_ms, "tflops": ach,
                       "frac_of_bf16_burst": ach / pk["bf16_tflops"] if cfg.dtype == "bf16" else None}
    out["calls_ms_per_step"] = {n: v[0] for n, v in calls.items()}
    return out


def dispatch_roofline(cfg, res, pk):
    """HBM fraction of the dispatch kernels (A4 permute, A6 combine, A7
    combine backward) from a one-stream pass: algorithmic bytes over the
    CUDA-event time of each call; the permute backward + router backward
    (A9 + A10) is given beside it."""
    calls = res["calls"]
    kinds = {"moe_permute": "permute", "moe_combine_fwd": "combine",
             "moe_combine_bwd": "combine_bwd", "moe_route_bwd": "route_bwd"}
    per = {}
    for n, kind in kinds.items():
        if n not in calls:
            continue
        ms, T = calls[n]
        byt = dispatch_bytes(cfg, kind, T)
        per[kind] = {"ms_per_step": ms, "bytes_per_step": byt,
                     "gbs": byt / (ms / 1e3) / 1e9, "frac": byt / (ms / 1e3) / 1e9 / pk["hbm_gbs"]}
    if "moe_route" in calls:
        ms, T = calls["moe_route"]
        fl = 2.0 * T * cfg.d * cfg.E
        per["route"] = {"ms_per_step": ms, "logits_flops_per_step": fl,
                        "tflops": fl / (ms / 1e3) / 1e12,
                        "note": "router logits (CUDA cores), gate, histogram, scan, rank"}
    names = [k for k in ("permute", "combine", "combine_bwd") if k in per]
    main = [per[k] for k in names]
    byt = sum(p["bytes_per_step"] for p in main)
    ms = sum(p["ms_per_step"] for p in main)
    ach = byt / (ms / 1e3) / 1e9 if ms > 0 else None
    label = {"permute": "permute (A4)", "combine": "combine (A6)",
             "combine_bwd": "combine backward (A7)"}
    kernels = ", ".join(label[k] for k in names)
    if "permute" not in per:
        kernels += "; the permute (A4) is fused into the expert GEMMs' operand loads"
    return {"bound": "hbm", "kernels": kernels,
            "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"] if ach else None,
            "algorithmic_bytes_per_step": byt, "ms_per_step": ms,
            "timing": "one-stream pass (no chunk pipelining), CUDA events around each call, "
                      "L2 flushed between steps",
            "per_kernel": per}


# ---- our arm -----------------------------------------------------------------------------

def run_ours(args, cfg):
    from mixture_experts_layer_11_gb300 import ops

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
    pk, pk_kind = peaks()

    if args.weights_on_host:
        return run_streaming(args, cfg, dev, rank, world, dist)
    # ---- the headline: the default router (CUDA cores), two-stream chunk
    # pipelining, one CUDA graph per step; clocks sampled over the timed steps
    sampler = ClockSampler(local)
    main = measure(cfg, dev, args.steps, args.warmup, sampler=sampler, e2e=True, dist=dist,
                   seed=rank, graph=not args.no_graph, recompute=args.recompute,
                   gemm_units=args.gemm_units,
                   defer_wgrad=False if args.per_chunk_wgrad else None)
    total_ms, e2e_ms = max_over_ranks([main["total_ms"], main["e2e_ms"]], dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0
    head = summarize(cfg, main, pk)
    sub_steps, sub_warm = min(args.steps, 10), 3
    # ---- the same workload with the router logits on the tensor cores (opt-in)
    tc = None
    if cfg.dtype == "bf16" and cfg.d % 64 == 0 and not args.no_sub_configs:
        r = measure(cfg, dev, sub_steps, sub_warm, router_tc=True)
        tc = summarize(cfg, r, pk)
        tc = {"tokens_per_s": tc["tokens_per_s"], "ms_per_step": tc["ms_per_step"],
              "route_ms_per_step": tc["calls_ms_per_step"].get("moe_route"),
              "note": "router logits as one segment of the tcgen05 grouped GEMM "
                      f"({ROUTER_TC_ENV}=1); not the default: the tensor cores are reserved "
                      "for the expert GEMMs"}
    # ---- the same workload with the permute fused into the GEMMs' loads (opt-in)
    fused = None
    if cfg.dtype == "bf16" and not args.no_sub_configs:
        r = summarize(cfg, measure(cfg, dev, sub_steps, sub_warm, gather=True), pk)
        c = r["calls_ms_per_step"]
        fused = {"tokens_per_s": r["tokens_per_s"], "ms_per_step": r["ms_per_step"],
                 "expert_ffn_fwd_ms_per_step": c.get("moe_expert_ffn_fwd_gather"),
                 "expert_ffn_bwd_weights_ms_per_step": c.get("moe_expert_ffn_bwd_weights_gather"),
                 "device_memory_gib": r["device_memory_gib"],
                 "note": "no moe_permute and no X_perm: the first expert GEMM and the dW1 GEMM "
                         "load x rows through the dispatch's perm (TMA tile::gather4); not the "
                         "default"}
    # ---- every call timed on one stream (the dispatch kernels' HBM fraction)
    serial = measure(cfg, dev, sub_steps, sub_warm, pipeline=False,
                     defer_wgrad=False if args.per_chunk_wgrad else None)
    disp = dispatch_roofline(cfg, serial, pk)
    serial_gemm = summarize(cfg, serial, pk).get("gemm", {})
    disp["serial_step_ms"] = serial["total_ms"] / serial["steps"]
    disp["serial_calls_ms_per_step"] = {n: v[0] for n, v in serial["calls"].items()}
    # ---- the other workloads
    per_config = {}
    if not args.no_sub_configs:
        for name, c in synth.CONFIGS.items():
            if name == cfg.name:
                continue
            r = summarize(c, measure(c, dev, sub_steps, sub_warm), pk)
            d = dispatch_roofline(c, measure(c, dev, sub_steps, sub_warm, pipeline=False), pk)
            per_config[name] = {
                "workload": workload_desc(c), "tokens_per_s": r["tokens_per_s"],
                "ms_per_step": r["ms_per_step"], "tflops": r["tflops"],
                "gemm_tflops": r.get("gemm", {}).get("tflops"),
                "gemm_frac_of_bf16_burst": r.get("gemm", {}).get("frac_of_bf16_burst"),
                "dispatch_gbs": d["achieved"], "dispatch_frac_of_hbm": d["frac"],
                "steps": sub_steps}

    traffic, traffic_note = gemm_traffic(cfg)
    value = whole_job_rate(cfg.T, args.steps, world, total_ms)
    flops = cfg.expert_flops() + cfg.router_flops()
    gemm = head.get("gemm", {})
    achieved = gemm.get("tflops")
    peak = pk["bf16_tflops"]
    elem = elem_bytes(cfg)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic (seeded N(0,1) inputs, N(0,1/fan_in) weights)",
        "tflops": flops * args.steps * world / (total_ms / 1e3) / 1e12,
        "device_memory_gib": main["device_memory_gib"],
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "d_model": cfg.d,
                   "d_ffn": cfg.f, "E": cfg.E, "k": cfg.k,
                   "router": "CUDA cores (fp32 FMA); tensor cores only for the expert GEMMs",
                   "l2": "flushed between steps (256 MiB write, outside the step timing)",
                   "launch": "eager" if args.no_graph else "one CUDA graph per step",
                   "chunks": (f"{main['chunks']}, pipelined on two streams, per-chunk expert "
                              f"GEMMs on {main['gemm_units'] or 'all'} CTA pairs"
                              if main["pipelined"] else f"{main['chunks']}, one stream"),
                   "activations": ("recomputed in the backward (routing kept)" if args.recompute
                                   else "kept from the forward for the backward"),
                   "weight_gradients": ("one pass over all chunks after the backward"
                                        if main["defer_wgrad"] else "accumulated per chunk"),
                   "permute": ("fused into the expert GEMMs' operand loads (TMA tile::gather4 "
                               "of x rows through the dispatch's perm; no X_perm)"
                               if main["gather"] else "its own kernel (X_perm written, read by "
                               "the expert GEMMs)"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {
            "bound": "tensor", "kernel": "grouped expert GEMM (tcgen05), all expert FFN calls",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak if achieved else None,
            "peak_kind": f"bf16 dense cuBLAS burst ({pk_kind}): each step lasts well under 1 s",
            "traffic": traffic,
            "traffic_note": traffic_note,
            "algorithmic_flops_per_step": cfg.expert_flops(),
            "gemm_ms_per_step": gemm.get("ms_per_step"),
            "timing": ("CUDA events around the expert GEMM calls of the timed (pipelined) steps; "
                       "there they share the GPU with the side stream's dispatch kernels"),
            "one_stream": {"achieved": serial_gemm.get("tflops"),
                           "frac": (serial_gemm["tflops"] / peak
                                    if serial_gemm.get("tflops") else None),
                           "gemm_ms_per_step": serial_gemm.get("ms_per_step"),
                           "timing": "the same calls in a one-stream pass (nothing beside them)"},
        },
        "dispatch_roofline": disp,
        "router_tensor_cores_variant": tc,
        "fused_permute_variant": fused,
        "per_config": per_config,
        "gpu_launches": main["launches"],
        "gpu_launches_source": ("launches_per_step() x steps; the formula matched the library "
                                "kernels of a profiled step on moe_s_bf16 (16) and on the "
                                "long-context workload (132)"),
        "e2e": {"value": whole_job_rate(cfg.T, main["e2e_steps"], world, e2e_ms),
                "unit": "tokens/s",
                "pipeline": "H2D of step i+1 and D2H of step i on copy streams, overlapping step i",
                "h2d_bytes_per_step": 2 * cfg.T * cfg.d * elem,
                "d2h_bytes_per_step": 2 * cfg.T * cfg.d * elem},
        "calls_ms_per_step": head["calls_ms_per_step"],
        "wall_s_timed_region": main["wall_s"],
        "clocks": main.get("clocks"),
    }
    if not args.no_cpu_baseline:
        r = oracle_rate(cfg, budget_s=20.0, max_runs=4)
        line["cpu_baseline"] = {"value": r["value"], "unit": "tokens/s", "cores": r["cores"],
                                "kind": "oracle", "sample": r["sample"]}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def run_streaming(args, cfg, dev, rank, world, dist):
    """--weights-on-host: the step with the expert weights streamed from host
    memory.  Prints one JSON line like the default mode (no per-workload table,
    no end-to-end leg: the weights already cross the host link every step)."""
    pk, pk_kind = peaks()
    sampler = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    r = measure_streaming(cfg, dev, args.steps, args.warmup, args.group, sampler=sampler,
                          seed=rank)
    total_ms, = max_over_ranks([r["total_ms"]], dist, dev)
    if rank != 0:
        return 0
    ms = total_ms / args.steps
    line = {
        "metric": METRIC, "value": whole_job_rate(cfg.T, args.steps, world, total_ms),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.dtype, "data": "synthetic (seeded N(0,1) inputs, N(0,1/fan_in) weights)",
        "tflops": (cfg.expert_flops() + cfg.router_flops()) / (ms / 1e3) / 1e12,
        "config": {"workload": workload_desc(cfg), "T": cfg.T, "d_model": cfg.d,
                   "d_ffn": cfg.f, "E": cfg.E, "k": cfg.k,
                   "weights": f"pinned host memory, streamed in groups of {args.group} experts "
                              f"({r['groups']} groups) per pass, fp32 weight gradients read back",
                   "launch": "eager", "parallelism": f"replicas x{world}"},
        "streaming": {k: r[k] for k in ("h2d_weight_bytes_per_step", "d2h_grad_bytes_per_step",
                                         "device_memory_gib", "groups")},
        "link_gbs_needed": (r["h2d_weight_bytes_per_step"] + r["d2h_grad_bytes_per_step"])
        / (ms / 1e3) / 1e9,
        "clocks": r["clocks"],
    }
    print(json.dumps(line), flush=True)
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
    ap.add_argument("--per-chunk-wgrad", action="store_true",
                    help="accumulate the weight gradients chunk by chunk instead of one pass "
                         "over all chunks after the backward")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels one by one instead of as one CUDA graph")
    ap.add_argument("--weights-on-host", action="store_true",
                    help="keep the expert weights in pinned host memory and stream them to "
                         "the GPU one group of experts at a time")
    ap.add_argument("--group", type=int, default=16,
                    help="experts per streamed group (--weights-on-host)")
    ap.add_argument("--gemm-units", type=int, default=None,
                    help="CTA pairs of the per-chunk expert GEMMs when chunks are pipelined "
                         "(default: the layer's choice; 0 = every pair)")
    ap.add_argument("--no-sub-configs", action="store_true",
                    help="time only the chosen workload (no per-workload table, no router "
                         "variant)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
