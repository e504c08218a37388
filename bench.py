#!/usr/bin/env python3
"""Throughput of the MXFP4 routed MoE block on GB300.

One step = one pass of the whole block (norm + router + top-k + softmax,
permutation, MXFP4 gate/up + SwiGLU, MXFP4 down, weighted combine + residual)
over one batch of the workload.  The headline workload is the largest
single-GPU one: the 24-layer stack of independently seeded gpt-oss MoE blocks
(hidden 2880, 32 experts, top-4, expert_hidden 2880, ~10 GB of MXFP4 expert
weights resident) decoding 16 tokens, each layer's output rounded to bf16 as
the next layer's input (written so by the layer itself, the "out_bf16" plan
option).  In the same run every other workload is measured too
(1-token decode, the 8-token hot-2 batch, the stack at 1 and 4 tokens, prefill
at 128 and 512 tokens, the DeepSeek-V4-Flash-shaped block at 1 and 2048
tokens) and reported under "configs", each with its own rate, roofline and
clock record.

Weights: router, gamma and router bias are drawn exactly as the seeded recipe
does on the host (they decide the routing, including the hot-2 and Zipf
skews); the expert matrices, gigabytes of them, are drawn on the device from
the same distributions.  Single-block workloads rotate over weight sets whose
touched experts together exceed twice the 129 MB L2, so no step finds its
weights in L2; the stack is itself ~10 GB.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the headline workload instead.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE block tokens/s; decode HBM GB/s and prefill TFLOP/s vs GB300 peak"
HEADLINE = (2, 16)           # (workload, tokens): the 24-layer stack decoding 16 tokens
# (workload, tokens, plan options): the FP4 rows run the same workloads on the
# block-scaled FP4 tensor-core path (activations FP4-encoded; its own oracle mode)
EXTRAS = [(0, 1, {}), (1, 8, {}), (2, 1, {}), (2, 4, {}), (3, 128, {}), (3, 512, {}), (4, 1, {}), (4, 2048, {}),
          (3, 128, {"act_fp4": 1}), (3, 512, {"act_fp4": 1}), (4, 2048, {"act_fp4": 1})]
KERNEL_SLOTS = ["route_permute", "gateup_swiglu", "down_weighted", "combine_residual"]
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=HEADLINE[0],
                    help="workload id of synth.WORKLOADS for the headline (default: the 24-layer stack)")
    ap.add_argument("--tokens", type=int, default=0, help="tokens per step (default: 16 for the stack, "
                                                          "else the workload's largest)")
    ap.add_argument("--no-extras", action="store_true", help="measure the headline workload only")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers of the stack workload (default: all 24); fewer only to keep an ncu capture small")
    ap.add_argument("--act-fp4", action="store_true",
                    help="run the headline workload on the block-scaled FP4 tensor-core path")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="timed region of the headline only (no clock pre-roll, kernel timing, e2e, CPU "
                         "baseline or extras); for ncu")
    ap.add_argument("--op", default="block", choices=["block", "mx_fp4_quantize", "attention", "attention_prefill", "expert_cache"],
                    help="block: the MoE block (the benchmark); mx_fp4_quantize: the FP4 activation "
                         "encoder alone, on --rows x --cols bf16 activations; attention: the gpt-oss "
                         "attention decode step alone; attention_prefill: its prefill of one 512-token prompt")
    ap.add_argument("--rows", type=int, default=14336, help="mx_fp4_quantize: rows (2048 tokens x 7 routes)")
    ap.add_argument("--cols", type=int, default=2048, help="mx_fp4_quantize: columns (expert_hidden)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def traffic_record(kernel: str, workload: str = "", tokens: int = 0, path: int = 0):
    """ncu DRAM bytes per launch of `kernel`, if taken on the current source, on
    this workload, token count and projection path."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    recs = json.load(open(p)).get(kernel) or []
    for rec in recs if isinstance(recs, list) else [recs]:
        src = os.path.join(ROOT, rec["source"])
        if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != rec["sha256"]:
            continue
        if rec.get("workload", workload) != workload or rec.get("tokens", tokens) != tokens:
            continue
        if path and rec.get("path", path) != path:
            continue
        return rec
    return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.p.terminate()
        self.p.wait()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_config(wl, tokens):
    """The `config` object of a line: what the workload is, from its shape."""
    sh = wl.shape
    return {"workload": wl.name, "tokens_per_step": tokens, "layers": wl.layers, "hidden": sh.hidden,
            "n_experts": sh.n_experts, "top_k": sh.top_k, "expert_hidden": sh.expert_hidden,
            "n_shared_experts": sh.n_shared, "weight_scale": sh.weight_scale, "swiglu_limit": sh.swiglu_limit,
            "routing": wl.router_skew, "weights": "mxfp4 (e2m1 + e8m0/32)"}


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world, wid, T):
    """The oracle, as it stands, on the host cores: each step one bounded sample
    of the step's tokens through the whole workload (every layer of the stack),
    sized so that the whole run takes a few minutes."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from mxfp4_mixture_experts_rms_gb300 import synth
    cores = os.cpu_count() or 1
    wl = synth.WORKLOADS[wid]
    shape = wl.shape
    n_steps = args.warmup + args.steps
    blk = synth.make_block(wid, layer=0)
    x = synth.make_tokens(wid, T, shape.hidden)
    oracle.moe_forward(blk, x[:1], nthreads=1)  # warm the library
    t0 = time.perf_counter()
    oracle.moe_forward(blk, x[:1], nthreads=1)
    t_tok = (time.perf_counter() - t0) * wl.layers   # one token through every layer
    budget = 150.0
    per_step = max(1, min(T, cores, int(budget * cores / max(1e-9, n_steps * t_tok))))
    # each step's sample: per_step consecutive tokens of the batch, rotating
    xs = [np.ascontiguousarray(np.roll(x, -(i * per_step) % T, axis=0)[:per_step]) for i in range(n_steps)]
    el = 0.0
    for layer in range(wl.layers):
        if layer:
            del blk
            blk = synth.make_block(wid, layer=layer)          # weight generation off the clock
        for i in range(n_steps):
            t0 = time.perf_counter()
            out = oracle.moe_forward(blk, xs[i], nthreads=per_step)["out"]
            if i >= args.warmup:
                el += time.perf_counter() - t0
            if layer + 1 < wl.layers:
                xs[i] = synth.f32_to_bf16_bits(out)
    value = per_step * args.steps / el
    sample = (f"{per_step} of the {T} tokens of each step through all {wl.layers} layer(s), "
              f"{per_step} threads, weight generation off the clock")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(wl, T),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": per_step, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def max_over_ranks(x: float) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's);
    x itself when there is no process group or a single rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens: int, steps: int, ms: float) -> float:
    """Tokens per second of the whole job: every rank processes `tokens` per step
    (weak scaling), the job takes the slowest rank's `ms` for `steps` steps."""
    return world * tokens * steps / (ms / 1e3)


def algorithmic_bytes(shape, counts, T, fp4=False):
    """Bytes the gate/up and down kernels must move at least once per launch
    (fp4: activations as FP4 codes + E8M0 scales, 17/32 bytes an element)."""
    H, F = shape.hidden, shape.expert_hidden
    distinct = int((counts > 0).sum()) + shape.n_shared
    routes = int(counts.sum()) + shape.n_shared * T
    mat = F * H // 2 + F * H // 32
    act = 17 / 32 if fp4 else 2
    gateup = distinct * (2 * mat + 2 * F * 4) + (routes if fp4 else T) * H * act + routes * F * act
    down = distinct * (mat + H * 4) + routes * F * act + routes * H * 4
    return gateup, down, distinct


def launches_per_forward(path: int, T: int) -> int:
    """Kernels one forward launches: routing (one kernel up to 32 tokens; above,
    norm, logits GEMM, top-k and the permutation), the x_hat gather (grouped-GEMM
    paths), gate/up, down, combine."""
    return (1 if T <= 32 else 4) + (1 if path in (2, 3) else 0) + 3


def n_weight_sets(wid, T):
    """Weight sets a single-block workload rotates over so that the experts
    touched between two uses of a set exceed 2.5 x L2."""
    from mxfp4_mixture_experts_rms_gb300 import synth
    wl = synth.WORKLOADS[wid]
    sh = wl.shape
    touched = (synth.distinct_uniform(sh.n_experts, sh.top_k, T) + sh.n_shared) * synth.expert_bytes(sh)
    return max(2, min(8, 1 + math.ceil(2.5 * L2_BYTES / touched)))


class Pool:
    """Device weight sets shared by every workload of one shape (drawn once)."""

    def __init__(self):
        self.sets = {}

    def experts(self, shape, i):
        from mxfp4_mixture_experts_rms_gb300 import synth
        key = (shape, i)
        if key not in self.sets:
            seed = 0x4D6F45 + 1009 * i + (0 if shape == synth.GPT_OSS else 500009)
            d = synth.expert_matrices_device(shape, shape.n_experts, seed)
            if shape.n_shared:
                d["shared"] = synth.expert_matrices_device(shape, 1, seed + 7919)
            self.sets[key] = d
        return self.sets[key]


class Workload:
    """Plans, inputs and buffers of one (workload, tokens) measurement."""

    def __init__(self, wid, T, pool, rank, opts=None, layers=0):
        import numpy as np
        import torch

        from mxfp4_mixture_experts_rms_gb300 import moe, synth
        self.wid, self.T = wid, T
        self.opts = dict(opts or {})
        self.wl = wl = synth.WORKLOADS[wid]
        self.shape = sh = wl.shape
        H, K = sh.hidden, sh.top_k
        self.layers = min(layers, wl.layers) if layers else wl.layers
        n_sets = 1 if wl.layers > 1 else n_weight_sets(wid, T)
        self.sets = []
        for s in range(n_sets):
            chain = []
            for layer in range(self.layers):
                li = layer if wl.layers > 1 else s
                blk = synth.make_router(wid, layer=li + 100 * rank)
                ex = pool.experts(sh, li + 30 * rank)
                blk.update({k: ex[k] for k in ("codes", "scales", "bias")})
                if sh.n_shared:
                    blk["shared"] = ex["shared"]
                # every layer but the last writes its output as the next layer's bf16 input
                last = layer == self.layers - 1
                plan = moe.Plan(sh, max_tokens=T, **self.opts, **({} if last else {"out_bf16": 1}))
                plan.alloc_workspace().load_weights(moe.DeviceBlock(blk))
                chain.append(dict(plan=plan, x=torch.empty((T, H), dtype=torch.int16, device="cuda"),
                                  out=torch.empty((T, H), dtype=torch.float32, device="cuda") if last else None,
                                  ids=torch.empty((T, K), dtype=torch.int32, device="cuda")))
            xb = synth.make_tokens(wid, T, H, layer=s + 100 * rank)
            chain[0]["x"].copy_(torch.from_numpy(xb.view(np.int16)))
            self.sets.append(dict(chain=chain, xb=xb))
        self.path = self.sets[0]["chain"][0]["plan"].path_for(T)

    def plans(self, d):
        return [ly["plan"] for ly in d["chain"]]

    def forward_set(self, d, stream):
        ls = d["chain"]
        for i, ly in enumerate(ls):
            out = ly["out"] if i + 1 == len(ls) else ls[i + 1]["x"]
            ly["plan"].forward(ly["x"], out, ly["ids"], stream=stream)

    def step(self, i, stream):
        self.forward_set(self.sets[i % len(self.sets)], stream)

    def capture(self, n):
        """One CUDA graph holding n consecutive steps (launch overhead off the clock)."""
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for i in range(n):
                self.step(i, cs)
        return g

    def close(self):
        for d in self.sets:
            for p in self.plans(d):
                p.close()
        self.sets = []


def measure(w, args, world, local, preroll_s):
    """Time exactly args.steps steps (one graph replay) between barriers and
    device synchronisations, then the same steps again with per-kernel events;
    returns the numbers of one line."""
    import torch
    st = torch.cuda.current_stream()
    sh, T = w.shape, w.T
    facts = []
    for i, d in enumerate(w.sets):
        w.forward_set(d, st)
        tot_f = [0, 0, 0]
        for p in w.plans(d):
            c = torch.empty(sh.n_experts, dtype=torch.int32, device="cuda")
            p.expert_counts(c)
            torch.cuda.synchronize()
            tot_f = [a + b for a, b in zip(tot_f, algorithmic_bytes(sh, c.cpu().numpy(), T, w.path == 3))]
        facts.append(tuple(tot_f))
        for p in w.plans(d):
            assert p.device_status() == 0
    for i in range(args.warmup):
        w.step(i, st)
    torch.cuda.synchronize()
    graph = w.capture(args.steps)
    graph.replay()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    t_end = time.perf_counter() + preroll_s
    while time.perf_counter() < t_end:      # clock samples see this load before and during the timed region
        graph.replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(st)
    graph.replay()
    ev1.record(st)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    ms = max_over_ranks(ms)
    del graph
    r = {"ms": ms, "clocks": clk, "facts": facts}
    if args.quick:
        return r
    # kernel durations over the same K steps: CUDA events the library records
    # around each launch on the launching stream (event nodes in the graph)
    for d in w.sets:
        for p in w.plans(d):
            p.set_i("profile", 1)
    pgraph = w.capture(args.steps)
    torch.cuda.synchronize()
    # the events keep their last recording: time the second replay (the first
    # launch of a graph also uploads it)
    pgraph.replay()
    torch.cuda.synchronize()
    pgraph.replay()
    torch.cuda.synchronize()
    tot, cnt = [0.0] * 4, [0] * 4
    for d in w.sets:
        for p in w.plans(d):
            m, c = p.profile_read()
            tot = [a + b for a, b in zip(tot, m)]
            cnt = [a + b for a, b in zip(cnt, c)]
            p.set_i("profile", 0)
    del pgraph
    r.update(tot=tot, cnt=cnt)
    return r


# fp32 FMA peak of the SIMT router: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz
# (the GB300's SM count and maximum SM clock)
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
# dense FP4 tensor peak taken as the measured bf16 peak x the nominal ratio (13.5 / 2.25)
FP4_OVER_BF16 = 13.5 / 2.25


def roofline(path, dom, avg_ms, achieved_gbs, hbm, bf16_peak, peak_kind, tr, dom_bytes, routes, H, F, router_macs):
    """Roofline of the dominant kernel: HBM for the GEMVs (decode path), the
    bf16 tensor peak for the grouped GEMMs (prefill path), the fp32 FMA peak
    when the SIMT routing kernel dominates a prefill step."""
    if path == 3 and dom in (1, 2):
        # the block-scaled FP4 GEMMs: far below the FP4 ridge (~1700 flop/B), so HBM binds
        flops = 2.0 * routes * (2 * F if dom == 1 else F) * H
        tf = flops / (avg_ms / 1e3) / 1e12 if avg_ms > 0 else 0.0
        fp4_peak = bf16_peak * FP4_OVER_BF16
        return {"bound": "hbm", "kernel": KERNEL_SLOTS[dom], "achieved": achieved_gbs, "peak": hbm,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved_gbs / hbm,
                "traffic": tr["bytes_per_launch"] if tr else None, "algorithmic_bytes_per_launch": dom_bytes,
                "avg_launch_ms": avg_ms, "tensor_tflops": tf, "fp4_peak_tflops": fp4_peak,
                "fp4_peak_kind": peak_kind + " bf16 x nominal fp4/bf16 ratio 6", "tensor_frac_of_fp4_peak": tf / fp4_peak}
    if path == 2 and dom in (1, 2):
        flops = 2.0 * routes * (2 * F if dom == 1 else F) * H
        ach = flops / (avg_ms / 1e3) / 1e12 if avg_ms > 0 else 0.0
        return {"bound": "tensor", "kernel": KERNEL_SLOTS[dom], "achieved": ach, "peak": bf16_peak,
                "peak_kind": peak_kind + " bf16 (burst)", "unit": "TFLOP/s", "frac": ach / bf16_peak,
                "traffic": tr["bytes_per_launch"] if tr else None,
                "algorithmic_flops_per_launch": flops, "avg_launch_ms": avg_ms,
                "hbm_frac_of_algorithmic_bytes": (dom_bytes / (avg_ms / 1e3) / 1e9 / hbm) if avg_ms > 0 else 0.0}
    if path in (2, 3) and dom == 0:
        flops = 2.0 * router_macs
        ach = flops / (avg_ms / 1e3) / 1e12 if avg_ms > 0 else 0.0
        return {"bound": "alu", "kernel": KERNEL_SLOTS[dom], "achieved": ach, "peak": ALU_FP32_TFLOPS,
                "peak_kind": "derived (SM count x fp32 lanes x 2 x max SM clock)", "unit": "TFLOP/s",
                "frac": ach / ALU_FP32_TFLOPS, "traffic": None, "algorithmic_flops_per_launch": flops,
                "avg_launch_ms": avg_ms}
    return {"bound": "hbm", "kernel": KERNEL_SLOTS[dom], "achieved": achieved_gbs, "peak": hbm,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved_gbs / hbm,
            "traffic": tr["bytes_per_launch"] if tr else None,
            "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": avg_ms}


def summarise(w, r, args, world):
    """value, roofline, kernels and step figures of one measurement."""
    sh, T = w.shape, w.T
    H, F, K = sh.hidden, sh.expert_hidden, sh.top_k
    steps = args.steps
    ms = r["ms"]
    n_blocks = w.layers
    facts = r["facts"]
    gu_bytes = sum(facts[i % len(facts)][0] for i in range(steps)) / steps / n_blocks
    dn_bytes = sum(facts[i % len(facts)][1] for i in range(steps)) / steps / n_blocks
    distinct = sum(facts[i % len(facts)][2] for i in range(steps)) / steps / n_blocks
    step_bytes = (gu_bytes + dn_bytes) * n_blocks
    step_s = ms / steps / 1e3
    routes = T * (K + sh.n_shared)
    step_flops = 6.0 * routes * H * F * n_blocks
    hbm, bf16_peak, peak_kind = peaks()
    out = {"value": whole_job_rate(world, T, steps, ms), "unit": "tokens/s", "ms_per_step": ms / steps,
           "path": {1: "gemv", 2: "grouped_gemm", 3: "fp4_grouped_gemm"}[w.path],
           "distinct_experts_per_block": distinct, "algorithmic_bytes_per_step": step_bytes,
           "step_hbm_gbs": step_bytes / step_s / 1e9, "step_frac_of_hbm": step_bytes / step_s / 1e9 / hbm,
           "algorithmic_flops_per_step": step_flops, "step_tflops": step_flops / step_s / 1e12,
           "step_frac_of_bf16_peak": step_flops / step_s / 1e12 / bf16_peak,
           "binding_roof_frac": max(step_bytes / (hbm * 1e9), step_flops / (bf16_peak * 1e12)) / step_s,
           "clocks": r["clocks"],
           "gpu_launches": launches_per_forward(w.path, T) * n_blocks * steps}
    if "tot" in r:
        tot, cnt = r["tot"], r["cnt"]
        avg_ms = [t / c if c else 0.0 for t, c in zip(tot, cnt)]
        share = [t / sum(tot) for t in tot] if sum(tot) > 0 else [0.0] * 4
        dom = max(range(4), key=lambda k: tot[k])
        dom_bytes = {1: gu_bytes, 2: dn_bytes}.get(dom, gu_bytes)
        achieved = dom_bytes / (avg_ms[dom] / 1e3) / 1e9 if avg_ms[dom] > 0 else 0.0
        tr = traffic_record(KERNEL_SLOTS[dom], w.wl.name, T, w.path)
        out["roofline"] = roofline(w.path, dom, avg_ms[dom], achieved, hbm, bf16_peak, peak_kind, tr, dom_bytes,
                                   routes, H, F, T * sh.n_experts * H)
        out["kernels"] = {KERNEL_SLOTS[k]: {"avg_us": 1e3 * avg_ms[k], "share": share[k], "launches": cnt[k]}
                          for k in range(4)}
    return out


def e2e_rate(w, args, world):
    """The same metric through the public API with host buffers: every step
    copies its inputs from pinned host memory and reads the outputs back."""
    import torch
    st = torch.cuda.current_stream()
    T, H, K = w.T, w.shape.hidden, w.shape.top_k
    hx = [d["chain"][0]["x"].cpu().pin_memory() for d in w.sets]
    hout = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in w.sets]
    hids = [torch.empty((T, K), dtype=torch.int32).pin_memory() for _ in w.sets]

    def e2e_step(i):
        j = i % len(w.sets)
        d = w.sets[j]
        d["chain"][0]["x"].copy_(hx[j], non_blocking=True)
        w.forward_set(d, st)
        hout[j].copy_(d["chain"][-1]["out"], non_blocking=True)
        hids[j].copy_(d["chain"][-1]["ids"], non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(st)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1))
    return {"value": whole_job_rate(world, T, args.steps, e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4 + T * K * 4}


def attention_bench(args, seqs: int = 16, ctx: int = 4096):
    """The attention half of the gpt-oss layer (moe_attn_decode), decode step:
    `seqs` sequences with ctx - 1 cached tokens each, one sliding-window layer
    (128 tokens) and one full-attention layer as in gpt-oss's alternation.
    Timed in a CUDA graph of the two steps; the roofline is HBM: both layers'
    projection weights once, the visible keys and values, activations."""
    import numpy as np
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe, synth
    A = synth.ATTN_GPT_OSS
    H, QH, KVH, D, window = A["hidden"], A["q_heads"], A["kv_heads"], A["head_dim"], A["window"]
    plans = []
    for layer, win in enumerate((window, 0)):
        w = synth.make_attention(200 + layer, H, QH, KVH)
        p = moe.AttnPlan(H, QH, KVH, seqs, ctx, sliding_window=win)
        p.load_weights({k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
                        for k, v in w.items()})
        kh, vh = synth.make_kv_history(200 + layer, seqs, ctx, KVH)
        p.k_cache.copy_(torch.from_numpy(kh))
        p.v_cache.copy_(torch.from_numpy(vh))
        plans.append(p)
    x = torch.from_numpy(synth.f32_to_bf16_bits(np.random.default_rng(0).normal(0, 1, (seqs, H))).view(np.int16)).cuda()
    pos = torch.full((seqs,), ctx - 1, dtype=torch.int32, device="cuda")
    out = torch.empty((seqs, H), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        for p in plans:
            p.decode(x, pos, out, stream=st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    reps = max(1, min(args.steps, 100))
    with torch.cuda.graph(g):
        for _ in range(reps):
            for p in plans:
                p.decode(x, pos, out, stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / reps
    weights = 2 * ((QH * D + 2 * KVH * D) * H * 2 + H * QH * D * 2 + 4 * (QH * D + 2 * KVH * D + 2 * H + QH))
    kv = seqs * (min(ctx, window) + ctx) * KVH * D * 2 * 2
    act = 2 * seqs * (H * 2 + H * 4 + 2 * KVH * D * 2)
    hbm, _, kind = peaks()
    gbs = (weights + kv + act) / (ms / 1e3) / 1e9
    for p in plans:
        p.close()
    del g
    return {"value": seqs / (ms / 1e3), "unit": "tokens/s (one sliding + one full attention layer)",
            "ms_per_step": ms, "path": "attention decode",
            "config": {"workload": f"gpt-oss attention decode, {seqs} sequences x {ctx - 1} cached tokens, "
                                   "one sliding-window (128) and one full layer",
                       "hidden": H, "q_heads": QH, "kv_heads": KVH, "head_dim": D, "weights": "bf16 (synthetic)",
                       "kv_cache": "fp16"},
            "algorithmic_bytes_per_step": weights + kv + act,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "peak_kind": kind, "unit": "GB/s",
                         "frac": gbs / hbm, "traffic": None},
            "clocks": clk, "gpu_launches": 2 * 5 * reps}


def expert_cache_bench(args, T: int = 4, slots: int = 16, n_sets: int = 64):
    """The gpt-oss block decoding T tokens with its expert matrices in pinned
    host memory behind a `slots`-slot device cache (plan option
    expert_cache_slots): the step with every routed expert resident (the same
    tokens each step: all hits after the first), and with fresh tokens each
    step (cycling over n_sets token sets: misses copied from host memory),
    beside the same block with its weights resident in HBM.  Each regime is
    timed in a CUDA graph; the hit rate and the misses come from the cache's
    own counters over the timed replay."""
    import numpy as np
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe, synth
    wid = 0
    blk = synth.make_block(wid)
    shape = blk["shape"]
    H, F = shape.hidden, shape.expert_hidden
    per_expert = 2 * F * (H // 2 + H // 32 + 4) + H * (F // 2 + F // 32 + 4)  # gate, up, down bytes
    ref = moe.Plan(shape, max_tokens=T).alloc_workspace().load_weights(moe.DeviceBlock(blk))
    cached = moe.Plan(shape, max_tokens=T, expert_cache_slots=slots).alloc_workspace()
    cached.load_weights(moe.HostStoreBlock(blk))
    xs = [torch.from_numpy(synth.make_tokens(wid, T, H, sub=500 + i).view(np.int16)).cuda() for i in range(n_sets)]
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    reps = n_sets
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(plan, rotate):
        for i in range(3):
            plan.forward(xs[i] if rotate else xs[0], out, stream=st)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                plan.forward(xs[i] if rotate else xs[0], out, stream=torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        before = plan.cache_state() if plan is cached else None
        clocks = Clocks(torch.cuda.current_device())
        e0.record(st)
        g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        clk = clocks.stop()
        after = plan.cache_state() if plan is cached else None
        del g
        return e0.elapsed_time(e1) / reps, before, after, clk

    ms_res, _, _, _ = timed(ref, True)
    ms_hit, b0, a0, _ = timed(cached, False)
    ms_miss, b1, a1, clk = timed(cached, True)
    hits, misses = a1[1] - b1[1], a1[2] - b1[2]
    moved = misses * per_expert / reps
    ref.close()
    cached.close()
    return {"value": T / (ms_miss / 1e3), "unit": "tokens/s", "ms_per_step": ms_miss, "path": "gemv + expert cache",
            "config": {"workload": f"gpt-oss MoE block decode, {T} tokens, experts in pinned host memory behind a "
                                   f"{slots}-slot device cache",
                       "tokens_per_step": T, "n_experts": shape.n_experts, "top_k": shape.top_k, "slots": slots,
                       "token_sets": n_sets, "weights": "mxfp4 (e2m1 + e8m0/32)"},
            "resident_ms_per_step": ms_res,
            "all_hits_ms_per_step": ms_hit,
            "all_hits_misses": a0[2] - b0[2],
            "hit_rate": hits / max(1, hits + misses),
            "misses_per_step": misses / reps,
            "store_bytes_per_step": moved,
            "store_gbs_over_hits": moved / max(1e-9, (ms_miss - ms_hit) / 1e3) / 1e9,
            "roofline": {"bound": "host link", "achieved": moved / (ms_miss / 1e3) / 1e9, "peak": None,
                         "peak_kind": "none measured (NVLink-C2C nominal 450 GB/s a direction)", "unit": "GB/s",
                         "frac": None, "traffic": None},
            "clocks": clk, "gpu_launches": 6 * reps}


def attention_prefill_bench(args, n: int = 512, ctx: int = 4096):
    """Prefill of the attention half (moe_attn_prefill): an n-token prompt into
    the empty cache of one sequence, one sliding-window (128) layer and one
    full-attention layer (one block of n rows: appended, then attended).
    Timed in a CUDA graph; HBM roofline of the algorithmic bytes (both layers'
    projection weights once, the keys and values each row sees, activations)."""
    import numpy as np
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe, synth
    A = synth.ATTN_GPT_OSS
    H, QH, KVH, D, window = A["hidden"], A["q_heads"], A["kv_heads"], A["head_dim"], A["window"]
    plans = []
    for layer, win in enumerate((window, 0)):
        p = moe.AttnPlan(H, QH, KVH, 32, ctx, sliding_window=win, prefill_rows=n)
        p.load_weights(synth.attention_device(300 + layer, H, QH, KVH, D))
        plans.append(p)
    x = torch.from_numpy(synth.f32_to_bf16_bits(np.random.default_rng(1).normal(0, 1, (n, H))).view(np.int16)).cuda()
    out = torch.empty((n, H), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        for p in plans:
            p.prefill(x, 0, 0, out, stream=st)
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 20))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            for p in plans:
                p.prefill(x, 0, 0, out, stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / reps
    weights = 2 * ((QH * D + 2 * KVH * D) * H * 2 + H * QH * D * 2)
    seen = sum(min(r + 1, window) for r in range(n)) + sum(r + 1 for r in range(n))
    kv = seen * KVH * D * 2 * 2
    act = 2 * n * (H * 2 + H * 4 + 2 * KVH * D * 2)
    hbm, _, kind = peaks()
    total = weights + kv + act
    for p in plans:
        p.close()
    del g
    return {"value": n / (ms / 1e3), "unit": "tokens/s (one sliding + one full attention layer)", "ms_per_step": ms,
            "path": "attention prefill (one block of the prompt's rows)",
            "config": {"workload": f"gpt-oss attention prefill, one {n}-token prompt into an empty cache, one "
                                   "sliding-window (128) and one full layer", "hidden": H, "q_heads": QH,
                       "kv_heads": KVH, "head_dim": D, "rows_per_block": n, "weights": "bf16 (synthetic)",
                       "kv_cache": "fp16"},
            "algorithmic_bytes_per_step": total,
            "roofline": {"bound": "hbm", "achieved": total / (ms / 1e3) / 1e9, "peak": hbm, "peak_kind": kind,
                         "unit": "GB/s", "frac": total / (ms / 1e3) / 1e9 / hbm, "traffic": None},
            "note": "the projections take the tokens 32 at a time: their weights come from HBM once and from "
                    "L2 for the other token blocks",
            "clocks": clk, "gpu_launches": reps * 2 * 6}


def decoder_bench(args, w, ctx: int = 4096):
    """The whole gpt-oss decoder stack's decode step: per layer the attention
    half (moe_attn_decode: sliding window of 128 on even layers, full
    attention on odd ones; the workload's tokens as that many sequences, each
    with ctx - 1 cached tokens) writing bf16 into the MoE block of the same
    layer (the stack workload's plans), whose bf16 output is the next layer's
    input.  Timed in one CUDA graph of K steps; HBM roofline of the step's
    algorithmic bytes (the MoE stack's, plus every layer's attention weights
    and visible keys and values)."""
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe, synth
    A = synth.ATTN_GPT_OSS
    H, QH, KVH, D, window = A["hidden"], A["q_heads"], A["kv_heads"], A["head_dim"], A["window"]
    T, d = w.T, w.sets[0]
    chain = d["chain"]
    L = len(chain)
    att = []
    for i in range(L):
        p = moe.AttnPlan(H, QH, KVH, T, ctx, sliding_window=window if i % 2 == 0 else 0, out_bf16=True)
        p.load_weights(synth.attention_device(7000 + i, H, QH, KVH, D))
        synth.kv_history_device(9000 + i, p.k_cache, p.v_cache)
        att.append(p)
    hs = [chain[0]["x"].clone()] + [torch.empty((T, H), dtype=torch.int16, device="cuda") for _ in range(L - 1)]
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    pos = torch.full((T,), ctx - 1, dtype=torch.int32, device="cuda")

    def step(st):
        for i in range(L):
            att[i].decode(hs[i], pos, chain[i]["x"], stream=st)
            chain[i]["plan"].forward(chain[i]["x"], out if i + 1 == L else hs[i + 1], chain[i]["ids"], stream=st)
    st = torch.cuda.current_stream()
    for _ in range(3):
        step(st)
    torch.cuda.synchronize()
    reps = max(1, min(args.steps, 50))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            step(torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / reps
    # algorithmic bytes: the MoE stack's (from its own measurement) and, per
    # layer, the attention weights once and the visible keys and values
    aw = (QH * D + 2 * KVH * D) * H * 2 + H * QH * D * 2 + 4 * (QH * D + 2 * KVH * D + 2 * H + QH)
    kv = sum(T * (min(ctx, window) if i % 2 == 0 else ctx) * KVH * D * 2 * 2 for i in range(L))
    hbm, _, kind = peaks()
    moe_bytes = 0
    for ly in chain:  # the MoE blocks' bytes from this run's own routing (the last step's counts)
        c = torch.empty(w.shape.n_experts, dtype=torch.int32, device="cuda")
        ly["plan"].expert_counts(c)
        torch.cuda.synchronize()
        gu, dn, _ = algorithmic_bytes(w.shape, c.cpu().numpy(), T)
        moe_bytes += gu + dn
    total = moe_bytes + L * aw + kv
    for p in att:
        p.close()
    del g
    return {"value": T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms, "path": "attention decode + MoE GEMV",
            "config": {"workload": f"{L}-layer gpt-oss decoder stack decode (attention + MoE), {T} sequences x "
                                   f"{ctx - 1} cached tokens", "layers": L, "sequences": T, "context": ctx,
                       "attention": "sliding window 128 on even layers, full on odd; bf16 weights (synthetic); "
                                    "fp16 caches", "moe": "the 24-layer stack workload's blocks"},
            "algorithmic_bytes_per_step": total,
            "roofline": {"bound": "hbm", "achieved": total / (ms / 1e3) / 1e9, "peak": hbm, "peak_kind": kind,
                         "unit": "GB/s", "frac": total / (ms / 1e3) / 1e9 / hbm, "traffic": None},
            "clocks": clk, "gpu_launches": reps * L * 9}


def locality_stats(w, steps: int = 16):
    """Expert-locality statistics of the stack's routing (the library's
    profiler attached to every layer; untimed, outside the measured steps):
    steps of the workload's tokens as consecutive positions, per-capacity hit
    rates of least-recently-used expert caches, the overlap of consecutive
    tokens' expert sets, and the recording cost per layer and step."""
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe
    sh = w.shape
    caps = [4, 8, 12, 16, 24]
    prof = moe.Locality(w.layers, sh.n_experts, sh.top_k, caps)
    d = w.sets[0]
    plans = w.plans(d)
    for i, p in enumerate(plans):
        prof.attach(p, i)
    st = torch.cuda.current_stream()
    for _ in range(steps):
        w.forward_set(d, st)
    torch.cuda.synchronize()
    got = prof.read()
    for p in plans:
        moe.load().moe_locality_attach(p.h, None, 0)
    # the recording alone (every layer's routes of the last step), in a CUDA
    # graph so that host launch costs stay off the clock
    wts = torch.zeros((w.T, sh.top_k), dtype=torch.float32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i, ly in enumerate(d["chain"]):
            prof.record(i, ly["ids"], wts, 0, stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(10):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    rec_us = 1e3 * e0.elapsed_time(e1) / (10 * len(plans))
    del g
    sel = float(got["hist"].sum())
    wsum = float(got["weight_hist"].sum())
    pairs = float(got["adjacent_pairs"].sum())
    prof.close()
    return {"tokens": int(steps * w.T), "layers": w.layers, "caps": [int(c) for c in got["caps"]],
            "hit_rate": [float(h) / sel for h in got["cache_hits"].sum(axis=1)],
            "weighted_hit_rate": [float(h) / wsum for h in got["cache_weight_hits"].sum(axis=1)],
            "adjacent_overlap": float(got["overlap_sum"].sum()) / pairs if pairs else None,
            "adjacent_jaccard": float(got["jaccard_sum"].sum()) / pairs if pairs else None,
            "unique_experts_per_layer": float((got["hist"] > 0).sum(axis=1).mean()),
            "record_us_per_layer_step": rec_us,
            "note": "synthetic router weights: the statistics show the profiler working, not a model's locality"}


def cpu_baseline(wid, T, w):
    """The oracle, as it stands, timed on the host cores for a bounded sample of
    the workload's tokens (about 10-30 s): as many tokens as there are cores
    (at most the step's), through every layer, on the seeded host-drawn weights
    of the same recipe (weight generation off the clock)."""
    import oracle
    from mxfp4_mixture_experts_rms_gb300 import synth
    cores = os.cpu_count() or 1
    wl = synth.WORKLOADS[wid]
    n = min(T, cores)
    xs = w.sets[0]["xb"][:n]
    el = 0.0
    for layer in range(wl.layers):
        blk = synth.make_block(wid, layer=layer)
        if layer == 0:
            oracle.moe_forward(blk, xs[:1], nthreads=1)
        t0 = time.perf_counter()
        out = oracle.moe_forward(blk, xs, nthreads=n)["out"]
        el += time.perf_counter() - t0
        xs = synth.f32_to_bf16_bits(out)
        del blk
    return {"value": n / el, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{n} of the {T} tokens of one step through all {wl.layers} layer(s), {el:.1f} s of oracle time"}


def run_ours(args, rank, world, local, wid, T):
    import torch

    from mxfp4_mixture_experts_rms_gb300 import moe, synth
    torch.cuda.set_device(local)
    moe.load()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pool = Pool()
    wl = synth.WORKLOADS[wid]
    w = Workload(wid, T, pool, rank, {"act_fp4": 1} if args.act_fp4 else None, args.layers)
    r = measure(w, args, world, local, 0.0 if args.quick else 1.0)
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": whole_job_rate(world, T, args.steps, r["ms"]),
                              "unit": "tokens/s", "ms_per_step": r["ms"] / args.steps, "quick": True,
                              "config": {"workload": wl.name, "tokens_per_step": T}}), flush=True)
        return
    head = summarise(w, r, args, world)
    e2e = e2e_rate(w, args, world)
    loc = locality_stats(w) if w.layers > 1 else None
    dec = decoder_bench(args, w) if w.layers > 1 and not args.no_extras else None
    extras = {}
    if not args.no_extras:
        for (ew, eT, eo) in EXTRAS:
            if (ew, eT) == (wid, T) and not eo:
                continue
            x = Workload(ew, eT, pool, rank, eo)
            xr = measure(x, args, world, local, 0.5)
            s = summarise(x, xr, args, world)
            s["config"] = workload_config(x.wl, eT)
            if eo.get("act_fp4"):
                s["config"]["activations"] = "fp4 (e2m1 + e8m0/32, the FP4 activation encoding)"
            s["weight_sets"] = len(x.sets)
            extras[f"{synth.WORKLOADS[ew].name} x{eT}" + (" fp4" if eo.get("act_fp4") else "")] = s
            x.close()
            torch.cuda.synchronize()
        att = attention_bench(args)
        extras[att["config"]["workload"]] = att
        apf = attention_prefill_bench(args)
        extras[apf["config"]["workload"]] = apf
        xc = expert_cache_bench(args)
        extras[xc["config"]["workload"]] = xc
        if dec:
            extras[dec["config"]["workload"]] = dec
    if rank != 0:
        return
    cpu = None if args.no_cpu_baseline else cpu_baseline(wid, T, w)
    cfg = workload_config(wl, T)
    cfg.update({"weight_sets": len(w.sets), "parallelism": f"replicas x{world}",
                "l2": ("inputs larger than L2: a stack of independently seeded layers (~10 GB)" if w.layers > 1 else
                       "inputs larger than L2: steps rotate over independently seeded weight sets "
                       "(> 2.5 x L2 touched between two uses of a set)"),
                "weights_drawn": "router/gamma/bias by the host recipe; expert matrices on the device, same "
                                 "distributions"})
    for k in ("distinct_experts_per_block", "algorithmic_bytes_per_step", "step_hbm_gbs", "step_frac_of_hbm",
              "algorithmic_flops_per_step", "step_tflops", "step_frac_of_bf16_peak", "binding_roof_frac", "path"):
        cfg[k] = head[k]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": head.get("roofline"), "kernels": head.get("kernels"),
        "cpu_baseline": cpu, "e2e": e2e, "clocks": head["clocks"], "gpu_launches": head["gpu_launches"],
        "configs": extras,
    }
    if loc:
        line["locality"] = loc
    print(json.dumps(line), flush=True)


def run_mx_fp4_quantize(args):
    """The FP4 activation encoder alone: bf16 [rows][cols] -> MXFP4 codes + E8M0
    scales, timed with CUDA events on the launching stream over input sets that
    together exceed twice the L2, so every launch reads from HBM."""
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe
    moe.load()
    R, Cc = args.rows, args.cols
    n = R * Cc
    algo = n * 2 + n // 2 + n // 32
    n_sets = max(2, -(-2 * L2_BYTES // algo) + 1)
    g = torch.Generator(device="cuda").manual_seed(0x4D6F45)
    xs = [(torch.randn((R, Cc), device="cuda", generator=g) * 4).to(torch.bfloat16).view(torch.int16)
          for _ in range(n_sets)]
    codes = [torch.empty(n // 2, dtype=torch.uint8, device="cuda") for _ in range(n_sets)]
    scales = [torch.empty(n // 32, dtype=torch.uint8, device="cuda") for _ in range(n_sets)]
    st = torch.cuda.current_stream()
    for i in range(max(3, args.warmup)):
        moe.mx_quantize_fp4(xs[i % n_sets], codes[i % n_sets], scales[i % n_sets], st)
    torch.cuda.synchronize()
    clk = Clocks(torch.cuda.current_device())
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < 1.0:   # clocks settle under load before the timed region
        for i in range(n_sets):
            moe.mx_quantize_fp4(xs[i], codes[i], scales[i], st)
        torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for i in range(args.steps):
        moe.mx_quantize_fp4(xs[i % n_sets], codes[i % n_sets], scales[i % n_sets], st)
    e1.record(st)
    torch.cuda.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1) / args.steps
    hbm, _, peak_kind = peaks()
    gbs = algo / (ms / 1e3) / 1e9
    workload = f"FP4 activation encoding, {R} x {Cc} bf16"
    tr = traffic_record("mx_fp4_quantize", workload)
    print(json.dumps({
        "op": "mx_fp4_quantize", "metric": "FP4 activation encoding bandwidth", "value": gbs, "unit": "GB/s",
        "higher_is_better": True, "steps": args.steps, "ms_per_launch": ms, "dtype": "bf16->fp4",
        "data": "synthetic", "gpu_launches": args.steps, "clocks": clocks,
        "config": {"workload": workload, "rows": R, "cols": Cc,
                   "l2": f"{n_sets} input sets rotated, {n_sets * algo / 1e6:.0f} MB > 2 x L2"},
        "roofline": {"bound": "hbm", "kernel": "mx_fp4_quantize", "achieved": gbs, "peak": hbm,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": tr["bytes_per_launch"] if tr else None,
                     "algorithmic_bytes_per_launch": algo, "avg_launch_ms": ms}}))


def main():
    args = parse()
    if args.op == "mx_fp4_quantize":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "op": "mx_fp4_quantize",
                              "unavailable": "the encoder is timed on the GPU only"}))
            return
        run_mx_fp4_quantize(args)
        return
    if args.op in ("attention", "attention_prefill", "expert_cache"):
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "op": args.op,
                              "unavailable": f"the {args.op.replace('_', ' ')} step is timed on the GPU only"}))
            return
        import torch
        from mxfp4_mixture_experts_rms_gb300 import moe
        moe.load()
        fn = {"attention": attention_bench, "attention_prefill": attention_prefill_bench,
              "expert_cache": expert_cache_bench}[args.op]
        print(json.dumps(fn(args)), flush=True)
        return
    from mxfp4_mixture_experts_rms_gb300 import synth
    wid = args.workload
    T = args.tokens or (HEADLINE[1] if wid == HEADLINE[0] else max(synth.WORKLOADS[wid].tokens))
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, wid, T)
        return
    run_ours(args, rank, world, local, wid, T)


if __name__ == "__main__":
    main()
