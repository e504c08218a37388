#!/usr/bin/env python3
"""Throughput of the MXFP4 routed MoE block on GB300.

One step = one forward of the whole block (norm + router + top-k + softmax,
permutation, MXFP4 gate/up + SwiGLU, MXFP4 down, weighted combine + residual)
over one batch of the workload: the gpt-oss MoE block decoding a batch of 8
tokens with two hot experts (hidden 2880, 32 experts, top-4, expert_hidden
2880).  Weights are seeded synthetic MXFP4 tensors of that architecture.  The
steps rotate over several independently seeded weight sets whose touched
experts together exceed the 129 MB L2, so no step finds its weights in L2.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
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
sys.path.insert(0, ROOT)

METRIC = "MoE block tokens/s; decode HBM GB/s and prefill TFLOP/s vs GB300 peak"
WORKLOAD = 1
TOKENS = 8
KERNEL_SLOTS = ["route_permute", "gateup_swiglu", "down_weighted", "combine_residual"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sets", type=int, default=4, help="weight sets rotated over the steps")
    ap.add_argument("--workload", type=int, default=WORKLOAD,
                    help="workload id of synth.WORKLOADS (default: the 8-token hot-2 decode batch)")
    ap.add_argument("--tokens", type=int, default=0, help="tokens per step (default: the workload's largest)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="timed region only (no clock pre-roll, kernel timing, e2e or CPU baseline); for ncu")
    ap.add_argument("--op", default="block", choices=["block", "mx_fp4_quantize"],
                    help="block: the MoE block (the benchmark); mx_fp4_quantize: the FP4 activation "
                         "encoder alone, on --rows x --cols bf16 activations")
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


def traffic_record(kernel: str, workload: str = "", tokens: int = 0):
    """ncu DRAM bytes per launch of `kernel`, if taken on the current source, on
    this workload and token count."""
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


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np

    import oracle
    from mxfp4_mixture_experts_rms_gb300 import synth
    cores = os.cpu_count() or 1
    wl = synth.WORKLOADS[WORKLOAD]
    if wl.layers > 1:
        return run_reference_stack(args, world, wl, cores)
    blk = synth.make_block(WORKLOAD)
    x = synth.make_tokens(WORKLOAD, TOKENS, blk["shape"].hidden)
    oracle.moe_forward(blk, x[:1], nthreads=1)  # warm the library
    t0 = time.perf_counter()
    oracle.moe_forward(blk, x[:1], nthreads=1)
    t_tok = time.perf_counter() - t0
    # tokens per step so that the whole run takes about three minutes on all cores
    budget = 180.0
    per_step = max(1, min(TOKENS, int(budget * cores / max(1e-9, (args.steps + args.warmup) * t_tok))))
    nthr = min(cores, per_step)
    for i in range(args.warmup):
        oracle.moe_forward(blk, np.ascontiguousarray(x[(i % TOKENS):(i % TOKENS) + 1].repeat(per_step, 0)), nthreads=nthr)
    t0 = time.perf_counter()
    for i in range(args.steps):
        xs = np.ascontiguousarray(np.roll(x, -i, axis=0)[:per_step]) if per_step <= TOKENS else x
        oracle.moe_forward(blk, xs, nthreads=nthr)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    sample = f"{per_step} of the {TOKENS} tokens of each step (full block per token), {nthr} threads"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": synth.WORKLOADS[WORKLOAD].name, "tokens_per_step": TOKENS,
                       "hidden": 2880, "n_experts": 32, "top_k": 4, "expert_hidden": 2880},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_stack(args, world, wl, cores):
    """The oracle through the whole stack for a bounded sample of each step's
    tokens; each layer's weights are regenerated from their seed off the clock
    (the stack does not fit comfortably in host memory twice)."""
    import numpy as np

    import oracle
    from mxfp4_mixture_experts_rms_gb300 import synth
    shape = wl.shape
    x = synth.make_tokens(WORKLOAD, TOKENS, shape.hidden)
    per_step = min(TOKENS, cores)
    el = 0.0
    for i in range(args.warmup + args.steps):
        xs = np.ascontiguousarray(np.roll(x, -i, axis=0)[:per_step])
        for l in range(wl.layers):
            blk = synth.make_block(WORKLOAD, layer=l)
            t0 = time.perf_counter()
            out = oracle.moe_forward(blk, xs, nthreads=per_step)["out"]
            if i >= args.warmup:
                el += time.perf_counter() - t0
            xs = synth.f32_to_bf16_bits(out)
            del blk
    value = per_step * args.steps / el
    sample = (f"{per_step} of the {TOKENS} tokens of each step through all {wl.layers} layers, "
              f"{per_step} threads (weight generation off the clock)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "tokens_per_step": TOKENS, "layers": wl.layers,
                       "hidden": shape.hidden, "n_experts": shape.n_experts, "top_k": shape.top_k,
                       "expert_hidden": shape.expert_hidden},
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


def algorithmic_bytes(shape, counts, T):
    """Bytes the gate/up and down kernels must move at least once per launch."""
    H, F = shape.hidden, shape.expert_hidden
    distinct = int((counts > 0).sum()) + shape.n_shared
    routes = int(counts.sum()) + shape.n_shared * T
    mat = F * H // 2 + F * H // 32
    gateup = distinct * (2 * mat + 2 * F * 4) + T * H * 2 + routes * F * 2
    down = distinct * (mat + H * 4) + routes * F * 2 + routes * H * 4
    return gateup, down, distinct


def cpu_baseline(blk, x):
    import oracle
    cores = os.cpu_count() or 1
    n = min(x.shape[0], cores)
    oracle.moe_forward(blk, x[:1], nthreads=1)
    t0 = time.perf_counter()
    oracle.moe_forward(blk, x[:n], nthreads=n)
    el = time.perf_counter() - t0
    return {"value": n / el, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{n} tokens of one step (weight set 0), whole block per token, {el:.1f} s wall"}


def cpu_baseline_stack(wl, x):
    """The oracle through the whole stack (each layer's fp32 output cast to bf16
    for the next), for as many of the step's tokens as there are cores."""
    import oracle
    from mxfp4_mixture_experts_rms_gb300 import synth
    cores = os.cpu_count() or 1
    n = min(x.shape[0], cores)
    xs = x[:n]
    el = 0.0
    for l in range(wl.layers):
        blk = synth.make_block(WORKLOAD, layer=l)
        t0 = time.perf_counter()
        out = oracle.moe_forward(blk, xs, nthreads=n)["out"]
        el += time.perf_counter() - t0
        xs = synth.f32_to_bf16_bits(out)
        del blk
    return {"value": n / el, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{n} tokens through all {wl.layers} layers, {el:.1f} s of oracle time"}


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from mxfp4_mixture_experts_rms_gb300 import moe, synth
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    wl = synth.WORKLOADS[WORKLOAD]
    shape = wl.shape
    H, K = shape.hidden, shape.top_k
    sets = []
    if wl.layers > 1:
        # a stack of independently seeded blocks: layer l's fp32 output, cast to
        # bf16, is layer l+1's input; the stack itself (~10 GB) is far larger than L2
        layers = []
        for l in range(wl.layers):
            blk = synth.make_block(WORKLOAD, layer=l + 100 * rank)
            plan = moe.Plan(shape, max_tokens=TOKENS).alloc_workspace().load_weights(moe.DeviceBlock(blk))
            layers.append(dict(plan=plan, x=torch.empty((TOKENS, H), dtype=torch.int16, device="cuda"),
                               out=torch.empty((TOKENS, H), dtype=torch.float32, device="cuda"),
                               ids=torch.empty((TOKENS, K), dtype=torch.int32, device="cuda")))
            del blk
        xb = synth.make_tokens(WORKLOAD, TOKENS, H, layer=100 * rank)
        layers[0]["x"].copy_(torch.from_numpy(xb.view(np.int16)))
        sets.append(dict(blk=None, xb=xb, plan=layers[0]["plan"], x=layers[0]["x"], out=layers[-1]["out"],
                         ids=layers[-1]["ids"], layers=layers))
    for s in range(args.sets if wl.layers == 1 else 0):
        layer = s + 100 * rank
        blk = synth.make_block(WORKLOAD, layer=layer)
        xb = synth.make_tokens(WORKLOAD, TOKENS, H, layer=layer)
        plan = moe.Plan(shape, max_tokens=TOKENS).alloc_workspace().load_weights(moe.DeviceBlock(blk))
        x = torch.from_numpy(xb.view(np.int16)).cuda()
        out = torch.empty((TOKENS, H), dtype=torch.float32, device="cuda")
        ids = torch.empty((TOKENS, K), dtype=torch.int32, device="cuda")
        sets.append(dict(blk=blk if s == 0 else None, xb=xb if s == 0 else None, plan=plan, x=x, out=out, ids=ids))
        del blk
    def plans_of(d):
        return [ly["plan"] for ly in d["layers"]] if "layers" in d else [d["plan"]]

    def forward_set(d, stream):
        if "layers" in d:
            ls = d["layers"]
            for l, ly in enumerate(ls):
                ly["plan"].forward(ly["x"], ly["out"], ly["ids"], stream=stream)
                if l + 1 < len(ls):
                    moe.cast_f32_to_bf16(ly["out"], ls[l + 1]["x"], stream=stream)
        else:
            d["plan"].forward(d["x"], d["out"], d["ids"], stream=stream)

    def step(i, stream):
        forward_set(sets[i % len(sets)], stream)

    def capture(n):
        """One CUDA graph holding n consecutive steps (launch overhead off the clock)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for i in range(n):
                step(i, cs)
        return g

    st = torch.cuda.current_stream()
    # per-set routing facts for the algorithmic byte counts
    facts = []
    for i, d in enumerate(sets):
        step(i, st)
        tot_f = [0, 0, 0]
        for p in plans_of(d):
            c = torch.empty(shape.n_experts, dtype=torch.int32, device="cuda")
            p.expert_counts(c)
            torch.cuda.synchronize()
            tot_f = [a + b for a, b in zip(tot_f, algorithmic_bytes(shape, c.cpu().numpy(), TOKENS))]
        facts.append(tuple(tot_f))
    n_blocks = len(plans_of(sets[0]))  # blocks per step (the stack's layers)
    for i in range(args.warmup):
        step(i, st)
    torch.cuda.synchronize()
    graph = capture(args.steps)
    graph.replay()
    torch.cuda.synchronize()
    # pre-roll so that the clock samples see this load for about a second
    clocks = Clocks(local)
    t_end = time.perf_counter() + (0.0 if args.quick else 1.0)
    while time.perf_counter() < t_end:
        graph.replay()
        torch.cuda.synchronize()
    # ---- timed region: exactly K steps (one graph replay)
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
    value = whole_job_rate(world, TOKENS, args.steps, ms)
    if args.quick:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "tokens/s", "ms_per_step": ms / args.steps,
                              "quick": True}), flush=True)
        return

    # ---- kernel durations over the same K steps: CUDA events the library
    # records around each launch (captured into the graph as event nodes)
    for d in sets:
        for p in plans_of(d):
            p.set_i("profile", 1)
    pgraph = capture(args.steps)
    torch.cuda.synchronize()
    pgraph.replay()
    torch.cuda.synchronize()
    tot = [0.0] * 4
    cnt = [0] * 4
    for d in sets:
        for p in plans_of(d):
            m, c = p.profile_read()
            tot = [a + b for a, b in zip(tot, m)]
            cnt = [a + b for a, b in zip(cnt, c)]
            p.set_i("profile", 0)
    del pgraph
    avg_ms = [t / c if c else 0.0 for t, c in zip(tot, cnt)]
    share = [t / sum(tot) for t in tot] if sum(tot) > 0 else [0.0] * 4
    # per launch of each kernel (a step launches each once per block)
    gu_bytes = sum(facts[i % len(sets)][0] for i in range(args.steps)) / args.steps / n_blocks
    dn_bytes = sum(facts[i % len(sets)][1] for i in range(args.steps)) / args.steps / n_blocks
    distinct = sum(facts[i % len(sets)][2] for i in range(args.steps)) / args.steps / n_blocks
    hbm, bf16_peak, peak_kind = peaks()
    dom = max(range(4), key=lambda k: tot[k])
    dom_bytes = {1: gu_bytes, 2: dn_bytes}.get(dom, gu_bytes)
    achieved = dom_bytes / (avg_ms[dom] / 1e3) / 1e9 if avg_ms[dom] > 0 else 0.0
    tr = traffic_record(KERNEL_SLOTS[dom], wl.name, TOKENS)
    path = sets[0]["plan"].path_for(TOKENS)  # 1 GEMV decode path, 2 tensor-core grouped GEMM
    step_bytes = (gu_bytes + dn_bytes) * n_blocks
    step_gbs = step_bytes / (ms / args.steps / 1e3) / 1e9
    routes = TOKENS * (K + shape.n_shared)
    step_flops = 6.0 * routes * H * shape.expert_hidden * n_blocks
    step_tflops = step_flops / (ms / args.steps / 1e3) / 1e12

    # ---- end to end through the public API with host buffers
    hx = [d["x"].cpu().pin_memory() for d in sets]
    hout = [torch.empty((TOKENS, H), dtype=torch.float32).pin_memory() for _ in sets]
    hids = [torch.empty((TOKENS, K), dtype=torch.int32).pin_memory() for _ in sets]

    def e2e_step(i):
        j = i % len(sets)
        d = sets[j]
        d["x"].copy_(hx[j], non_blocking=True)
        forward_set(d, st)
        hout[j].copy_(d["out"], non_blocking=True)
        hids[j].copy_(d["ids"], non_blocking=True)

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
    e2e = {"value": whole_job_rate(world, TOKENS, args.steps, e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": TOKENS * H * 2, "d2h_bytes_per_step": TOKENS * H * 4 + TOKENS * K * 4}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world >= 1:
        cpu = (cpu_baseline_stack(wl, sets[0]["xb"]) if n_blocks > 1
               else cpu_baseline(sets[0]["blk"], sets[0]["xb"]))
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "tokens_per_step": TOKENS, "hidden": H, "n_experts": shape.n_experts,
                   "top_k": K, "expert_hidden": shape.expert_hidden, "weights": "mxfp4 (e2m1 + e8m0/32)",
                   "weight_sets": len(sets), "layers": n_blocks,
                   "l2": ("inputs larger than L2: a stack of independently seeded layers" if n_blocks > 1 else
                          "inputs larger than L2: steps rotate over independently seeded weight sets"),
                   "distinct_experts_per_block": distinct,
                   "algorithmic_bytes_per_step": step_bytes, "step_hbm_gbs": step_gbs,
                   "algorithmic_flops_per_step": step_flops, "step_tflops": step_tflops,
                   "step_tensor_frac_of_bf16_peak": step_tflops / peaks()[1],
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline(path, dom, avg_ms[dom], achieved, hbm, bf16_peak, peak_kind, tr, dom_bytes,
                             routes, H, shape.expert_hidden, TOKENS * shape.n_experts * H),
        "kernels": {KERNEL_SLOTS[k]: {"avg_us": 1e3 * avg_ms[k], "share": share[k], "launches": cnt[k]}
                    for k in range(4)},
        "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "gpu_launches": int(sum(cnt)) + (n_blocks - 1) * args.steps,  # + the stack's casts between layers
    }
    print(json.dumps(line), flush=True)


# fp32 FMA peak of the SIMT router: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz
# (the GB300's SM count and maximum SM clock)
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def roofline(path, dom, avg_ms, achieved_gbs, hbm, bf16_peak, peak_kind, tr, dom_bytes, routes, H, F, router_macs):
    """Roofline of the dominant kernel: HBM for the GEMVs (decode path), the
    bf16 tensor peak for the grouped GEMMs (prefill path), the fp32 FMA peak
    when the SIMT routing kernel dominates a prefill step."""
    if path == 2 and dom in (1, 2):
        flops = 2.0 * routes * (2 * F if dom == 1 else F) * H
        ach = flops / (avg_ms / 1e3) / 1e12 if avg_ms > 0 else 0.0
        return {"bound": "tensor", "kernel": KERNEL_SLOTS[dom], "achieved": ach, "peak": bf16_peak,
                "peak_kind": peak_kind, "unit": "TFLOP/s", "frac": ach / bf16_peak,
                "traffic": tr["bytes_per_launch"] if tr else None,
                "algorithmic_flops_per_launch": flops, "avg_launch_ms": avg_ms}
    if path == 2 and dom == 0:
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


def run_mx_fp4_quantize(args):
    """The FP4 activation encoder alone: bf16 [rows][cols] -> MXFP4 codes + E8M0
    scales, timed with CUDA events on the launching stream over input sets that
    together exceed twice the L2, so every launch reads from HBM."""
    import numpy as np
    import torch
    from mxfp4_mixture_experts_rms_gb300 import moe
    moe.load()
    R, Cc = args.rows, args.cols
    n = R * Cc
    algo = n * 2 + n // 2 + n // 32
    n_sets = max(2, -(-2 * 129 * 2 ** 20 // algo) + 1)
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
    from mxfp4_mixture_experts_rms_gb300 import synth
    global WORKLOAD, TOKENS
    WORKLOAD = args.workload
    TOKENS = args.tokens or max(synth.WORKLOADS[WORKLOAD].tokens)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
