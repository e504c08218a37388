"""Shared helpers of the GPU parity tests: run the CUDA library through the
C-ABI binding and compare with the CPU oracle on the same seeded inputs."""
import os

import numpy as np

import oracle
from mxfp4_mixture_experts_rms_gb300 import moe, synth

NTHREADS = os.cpu_count() or 4

# Tolerance of the block output (float32 accumulation against the fp64 oracle):
# relative L2 <= 1e-3 and max abs <= 2e-3 * max|ref|.
REL_L2 = 1e-3
MAX_ABS_FRAC = 2e-3


def run_gpu(blk, x_bits, max_tokens=None, plan=None, dev=None, **opts):
    import torch
    shape = blk["shape"]
    T = x_bits.shape[0]
    if plan is None:
        plan = moe.Plan(shape, max_tokens=max_tokens or max(T, 1), **opts).alloc_workspace()
        dev = dev or moe.DeviceBlock(blk)
        plan.load_weights(dev)
    K, H, E = shape.top_k, shape.hidden, shape.n_experts
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    rw = torch.empty((T, K), dtype=torch.float32, device="cuda")
    xh = torch.empty((T, H), dtype=torch.int16, device="cuda")
    plan.forward_ex(x, out, ids, rw, xh)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    plan.expert_counts(counts)
    EE = E + shape.n_shared
    R = plan.max_tokens * (K + shape.n_shared)
    offs = torch.empty(EE + 1, dtype=torch.int32, device="cuda")
    pt = torch.empty(R, dtype=torch.int32, device="cuda")
    ps = torch.empty(R, dtype=torch.int32, device="cuda")
    plan.permutation(offs, pt, ps)
    torch.cuda.synchronize()
    status = plan.device_status()
    r = dict(out=out.cpu().numpy(), ids=ids.cpu().numpy(), route_w=rw.cpu().numpy(),
             xhat=xh.cpu().numpy().view(np.uint16), counts=counts.cpu().numpy(), offsets=offs.cpu().numpy(),
             perm_token=pt.cpu().numpy(), perm_slot=ps.cpu().numpy(), status=status)
    return r, plan, dev


def check_close(got, ref, x_bits=None, what="out"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = got - ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(err).max() / max(np.abs(ref).max(), 1e-300)
    assert rel <= REL_L2 and mx <= MAX_ABS_FRAC, f"{what}: rel L2 {rel:.3e}, max abs/max|ref| {mx:.3e}"
    if x_bits is not None:  # the MoE delta alone, as a diagnostic that must also hold
        x = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
        d_ref = ref - x
        d_rel = np.linalg.norm(got - x - d_ref) / max(np.linalg.norm(d_ref), 1e-300)
        assert d_rel <= REL_L2, f"{what} delta: rel L2 {d_rel:.3e}"
    return rel, mx


def oracle_routes(blk, x_bits):
    """Routing-only oracle (norm, logits, top-k, weights) per token."""
    shape = blk["shape"]
    T = x_bits.shape[0]
    ids = np.empty((T, shape.top_k), np.int32)
    rw = np.empty((T, shape.top_k))
    xh = np.empty_like(x_bits)
    for t in range(T):
        xh[t], _ = oracle.rmsnorm(x_bits[t], blk["gamma"], shape.rms_eps)
        lg = oracle.router_logits(xh[t], blk["router_w"], blk["router_b"])
        ids[t], vals = oracle.topk(lg, shape.top_k)
        rw[t] = oracle.route_weights(vals, shape.weight_scale)
    return ids, rw, xh


def check_permutation(r, ids, shape):
    E, K, ns = shape.n_experts, shape.top_k, shape.n_shared
    T = ids.shape[0]
    p = oracle.permutation(ids, E)
    assert np.array_equal(r["counts"], p["counts"])
    assert np.array_equal(r["offsets"][:E + 1], p["offsets"])
    n = T * K
    assert np.array_equal(r["perm_token"][:n], p["perm_token"])
    assert np.array_equal(r["perm_slot"][:n], p["perm_slot"])
    if ns:
        assert r["offsets"][E + 1] == n + T
        assert np.array_equal(r["perm_token"][n:n + T], np.arange(T))
        assert np.all(r["perm_slot"][n:n + T] == K)


def tiny_block(seed, shape, elo=118, ehi=124):
    """Random canonical weights for arbitrary small shapes (same recipe as the workloads)."""
    rng = np.random.default_rng(seed)
    H, E = shape.hidden, shape.n_experts
    blk = {"shape": shape,
           "gamma": (1 + rng.normal(0, 0.1, H)).astype(np.float32),
           "router_w": synth.f32_to_bf16_bits(rng.normal(0, 0.3, (E, H))),
           "router_b": rng.normal(0, 0.5, E).astype(np.float32),
           "codes": {}, "scales": {}, "bias": {}}

    def mats(n):
        d = {"codes": {}, "scales": {}, "bias": {}}
        for m in synth.MATS:
            rows, cols = shape.mat_shape(m)
            d["codes"][m] = rng.integers(0, 256, (n, rows, cols // 2), dtype=np.uint8)
            d["scales"][m] = rng.integers(elo, ehi + 1, (n, rows, cols // 32), dtype=np.uint8)
            d["bias"][m] = rng.normal(0, 0.02, (n, rows)).astype(np.float32)
        return d

    blk.update(mats(E))
    if shape.n_shared:
        blk["shared"] = mats(1)
    return blk
