"""GPU parity at the sizes the benchmark measures, in the launch configuration
it times (moe_forward on a plan sized for the batch):

* the gpt-oss block prefill at 512 tokens (grouped GEMM, ~64 routes per expert);
* the DeepSeek-V4-Flash-shaped block at 2048 tokens (256 experts, top-6, one
  shared expert, Zipf(1.1) routing: many route tiles per hot expert);
* the 24-layer gpt-oss stack decoding 16 tokens (16-route GEMV tiles), each
  layer's fp32 output cast to bf16 as the next layer's input.

Routing (x_hat, expert ids, counts, permutation) is compared bit-exactly for
every token; block outputs within the tolerance (relative L2 <= 1e-3 and max
abs <= 2e-3 * max|ref|) on tokens the oracle computes one by one.
"""
import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import NTHREADS, check_close, check_permutation, oracle_routes, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


def _sample(T, ids, n_random, n_hot, seed):
    """n_random tokens at random plus n_hot tokens routed to the most used expert."""
    rng = np.random.default_rng(seed)
    counts = np.bincount(ids.ravel(), minlength=ids.max() + 1)
    hot = int(np.argmax(counts))
    hot_tokens = np.nonzero((ids == hot).any(axis=1))[0]
    pick = set(rng.choice(T, n_random, replace=False).tolist())
    pick |= set(rng.choice(hot_tokens, min(n_hot, len(hot_tokens)), replace=False).tolist())
    return np.array(sorted(pick)), hot, int(counts[hot])


@pytest.mark.parametrize("cfg,T,n_random,n_hot", [(3, 512, 8, 6), (4, 2048, 8, 6)])
def test_block_parity_at_bench_size(cfg, T, n_random, n_hot):
    blk = synth.make_block(cfg)
    shape = blk["shape"]
    x = synth.make_tokens(cfg, T, shape.hidden)
    r, plan, _ = run_gpu(blk, x)
    assert plan.path_for(T) == 2          # the benchmark's grouped-GEMM path
    assert r["status"] == 0
    ids, rw, xh = oracle_routes(blk, x)
    assert np.array_equal(r["xhat"], xh)
    assert np.array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["route_w"], rw, rtol=2e-6, atol=1e-7)
    check_permutation(r, ids, shape)
    sample, hot, n_hot_routes = _sample(T, ids, n_random, n_hot, cfg)
    assert n_hot_routes > 128 or cfg == 3  # the Zipf-hot expert spans several 128-route tiles
    ref = oracle.moe_forward(blk, np.ascontiguousarray(x[sample]), nthreads=NTHREADS)
    assert np.array_equal(r["ids"][sample], ref["ids"])
    check_close(r["out"][sample], ref["out"], x[sample], what=f"cfg{cfg} x{T} sampled tokens")


def _route_margin(blk, x_bits, K):
    """Smallest gap between consecutive logits among the K + 1 largest (the
    margin by which the top-K set and its order are decided) and the logits."""
    xh, _ = oracle.rmsnorm(x_bits, blk["gamma"], blk["shape"].rms_eps)
    lg = oracle.router_logits(xh, blk["router_w"], blk["router_b"])
    top = np.sort(lg)[::-1][:K + 1]
    return float(np.min(top[:-1] - top[1:])), lg


def test_stack_24_layers_16_tokens():
    """Every layer teacher-forced: the oracle is fed the GPU's own bf16 input of
    that layer (routing for all 16 tokens bit-exact, outputs of sampled tokens
    within tolerance).  End to end, the oracle's own chain for four tokens
    through all 24 layers against the GPU's chain: equal routes give outputs
    within the accumulated tolerance; where the chains' routes part, the two
    inputs of that layer must still agree within the accumulated tolerance and
    the oracle's routing margin must be smaller than the logit change the
    input difference causes (a near tie decided the other way, not an error)."""
    import torch
    cfg, T = 2, 16
    wl = synth.WORKLOADS[cfg]
    shape, H, K = wl.shape, wl.shape.hidden, wl.shape.top_k
    x0 = synth.make_tokens(cfg, T, H)
    x = torch.from_numpy(x0.view(np.int16)).cuda()
    tf = np.array([0, 7, 13])             # teacher-forced sample
    ch = np.array([2, 5, 10, 15])         # tokens of the oracle's own chain
    xr = np.ascontiguousarray(x0[ch])
    parted = {}                           # chain token -> layer where the routes parted
    for layer in range(wl.layers):
        blk = synth.make_block(cfg, layer=layer)
        plan = moe.Plan(shape, max_tokens=T).alloc_workspace().load_weights(moe.DeviceBlock(blk))
        assert plan.path_for(T) == 1      # the benchmark's GEMV path (16-route tiles)
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        plan.forward(x, out, ids)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        xin = x.cpu().numpy().view(np.uint16)
        gids = ids.cpu().numpy()
        want_ids, _, _ = oracle_routes(blk, xin)
        assert np.array_equal(gids, want_ids), f"layer {layer}: expert ids"
        # one oracle call: the teacher-forced rows and the chain rows
        both = np.ascontiguousarray(np.concatenate([xin[tf], xr]))
        ref = oracle.moe_forward(blk, both, nthreads=NTHREADS)
        got = out.cpu().numpy()
        check_close(got[tf], ref["out"][:len(tf)], xin[tf], what=f"layer {layer} (teacher-forced)")
        for i, t in enumerate(ch):
            if t in parted or np.array_equal(ref["ids"][len(tf) + i], gids[t]):
                continue
            a = synth.bf16_bits_to_f32(xr[i]).astype(np.float64)
            b = synth.bf16_bits_to_f32(xin[t]).astype(np.float64)
            rel_in = np.linalg.norm(a - b) / np.linalg.norm(a)
            assert rel_in < wl.layers * 1e-3, (layer, t, rel_in)
            margin, lo = _route_margin(blk, xr[i], K)
            _, lg = _route_margin(blk, xin[t], K)
            assert margin <= 2 * np.abs(lo - lg).max(), (layer, t, margin, np.abs(lo - lg).max())
            parted[t] = layer
        xr = synth.f32_to_bf16_bits(ref["out"][len(tf):])
        nxt = torch.empty((T, H), dtype=torch.int16, device="cuda")
        moe.cast_f32_to_bf16(out, nxt)
        x = nxt
        plan.close()
        del blk
    torch.cuda.synchronize()
    got = x.cpu().numpy().view(np.uint16)[ch]
    g = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = (xr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # end to end each layer adds its own rounding differences on top of what it
    # inherits; a route chosen differently would show as an error orders of
    # magnitude above this
    for i, t in enumerate(ch):
        if t in parted:
            continue
        rel = np.linalg.norm(g[i] - r[i]) / np.linalg.norm(r[i])
        assert rel < wl.layers * 1e-3, (t, rel)
