"""GPU parity: the CUDA library (through the C-ABI) against the CPU oracle.

Bit-exact: MXFP4 dequantisation, x_hat, expert ids, per-expert counts and the
token->expert permutation.  Within tolerance (relative L2 <= 1e-3 and max abs
<= 2e-3 * max|ref|): the block output and the MoE delta.
"""
import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import (NTHREADS, check_close, check_permutation, oracle_routes, run_gpu, tiny_block)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


# ------------------------------------------------------------- dequantisation
def test_dequant_bitexact_all_codes_and_exponents():
    import torch
    # gate rows r = 0..252 carry E8M0 exponent r, each row holds all 16 codes twice
    shape = synth.tiny_shape(32, 256, 1, 1)
    blk = tiny_block(1, shape)
    nib = np.arange(32) % 16
    row = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    blk["codes"]["gate"][0] = row[None, :]
    sc = np.minimum(np.arange(256), 252).astype(np.uint8)
    blk["scales"]["gate"][0] = sc[:, None]
    dev = moe.DeviceBlock(blk)
    plan = moe.Plan(shape, max_tokens=1).alloc_workspace().load_weights(dev)
    out = torch.empty((256, 32), dtype=torch.float32, device="cuda")
    plan.debug_dequant(0, 0, out)
    torch.cuda.synchronize()
    want = oracle.mxfp4_dequant(blk["codes"]["gate"][0], blk["scales"]["gate"][0]).astype(np.float32)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("cfg", [0, 4])
def test_dequant_bitexact_workload_weights(cfg):
    import torch
    blk = synth.make_block(cfg)
    shape = blk["shape"]
    dev = moe.DeviceBlock(blk)
    plan = moe.Plan(shape, max_tokens=1).alloc_workspace().load_weights(dev)
    experts = [0, 5, shape.n_experts - 1] + ([shape.n_experts] if shape.n_shared else [])
    for e in experts:
        for which, m in enumerate(synth.MATS):
            rows, cols = shape.mat_shape(m)
            out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
            plan.debug_dequant(e, which, out)
            src = blk["shared"] if e == shape.n_experts else None
            codes = src["codes"][m][0] if src else blk["codes"][m][e]
            scales = src["scales"][m][0] if src else blk["scales"][m][e]
            want = oracle.mxfp4_dequant(codes, scales).astype(np.float32)
            assert np.array_equal(out.cpu().numpy(), want), (e, m)


# --------------------------------------------------------------------- routing
# 1300 / 1400 tokens: the large-batch routing configuration (8 tokens per CTA)
@pytest.mark.parametrize("cfg,T", [(0, 1), (1, 8), (3, 128), (4, 40), (3, 1300), (4, 1400)])
def test_routing_bitexact(cfg, T):
    blk = synth.make_block(cfg)
    x = synth.make_tokens(cfg, T, blk["shape"].hidden)
    r, plan, _ = run_gpu(blk, x)
    ids, rw, xh = oracle_routes(blk, x)
    assert r["status"] == 0
    assert np.array_equal(r["xhat"], xh)
    assert np.array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["route_w"], rw, rtol=2e-6, atol=1e-7)
    check_permutation(r, ids, blk["shape"])


def test_router_exact_mode_gives_same_routes():
    blk = synth.make_block(3)
    x = synth.make_tokens(3, 64, 2880)
    a, _, dev = run_gpu(blk, x)
    b, _, _ = run_gpu(blk, x, dev=dev, router_exact=1)
    assert np.array_equal(a["ids"], b["ids"])
    np.testing.assert_allclose(a["route_w"], b["route_w"], rtol=2e-6)


@pytest.mark.parametrize("T", [33, 1300])
def test_routing_near_ties_are_resolved_exactly(T):
    # two router rows identical except one tiny bf16 step: fp32 cannot order them
    # reliably, the certified path must fall back to exact logits
    shape = synth.tiny_shape(256, 64, 8, 2)
    blk = tiny_block(3, shape)
    blk["router_w"][1] = blk["router_w"][0]
    blk["router_w"][1, 7] ^= 1
    blk["router_b"][:] = 0
    blk["router_b"][[0, 1]] = 5.0
    x = synth.make_tokens(3, T, 256)
    r, _, _ = run_gpu(blk, x)
    ids, _, _ = oracle_routes(blk, x)
    assert np.array_equal(r["ids"], ids)


# ------------------------------------------------------------------ full block
@pytest.mark.parametrize("H,F,E,K,T,ns,scale,path", [
    (64, 96, 5, 3, 1, 0, 1.0, 0), (64, 96, 5, 3, 3, 0, 1.0, 0), (96, 64, 5, 3, 9, 0, 1.0, 0),
    (64, 96, 5, 3, 17, 1, 1.5, 0), (128, 64, 8, 2, 33, 0, 1.0, 0), (32, 32, 4, 2, 40, 1, 2.5, 0),
    (64, 64, 1, 1, 5, 0, 1.0, 0), (160, 96, 16, 8, 12, 0, 1.0, 0),
    # the grouped GEMM on ragged token counts, several route tiles, the shared expert
    (128, 64, 8, 2, 33, 0, 1.0, 2), (64, 128, 6, 2, 50, 1, 1.5, 2), (128, 192, 5, 3, 70, 0, 1.0, 2),
    (192, 320, 3, 2, 200, 0, 1.0, 2)])
def test_block_parity_ragged_shapes(H, F, E, K, T, ns, scale, path):
    shape = synth.tiny_shape(H, F, E, K, n_shared=ns, weight_scale=scale)
    blk = tiny_block(H * 7 + T, shape)
    x = synth.f32_to_bf16_bits(np.random.default_rng(T).normal(0, 1, (T, H)))
    r, _, _ = run_gpu(blk, x, path=path)
    ref = oracle.moe_forward(blk, x, nthreads=NTHREADS)
    assert r["status"] == 0
    assert np.array_equal(r["ids"], ref["ids"])
    check_close(r["out"], ref["out"], x)


@pytest.mark.parametrize("cfg,T", [(0, 1), (1, 8), (4, 1)])
def test_block_parity_workloads(cfg, T):
    blk = synth.make_block(cfg)
    x = synth.make_tokens(cfg, T, blk["shape"].hidden)
    r, _, _ = run_gpu(blk, x)
    ref = oracle.moe_forward(blk, x, nthreads=NTHREADS)
    assert np.array_equal(r["ids"], ref["ids"])
    check_close(r["out"], ref["out"], x)


@pytest.mark.parametrize("cfg,T,n_sample", [(3, 128, 12), (4, 64, 6)])
def test_block_parity_sampled_tokens(cfg, T, n_sample):
    blk = synth.make_block(cfg)
    x = synth.make_tokens(cfg, T, blk["shape"].hidden)
    r, _, _ = run_gpu(blk, x)
    sample = np.random.default_rng(cfg).choice(T, n_sample, replace=False)
    ref = oracle.moe_forward(blk, np.ascontiguousarray(x[sample]), nthreads=NTHREADS)
    assert np.array_equal(r["ids"][sample], ref["ids"])
    check_close(r["out"][sample], ref["out"], x[sample])


def test_edge_token_counts():
    import torch
    shape = synth.tiny_shape(64, 64, 4, 2)
    blk = tiny_block(5, shape)
    plan = moe.Plan(shape, max_tokens=4).alloc_workspace().load_weights(moe.DeviceBlock(blk))
    x = torch.zeros((5, 64), dtype=torch.int16, device="cuda")
    out = torch.empty((5, 64), dtype=torch.float32, device="cuda")
    plan.forward(x[:0], out[:0])                     # empty batch: no-op
    with pytest.raises(moe.MoeError) as ei:
        plan.forward(x, out)                         # above max_tokens
    assert ei.value.status == moe.MOE_ENOMEM
    with pytest.raises(moe.MoeError):
        plan.forward(x[:2], x[:2].view(torch.float32).view(2, 32))  # x aliases out
    assert plan.device_status() == 0


def test_misaligned_or_overlapping_outputs_rejected_before_launch():
    """ids / route weights are written with 4-byte stores and x_hat with 16-byte
    stores: misaligned output pointers are refused on the host, nothing runs."""
    import ctypes as C
    import torch
    shape = synth.tiny_shape(64, 64, 4, 2)
    blk = tiny_block(6, shape)
    plan = moe.Plan(shape, max_tokens=4).alloc_workspace().load_weights(moe.DeviceBlock(blk))
    x = torch.zeros((2, 64), dtype=torch.int16, device="cuda")
    out = torch.empty((2, 64), dtype=torch.float32, device="cuda")
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    P = lambda t, off=0: C.c_void_p(t.data_ptr() + off)  # noqa: E731
    L, h, N = plan.L, plan.h, None
    assert L.moe_forward_ex(h, P(x), 2, P(out), P(buf, 2), N, N, N) == moe.MOE_EINVAL
    assert L.moe_forward_ex(h, P(x), 2, P(out), N, P(buf, 6), N, N) == moe.MOE_EINVAL
    assert L.moe_forward_ex(h, P(x), 2, P(out), N, N, P(buf, 8), N) == moe.MOE_EINVAL
    assert L.moe_forward_ex(h, P(x), 2, P(out), N, N, P(x, 16), N) == moe.MOE_EINVAL   # x_hat over x
    assert L.moe_forward_noalloc(h, P(x), 2, P(out), P(buf, 1), N) == moe.MOE_EINVAL
    assert L.moe_debug_dequant(h, 0, 0, P(buf, 2), N) == moe.MOE_EINVAL
    torch.cuda.synchronize()
    assert int(buf.sum()) == 0 and plan.device_status() == 0
    plan.forward_ex(x, out, ids=torch.empty((2, 2), dtype=torch.int32, device="cuda"),
                    route_w=torch.empty((2, 2), dtype=torch.float32, device="cuda"),
                    xhat=torch.empty((2, 64), dtype=torch.int16, device="cuda"))
    torch.cuda.synchronize()
    assert plan.device_status() == 0


def test_nan_scale_rejected_at_load():
    shape = synth.tiny_shape(64, 64, 4, 2)
    blk = tiny_block(6, shape)
    blk["scales"]["down"][2, 5, 1] = 0xFF
    plan = moe.Plan(shape, max_tokens=4).alloc_workspace()
    with pytest.raises(moe.MoeError) as ei:
        plan.load_weights(moe.DeviceBlock(blk))
    assert ei.value.status == moe.MOE_EINVAL


def test_repeated_forward_is_deterministic():
    blk = synth.make_block(1)
    x = synth.make_tokens(1, 8, 2880)
    a, plan, dev = run_gpu(blk, x)
    b, _, _ = run_gpu(blk, x, plan=plan, dev=dev)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["ids"], b["ids"])


@pytest.mark.parametrize("cfg,T", [(3, 48), (4, 24)])
def test_decode_and_prefill_paths_agree(cfg, T):
    blk = synth.make_block(cfg)
    x = synth.make_tokens(cfg, T, blk["shape"].hidden, sub=7)
    dev = moe.DeviceBlock(blk)
    a, _, _ = run_gpu(blk, x, dev=dev, path=1)
    b, _, _ = run_gpu(blk, x, dev=dev, path=2)
    assert a["status"] == 0 and b["status"] == 0
    assert np.array_equal(a["ids"], b["ids"])
    check_close(b["out"], a["out"], what="prefill vs decode")
    sample = np.arange(0, T, max(1, T // 4))
    ref = oracle.moe_forward(blk, np.ascontiguousarray(x[sample]), nthreads=NTHREADS)
    check_close(b["out"][sample], ref["out"], x[sample], what="prefill vs oracle")
    check_close(a["out"][sample], ref["out"], x[sample], what="decode vs oracle")


@pytest.mark.parametrize("H,F,gamma_mul,limit,T", [
    (96, 64, 8000.0, 7.0, 5),      # |x_hat| beyond fp16: bf16 gate/up GEMV
    (96, 64, 1.0, 300.0, 9),       # |h| beyond fp16: bf16 down GEMV
    (128, 128, 8000.0, 300.0, 12)])
def test_block_parity_bf16_activation_gemvs(H, F, gamma_mul, limit, T):
    # activations that can leave the fp16 range switch the decode GEMVs to bf16 operands
    shape = synth.tiny_shape(H, F, 4, 2, swiglu_limit=limit)
    blk = tiny_block(H + T, shape)
    blk["gamma"] = (blk["gamma"] * np.float32(gamma_mul)).astype(np.float32)
    x = synth.f32_to_bf16_bits(np.random.default_rng(T).normal(0, 1, (T, H)))
    r, _, _ = run_gpu(blk, x, path=1)
    ref = oracle.moe_forward(blk, x, nthreads=NTHREADS)
    assert r["status"] == 0
    assert np.array_equal(r["ids"], ref["ids"])
    check_close(r["out"], ref["out"], x)


@pytest.mark.parametrize("elo,ehi", [(118, 124), (90, 150)])
def test_grouped_gemm_fp16_and_bf16_variants(elo, ehi):
    # exponents inside [104, 140] take the fp16-operand grouped GEMM, wider ones the bf16 one
    shape = synth.tiny_shape(128, 192, 6, 2)
    blk = tiny_block(elo, shape, elo=elo, ehi=ehi)
    x = synth.f32_to_bf16_bits(np.random.default_rng(elo).normal(0, 1, (45, 128)))
    r, _, _ = run_gpu(blk, x, path=2)
    ref = oracle.moe_forward(blk, x, nthreads=NTHREADS)
    assert r["status"] == 0
    assert np.array_equal(r["ids"], ref["ids"])
    check_close(r["out"], ref["out"], x)


# ------------------------------------------------------------ stacked blocks
def test_cast_f32_to_bf16_matches_round_to_nearest_even():
    import torch
    rng = np.random.default_rng(11)
    v = rng.normal(0, 3, 4099).astype(np.float32)
    # exact halfway cases (ties to even), both parities, signs, large and tiny values
    v[:8] = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3.0e38, -3.0e38, 1e-40, -1e-40, 0.0], np.float32)
    src = torch.from_numpy(v).cuda()
    dst = torch.empty(v.size, dtype=torch.int16, device="cuda")
    moe.cast_f32_to_bf16(src, dst)
    got = dst.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, synth.f32_to_bf16_bits(v))
    nan = torch.full((5,), float("nan"), device="cuda")
    out = torch.empty(5, dtype=torch.int16, device="cuda")
    moe.cast_f32_to_bf16(nan, out)
    b = out.cpu().numpy().view(np.uint16)
    assert np.all((b & 0x7F80) == 0x7F80) and np.all(b & 0x7F)


def test_stacked_blocks_residual_chain():
    """Config 2's chain: layer l's fp32 output, cast to bf16, is layer l+1's
    input.  Each layer is checked against the oracle fed the GPU's own input
    (teacher-forced), and the last output against the oracle's own chain."""
    import torch
    cfg, T, n_layers = 2, 4, 4
    shape = synth.WORKLOADS[cfg].shape
    H = shape.hidden
    x0 = synth.make_tokens(cfg, T, H)
    x = torch.from_numpy(x0.view(np.int16)).cuda()
    xr = x0
    for layer in range(n_layers):
        blk = synth.make_block(cfg, layer=layer)
        plan = moe.Plan(shape, max_tokens=T).alloc_workspace().load_weights(moe.DeviceBlock(blk))
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        plan.forward(x, out)
        torch.cuda.synchronize()
        xin = x.cpu().numpy().view(np.uint16)
        ref = oracle.moe_forward(blk, xin, nthreads=NTHREADS)
        check_close(out.cpu().numpy(), ref["out"], xin, what="layer %d (teacher-forced)" % layer)
        xr = synth.f32_to_bf16_bits(oracle.moe_forward(blk, xr, nthreads=NTHREADS)["out"])
        nxt = torch.empty((T, H), dtype=torch.int16, device="cuda")
        moe.cast_f32_to_bf16(out, nxt)
        x = nxt
        plan.close()
    torch.cuda.synchronize()
    got = x.cpu().numpy().view(np.uint16)
    # end to end: each layer adds its own rounding differences (within the
    # per-block 1e-3) on top of what it inherits, so the chains may drift apart
    # by up to about n_layers x 1e-3; a route chosen differently would show up
    # as an error orders of magnitude larger
    g = (got.astype(np.uint32) << 16).view(np.float32)
    r = (xr.astype(np.uint32) << 16).view(np.float32)
    rel = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert rel < n_layers * 1e-3, rel


# ------------------------------------------------------- device-side failure
def test_bounded_wait_timeout_is_reported_and_the_plan_recovers():
    """The test hook makes the decode gate/up kernel's consumer warps wait on a
    barrier nothing completes: a bounded wait (about 2 s) runs out -- theirs
    (detail 59) or the epilogue warp's wait for their partial sums (detail 54),
    whichever limit expires first -- the kernel records MOE_DEV_WAIT_TIMEOUT,
    lets the copies it issued land and exits; the host reads the status (and
    clears it) and the next forward is correct."""
    import torch
    blk = synth.make_block(1)
    x_bits = synth.make_tokens(1, 8, 2880)
    ref, plan, dev = run_gpu(blk, x_bits)
    assert ref["status"] == 0
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    out = torch.empty((8, 2880), dtype=torch.float32, device="cuda")
    ids = torch.empty((8, 4), dtype=torch.int32, device="cuda")
    plan.set_i("test_stall_wait", 1)
    plan.forward(x, out, ids)
    torch.cuda.synchronize()
    assert plan.device_status() == 1            # MOE_DEV_WAIT_TIMEOUT
    msg = moe.load().moe_last_error()
    assert b"detail 59" in msg or b"detail 54" in msg, msg
    assert plan.device_status() == 0            # cleared by the read
    plan.set_i("test_stall_wait", 0)
    again, _, _ = run_gpu(blk, x_bits, plan=plan, dev=dev)
    assert again["status"] == 0
    assert np.array_equal(again["ids"], ref["ids"]) and np.array_equal(again["out"], ref["out"])


# ------------------------------------------------------------ bf16 output
@pytest.mark.parametrize("cfg,T", [(1, 8), (3, 128)])
def test_out_bf16_is_the_rounded_fp32_output(cfg, T):
    """With the out_bf16 option the forward writes x + MoE(x) rounded to bf16:
    bit for bit what moe_cast_f32_to_bf16 makes of the fp32 output (GEMV and
    grouped-GEMM paths), and the no-alloc forward does the same."""
    import torch
    blk = synth.make_block(cfg)
    shape = blk["shape"]
    H = shape.hidden
    x_bits = synth.make_tokens(cfg, T, H)
    ref, plan, dev = run_gpu(blk, x_bits)
    want = torch.empty((T, H), dtype=torch.int16, device="cuda")
    moe.cast_f32_to_bf16(torch.from_numpy(ref["out"]).cuda(), want)
    p16 = moe.Plan(shape, max_tokens=T, out_bf16=1).alloc_workspace().load_weights(dev)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    got = torch.empty((T, H), dtype=torch.int16, device="cuda")
    p16.forward(x, got)
    torch.cuda.synchronize()
    assert p16.device_status() == 0
    assert torch.equal(got, want)
    got.zero_()
    L = moe.load()
    import ctypes as C
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.moe_forward_noalloc(p16.h, C.c_void_p(x.data_ptr()), T, C.c_void_p(got.data_ptr()), None,
                                 st) == moe.MOE_OK
    torch.cuda.synchronize()
    assert p16.device_status() == 0
    assert torch.equal(got, want)
    p16.close()
