"""The allocation-free forward (moe_forward_noalloc) against moe_forward.

moe_forward_noalloc serves callers that may not allocate device memory: a
runtime that owns all device memory through its own pool, or code that must
not risk the implicit synchronisation an allocation can bring.  It runs the
same kernels on a static device scratch array instead of a caller-provided
workspace.  Two calls in a row must match moe_forward within the block's
output tolerance (the array keeps the previous call's contents, so the second
call checks that everything that must start at zero is cleared), the calls
must leave the device's free memory unchanged, and the kernels' status word
in the array must be readable through moe_get_device_status.  This file is
named so that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest

from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import check_close, tiny_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


def _noalloc(L, plan, x, out, ids):
    import torch
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.moe_forward_noalloc(plan.h, C.c_void_p(x.data_ptr()), int(x.shape[0]), C.c_void_p(out.data_ptr()),
                                 C.c_void_p(ids.data_ptr()) if ids is not None else None, st)


def _forward_both(blk, x_bits, **opts):
    import torch
    shape = blk["shape"]
    T, H, K = x_bits.shape[0], shape.hidden, shape.top_k
    dev = moe.DeviceBlock(blk)
    ref_plan = moe.Plan(shape, max_tokens=T, **opts).alloc_workspace().load_weights(dev)
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    out_ref = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids_ref = torch.empty((T, K), dtype=torch.int32, device="cuda")
    ref_plan.forward(x, out_ref, ids_ref)
    # the caller this entry point is for: weights loaded, no workspace ever set
    plan = moe.Plan(shape, max_tokens=T, **opts).load_weights(dev)
    L = moe.load()
    outs = [torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    idss = [torch.full((T, K), -1, dtype=torch.int32, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free0 = None
    results = []
    for i in range(2):
        rc = _noalloc(L, plan, x, outs[i], idss[i])
        assert rc == moe.MOE_OK, L.moe_last_error().decode()
        torch.cuda.synchronize()
        if i == 0:
            free0 = torch.cuda.mem_get_info()[0]   # after the first call resolved the array's address
        results.append((outs[i].cpu().numpy(), idss[i].cpu().numpy()))
    rc = _noalloc(L, plan, x, outs[1], idss[1])
    assert rc == moe.MOE_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "moe_forward_noalloc changed the device's free memory"
    # the status word of the calls above: the static array's, read through this plan
    assert plan.device_status() == 0
    return out_ref.cpu().numpy(), ids_ref.cpu().numpy(), results, plan


@pytest.mark.parametrize("cfg,T", [(1, 8), (0, 1)])
def test_noalloc_matches_forward_on_two_calls(cfg, T):
    blk = synth.make_block(cfg)
    x = synth.make_tokens(cfg, T, blk["shape"].hidden)
    out_ref, ids_ref, results, _ = _forward_both(blk, x)
    for out, ids in results:
        assert np.array_equal(ids, ids_ref)
        check_close(out, out_ref, what="noalloc vs forward")


def test_noalloc_prefill_path_and_size_limit():
    import torch
    shape = synth.tiny_shape(128, 64, 8, 2)
    blk = tiny_block(21, shape)
    x = synth.f32_to_bf16_bits(np.random.default_rng(21).normal(0, 1, (40, 128)))
    out_ref, ids_ref, results, plan = _forward_both(blk, x)
    for out, ids in results:
        assert np.array_equal(ids, ids_ref)
        check_close(out, out_ref, what="noalloc vs forward (grouped GEMM path)")
    # a token count whose workspace exceeds the static array, and one above the
    # grid limit, are refused on the host before any launch (these addresses
    # are never dereferenced)
    L = moe.load()
    rc = L.moe_forward_noalloc(plan.h, C.c_void_p(256), 60000, C.c_void_p(1 << 40), None, None)
    assert rc == moe.MOE_ENOMEM
    assert b"static array" in L.moe_last_error()
    rc = L.moe_forward_noalloc(plan.h, C.c_void_p(256), 1 << 20, C.c_void_p(1 << 40), None, None)
    assert rc == moe.MOE_ENOMEM
    torch.cuda.synchronize()
    assert plan.device_status() == 0


def test_noalloc_reports_a_device_side_wait_timeout():
    """A bounded wait that runs out inside a no-alloc forward (the test hook
    makes the gate/up GEMV wait on a barrier nothing completes) is reported by
    moe_get_device_status on the plan, from the static array's status word;
    reading it clears it and the next no-alloc forward is correct again."""
    import torch
    blk = synth.make_block(0)
    x_bits = synth.make_tokens(0, 2, 2880)
    out_ref, ids_ref, _, plan = _forward_both(blk, x_bits)
    L = moe.load()
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    out = torch.empty((2, 2880), dtype=torch.float32, device="cuda")
    ids = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    plan.set_i("test_stall_wait", 1)
    assert _noalloc(L, plan, x, out, ids) == moe.MOE_OK
    torch.cuda.synchronize()
    assert plan.device_status() == 1                  # MOE_DEV_WAIT_TIMEOUT
    msg = L.moe_last_error()
    # the consumers' stalled wait (59) or the epilogue's wait for them (54)
    assert (b"detail 59" in msg or b"detail 54" in msg) and b"noalloc" in msg, msg
    assert plan.device_status() == 0                  # read once, cleared
    plan.set_i("test_stall_wait", 0)
    assert _noalloc(L, plan, x, out, ids) == moe.MOE_OK
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    check_close(out.cpu().numpy(), out_ref, what="noalloc after a reported timeout")


def test_noalloc_through_the_expert_cache():
    """A plan with an expert cache (its store in pinned host memory) and no
    workspace runs the allocation-free forward too: the output of moe_forward
    on a plan with resident weights, bit for bit, and the cache counts it."""
    import torch
    L = moe.load()
    blk = synth.make_block(0)
    shape = blk["shape"]
    ref = moe.Plan(shape, max_tokens=2).alloc_workspace().load_weights(moe.DeviceBlock(blk))
    plan = moe.Plan(shape, max_tokens=2, expert_cache_slots=8)
    plan.load_weights(moe.HostStoreBlock(blk))
    x = torch.from_numpy(synth.make_tokens(0, 2, shape.hidden, sub=9).view(np.int16)).cuda()
    got = torch.empty((2, shape.hidden), dtype=torch.float32, device="cuda")
    want = torch.empty_like(got)
    ids = torch.empty((2, shape.top_k), dtype=torch.int32, device="cuda")
    assert _noalloc(L, plan, x, got, ids) == moe.MOE_OK
    ref.forward(x, want)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    _, hits, misses, fwds = plan.cache_state()
    assert (hits, fwds) == (0, 1) and misses == len(set(ids.cpu().numpy().ravel().tolist()))
    assert plan.device_status() == 0
    plan.close()
    ref.close()
