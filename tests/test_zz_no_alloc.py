"""The allocation-free forward (moe_forward_noalloc) against moe_forward.

moe_forward_noalloc serves callers that may not allocate device memory: it
runs the same kernels on a static device scratch array instead of a
caller-provided workspace.  Two calls in a row must match moe_forward within
the block's output tolerance (the array keeps the previous call's contents, so
the second call checks that everything that must start at zero is cleared).
This file is named so that pytest collects it last.
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


def _forward_both(blk, x_bits, **opts):
    import torch
    shape = blk["shape"]
    T, H, K = x_bits.shape[0], shape.hidden, shape.top_k
    plan = moe.Plan(shape, max_tokens=T, **opts).alloc_workspace().load_weights(moe.DeviceBlock(blk))
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    out_ref = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids_ref = torch.empty((T, K), dtype=torch.int32, device="cuda")
    plan.forward(x, out_ref, ids_ref)
    L = moe.load()
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    results = []
    for _ in range(2):
        out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        ids = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
        rc = L.moe_forward_noalloc(plan.h, C.c_void_p(x.data_ptr()), T, C.c_void_p(out.data_ptr()),
                                   C.c_void_p(ids.data_ptr()), st)
        assert rc == moe.MOE_OK, L.moe_last_error().decode()
        torch.cuda.synchronize()
        results.append((out.cpu().numpy(), ids.cpu().numpy()))
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
    # a token count whose workspace exceeds the static array is refused before any launch
    big = 1 << 20
    L = moe.load()
    rc = L.moe_forward_noalloc(plan.h, C.c_void_p(256), big, C.c_void_p(1 << 40), None, None)
    assert rc == moe.MOE_ENOMEM
    assert b"static array" in L.moe_last_error()
    torch.cuda.synchronize()
