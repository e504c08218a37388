"""Host-side checks of the C-ABI library (no GPU needed).

The library must build for sm_103a, load, export every function that
include/moe.h declares, and reject bad arguments with the documented status
codes before touching the device.
"""
import ctypes as C
import os
import re

import pytest

from mxfp4_mixture_experts_rms_gb300 import build, moe, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.load()


def test_library_exports_every_declared_function(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.EXPORTS)


def test_plan_create_rejects_bad_shapes(L):
    bad = [(30, 64, 4, 2), (64, 0, 4, 2), (64, 64, 0, 1), (64, 64, 4, 5), (64, 64, 300, 4), (64, 64, 16, 9)]
    for H, F, E, K in bad:
        assert not L.moe_plan_create(H, F, E, K, 1.702, 7.0, 1.0)
        assert L.moe_last_error()
    assert not L.moe_plan_create(64, 64, 4, 2, 1.702, 0.0, 1.0)


def test_options_and_workspace_sizing(L):
    h = L.moe_plan_create(2880, 2880, 32, 4, 1.702, 7.0, 1.0)
    assert h
    h = C.c_void_p(h)
    assert L.moe_plan_set_i(h, b"n_shared_experts", 2) == moe.MOE_EINVAL
    assert L.moe_plan_set_i(h, b"no_such_key", 1) == moe.MOE_EINVAL
    assert L.moe_plan_set_f(h, b"rms_eps", -1.0) == moe.MOE_EINVAL
    assert L.moe_plan_set_i(h, b"max_tokens", 65536) == moe.MOE_EINVAL   # one combine grid row per token
    assert L.moe_plan_set_i(h, b"max_tokens", 0) == moe.MOE_EINVAL
    assert L.moe_plan_set_i(h, b"max_tokens", 8) == moe.MOE_OK
    small = L.moe_workspace_bytes(h, 0)
    assert L.moe_plan_set_i(h, b"max_tokens", 512) == moe.MOE_OK
    big = L.moe_workspace_bytes(h, 0)
    assert 0 < small < big
    # the per-route fp32 outputs dominate: T*K*H*4 bytes
    assert big >= 512 * 4 * 2880 * 4
    L.moe_plan_destroy(h)


def test_forward_before_weights_is_not_ready(L):
    h = C.c_void_p(L.moe_plan_create(64, 64, 4, 2, 1.702, 7.0, 1.0))
    rc = L.moe_forward(h, C.c_void_p(256), 1, C.c_void_p(4096), None, None)
    assert rc == moe.MOE_ENOTREADY
    assert b"moe_load_weights" in L.moe_last_error()
    assert L.moe_forward(h, C.c_void_p(256), -1, C.c_void_p(4096), None, None) == moe.MOE_EINVAL
    assert L.moe_forward(h, None, 0, None, None, None) == moe.MOE_OK   # empty batch: no-op
    assert L.moe_load_weights(h, None) == moe.MOE_EINVAL
    w = moe.Weights()
    assert L.moe_load_weights(h, C.byref(w)) == moe.MOE_EINVAL       # NULL pointers
    w.gamma = w.router_w = w.router_b = 0x1001                        # misaligned
    assert L.moe_load_weights(h, C.byref(w)) == moe.MOE_EINVAL
    assert L.moe_set_workspace(h, C.c_void_p(0x1008), 1 << 20) == moe.MOE_EINVAL  # misaligned
    assert L.moe_debug_dequant(h, 0, 0, C.c_void_p(256), None) == moe.MOE_ENOTREADY
    # neither a workspace nor a no-alloc call: there is no status word to read
    st = C.c_int(7)
    assert L.moe_get_device_status(h, C.byref(st), None) == moe.MOE_ENOTREADY
    assert L.moe_forward_noalloc(h, C.c_void_p(256), 1, C.c_void_p(4096), None, None) == moe.MOE_ENOTREADY
    assert L.moe_plan_set_i(h, b"test_stall_wait", 1) == moe.MOE_OK
    assert L.moe_plan_set_i(h, b"test_stall_wait", 0) == moe.MOE_OK
    assert L.moe_plan_set_i(h, b"out_bf16", 1) == moe.MOE_OK      # out written as bf16
    assert L.moe_plan_set_i(h, b"out_bf16", 0) == moe.MOE_OK
    # the expert cache: 0 (off) .. n_experts slots; its state only once loaded
    assert L.moe_plan_set_i(h, b"expert_cache_slots", -1) == moe.MOE_EINVAL
    assert L.moe_plan_set_i(h, b"expert_cache_slots", 5) == moe.MOE_EINVAL   # 4 experts
    assert L.moe_plan_set_i(h, b"expert_cache_slots", 4) == moe.MOE_OK
    stats = (C.c_longlong * 3)()
    assert L.moe_get_cache_state(h, None, stats, None) == moe.MOE_ENOTREADY
    assert L.moe_plan_set_i(h, b"expert_cache_slots", 0) == moe.MOE_OK
    assert L.moe_get_cache_state(None, None, None, None) == moe.MOE_EINVAL
    L.moe_plan_destroy(h)


def test_token_counts_above_the_grid_limit_are_refused(L):
    h = C.c_void_p(L.moe_plan_create(64, 64, 4, 2, 1.702, 7.0, 1.0))
    assert L.moe_workspace_bytes(h, 65535) > 0
    assert L.moe_workspace_bytes(h, 65536) == 0          # the combine grid's y extent
    assert b"65535" in L.moe_last_error()
    assert L.moe_workspace_bytes(h, 2 ** 31 - 1) == 0
    L.moe_plan_destroy(h)


def test_generated_shapes_match_layout():
    blk = synth.make_block(0)
    assert blk["codes"]["gate"].shape == (32, 2880, 1440)
    assert blk["scales"]["down"].shape == (32, 2880, 90)
    assert synth.expert_bytes(synth.GPT_OSS) == 3 * (2880 * 1440 + 2880 * 90)


def test_standalone_ops_reject_bad_arguments_before_touching_the_device(L):
    """The encoder and the cast validate sizes, alignment and overlap on the
    host; these addresses are never dereferenced."""
    X, Cd, S = C.c_void_p(0x100000), C.c_void_p(0x200000), C.c_void_p(0x300000)
    assert L.moe_mx_quantize_fp4(X, 0, 64, Cd, S, None) == moe.MOE_OK           # empty: no-op
    assert L.moe_mx_quantize_fp4(X, 4, 48, Cd, S, None) == moe.MOE_ESHAPE
    assert L.moe_mx_quantize_fp4(X, 4, 0, Cd, S, None) == moe.MOE_ESHAPE
    assert L.moe_mx_quantize_fp4(None, 4, 64, Cd, S, None) == moe.MOE_EINVAL
    assert L.moe_mx_quantize_fp4(C.c_void_p(0x100008), 4, 64, Cd, S, None) == moe.MOE_EINVAL
    assert L.moe_mx_quantize_fp4(X, 4, 64, C.c_void_p(0x200004), S, None) == moe.MOE_EINVAL
    assert L.moe_mx_quantize_fp4(X, 4, 64, C.c_void_p(0x100100), S, None) == moe.MOE_EINVAL  # inside x
    assert L.moe_mx_quantize_fp4(X, 4, 64, Cd, C.c_void_p(0x200010), None) == moe.MOE_EINVAL  # inside codes
    assert L.moe_mx_quantize_fp4(X, 2 ** 62, 64, Cd, S, None) == moe.MOE_EINVAL
    assert b"overflow" in L.moe_last_error()
    assert L.moe_cast_f32_to_bf16(X, Cd, 0, None) == moe.MOE_OK
    assert L.moe_cast_f32_to_bf16(None, Cd, 16, None) == moe.MOE_EINVAL
    assert L.moe_cast_f32_to_bf16(C.c_void_p(0x100004), Cd, 16, None) == moe.MOE_EINVAL
    assert L.moe_cast_f32_to_bf16(X, C.c_void_p(0x100020), 16, None) == moe.MOE_EINVAL   # overlap


def test_binding_refuses_strided_tensors(L):
    torch = pytest.importorskip("torch")
    src = torch.zeros((8, 4), dtype=torch.float32).t()          # a transposed view
    dst = torch.zeros((4, 8), dtype=torch.int16)
    with pytest.raises(moe.MoeError) as ei:
        moe.cast_f32_to_bf16(src, dst)
    assert ei.value.status == moe.MOE_EINVAL


def test_locality_profiler_refuses_bad_arguments(L):
    """Refusals happen on the host before any device memory is touched."""
    import ctypes as C
    caps = (C.c_int * 2)(4, 8)
    assert not L.moe_locality_create(0, 32, 4, caps, 2)            # no layer
    assert b"bad arguments" in L.moe_last_error()
    assert not L.moe_locality_create(2, 300, 4, caps, 2)           # too many experts
    assert not L.moe_locality_create(2, 32, 9, caps, 2)            # top_k above 8
    assert not L.moe_locality_create(2, 4, 5, caps, 2)             # top_k above n_experts
    assert not L.moe_locality_create(2, 32, 4, None, 2)            # capacities missing
    assert not L.moe_locality_create(2, 32, 4, caps, 17)           # too many capacities
    assert L.moe_locality_record(None, 0, None, None, 1, 0, None) == moe.MOE_EINVAL
    assert L.moe_locality_attach(None, None, 0) == moe.MOE_EINVAL
    assert L.moe_locality_read(None, None) == moe.MOE_EINVAL
    assert L.moe_locality_reset(None, None) == moe.MOE_EINVAL
    L.moe_locality_destroy(None)                                    # no-op
