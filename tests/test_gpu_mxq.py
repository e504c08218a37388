"""GPU parity of the FP4 activation encoding (moe_mx_quantize_fp4, through the
C-ABI) against the oracle: codes and E8M0 scales bit-exact, every byte.

The encoding decides integers (a code, an exponent) from floating point; both
sides take those decisions from exact quantities (|x| of bf16 values; the
exponent of amax / 6, from a float32 division in the oracle and from amax's
bits on the GPU, equal for every bf16 amax; a power-of-two scaling), so they
must agree bit for bit on every input, NaN and infinity included.
"""
import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import moe, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


def _f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _gpu(bits: np.ndarray):
    import torch
    rows, cols = bits.shape
    x = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    # pre-filled, so that a byte the kernel leaves unwritten shows
    codes = torch.full((rows * cols // 2,), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows * cols // 32,), 0xA5, dtype=torch.uint8, device="cuda")
    moe.mx_quantize_fp4(x, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy().reshape(rows, cols // 2), scales.cpu().numpy().reshape(rows, cols // 32)


def _check(bits: np.ndarray):
    got_c, got_s = _gpu(bits)
    ref_c, ref_s = oracle.mx_fp4_quantize(_f32(bits))
    bad = np.argwhere(got_s != ref_s)
    assert bad.size == 0, f"scales differ at {bad[:5].tolist()}"
    bad = np.argwhere(got_c != ref_c)
    assert bad.size == 0, f"codes differ at {bad[:5].tolist()}: {got_c[tuple(bad[0])]:#x} vs {ref_c[tuple(bad[0])]:#x}"


@pytest.mark.parametrize("order", ["sorted", "shuffled"])
def test_all_bf16_bit_patterns(order):
    """Every bf16 pattern: in order (blocks of subnormals only, of NaNs only, the
    infinities, runs across every exponent) and shuffled (mixed blocks)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if order == "shuffled":
        bits = np.random.default_rng(21).permutation(bits)
    _check(bits.reshape(32, 2048))


def _scaled_blocks(rng, rows, cols, lo, hi):
    x = rng.standard_normal((rows, cols))
    e = rng.integers(lo, hi, size=(rows, cols // 32))
    return synth.f32_to_bf16_bits((x * np.repeat(np.exp2(e.astype(np.float64)), 32, axis=1)).astype(np.float32))


@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 2880), (130, 4096), (257, 2048), (5, 32 * 129)])
def test_ragged_shapes_and_block_exponents(rows, cols):
    rng = np.random.default_rng(rows * 7919 + cols)
    _check(_scaled_blocks(rng, rows, cols, -135, 126))


def test_grid_midpoints_and_clamp():
    """Blocks whose largest element is exactly 6 * 2^k: every E2M1 midpoint (a
    tie) and grid point at that scale, both signs, and values just off them."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)
    rows = []
    for k in (-120, -3, 0, 1, 17, 100):
        s = 2.0 ** k
        for sign in (1.0, -1.0):
            blk = np.zeros(32)
            blk[:14] = sign * mids * s
            blk[14:28] = sign * (mids * s) * (1 + 2.0 ** -7)   # one bf16 ulp above
            blk[28] = 6.0 * s
            blk[29] = -6.0 * s * (1 - 2.0 ** -8)
            rows.append(blk)
    bits = synth.f32_to_bf16_bits(np.array(rows, np.float32))
    assert np.all(_f32(bits).astype(np.float64)[:, :14] == np.array(rows)[:, :14])   # ties are exact in bf16
    _check(bits)


def test_activation_sized_inputs():
    """The largest activations the expert projections take at the measured
    sizes: x_hat of 2048 tokens at hidden 4096, and h of 2048 tokens x 7
    routes at expert_hidden 2048."""
    rng = np.random.default_rng(23)
    xhat = synth.f32_to_bf16_bits((rng.standard_normal((2048, 4096)) * 1.1).astype(np.float32))
    _check(xhat)
    h = rng.standard_normal((2048 * 7, 2048)) * np.exp2(rng.integers(-6, 5, size=(2048 * 7, 1)))
    _check(synth.f32_to_bf16_bits(h.astype(np.float32)))


def test_arguments_and_empty_input():
    import torch
    x = torch.zeros((4, 64), dtype=torch.int16, device="cuda")
    codes = torch.zeros(4 * 32, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(4 * 2, dtype=torch.uint8, device="cuda")
    L = moe.load()
    import ctypes as C
    p = lambda t, off=0: C.c_void_p(t.data_ptr() + off)  # noqa: E731
    assert L.moe_mx_quantize_fp4(p(x), 0, 64, p(codes), p(scales), None) == moe.MOE_OK
    assert L.moe_mx_quantize_fp4(p(x), 4, 48, p(codes), p(scales), None) == moe.MOE_ESHAPE
    assert L.moe_mx_quantize_fp4(p(x), 4, 0, p(codes), p(scales), None) == moe.MOE_ESHAPE
    assert L.moe_mx_quantize_fp4(p(x, 2), 2, 32, p(codes), p(scales), None) == moe.MOE_EINVAL
    assert L.moe_mx_quantize_fp4(p(x), 2, 32, p(codes, 4), p(scales), None) == moe.MOE_EINVAL
    assert L.moe_mx_quantize_fp4(p(x), 4, 64, p(x, 64), p(scales), None) == moe.MOE_EINVAL   # overlap
    assert L.moe_mx_quantize_fp4(None, 4, 64, p(codes), p(scales), None) == moe.MOE_EINVAL
    assert L.moe_mx_quantize_fp4(p(x), 2 ** 62, 64, p(codes), p(scales), None) == moe.MOE_EINVAL
    torch.cuda.synchronize()
    assert codes.cpu().numpy().max() == 0 and scales.cpu().numpy().max() == 0   # nothing written
