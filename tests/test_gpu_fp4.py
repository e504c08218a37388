"""GPU parity of the block-scaled FP4 grouped GEMM (plan option act_fp4:
tcgen05.mma kind::mxf4, activations FP4-encoded along the contracted
dimension, ds4.c FP4 activation quantisation) against the oracle's FP4
activation mode (x_hat before gate/up and h, after its bf16 rounding, before
down each pass through the same encoding).

Routing is untouched by the mode and stays bit-exact; the block output is held
to the block's tolerance (relative L2 <= 1e-3 and max abs <= 2e-3 * max|ref|):
products of E2M1 values are exact, so what remains is fp32 accumulation.
"""
import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import NTHREADS, check_close, run_gpu, tiny_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


# K stages of 256 with a short last stage (H = 192, F = 320), down row blocks of
# 128 with a partial last one, several 128-route tiles per expert, the shared
# expert, one token
@pytest.mark.parametrize("H,F,E,K,T,ns,scale", [
    (64, 64, 4, 2, 1, 0, 1.0), (128, 64, 8, 2, 33, 0, 1.0), (64, 128, 6, 2, 50, 1, 1.5),
    (192, 320, 5, 3, 70, 0, 1.0), (192, 320, 3, 2, 200, 0, 1.0), (256, 128, 4, 4, 300, 1, 2.5)])
def test_fp4_block_parity_ragged_shapes(H, F, E, K, T, ns, scale):
    shape = synth.tiny_shape(H, F, E, K, n_shared=ns, weight_scale=scale)
    blk = tiny_block(H * 3 + T, shape)
    x = synth.f32_to_bf16_bits(np.random.default_rng(T + 1).normal(0, 1, (T, H)))
    r, plan, _ = run_gpu(blk, x, act_fp4=1)
    assert plan.path_for(T) == 3
    ref = oracle.moe_forward(blk, x, nthreads=NTHREADS, act_fp4=True)
    assert r["status"] == 0
    assert np.array_equal(r["ids"], ref["ids"])
    check_close(r["out"], ref["out"], x, what="FP4 path")


def test_fp4_mode_differs_from_the_bf16_contract():
    """The FP4 path is the oracle's FP4 mode, not the bf16-activation block:
    against the bf16 oracle it is off by the FP4 encoding's error (well above
    the tolerance), so the parity above really checks the FP4 arithmetic."""
    shape = synth.tiny_shape(128, 128, 4, 2)
    blk = tiny_block(7, shape)
    x = synth.f32_to_bf16_bits(np.random.default_rng(7).normal(0, 1, (40, 128)))
    r, _, _ = run_gpu(blk, x, act_fp4=1)
    ref_bf16 = oracle.moe_forward(blk, x, nthreads=NTHREADS)
    d = r["out"] - ref_bf16["out"]
    x32 = synth.bf16_bits_to_f32(x)
    assert np.linalg.norm(d) / np.linalg.norm(ref_bf16["out"] - x32) > 1e-2


@pytest.mark.parametrize("cfg,T,n_sample", [(3, 512, 10), (4, 2048, 8)])
def test_fp4_block_parity_at_bench_size(cfg, T, n_sample):
    blk = synth.make_block(cfg)
    shape = blk["shape"]
    x = synth.make_tokens(cfg, T, shape.hidden)
    r, _, _ = run_gpu(blk, x, act_fp4=1)
    assert r["status"] == 0
    ids = r["ids"]
    hot = np.bincount(ids.ravel()).argmax()
    rng = np.random.default_rng(cfg)
    sample = np.union1d(rng.choice(T, n_sample, replace=False),
                        rng.choice(np.nonzero((ids == hot).any(axis=1))[0], 4, replace=False))
    ref = oracle.moe_forward(blk, np.ascontiguousarray(x[sample]), nthreads=NTHREADS, act_fp4=True)
    assert np.array_equal(ids[sample], ref["ids"])
    check_close(r["out"][sample], ref["out"], x[sample], what=f"FP4 path cfg{cfg} x{T}")
