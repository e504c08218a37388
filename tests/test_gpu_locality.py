"""GPU expert-locality profiler (moe_locality_*) against the oracle's plain
restatement of the ds4.c expert locality profiler (oracle/locality.py):
counts, record counts, adjacent pairs and cache hits bit-exact; the weight
totals (per expert and of the cache hits, summed on the device in another
order than the page's) and the overlap sums to 1e-12 relative."""
import numpy as np
import pytest

from oracle.locality import Locality as OracleLocality
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


def _compare(got, ref: OracleLocality):
    L = ref.L
    assert np.array_equal(got["hist"], np.array(ref.hist, np.uint64))
    np.testing.assert_allclose(got["weight_hist"], np.array(ref.weight_hist), rtol=1e-12, atol=0)
    assert np.array_equal(got["layer_records"], np.array(ref.layer_records, np.uint64))
    assert np.array_equal(got["adjacent_pairs"], np.array(ref.adjacent_pairs, np.uint64))
    np.testing.assert_allclose(got["overlap_sum"], np.array(ref.adjacent_overlap_sum), rtol=1e-12, atol=0)
    np.testing.assert_allclose(got["jaccard_sum"], np.array(ref.adjacent_jaccard_sum), rtol=1e-12, atol=0)
    assert list(got["caps"]) == ref.caps
    assert np.array_equal(got["cache_hits"], np.array(ref.cache_hits, np.uint64).reshape(len(ref.caps), L))
    np.testing.assert_allclose(got["cache_weight_hits"],
                               np.array(ref.cache_weight_hits, np.float64).reshape(len(ref.caps), L),
                               rtol=1e-12, atol=0)


def _trace(rng, T, E, k, invalid=0.0):
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    if invalid:
        bad = rng.random(ids.shape) < invalid
        ids[bad] = rng.choice([-1, E, E + 5], bad.sum())
    w = rng.random((T, k)).astype(np.float32)
    return ids, w


@pytest.mark.parametrize("E,k,caps", [(32, 4, [1, 2, 4, 8, 16, 32, 40]), (256, 6, [6, 8, 32, 64, 128, 256]),
                                      (8, 2, [1, 3, 8])])
def test_random_traces_match_the_oracle(E, k, caps):
    """Three layers, several batches each: consecutive positions, a gap, a
    one-token batch, experts outside [0, E) mixed in."""
    import torch
    rng = np.random.default_rng(E + k)
    prof = moe.Locality(3, E, k, caps)
    ref = OracleLocality(3, E, k, caps)
    for layer, first_pos, T in [(0, 0, 17), (0, 17, 40), (1, 0, 5), (0, 60, 33), (2, 100, 1), (2, 101, 64),
                                (1, 5, 128), (0, 93, 2)]:
        ids, w = _trace(rng, T, E, k, invalid=0.03)
        prof.record(layer, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), first_pos)
        ref.record_batch(layer, first_pos, ids, w)
    _compare(prof.read(), ref)
    prof.reset()
    got = prof.read()
    assert got["hist"].sum() == 0 and got["cache_hits"].sum() == 0 and got["adjacent_pairs"].sum() == 0
    prof.close()


def test_large_batch_matches_the_oracle():
    """2048 tokens x 6 slots over 256 experts in one record (the cache pass
    runs 12 288 dependent steps), Zipf-skewed like the DeepSeek-shaped
    workload's routing."""
    import torch
    E, k, T = 256, 6, 2048
    rng = np.random.default_rng(11)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    perm = rng.permutation(E)
    ids = np.stack([perm[rng.choice(E, k, replace=False, p=p)] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    caps = [8, 16, 32, 64, 128]
    prof = moe.Locality(1, E, k, caps)
    ref = OracleLocality(1, E, k, caps)
    prof.record(0, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), 0)
    ref.record_batch(0, 0, ids, w)
    _compare(prof.read(), ref)
    prof.close()


def test_attached_profiler_records_every_forward():
    """Attached to a plan, the profiler records each forward's routes (the
    ids and route weights the forward returns) at positions that continue
    from one forward to the next, on the GEMV and the grouped-GEMM paths."""
    import torch
    for cfg, T in [(1, 8), (3, 70)]:
        blk = synth.make_block(cfg)
        sh = blk["shape"]
        caps = [2, 4, 8, 16]
        prof = moe.Locality(2, sh.n_experts, sh.top_k, caps)
        ref = OracleLocality(2, sh.n_experts, sh.top_k, caps)
        plan = None
        dev = None
        pos = 0
        for step in range(3):
            x = synth.make_tokens(cfg, T, sh.hidden, sub=step)
            if plan is None:
                r, plan, dev = run_gpu(blk, x)
                prof.attach(plan, 1)
                r, _, _ = run_gpu(blk, x, plan=plan, dev=dev)
            else:
                r, _, _ = run_gpu(blk, x, plan=plan, dev=dev)
            ref.record_batch(1, pos, r["ids"], r["route_w"])
            pos += T
        _compare(prof.read(), ref)
        assert prof.read()["layer_records"][1] == 3 * T
        plan.close()
        prof.close()
