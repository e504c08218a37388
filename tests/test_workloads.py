"""The seeded synthetic inputs follow their stated recipe.

Value distributions of the generated tensors, and the routing structure the
two skewed workloads are built to have, measured with the oracle's routing
steps (rms_norm, router logits, top-k, softmax): the hot-2 decode batch puts
about 60 % of the routing weight on two experts, and the DeepSeek-shaped
block's Zipf(1.1) prior concentrates routes on the experts it ranks first.
"""
import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import synth


def _route(blk, x):
    shape = blk["shape"]
    ids, ws = [], []
    for t in range(x.shape[0]):
        xh, _ = oracle.rmsnorm(x[t], blk["gamma"], shape.rms_eps)
        lg = oracle.router_logits(xh, blk["router_w"], blk["router_b"])
        i, v = oracle.topk(lg, shape.top_k)
        ids.append(i)
        ws.append(oracle.route_weights(v, shape.weight_scale))
    return np.array(ids), np.array(ws)


def test_router_generator_is_make_block_without_the_experts():
    shape = synth.BlockShape(64, 64, 8, 2)
    r, b = synth.make_router(1, layer=3, shape=shape), synth.make_block(1, layer=3, shape=shape)
    for k in ("gamma", "router_w", "router_b"):
        assert np.array_equal(r[k], b[k]), k


def test_value_recipes():
    shape = synth.BlockShape(256, 256, 4, 2)
    blk = synth.make_block(0, shape=shape)
    for m in synth.MATS:
        sc = blk["scales"][m].ravel()
        assert sc.min() == 118 and sc.max() == 124
        freq = np.bincount(sc, minlength=125)[118:] / sc.size
        assert np.all(np.abs(freq - 1 / 7) < 0.01)
        c = blk["codes"][m].ravel()
        for nib in (c & 15, c >> 4):
            assert np.all(np.abs(np.bincount(nib, minlength=16) / nib.size - 1 / 16) < 0.005)
        b = blk["bias"][m]
        assert abs(b.mean()) < 0.003 and abs(b.std() - 0.02) < 0.003
    g = blk["gamma"]
    assert abs(g.mean() - 1.0) < 0.02 and abs(g.std() - 0.1) < 0.02
    rw = synth.bf16_bits_to_f32(blk["router_w"])
    assert abs(rw.std() - 0.02) < 0.002
    rb = synth.router_bias(synth.GPT_OSS, "none", 0, 0)
    assert abs(rb.std() - 0.5) < 0.25
    x = synth.bf16_bits_to_f32(synth.make_tokens(0, 64, 2880)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01


def test_hot2_decode_batch_routes_about_60_percent_of_weight_to_two_experts():
    blk = synth.make_router(1)
    b = blk["router_b"]
    hot = np.argsort(b)[-2:]
    assert np.sort(b)[-2] - np.sort(b)[-3] > 1.0        # the two boosted biases stand apart
    ids, w = _route(blk, synth.make_tokens(1, 1024, synth.GPT_OSS.hidden))
    on_hot = np.isin(ids, hot)
    share = w[on_hot].sum() / w.sum()
    assert 0.55 < share < 0.68, share
    assert 0.35 < on_hot.mean() <= 0.5                    # two of four slots at most


def test_zipf_prior_concentrates_routes_on_its_first_ranks():
    from mxfp4_mixture_experts_rms_gb300.synth import DSV4_FLASH_SHAPE as S
    blk = synth.make_router(4)
    b = blk["router_b"].astype(np.float64)
    ranks = np.rint(np.exp(-b / 1.1)).astype(np.int64)   # the prior is -1.1 ln(rank)
    assert sorted(ranks.tolist()) == list(range(1, S.n_experts + 1))
    ids, w = _route(blk, synth.make_tokens(4, 128, S.hidden))
    np.testing.assert_allclose(w.sum(axis=1), S.weight_scale, rtol=1e-12)
    cnt = np.bincount(ids.ravel(), minlength=S.n_experts)
    order = np.argsort(ranks)
    assert cnt[order[:8]].sum() / cnt.sum() > 0.4         # 8 of 256 experts
    assert cnt[order[128:]].sum() / cnt.sum() < 0.05      # the lower half of the prior
    scipy_stats = pytest.importorskip("scipy.stats")
    assert scipy_stats.spearmanr(cnt, -ranks).correlation > 0.5
