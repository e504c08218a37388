"""Pins of the oracle's gpt-oss attention decode step (goosedump gpt_oss.rs
`Rope::new`, `apply_rope`, `causal_gqa`, `attention_head`, `forward`) against
facts that are not its own code: the YaRN correction dimensions and ramp at
the page's constants worked out by hand, rotation at position 0 and norm
preservation, a sink that vanishes or dominates, tokens outside the sliding
window that cannot matter, one visible token giving its value exactly,
query heads of one group reading the same keys, and a dense restatement of the
whole step with einsum over every head at once."""
import math

import numpy as np
import pytest

from oracle import attention as A
from mxfp4_mixture_experts_rms_gb300 import synth

D = 64


def test_yarn_correction_dimensions_and_ramp():
    """ln(4096 / (32 * 2 pi)) and ln(4096 / (2 pi)) over 2 ln(150000), times 64:
    the ramp runs between pairs 8.09.. and 17.40..; below it the frequency is
    150000^(-2p/64), above it that over 32."""
    low = 64 * math.log(4096 / (32 * 2 * math.pi)) / (2 * math.log(150000))
    high = 64 * math.log(4096 / (2 * math.pi)) / (2 * math.log(150000))
    assert low == pytest.approx(8.0928, abs=1e-3) and high == pytest.approx(17.398, abs=1e-3)
    assert A.correction_dimension(32.0, D) == pytest.approx(low, rel=1e-15)
    pos = 1000
    cos, sin = A.rope_tables(pos, D)
    af = 0.1 * math.log(32) + 1
    for p in (0, 3, 8):                     # ramp 0: the plain frequency
        ang = pos * 150000 ** (-2 * p / 64)
        assert cos[p] == pytest.approx(math.cos(ang) * af, abs=1e-12)
        assert sin[p] == pytest.approx(math.sin(ang) * af, abs=1e-12)
    for p in (18, 25, 31):                  # ramp 1: divided by the factor
        ang = pos * 150000 ** (-2 * p / 64) / 32
        assert cos[p] == pytest.approx(math.cos(ang) * af, abs=1e-12)
    p = 12                                  # inside the ramp: the linear blend
    r = (p - low) / (high - low)
    ang = pos * 150000 ** (-2 * p / 64) * (1 - r + r / 32)
    assert sin[p] == pytest.approx(math.sin(ang) * af, abs=1e-12)


def test_rope_at_zero_scales_and_rotation_keeps_norms():
    rng = np.random.default_rng(0)
    v = rng.normal(size=3 * D)
    af = 0.1 * math.log(32) + 1
    c0, s0 = A.rope_tables(0, D)
    assert np.allclose(A.apply_rope(v, c0, s0), af * v, rtol=0, atol=1e-15)
    c, s = A.rope_tables(12345, D)
    r = A.apply_rope(v, c, s).reshape(3, D)
    vv = v.reshape(3, D)
    # each (first-half, second-half) pair keeps its length times the attention factor
    assert np.allclose(np.hypot(r[:, :32], r[:, 32:]), af * np.hypot(vv[:, :32], vv[:, 32:]), rtol=1e-12)


def _weights(rng, H, QH, KVH, sink=0.0):
    def bf(shape, s):
        return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.normal(0, s, shape))).astype(np.float64)
    return dict(gamma=(1 + 0.1 * rng.normal(size=H)).astype(np.float32),
                wq=bf((QH * D, H), 0.05), bq=rng.normal(0, 0.02, QH * D).astype(np.float32).astype(np.float64),
                wk=bf((KVH * D, H), 0.05), bk=rng.normal(0, 0.02, KVH * D).astype(np.float32).astype(np.float64),
                wv=bf((KVH * D, H), 0.05), bv=rng.normal(0, 0.02, KVH * D).astype(np.float32).astype(np.float64),
                wo=bf((H, QH * D), 0.02), bo=rng.normal(0, 0.02, H).astype(np.float32).astype(np.float64),
                sinks=np.full(QH, sink))


def _step(wts, x, n_ctx, kc, vc, sliding=False, QH=8, KVH=2, window=128):
    return A.decode_step(wts, x, kc, vc, n_ctx, q_heads=QH, kv_heads=KVH, head_dim=D, sliding=sliding,
                         window=window, eps=1e-5)


def _cache(rng, n, KVH):
    kc = A.to_fp16(rng.normal(0, 1, (n + 1, KVH, D)))
    vc = A.to_fp16(rng.normal(0, 1, (n + 1, KVH, D)))
    return kc, vc


def test_one_visible_token_gives_its_value():
    """Empty cache and a sink at -inf: every head's output is the new token's
    own value row exactly."""
    rng = np.random.default_rng(1)
    H = 64
    wts = _weights(rng, H, 8, 2, sink=-np.inf)
    x = synth.f32_to_bf16_bits(rng.normal(size=H))
    kc, vc = _cache(rng, 0, 2)
    out, q, ob = _step(wts, x, 0, kc, vc)
    o = ob.reshape(8, D)
    for h in range(8):
        assert np.array_equal(o[h], A.bf16_round(vc[0, h // 4]))


def test_sink_vanishing_or_dominating():
    rng = np.random.default_rng(2)
    H = 64
    x = synth.f32_to_bf16_bits(rng.normal(size=H))
    w0 = _weights(rng, H, 8, 2, sink=-np.inf)
    kc, vc = _cache(rng, 40, 2)
    kc1, vc1 = kc.copy(), vc.copy()
    _, q, ob_plain = _step(w0, x, 40, kc1, vc1)                      # appends the new token's k, v at 40
    # the plain softmax attention, written out with einsum over every head at once
    keys = kc1[:41][:, np.arange(8) // 4, :].transpose(1, 0, 2)     # [head][token][dim]
    scores = np.einsum("hd,htd->ht", q.reshape(8, D), keys) / math.sqrt(D)
    p = np.exp(scores - scores.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    o = np.einsum("ht,htd->hd", p, vc1[:41][:, np.arange(8) // 4, :].transpose(1, 0, 2))
    assert np.array_equal(ob_plain, A.bf16_round(o.reshape(-1)))
    w_big = dict(w0, sinks=np.full(8, 1e4))
    _, _, ob_big = _step(w_big, x, 40, kc.copy(), vc.copy())
    assert np.all(ob_big == 0)


def test_tokens_outside_the_window_do_not_matter():
    rng = np.random.default_rng(3)
    H = 64
    wts = _weights(rng, H, 8, 2, sink=0.5)
    x = synth.f32_to_bf16_bits(rng.normal(size=H))
    n = 300
    kc, vc = _cache(rng, n, 2)
    out1, _, _ = _step(wts, x, n, kc.copy(), vc.copy(), sliding=True)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[: n + 1 - 128] = A.to_fp16(rng.normal(0, 5, kc2[: n + 1 - 128].shape))
    vc2[: n + 1 - 128] = A.to_fp16(rng.normal(0, 5, vc2[: n + 1 - 128].shape))
    out2, _, _ = _step(wts, x, n, kc2, vc2, sliding=True)
    assert np.array_equal(out1, out2)
    out3, _, _ = _step(wts, x, n, kc2, vc2, sliding=False)   # full attention sees them
    assert not np.array_equal(out1, out3)


def test_heads_of_one_group_read_the_same_keys():
    """Query heads 0..3 share kv head 0: equal queries give equal outputs;
    head 4 (kv head 1) differs."""
    rng = np.random.default_rng(4)
    H = 64
    wts = _weights(rng, H, 8, 2)
    wts["wq"][D:4 * D] = np.tile(wts["wq"][:D], (3, 1))
    wts["bq"][D:4 * D] = np.tile(wts["bq"][:D], 3)
    wts["wq"][4 * D:5 * D] = wts["wq"][:D]
    wts["bq"][4 * D:5 * D] = wts["bq"][:D]
    x = synth.f32_to_bf16_bits(rng.normal(size=H))
    kc, vc = _cache(rng, 20, 2)
    _, _, ob = _step(wts, x, 20, kc, vc)
    o = ob.reshape(8, D)
    for h in (1, 2, 3):
        assert np.array_equal(o[h], o[0])
    assert not np.array_equal(o[4], o[0])


def test_prefill_equals_masked_attention_written_as_matrices():
    """The oracle's prefill of n tokens (sequential decode steps) against a
    restatement with matrices: all new tokens' q, k, v at once, one score
    matrix per head with the causal mask (and, on a sliding layer, the
    window) applied as -inf, the sink as an extra column."""
    rng = np.random.default_rng(7)
    H, QH, KVH, n, pos0 = 64, 8, 2, 7, 5
    for sliding, window in ((False, 128), (True, 4)):
        wts = _weights(rng, H, QH, KVH, sink=0.3)
        x = synth.f32_to_bf16_bits(rng.normal(size=(n, H)))
        kc, vc = _cache(rng, pos0 + n - 1, KVH)
        kc1, vc1 = kc.copy(), vc.copy()
        got = A.prefill(wts, x, kc1, vc1, pos0, q_heads=QH, kv_heads=KVH, head_dim=D, sliding=sliding,
                        window=window, eps=1e-5)
        # the matrix form
        import oracle as O
        xs = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        xh = np.stack([(O.rmsnorm(x[r], wts["gamma"], 1e-5)[0].astype(np.uint32) << 16).view(np.float32)
                       for r in range(n)]).astype(np.float64)
        q = xh @ wts["wq"].T + wts["bq"]
        k = xh @ wts["wk"].T + wts["bk"]
        v = xh @ wts["wv"].T + wts["bv"]
        for r in range(n):
            c, s_ = A.rope_tables(pos0 + r, D)
            q[r] = A.apply_rope(q[r], c, s_)
            k[r] = A.apply_rope(k[r], c, s_)
        keys = kc.copy()
        vals = vc.copy()
        keys[pos0:] = A.to_fp16(k).reshape(n, KVH, D)
        vals[pos0:] = A.to_fp16(v).reshape(n, KVH, D)
        assert np.array_equal(keys, kc1) and np.array_equal(vals, vc1)
        T = pos0 + n
        t = np.arange(T)
        o = np.zeros((n, QH * D))
        for h in range(QH):
            g = h // (QH // KVH)
            sc = q[:, h * D:(h + 1) * D] @ keys[:, g, :].T / math.sqrt(D)        # [n][T]
            pos = pos0 + np.arange(n)[:, None]
            mask = t[None, :] <= pos
            if sliding:
                mask &= t[None, :] > pos - window
            sc = np.where(mask, sc, -np.inf)
            full = np.concatenate([sc, np.full((n, 1), wts["sinks"][h])], axis=1)
            p = np.exp(full - full.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o[:, h * D:(h + 1) * D] = p[:, :T] @ vals[:, g, :]
        ob = A.bf16_round(o)
        want = xs + ob @ wts["wo"].T + wts["bo"]
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
