"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the E2M1
table printed on the ds4.c page, library routines (numpy matmul, a stable
sort, scipy softmax, torch's float32->bf16 rounding and rms_norm), closed
forms, invariants, and a dense brute-force formulation of the whole block on a
tiny shape.  A plausible slip anywhere in the oracle (a swapped nibble, a wrong
scale index, a transposed matrix, a dropped bias, a wrong tie rule, a double
rounding) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_table():
    vals = {}
    for line in open(os.path.join(GOLDEN, "e2m1_table.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        i, v = line.split()
        vals[int(i)] = float(v)
    return [vals[i] for i in range(8)]


TABLE = _golden_table()


def _pack(idx: np.ndarray, sign: np.ndarray, exps: np.ndarray):
    """Test-side packer: magnitude indices [rows][cols], signs, E8M0 [rows][cols/32]
    -> canonical codes [rows][cols/2] (even element in the low nibble)."""
    nib = (idx.astype(np.uint8) & 7) | (sign.astype(np.uint8) << 3)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return codes, exps.astype(np.uint8)


def _dense(idx, sign, exps):
    rows, cols = idx.shape
    out = np.empty((rows, cols))
    for r in range(rows):
        for c in range(cols):
            v = math.ldexp(TABLE[idx[r, c]], int(exps[r, c // 32]) - 127)
            out[r, c] = -v if sign[r, c] else v
    return out


def _random_mxfp4(rng, rows, cols, elo=118, ehi=124):
    idx = rng.integers(0, 8, size=(rows, cols))
    sign = rng.integers(0, 2, size=(rows, cols))
    exps = rng.integers(elo, ehi + 1, size=(rows, cols // 32))
    return idx, sign, exps


# ------------------------------------------------------------------ MXFP4
def test_golden_table_is_the_e2m1_format():
    # E2M1: 2 exponent bits (bias 1), 1 mantissa bit; subnormal when exponent bits are 0.
    for m in range(8):
        e, f = m >> 1, m & 1
        v = (f * 0.5) if e == 0 else 2.0 ** (e - 1) * (1 + f / 2)
        assert TABLE[m] == v


def test_e2m1_all_codes_match_page_table():
    for nib in range(16):
        want = TABLE[nib & 7] * (-1.0 if nib & 8 else 1.0)
        got = oracle.e2m1_value(nib)
        assert got == want and math.copysign(1, got) == math.copysign(1, want) or want == 0


def test_mxfp4_exhaustive_codes_times_exponents():
    # every 4-bit code x every finite E8M0 exponent, against ldexp
    for e in range(0, 255):
        nibs = np.arange(32) % 16
        codes = (nibs[0::2] | (nibs[1::2] << 4)).astype(np.uint8)[None, :]
        scales = np.array([[e]], np.uint8)
        got = oracle.mxfp4_dequant(codes, scales)[0]
        want = np.array([math.ldexp(TABLE[n & 7], e - 127) * (-1 if n & 8 else 1) for n in nibs])
        assert np.array_equal(got, want), e
    nan = oracle.mxfp4_dequant(np.array([[0x11] * 16], np.uint8), np.array([[255]], np.uint8))
    assert np.all(np.isnan(nan))


def test_mxfp4_nibble_order_and_scale_index():
    rng = np.random.default_rng(1)
    idx, sign, exps = _random_mxfp4(rng, 7, 96, 100, 140)
    codes, scales = _pack(idx, sign, exps)
    assert np.array_equal(oracle.mxfp4_dequant(codes, scales), _dense(idx, sign, exps))


# ------------------------------------------------------------------- bf16
def test_bf16_rne_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 1e-38, 500), rng.normal(0, 1e30, 500),
                        np.array([0.0, -0.0, 1.0, -1.5, 3.0e38, -3.3e38, 1e-45, 2.0 ** -133])]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rne_single_rounding_from_double():
    # ties to even, and a value just above a tie that float-first rounding would lose
    one = 1.0
    assert oracle.bf16_rne(one + 2.0 ** -8) == 0x3F80            # tie -> even (1.0)
    assert oracle.bf16_rne(one + 3 * 2.0 ** -8) == 0x3F82        # tie -> even (1+2^-6)
    assert oracle.bf16_rne(one + 2.0 ** -8 + 2.0 ** -40) == 0x3F81  # above tie -> up
    assert oracle.bf16_rne(-(one + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    # subnormal bf16 range: quantum 2^-133
    assert oracle.bf16_rne(2.0 ** -133) == 0x0001
    assert oracle.bf16_rne(1.5 * 2.0 ** -133) == 0x0002          # tie -> even
    assert oracle.bf16_rne(0.5 * 2.0 ** -133) == 0x0000          # tie -> even (0)
    assert oracle.bf16_rne(2.0 ** -127) == 0x0040
    # overflow
    assert oracle.bf16_rne(2.0 ** 128) == 0x7F80
    assert oracle.bf16_rne(-(2.0 ** 127) * (2 - 2.0 ** -8)) == 0xFF80   # rounds up past max
    assert oracle.bf16_rne(2.0 ** 127 * (2 - 2.0 ** -7)) == 0x7F7F
    for b in (0x0001, 0x3F80, 0x7F7F, 0xC2F7, 0x0080):
        assert oracle.bf16_rne(oracle.bf16_to_double(b)) == b


# ---------------------------------------------------------------- rmsnorm
def test_rmsnorm_matches_torch_rms_norm_in_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    for H in (32, 2880, 4096):
        x = synth.f32_to_bf16_bits(rng.normal(0, 1, H))
        gamma = (1 + rng.normal(0, 0.1, H)).astype(np.float32)
        xh, pre = oracle.rmsnorm(x, gamma, 1e-5)
        xt = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
        want = torch.nn.functional.rms_norm(xt, (H,), torch.from_numpy(gamma.astype(np.float64)), eps=1e-5)
        np.testing.assert_allclose(pre, want.numpy(), rtol=1e-14, atol=0)
        # the rounding point: x_hat is the bf16 of the unrounded value
        assert np.array_equal(xh, np.array([oracle.bf16_rne(v) for v in pre], np.uint16))


def test_rmsnorm_scale_invariance_without_eps():
    rng = np.random.default_rng(4)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, 256))
    gamma = (1 + rng.normal(0, 0.1, 256)).astype(np.float32)
    x8 = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * 8.0)   # exact power-of-two scaling
    assert np.array_equal(oracle.rmsnorm(x, gamma, 0.0)[0], oracle.rmsnorm(x8, gamma, 0.0)[0])


def test_rmsnorm_constant_vector_closed_form():
    # x = c * 1 -> mean(x^2) = c^2, so x_hat = c / sqrt(c^2 + eps) * gamma
    c, H, eps = 0.75, 64, 1e-5
    x = np.full(H, synth.f32_to_bf16_bits(np.array([c], np.float32))[0], np.uint16)
    gamma = np.linspace(0.5, 1.5, H).astype(np.float32)
    _, pre = oracle.rmsnorm(x, gamma, eps)
    np.testing.assert_allclose(pre, c / math.sqrt(c * c + eps) * gamma.astype(np.float64), rtol=1e-15)


# ----------------------------------------------------------------- router
def test_router_logits_match_numpy_matmul():
    rng = np.random.default_rng(5)
    E, H = 32, 2880
    xh = synth.f32_to_bf16_bits(rng.normal(0, 1, H))
    W = synth.f32_to_bf16_bits(rng.normal(0, 0.02, (E, H)))
    b = rng.normal(0, 0.5, E).astype(np.float32)
    got = oracle.router_logits(xh, W, b)
    want = synth.bf16_bits_to_f32(W).astype(np.float64) @ synth.bf16_bits_to_f32(xh).astype(np.float64) + b
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def _brute_topk(v, k):
    # full stable sort by (-value, index); NaN and -inf can never beat an empty
    # slot (which starts at -inf under a strict comparison), so they are never selected
    order = sorted([i for i in range(len(v)) if v[i] > -math.inf], key=lambda i: (-v[i], i))
    ids = order[:k]
    vals = [v[i] for i in ids]
    while len(ids) < k:
        ids.append(0)
        vals.append(-math.inf)
    return ids, vals


def test_topk_matches_brute_force_sort_with_ties_and_nan():
    rng = np.random.default_rng(6)
    cases = [rng.normal(0, 1, 32) for _ in range(200)]
    cases += [np.round(rng.normal(0, 1, 32), 1) for _ in range(200)]      # many ties
    cases += [rng.integers(0, 3, 16).astype(float) for _ in range(100)]  # heavy ties
    c = rng.normal(0, 1, 32)
    c[[3, 9, 20]] = np.nan
    cases.append(c)
    cases.append(np.array([np.nan, 1.0, np.nan, 1.0]))
    cases.append(np.array([-np.inf, -np.inf, 2.0, -np.inf]))
    for v in cases:
        for k in (1, 2, 4, 6):
            if k > len(v):
                continue
            ids, vals = oracle.topk(v, k)
            bi, bv = _brute_topk(list(v), k)
            assert list(ids) == bi
            assert np.array_equal(vals, np.array(bv))


def test_topk_all_nan_keeps_initial_slots():
    ids, vals = oracle.topk(np.full(8, np.nan), 3)
    assert list(ids) == [0, 0, 0] and np.all(np.isneginf(vals))


def test_route_weights_softmax_and_scale():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    for k in (1, 2, 4, 6):
        for s in (1.0, 1.5, 2.5):
            v = np.sort(rng.normal(0, 3, k))[::-1].copy()
            w = oracle.route_weights(v, s)
            np.testing.assert_allclose(w, s * sp.softmax(v), rtol=1e-14)
            assert abs(w.sum() - s) < 1e-14 * s * k
    assert oracle.route_weights(np.array([0.3]), 1.5)[0] == 1.5
    np.testing.assert_array_equal(oracle.route_weights(np.array([2.0, 2.0]), 1.0), [0.5, 0.5])
    np.testing.assert_array_equal(oracle.route_weights(np.array([1.0, -np.inf]), 1.0), [1.0, 0.0])
    np.testing.assert_array_equal(oracle.route_weights(np.array([-np.inf, -np.inf]), 1.0), [0.0, 0.0])


# ----------------------------------------------------------------- SwiGLU
@pytest.mark.parametrize("alpha,L", [(1.702, 7.0), (1.702, 10.0)])
def test_swiglu_clamp_closed_forms(alpha, L):
    def sig(z):
        return 1.0 / (1.0 + math.exp(-z)) if z > -700 else 0.0
    eps = 1e-9
    glu_L = L * sig(alpha * L)
    for g in (L, L + 1, 1e30):
        for u in (-L - 1, -L, 0.0, L, L + 1, 1e30, -1e30):
            uc = max(-L, min(L, u))
            assert oracle.swiglu(g, u, alpha, L) == pytest.approx(glu_L * (uc + 1), rel=1e-15)
    # gate is not clamped from below
    for g in (-L - 1, -20.0, -1e3):
        assert oracle.swiglu(g, 0.0, alpha, L) == pytest.approx(g * sig(alpha * g), rel=1e-12, abs=1e-300)
    # up clamps on both sides; continuity at the clamps
    for u in (-L, L):
        a = oracle.swiglu(1.3, u, alpha, L)
        b = oracle.swiglu(1.3, u + (eps if u < 0 else -eps), alpha, L)
        assert abs(a - b) < 1e-8
    assert oracle.swiglu(L - eps, 0.0, alpha, L) == pytest.approx(glu_L, rel=1e-8)
    # monotone non-decreasing in u for positive glu
    us = np.linspace(-2 * L, 2 * L, 401)
    hs = [oracle.swiglu(2.0, u, alpha, L) for u in us]
    assert all(b >= a for a, b in zip(hs, hs[1:]))
    # the gelu-like core: g * sigmoid(alpha g) at u = 0
    for g in (-3.0, -0.5, 0.0, 0.7, 3.0):
        assert oracle.swiglu(g, 0.0, alpha, L) == pytest.approx(g * sig(alpha * g), rel=1e-14, abs=0)
    assert math.isnan(oracle.swiglu(float("nan"), 0.0, alpha, L))


# ---------------------------------------------------------- expert + block
def _tiny_block(rng, shape: synth.BlockShape, identical=False):
    H, F, E = shape.hidden, shape.expert_hidden, shape.n_experts
    blk = {"shape": shape,
           "gamma": (1 + rng.normal(0, 0.1, H)).astype(np.float32),
           "router_w": synth.f32_to_bf16_bits(rng.normal(0, 0.3, (E, H))),
           "router_b": rng.normal(0, 0.5, E).astype(np.float32),
           "codes": {}, "scales": {}, "bias": {}, "dense": {}}
    for m in synth.MATS:
        rows, cols = shape.mat_shape(m)
        nE = 1 if identical else E
        parts = [_random_mxfp4(rng, rows, cols, 123, 127) for _ in range(nE)]
        packed = [_pack(*p) for p in parts]
        dense = [_dense(*p) for p in parts]
        if identical:
            packed, dense = packed * E, dense * E
        blk["codes"][m] = np.stack([p[0] for p in packed])
        blk["scales"][m] = np.stack([p[1] for p in packed])
        blk["dense"][m] = np.stack(dense)
        bias = rng.normal(0, 0.05, (nE, rows)).astype(np.float32)
        blk["bias"][m] = np.repeat(bias, E, 0) if identical else bias
    if shape.n_shared:
        sh = {"codes": {}, "scales": {}, "bias": {}, "dense": {}}
        for m in synth.MATS:
            rows, cols = shape.mat_shape(m)
            p = _random_mxfp4(rng, rows, cols, 123, 127)
            c, s = _pack(*p)
            sh["codes"][m], sh["scales"][m] = c[None], s[None]
            sh["dense"][m] = _dense(*p)[None]
            sh["bias"][m] = rng.normal(0, 0.05, (1, rows)).astype(np.float32)
        blk["shared"] = sh
    return blk


def _bf16_round_array(v):
    return np.array([oracle.bf16_to_double(oracle.bf16_rne(a)) for a in np.ravel(v)]).reshape(np.shape(v))


def _fp4_rows(v):
    """Each row through the (separately pinned) FP4 activation encoding and back."""
    c, s = oracle.mx_fp4_quantize(np.atleast_2d(v).astype(np.float32))   # exact: bf16 values
    return oracle.mxfp4_dequant(c, s)


def _dense_block(blk, x_bits, act_fp4=False):
    """Dense brute force: every expert on every token (numpy matmul on the test's
    own dense matrices), then a top-k mask from a full stable sort, scipy softmax.
    act_fp4: the expert inputs (x_hat; h after its bf16 rounding) go through the
    FP4 activation encoding row by row first."""
    import scipy.special as sp
    shape = blk["shape"]
    H, E, K = shape.hidden, shape.n_experts, shape.top_k
    x = synth.bf16_bits_to_f32(x_bits).astype(np.float64)
    g = blk["gamma"].astype(np.float64)
    rms = np.sqrt((x * x).mean(axis=1, keepdims=True) + shape.rms_eps)
    xh = _bf16_round_array(x / rms * g)
    logits = xh @ synth.bf16_bits_to_f32(blk["router_w"]).astype(np.float64).T + blk["router_b"]

    def ffn(d, b, xin):
        if act_fp4:
            xin = _fp4_rows(xin)
        gg = xin @ d["gate"].T + b["gate"]
        uu = xin @ d["up"].T + b["up"]
        gc = np.minimum(gg, shape.swiglu_limit)
        uc = np.clip(uu, -shape.swiglu_limit, shape.swiglu_limit)
        h = _bf16_round_array(gc * sp.expit(shape.swiglu_alpha * gc) * (uc + 1))
        if act_fp4:
            h = _fp4_rows(h)
        return h @ d["down"].T + b["down"]

    ys = np.stack([ffn({m: blk["dense"][m][e] for m in synth.MATS},
                       {m: blk["bias"][m][e].astype(np.float64) for m in synth.MATS}, xh)
                   for e in range(E)], axis=1)              # [T][E][H]
    out = x.copy()
    ids = np.zeros((x.shape[0], K), np.int32)
    for t in range(x.shape[0]):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))[:K]
        ids[t] = order
        w = shape.weight_scale * sp.softmax(logits[t, order])
        mask = np.zeros(E)
        mask[order] = w
        out[t] += mask @ ys[t]
    if shape.n_shared:
        sh = blk["shared"]
        out += ffn({m: sh["dense"][m][0] for m in synth.MATS},
                   {m: sh["bias"][m][0].astype(np.float64) for m in synth.MATS}, xh)
    return out, ids, xh


@pytest.mark.parametrize("shared,scale", [(0, 1.0), (1, 1.5)])
def test_tiny_block_matches_dense_brute_force(shared, scale):
    pytest.importorskip("scipy")
    rng = np.random.default_rng(8 + shared)
    shape = synth.tiny_shape(32, 32, 4, 2, n_shared=shared, weight_scale=scale)
    blk = _tiny_block(rng, shape)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (9, 32)))
    r = oracle.moe_forward(blk, x)
    want, ids, xh = _dense_block(blk, x)
    assert np.array_equal(r["ids"], ids)
    assert np.array_equal(synth.bf16_bits_to_f32(r["xhat"]).astype(np.float64), xh)
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)


def test_tiny_block_rectangular_expert_hidden():
    # hidden != expert_hidden catches a transposed gate/up or down
    pytest.importorskip("scipy")
    rng = np.random.default_rng(10)
    shape = synth.tiny_shape(64, 32, 5, 3)
    blk = _tiny_block(rng, shape)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (6, 64)))
    r = oracle.moe_forward(blk, x)
    want, ids, _ = _dense_block(blk, x)
    assert np.array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("H,F,E,K,shared,scale", [(32, 32, 4, 2, 0, 1.0), (64, 32, 5, 3, 0, 1.0),
                                                  (32, 64, 4, 2, 1, 1.5)])
def test_fp4_activation_mode_matches_dense_brute_force(H, F, E, K, shared, scale):
    """The FP4 activation mode of the block (expert inputs encoded as the ds4.c
    FP4 activation quantisation does) against the dense formulation."""
    pytest.importorskip("scipy")
    rng = np.random.default_rng(31 + H + F + shared)
    shape = synth.tiny_shape(H, F, E, K, n_shared=shared, weight_scale=scale)
    blk = _tiny_block(rng, shape)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (7, H)))
    r = oracle.moe_forward(blk, x, act_fp4=True)
    want, ids, _ = _dense_block(blk, x, act_fp4=True)
    assert np.array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["out"], want, rtol=1e-12, atol=1e-12)


def test_fp4_activation_mode_changes_only_the_expert_outputs():
    rng = np.random.default_rng(37)
    shape = synth.tiny_shape(64, 64, 6, 2)
    blk = _tiny_block(rng, shape)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (5, 64)))
    r0 = oracle.moe_forward(blk, x)
    r1 = oracle.moe_forward(blk, x, act_fp4=True)
    for key in ("ids", "route_w", "xhat", "logits"):
        assert np.array_equal(r0[key], r1[key]), key
    d0, d1 = r0["out"] - synth.bf16_bits_to_f32(x), r1["out"] - synth.bf16_bits_to_f32(x)
    assert not np.array_equal(d0, d1)
    # E2M1 keeps ~2 significant bits of each activation: the deltas agree to tens of percent
    assert np.linalg.norm(d1 - d0) < 0.5 * np.linalg.norm(d0)


def test_identical_experts_collapse_to_one_expert():
    rng = np.random.default_rng(11)
    shape = synth.tiny_shape(64, 64, 6, 3, weight_scale=1.5)
    blk = _tiny_block(rng, shape, identical=True)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, (5, 64)))
    r = oracle.moe_forward(blk, x)
    one = dict(blk)
    one["router_w"], one["router_b"] = blk["router_w"][:1], blk["router_b"][:1]
    for key in ("codes", "scales", "bias"):
        one[key] = {m: blk[key][m][:1] for m in synth.MATS}
    r1 = oracle.moe_forward(one, x, shape=synth.tiny_shape(64, 64, 1, 1))
    x64 = synth.bf16_bits_to_f32(x).astype(np.float64)
    np.testing.assert_allclose(r["out"] - x64, 1.5 * (r1["out"] - x64), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["route_w"].sum(axis=1), 1.5, rtol=1e-15)


def test_down_scale_exponent_doubles_output():
    rng = np.random.default_rng(12)
    shape = synth.tiny_shape(64, 32, 4, 2)
    blk = _tiny_block(rng, shape)
    x = synth.f32_to_bf16_bits(rng.normal(0, 1, 64))
    y, h, gu = oracle.expert_ffn(blk["codes"], blk["scales"], blk["bias"], 2, oracle.rmsnorm(x, blk["gamma"], 1e-5)[0], 1.702, 7.0)
    sc = {m: blk["scales"][m].copy() for m in synth.MATS}
    sc["down"] = sc["down"] + 1
    y2, h2, _ = oracle.expert_ffn(blk["codes"], sc, blk["bias"], 2, oracle.rmsnorm(x, blk["gamma"], 1e-5)[0], 1.702, 7.0)
    bd = blk["bias"]["down"][2].astype(np.float64)
    assert np.array_equal(h, h2)
    np.testing.assert_allclose(y2 - bd, 2 * (y - bd), rtol=1e-14, atol=1e-15)
    # the ffn against numpy on the test's own dense matrices
    xh = synth.bf16_bits_to_f32(oracle.rmsnorm(x, blk["gamma"], 1e-5)[0]).astype(np.float64)
    np.testing.assert_allclose(gu[:32], blk["dense"]["gate"][2] @ xh + blk["bias"]["gate"][2], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(gu[32:], blk["dense"]["up"][2] @ xh + blk["bias"]["up"][2], rtol=1e-13, atol=1e-14)
    hv = synth.bf16_bits_to_f32(h).astype(np.float64)
    np.testing.assert_allclose(y, blk["dense"]["down"][2] @ hv + bd, rtol=1e-13, atol=1e-14)


def test_permutation_invariants_and_stable_order():
    rng = np.random.default_rng(13)
    for T, K, E in ((1, 4, 32), (8, 4, 32), (37, 6, 256), (300, 2, 4)):
        ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
        p = oracle.permutation(ids, E)
        assert p["counts"].sum() == T * K
        assert np.array_equal(p["counts"], np.bincount(ids.ravel(), minlength=E))
        assert np.array_equal(p["offsets"], np.concatenate([[0], np.cumsum(p["counts"])]))
        order = np.argsort(ids.ravel(), kind="stable")   # library stable sort
        assert np.array_equal(p["perm_token"], order // K)
        assert np.array_equal(p["perm_slot"], order % K)
        assert np.array_equal(np.sort(p["loc"]), np.arange(T * K))
        assert np.array_equal(p["perm_token"][p["loc"]], np.repeat(np.arange(T), K))


def test_thread_count_does_not_change_results():
    blk = synth.make_block(0)
    x = synth.make_tokens(0, 3, 2880)
    a = oracle.moe_forward(blk, x, nthreads=1)
    b = oracle.moe_forward(blk, x, nthreads=3)
    for k in a:
        assert np.array_equal(a[k], b[k])


def test_golden_constants_match_workload_shapes():
    want = {}
    for line in open(os.path.join(GOLDEN, "block_constants.txt")):
        if line.strip() and not line.startswith("#"):
            name, key, val = line.split()
            want[(name, key)] = float(val)
    shapes = {"gpt-oss": synth.GPT_OSS, "dsv4-flash": synth.DSV4_FLASH_SHAPE}
    for (name, key), v in want.items():
        assert float(getattr(shapes[name], key)) == v, (name, key)


# ------------------------------------------------ FP4 activation encoding
# ds4.c, FP4 activation quantisation: per 32-element block the scale is the
# power of two 2^ceil(log2(amax / 6)) and each element is the nearest E2M1
# value (ties to even) of x / scale, clamped to +-6.

def _mx_blocks(rng, rows, cols, lo=-130, hi=120):
    """float32 rows whose 32-element blocks each have their own magnitude."""
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    e = rng.integers(lo, hi, size=(rows, cols // 32))
    return (x * np.repeat(np.exp2(e.astype(np.float64)), 32, axis=1)).astype(np.float32)


def test_mx_fp4_scale_is_the_smallest_power_of_two_covering_amax_over_6():
    rng = np.random.default_rng(11)
    x = _mx_blocks(rng, 64, 256)
    x[0, :32] = 0.0                       # all-zero block: the 6 * 2^-126 floor
    x[1, :32] = np.float32(6.0)           # q = 1 exactly
    x[2, 32:64] = np.float32(3.0) * np.float32(2.0) ** 20   # q a power of two
    _, sc = oracle.mx_fp4_quantize(x)
    amax = np.abs(x).reshape(64, 8, 32).max(axis=2)
    amax = np.maximum(amax, np.float32(6.0 * 2.0 ** -126))
    q = (amax / np.float32(6.0)).astype(np.float32)      # one float32 rounding
    k = sc.astype(np.int64) - 127
    for qi, ki in zip(q.ravel(), k.ravel()):
        assert math.ldexp(1.0, int(ki) - 1) < float(qi) <= math.ldexp(1.0, int(ki))
        lg = math.log2(float(qi))
        if abs(lg - round(lg)) > 1e-4:
            assert ki == math.ceil(lg)
    assert sc[0, 0] == 1 and sc[1, 0] == 127 and sc[2, 1] == 127 + 19


def _decode(codes, scales):
    return oracle.mxfp4_dequant(codes, scales)


def test_mx_fp4_codes_are_the_nearest_values_with_ties_to_even():
    rng = np.random.default_rng(12)
    x = _mx_blocks(rng, 32, 128, -20, 20)
    # every tie of the E2M1 grid (midpoints) and the grid itself, scale 2^0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2, 3, 4, 6], np.float32)
    x[0, :14], x[0, 14:28] = mids, -mids
    x[0, 28:32] = [6.0, 0.1, -0.2, 5.9]
    codes, sc = oracle.mx_fp4_quantize(x)
    nib = np.stack([codes & 15, codes >> 4], axis=2).reshape(x.shape).astype(np.int64)
    k = np.repeat(sc.astype(np.int64) - 127, 32, axis=1)
    cand_mag = np.array(TABLE)
    for (r, c), xv in np.ndenumerate(x):
        s = math.ldexp(1.0, int(k[r, c]))
        xc = min(max(float(xv), -6 * s), 6 * s)
        cands = np.concatenate([cand_mag, -cand_mag]) * s
        dist = np.abs(cands - xc)
        got = TABLE[nib[r, c] & 7] * s * (-1.0 if nib[r, c] & 8 else 1.0)
        assert abs(got - xc) == dist.min(), (r, c, xv)
        ties = {i % 8 for i in np.flatnonzero(dist == dist.min())}
        if len(ties) > 1:
            assert (nib[r, c] & 7) % 2 == 0, (r, c, xv)
        assert bool(nib[r, c] & 8) == bool(xv < 0)


def test_mx_fp4_worked_cases():
    x = np.zeros((4, 32), np.float32)
    x[0, :12] = [0.5, 6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -5, -0.0, -1e-30]
    x[1, :2] = [12.0, -1.0]               # q = 2 -> k = 1
    x[2, :2] = [np.nan, 1.0]              # NaN ignored by amax, encoded +6
    x[3, :3] = [-np.inf, 1.0, 2.0 ** 120]
    codes, sc = oracle.mx_fp4_quantize(x)
    # scale 2^0: 0.5|6 -> 0x71, 0.25->0 | 0.75->1.0 -> 0x20, 1.25->1.0 | 1.75->2.0 -> 0x42,
    # 2.5->2.0 | 3.5->4.0 -> 0x64, 5->4.0 | -5->-4.0 -> 0xE6, -0.0 -> +0 | -1e-30 -> -0 -> 0x80
    assert sc[0, 0] == 127
    assert codes[0, :8].tolist() == [0x71, 0x20, 0x42, 0x64, 0xE6, 0x80, 0, 0]
    # 12 / 2 = 6 -> 7; -1 / 2 = -0.5 -> sign | 1
    assert sc[1, 0] == 128 and codes[1, 0] == 0x97
    # amax 1: q = 1/6 -> k = -2 (scale 2^-2); NaN -> +6 (7), 1 / 0.25 = 4 -> 6
    assert sc[2, 0] == 125 and codes[2, 0] == 0x67
    # an infinite element saturates the exponent at 127: -inf -> -6, the rest -> 0
    assert sc[3, 0] == 254 and codes[3, 0] == 0x0F and codes[3, 1] == 0
    with pytest.raises(ValueError):
        oracle.mx_fp4_quantize(np.zeros((1, 48), np.float32))


def test_mx_fp4_round_trip_is_idempotent_and_within_half_a_step():
    rng = np.random.default_rng(13)
    x = _mx_blocks(rng, 48, 320, -60, 60)
    y = _decode(*oracle.mx_fp4_quantize(x))
    y2 = _decode(*oracle.mx_fp4_quantize(y.astype(np.float32)))
    np.testing.assert_array_equal(y2, y)
    _, sc = oracle.mx_fp4_quantize(x)
    s = np.exp2(np.repeat(sc.astype(np.float64) - 127, 32, axis=1))
    v = np.abs(x.astype(np.float64)) / s
    half_step = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0)) * s
    assert np.all(np.abs(x - y) <= half_step)


def test_mx_fp4_is_monotone_within_a_block():
    rng = np.random.default_rng(14)
    for _ in range(50):
        b = np.sort(rng.uniform(-7.0, 7.0, 32)).astype(np.float32)
        b[0], b[-1] = -7.5, 7.5          # fixed amax: one scale for the block
        y = _decode(*oracle.mx_fp4_quantize(b[None, :]))[0]
        assert np.all(np.diff(y) >= 0)
