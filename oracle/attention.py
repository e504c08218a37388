"""The attention half of the gpt-oss layer, decode step, written plainly from
the pages in float64 (TEST INFRASTRUCTURE ONLY, like the rest of this folder:
the tests are its only users; the CUDA library never imports it and it never
imports the library).

goosedump gpt_oss.rs, `forward` (the per-layer attention step), `Rope::new`,
`correction_dimension`, `apply_rope`, `LayerCache::append`, `causal_gqa`,
`attention_window`, `attention_head`; turbospark-runtime gptoss/mod.rs module
doc comment (the per-layer formula).  For one new token of a sequence whose
cache holds n - 1 earlier tokens (its position is n - 1):

    x_hat = bf16(rms_norm(x) * gamma)                      (as for the MoE block)
    q = Wq x_hat + bq, k = Wk x_hat + bk, v = Wv x_hat + bv
    q, k rotated by YaRN RoPE at the token's position
    k, v appended to the cache as fp16
    per query head h (kv head h / group): scores over the visible cached
      tokens (the last `window` of them on sliding layers, all otherwise)
      = q_h . k_t / sqrt(head_dim), plus the head's sink logit; softmax over
      all of them; o_h = sum_t p_t v_t (the sink's share is dropped)
    out = x + Wo bf16(o) + bo

Readings (where the pages leave a step open): q, k, v, the scores and o are
exact (float64) values of the stated sums; the cache holds k and v rounded to
fp16 (the page's `Fp16::from`); o is rounded once to bf16 before the output
projection (as h before the MoE's down projection: the tensor-core input);
the RoPE angles, cosines and sines are the exact values of the page's
formulas (the page evaluates them in f32).
"""
from __future__ import annotations

import math

import numpy as np

import oracle

# [gpt_oss.rs] constants block
ROPE_BASE = 150_000.0
ROPE_FACTOR = 32.0
ROPE_ORIGINAL_CONTEXT = 4_096.0
ROPE_BETA_FAST = 32.0
ROPE_BETA_SLOW = 1.0


def correction_dimension(rotations: float, head_dim: int, base=ROPE_BASE, orig=ROPE_ORIGINAL_CONTEXT) -> float:
    return head_dim * math.log(orig / (rotations * 2.0 * math.pi)) / (2.0 * math.log(base))


def rope_tables(position: int, head_dim: int, base=ROPE_BASE, factor=ROPE_FACTOR, orig=ROPE_ORIGINAL_CONTEXT,
                beta_fast=ROPE_BETA_FAST, beta_slow=ROPE_BETA_SLOW):
    """cos and sin per pair (head_dim / 2 of them), times the attention factor."""
    attention_factor = 0.1 * math.log(factor) + 1.0
    low = max(correction_dimension(beta_fast, head_dim, base, orig), 0.0)
    high = min(correction_dimension(beta_slow, head_dim, base, orig), head_dim - 1.0)
    cos = np.zeros(head_dim // 2)
    sin = np.zeros(head_dim // 2)
    for pair in range(head_dim // 2):
        base_frequency = base ** (-(2.0 * pair / head_dim))
        ramp = min(max((pair - low) / (high - low), 0.0), 1.0)
        frequency = base_frequency * (1.0 - ramp + ramp / factor)
        angle = position * frequency
        cos[pair] = math.cos(angle) * attention_factor
        sin[pair] = math.sin(angle) * attention_factor
    return cos, sin


def apply_rope(values: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Each head's first half l and second half r become l cos - r sin and
    l sin + r cos, pair by pair."""
    d = 2 * cos.shape[0]
    v = values.reshape(-1, d).astype(np.float64)
    left, right = v[:, :d // 2].copy(), v[:, d // 2:].copy()
    out = np.empty_like(v)
    out[:, :d // 2] = left * cos - right * sin
    out[:, d // 2:] = left * sin + right * cos
    return out.reshape(values.shape)


def to_fp16(v: np.ndarray) -> np.ndarray:
    """Round to the nearest fp16 (ties to even) and back to float64."""
    return v.astype(np.float64).astype(np.float16).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round float64 values once to bf16 (nearest, ties to even), as float64."""
    bits = np.array([oracle.bf16_rne(float(t)) for t in np.ravel(v)], np.uint32).reshape(np.shape(v))
    return (bits << 16).view(np.float32).astype(np.float64)


def attention_window(token_count: int, sliding: bool, window: int):
    first = max(0, token_count - window) if sliding else 0
    return first, token_count - first


def softmax(z: np.ndarray) -> np.ndarray:
    m = np.max(z)
    e = np.exp(z - m)
    return e / e.sum()


def decode_step(wts: dict, x_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, n_ctx: int, *,
                q_heads: int, kv_heads: int, head_dim: int, sliding: bool, window: int, eps: float,
                rope=None):
    """One new token (bf16 bits x [H]) of a sequence with n_ctx cached tokens
    (k_cache, v_cache float64 fp16 values [n_ctx + 1][kv_heads][head_dim];
    row n_ctx receives the new token's k and v).  Returns the block output
    (float64 [H]), q after RoPE, and the bf16-rounded o fed to the output
    projection."""
    rope = rope or {}
    x = (x_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xh, _ = oracle.rmsnorm(x_bits, wts["gamma"], eps)
    xh = (xh.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q = wts["wq"] @ xh + wts["bq"]
    k = wts["wk"] @ xh + wts["bk"]
    v = wts["wv"] @ xh + wts["bv"]
    cos, sin = rope_tables(n_ctx, head_dim, **rope)
    q = apply_rope(q, cos, sin)
    k = apply_rope(k, cos, sin)
    k_cache[n_ctx] = to_fp16(k).reshape(kv_heads, head_dim)
    v_cache[n_ctx] = to_fp16(v).reshape(kv_heads, head_dim)
    count = n_ctx + 1
    first, visible = attention_window(count, sliding, window)
    scale = 1.0 / math.sqrt(head_dim)
    group = q_heads // kv_heads
    o = np.zeros(q_heads * head_dim)
    for h in range(q_heads):
        g = h // group
        qh = q[h * head_dim:(h + 1) * head_dim]
        keys = k_cache[first:first + visible, g, :]
        scores = np.empty(visible + 1)
        scores[:visible] = keys @ qh * scale
        scores[visible] = wts["sinks"][h]
        p = softmax(scores)
        o[h * head_dim:(h + 1) * head_dim] = p[:visible] @ v_cache[first:first + visible, g, :]
    ob = bf16_round(o)
    out = x + wts["wo"] @ ob + wts["bo"]
    return out, q, ob


def prefill(wts: dict, x_rows: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, pos0: int, *,
            q_heads: int, kv_heads: int, head_dim: int, sliding: bool, window: int, eps: float):
    """goosedump gpt_oss.rs `prefill_attention_layer` with `causal_gqa_batch`:
    new tokens x_rows (bf16 bits [n][H]) of one sequence whose cache holds
    pos0 tokens.  Every new token's k and v go to the cache; token r attends
    over the tokens 0 .. pos0 + r (the last `window` of them on sliding
    layers) and the sink -- the same as n decode steps in order, which is how
    this restates it.  k_cache, v_cache: float64 [pos0 + n][kv_heads][64]
    (rows pos0 .. receive the new keys and values).  Returns the outputs
    [n][H]."""
    out = []
    for r in range(x_rows.shape[0]):
        o, _, _ = decode_step(wts, x_rows[r], k_cache, v_cache, pos0 + r, q_heads=q_heads, kv_heads=kv_heads,
                              head_dim=head_dim, sliding=sliding, window=window, eps=eps)
        out.append(o)
    return np.stack(out)
