"""Seeded synthetic inputs for the MXFP4 routed MoE block.

This module only draws random numbers and stores them in the block's input
formats.  It holds none of the block's arithmetic: no normalisation, no
routing, no dequantisation, no activation.  Both the CPU oracle (through the
tests) and the CUDA library (through the tests, ``bench.py`` and
``smoke()``) consume exactly the arrays produced here.

Formats (the canonical layout of the C-ABI, see ``include/moe.h``):

* ``x``          bf16 bit patterns, uint16 ``[T][H]``
* ``gamma``      float32 ``[H]``
* ``router_w``   bf16 bit patterns, uint16 ``[E][H]``
* ``router_b``   float32 ``[E]``
* per matrix ``m`` in (gate, up, down):
    ``codes[m]``  uint8 ``[E][rows][cols/2]``; element ``2i`` of a row sits in
                  the low nibble of byte ``i``, element ``2i+1`` in the high one;
                  nibble bit 3 is the sign, bits 0..2 the E2M1 magnitude index
    ``scales[m]`` uint8 E8M0 ``[E][rows][cols/32]``
    ``bias[m]``   float32 ``[E][rows]``
  gate and up are ``[F][H]`` (rows = expert_hidden), down is ``[H][F]``.
* the always-on shared expert (``n_shared == 1``) uses the same three matrices
  with a leading dimension of 1.

Value recipes follow the workloads of the gpt-oss MoE block (goosedump
``gpt_oss.rs``, constants block and ``mixture_of_experts``) and the
DeepSeek-V4-Flash shape profile (ds4 ``ds4.c``, ``DS4_SHAPE_FLASH``):
x ~ N(0,1); gamma = 1 + N(0, 0.1); router weights N(0, 0.02); router bias
N(0, 0.5); expert biases N(0, 0.02); code nibbles uniform over all 16 values;
E8M0 exponents uniform over [118, 124].
"""
from __future__ import annotations

import dataclasses

import numpy as np

BASE_SEED = 0x4D6F45

# tensor ids for the per-tensor random streams
_T_GAMMA, _T_RW, _T_RB, _T_X, _T_SKEW = 1, 2, 3, 4, 5
_T_CODES, _T_SCALES, _T_BIAS = 10, 20, 30
MATS = ("gate", "up", "down")


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """Shape and scalar parameters of one MoE block."""

    hidden: int
    expert_hidden: int
    n_experts: int
    top_k: int
    swiglu_alpha: float = 1.702
    swiglu_limit: float = 7.0
    weight_scale: float = 1.0
    rms_eps: float = 1e-5
    n_shared: int = 0

    def mat_shape(self, m: str) -> tuple[int, int]:
        """(rows, cols) of matrix ``m`` of one expert."""
        if m in ("gate", "up"):
            return self.expert_hidden, self.hidden
        return self.hidden, self.expert_hidden


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: BlockShape
    tokens: tuple[int, ...]
    router_skew: str = "none"  # "none" | "hot2" | "zipf1.1"
    layers: int = 1


GPT_OSS = BlockShape(2880, 2880, 32, 4)
DSV4_FLASH_SHAPE = BlockShape(4096, 2048, 256, 6, swiglu_limit=10.0, weight_scale=1.5, n_shared=1)

# Hot-expert boost of the skewed decode batch.  Two experts get this added to
# their router bias; with it they carry about 60% of the routing weight
# (measured over 4096 tokens: 0.61 of the weight, 0.42 of the slots; two
# experts can hold at most half of the top-4 slots).
HOT2_BOOST = 2.75

WORKLOADS = {
    0: Workload("gpt-oss MoE block decode, 1 token", GPT_OSS, (1,)),
    1: Workload("gpt-oss MoE block decode, 8 tokens, 2 hot experts", GPT_OSS, (8,), "hot2"),
    2: Workload("24-layer gpt-oss MoE stack decode", GPT_OSS, (1, 4, 16), layers=24),
    3: Workload("gpt-oss MoE block prefill", GPT_OSS, (128, 512)),
    4: Workload("DeepSeek-V4-Flash-shaped MoE block, Zipf(1.1) routing", DSV4_FLASH_SHAPE, (1, 2048), "zipf1.1"),
}


def _rng(config: int, layer: int, tensor: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([BASE_SEED, config, layer, tensor, sub])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 samples to bf16 (nearest, ties to even); returns uint16 bits.

    Only used to store generated samples in bf16; finite inputs only.
    """
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def router_bias(shape: BlockShape, skew: str, config: int, layer: int) -> np.ndarray:
    E = shape.n_experts
    if skew == "zipf1.1":
        ranks = _rng(config, layer, _T_SKEW).permutation(E) + 1
        return (-1.1 * np.log(ranks.astype(np.float64))).astype(np.float32)
    b = _rng(config, layer, _T_RB).normal(0.0, 0.5, size=E).astype(np.float32)
    if skew == "hot2":
        hot = _rng(config, layer, _T_SKEW).choice(E, size=2, replace=False)
        b[hot] += np.float32(HOT2_BOOST)
    return b


def expert_matrices(shape: BlockShape, n: int, config: int, layer: int, sub: int) -> dict:
    """Codes, scales and biases of ``n`` experts (``sub`` separates routed/shared)."""
    out = {"codes": {}, "scales": {}, "bias": {}}
    for mi, m in enumerate(MATS):
        rows, cols = shape.mat_shape(m)
        out["codes"][m] = _rng(config, layer, _T_CODES + mi, sub).integers(
            0, 256, size=(n, rows, cols // 2), dtype=np.uint8)
        out["scales"][m] = _rng(config, layer, _T_SCALES + mi, sub).integers(
            118, 125, size=(n, rows, cols // 32), dtype=np.uint8)
        out["bias"][m] = _rng(config, layer, _T_BIAS + mi, sub).normal(
            0.0, 0.02, size=(n, rows)).astype(np.float32)
    return out


def make_router(config: int, layer: int = 0, shape: BlockShape | None = None,
                skew: str | None = None) -> dict:
    """The norm and router weights of one block (``make_block`` without the
    experts; the same arrays)."""
    wl = WORKLOADS.get(config)
    shape = shape or wl.shape
    skew = skew if skew is not None else (wl.router_skew if wl else "none")
    H, E = shape.hidden, shape.n_experts
    return {
        "shape": shape,
        "gamma": (1.0 + _rng(config, layer, _T_GAMMA).normal(0.0, 0.1, size=H)).astype(np.float32),
        "router_w": f32_to_bf16_bits(_rng(config, layer, _T_RW).normal(0.0, 0.02, size=(E, H))),
        "router_b": router_bias(shape, skew, config, layer),
    }


def make_block(config: int, layer: int = 0, shape: BlockShape | None = None,
               skew: str | None = None) -> dict:
    """All weights of one block of workload ``config`` (layer ``layer``)."""
    blk = make_router(config, layer, shape, skew)
    shape = blk["shape"]
    blk.update(expert_matrices(shape, shape.n_experts, config, layer, 0))
    if shape.n_shared:
        sh = expert_matrices(shape, 1, config, layer, 1)
        blk["shared"] = sh
    return blk


def expert_matrices_device(shape: BlockShape, n: int, seed: int, device="cuda") -> dict:
    """The same recipe as ``expert_matrices`` drawn on the device with torch's
    generator (another random stream: only the distributions are shared).
    For benchmark weight sets too large to draw on the host in reasonable time;
    nothing that is compared with the oracle uses these."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = {"codes": {}, "scales": {}, "bias": {}}
    for m in MATS:
        rows, cols = shape.mat_shape(m)
        out["codes"][m] = torch.randint(0, 256, (n, rows, cols // 2), dtype=torch.uint8, device=device, generator=g)
        out["scales"][m] = torch.randint(118, 125, (n, rows, cols // 32), dtype=torch.uint8, device=device,
                                         generator=g)
        out["bias"][m] = torch.randn((n, rows), dtype=torch.float32, device=device, generator=g) * 0.02
    return out


def make_block_device(config: int, layer: int, expert_seed: int, device="cuda") -> dict:
    """Norm and router weights of workload ``config`` (layer ``layer``) drawn
    exactly as ``make_router`` does, with expert matrices from
    ``expert_matrices_device`` (seeded by ``expert_seed``)."""
    blk = make_router(config, layer)
    shape = blk["shape"]
    blk.update(expert_matrices_device(shape, shape.n_experts, expert_seed, device))
    if shape.n_shared:
        blk["shared"] = expert_matrices_device(shape, 1, expert_seed + 7919, device)
    return blk


# The attention half of the gpt-oss layer (goosedump gpt_oss.rs constants block:
# 64 query heads, 8 key/value heads, head dimension 64).
_T_ATTN = 40
ATTN_GPT_OSS = dict(hidden=2880, q_heads=64, kv_heads=8, head_dim=64, window=128)


def make_attention(seed: int, hidden: int = 2880, q_heads: int = 64, kv_heads: int = 8, head_dim: int = 64) -> dict:
    """Seeded attention weights: gamma = 1 + N(0, 0.1) (f32); Wq, Wk, Wv, Wo ~
    N(0, 0.02) as bf16 bits (Wq [q_heads*64][H], Wk/Wv [kv_heads*64][H],
    Wo [H][q_heads*64]); biases N(0, 0.02) (f32); sinks N(0, 1) (f32)."""
    r = lambda t: _rng(_T_ATTN, seed, t)  # noqa: E731
    QD, KD = q_heads * head_dim, kv_heads * head_dim
    return dict(gamma=(1.0 + r(0).normal(0.0, 0.1, hidden)).astype(np.float32),
                wq=f32_to_bf16_bits(r(1).normal(0.0, 0.02, (QD, hidden))),
                wk=f32_to_bf16_bits(r(2).normal(0.0, 0.02, (KD, hidden))),
                wv=f32_to_bf16_bits(r(3).normal(0.0, 0.02, (KD, hidden))),
                wo=f32_to_bf16_bits(r(4).normal(0.0, 0.02, (hidden, QD))),
                bq=r(5).normal(0.0, 0.02, QD).astype(np.float32),
                bk=r(6).normal(0.0, 0.02, KD).astype(np.float32),
                bv=r(7).normal(0.0, 0.02, KD).astype(np.float32),
                bo=r(8).normal(0.0, 0.02, hidden).astype(np.float32),
                sinks=r(9).normal(0.0, 1.0, q_heads).astype(np.float32))


def make_kv_history(seed: int, seqs: int, ctx: int, kv_heads: int = 8, head_dim: int = 64) -> tuple:
    """Cached keys and values of earlier tokens: N(0, 1) rounded to fp16,
    [seqs][ctx][kv_heads][head_dim] each."""
    k = _rng(_T_ATTN, seed, 20).normal(0.0, 1.0, (seqs, ctx, kv_heads, head_dim)).astype(np.float16)
    v = _rng(_T_ATTN, seed, 21).normal(0.0, 1.0, (seqs, ctx, kv_heads, head_dim)).astype(np.float16)
    return k, v


def attention_device(seed: int, hidden: int = 2880, q_heads: int = 64, kv_heads: int = 8, head_dim: int = 64,
                     device="cuda") -> dict:
    """The ``make_attention`` recipe drawn on the device with torch's generator
    (another random stream: only the distributions are shared), bf16 bits as
    int16.  For benchmark stacks; nothing compared with the oracle uses it."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    QD, KD = q_heads * head_dim, kv_heads * head_dim

    def n(shape, s):
        return torch.randn(shape, dtype=torch.float32, device=device, generator=g) * s

    def bf(shape):
        return n(shape, 0.02).to(torch.bfloat16).view(torch.int16)
    return dict(gamma=1.0 + n(hidden, 0.1), wq=bf((QD, hidden)), wk=bf((KD, hidden)), wv=bf((KD, hidden)),
                wo=bf((hidden, QD)), bq=n(QD, 0.02), bk=n(KD, 0.02), bv=n(KD, 0.02), bo=n(hidden, 0.02),
                sinks=n(q_heads, 1.0))


def kv_history_device(seed: int, k_cache, v_cache) -> None:
    """Fill a plan's key and value caches with N(0, 1) rounded to fp16 on the
    device (the ``make_kv_history`` distributions, torch's generator)."""
    import torch
    g = torch.Generator(device=k_cache.device)
    g.manual_seed(int(seed))
    for c in (k_cache, v_cache):
        c.copy_(torch.randn(c.shape, dtype=torch.float32, device=c.device, generator=g).to(torch.float16))


def make_tokens(config: int, tokens: int, hidden: int, layer: int = 0, sub: int = 0) -> np.ndarray:
    """Input activations x ~ N(0,1) as bf16 bits ``[tokens][hidden]``."""
    return f32_to_bf16_bits(_rng(config, layer, _T_X, sub).normal(0.0, 1.0, size=(tokens, hidden)))


def tiny_shape(hidden=32, expert_hidden=32, n_experts=4, top_k=2, **kw) -> BlockShape:
    """Small shapes for brute-force and edge-case tests."""
    return BlockShape(hidden, expert_hidden, n_experts, top_k, **kw)


def expert_bytes(shape: BlockShape) -> int:
    """HBM bytes of one expert's packed MXFP4 matrices (codes + E8M0 scales)."""
    H, F = shape.hidden, shape.expert_hidden
    return 3 * (F * H // 2 + F * H // 32)


def expert_bias_bytes(shape: BlockShape) -> int:
    return 4 * (2 * shape.expert_hidden + shape.hidden)


def distinct_uniform(E: int, K: int, T: int) -> float:
    """Expected distinct experts touched by T tokens under uniform top-K routing."""
    return E * (1.0 - (1.0 - K / E) ** T)


__all__ = [
    "BlockShape", "Workload", "WORKLOADS", "GPT_OSS", "DSV4_FLASH_SHAPE", "MATS", "ATTN_GPT_OSS", "make_attention",
    "make_kv_history",
    "make_block", "make_router", "make_tokens", "make_block_device", "expert_matrices_device", "tiny_shape", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "expert_bytes", "expert_bias_bytes", "distinct_uniform",
]
