"""One gpt-oss decoder layer through the library, as the pages chain it
(goosedump gpt_oss.rs `forward`: the attention step, then the MoE block on
its output; turbospark-runtime gptoss/mod.rs module doc comment, the
per-layer formula): moe_attn_decode writes x + attention(x) rounded to bf16
(`out_bf16`), which is the MoE plan's input as it stands.  Checked against
the oracle, teacher-forced at the hand-off: the attention's fp32 output
(same plan, fp32 out) within the block tolerance and its bf16 output equal
to that rounded once; the MoE block on the GPU's bf16 hand-off with ids and
permutation bit-exact and the output within the block tolerance."""
import numpy as np
import pytest

import oracle
from oracle import attention as A
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import check_close, check_permutation, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


def _as64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("window", [128, 0])
def test_attention_then_moe_block(window):
    import torch
    cfg, B, ctx = 0, 8, 300
    blk = synth.make_block(cfg)
    sh = blk["shape"]
    a = synth.ATTN_GPT_OSS
    H, QH, KVH = a["hidden"], a["q_heads"], a["kv_heads"]
    assert H == sh.hidden
    w = synth.make_attention(41 + window, H, QH, KVH)
    kh, vh = synth.make_kv_history(41, B, ctx, KVH)
    x = synth.make_tokens(cfg, B, H, sub=3)
    positions = [5, 40, 127, 128, 200, 256, 270, 299]
    dev = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda() for k, v in w.items()}
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    outs = {}
    for bf in (False, True):
        plan = moe.AttnPlan(H, QH, KVH, B, ctx, sliding_window=window, out_bf16=bf)
        plan.load_weights(dev)
        plan.k_cache.copy_(torch.from_numpy(kh))
        plan.v_cache.copy_(torch.from_numpy(vh))
        o = torch.empty((B, H), dtype=torch.int16 if bf else torch.float32, device="cuda")
        plan.decode(xd, pos, o)
        torch.cuda.synchronize()
        outs[bf] = o.cpu().numpy()
        plan.close()
    # the attention half against the oracle, and the hand-off as its rounding
    wts = dict(gamma=w["gamma"], wq=_as64(w["wq"]), wk=_as64(w["wk"]), wv=_as64(w["wv"]), wo=_as64(w["wo"]),
               bq=w["bq"].astype(np.float64), bk=w["bk"].astype(np.float64), bv=w["bv"].astype(np.float64),
               bo=w["bo"].astype(np.float64), sinks=w["sinks"].astype(np.float64))
    ref = np.stack([A.decode_step(wts, x[b], kh[b, :p + 1].astype(np.float64), vh[b, :p + 1].astype(np.float64), p,
                                  q_heads=QH, kv_heads=KVH, head_dim=64, sliding=window > 0, window=window or 1,
                                  eps=1e-5)[0] for b, p in enumerate(positions)])
    check_close(outs[False], ref, x, what="attention half")
    hand_off = outs[True].view(np.uint16)
    assert np.array_equal(hand_off, synth.f32_to_bf16_bits(outs[False]))
    # the MoE block on the GPU's hand-off
    got, plan, _ = run_gpu(blk, hand_off)
    want = oracle.moe_forward(blk, hand_off)
    assert np.array_equal(got["ids"], want["ids"])
    check_permutation(got, want["ids"], sh)
    check_close(got["out"], want["out"], hand_off, what="MoE block on the attention output")
    plan.close()
