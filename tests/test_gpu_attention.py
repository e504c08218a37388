"""GPU parity of the attention decode step (moe_attn_decode) against the
oracle's plain float64 restatement of goosedump gpt_oss.rs (`forward`'s
attention step: norm, projections, YaRN RoPE, fp16 cache append, grouped
attention with sinks over the full or the sliding window, output projection,
residual).  Outputs within the block tolerance (relative L2 <= 1e-3, max abs
<= 2e-3 max|ref|, on the output and on the attention's own contribution;
the bf16 output bit-equal to the fp32 output rounded once);
the appended cache rows within one fp16 rounding of the oracle's; cache rows
the step must not touch unchanged."""
import numpy as np
import pytest

from oracle import attention as A
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


def _as64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def _run(H, QH, KVH, positions, max_ctx, window, seed, out_bf16=False):
    import torch
    B = len(positions)
    w = synth.make_attention(seed, H, QH, KVH)
    kh, vh = synth.make_kv_history(seed, B, max_ctx, KVH)
    x = synth.f32_to_bf16_bits(np.random.default_rng(seed).normal(0.0, 1.0, (B, H)))
    plan = moe.AttnPlan(H, QH, KVH, B, max_ctx, sliding_window=window, out_bf16=out_bf16)
    dev = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda() for k, v in w.items()}
    plan.load_weights(dev)
    plan.k_cache.copy_(torch.from_numpy(kh))
    plan.v_cache.copy_(torch.from_numpy(vh))
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    out = torch.empty((B, H), dtype=torch.int16 if out_bf16 else torch.float32, device="cuda")
    plan.decode(xd, pos, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    kc, vc = plan.k_cache.cpu().numpy(), plan.v_cache.cpu().numpy()
    wts = dict(gamma=w["gamma"], wq=_as64(w["wq"]), wk=_as64(w["wk"]), wv=_as64(w["wv"]), wo=_as64(w["wo"]),
               bq=w["bq"].astype(np.float64), bk=w["bk"].astype(np.float64), bv=w["bv"].astype(np.float64),
               bo=w["bo"].astype(np.float64), sinks=w["sinks"].astype(np.float64))
    refs = []
    for b, p in enumerate(positions):
        kr = kh[b, :p + 1].astype(np.float64)
        vr = vh[b, :p + 1].astype(np.float64)
        out_r, _, _ = A.decode_step(wts, x[b], kr, vr, p, q_heads=QH, kv_heads=KVH, head_dim=64,
                                    sliding=window > 0, window=window or 1, eps=1e-5)
        refs.append((out_r, kr[p], vr[p]))
        # the appended rows: within one fp16 rounding of the oracle's, beyond
        # the fp32 accumulation error of the projection (1e-5 of the row's
        # largest entry: entries near zero come from cancelling sums)
        for got_row, ref_row in ((kc[b, p], kr[p]), (vc[b, p], vr[p])):
            g = got_row.astype(np.float64)
            assert np.all(np.abs(g - ref_row) <= 2.0 ** -10 * np.abs(ref_row) + 1e-5 * np.abs(ref_row).max()), (b, p)
        # every other row as it was
        others = np.ones(max_ctx, bool)
        others[p] = False
        assert np.array_equal(kc[b, others], kh[b, others]) and np.array_equal(vc[b, others], vh[b, others])
    ref = np.stack([r[0] for r in refs])
    if out_bf16:
        # the bf16 output is the fp32 output rounded once (a second plan with
        # the same weights and history, fp32 out), and that is within tolerance
        plan32 = moe.AttnPlan(H, QH, KVH, B, max_ctx, sliding_window=window)
        plan32.load_weights(dev)
        plan32.k_cache.copy_(torch.from_numpy(kh))
        plan32.v_cache.copy_(torch.from_numpy(vh))
        out32 = torch.empty((B, H), dtype=torch.float32, device="cuda")
        plan32.decode(xd, pos, out32)
        torch.cuda.synchronize()
        got32 = out32.cpu().numpy()
        assert np.array_equal(got.view(np.uint16), synth.f32_to_bf16_bits(got32))
        check_close(got32, ref, x, what=f"attention out (window {window})")
        plan32.close()
    else:
        check_close(got, ref, x, what=f"attention out (window {window})")
    plan.close()


@pytest.mark.parametrize("window", [0, 128])
def test_gpt_oss_attention_decode(window):
    """gpt-oss shape (2880 hidden, 64 query heads over 8 kv heads): an empty
    cache, short contexts, contexts across the 256-token chunk boundary and
    beyond the 128-token window, and a position near the end of the cache."""
    _run(2880, 64, 8, [0, 5, 127, 128, 255, 256, 300, 1022], 1024, window, seed=1 + window)


@pytest.mark.parametrize("window", [0, 128])
def test_decode_at_the_benchmark_size(window):
    """The benchmark's own launch: 16 sequences whose new token is the last
    row of a 4096-row cache (the streamed kernel's split count and chunking
    as timed), full and sliding."""
    _run(2880, 64, 8, [4095] * 16, 4096, window, seed=7 + window)


def test_ragged_batch_sizes_and_small_shapes():
    """Every MMA column tile count (1..32 sequences), a smaller head layout
    (4 query heads per kv head), the bf16 output."""
    _run(256, 8, 2, [3], 64, 0, seed=5)
    _run(256, 8, 2, list(range(9)), 64, 16, seed=6)
    _run(512, 16, 4, [i * 7 % 300 for i in range(17)], 320, 0, seed=7)
    _run(512, 16, 1, [i * 13 % 300 for i in range(32)], 320, 100, seed=8)
    _run(2880, 64, 8, [10, 700], 768, 128, seed=9, out_bf16=True)


def test_position_outside_the_cache_is_skipped():
    """A position at or beyond max_ctx writes nothing into the caches."""
    import torch
    H, QH, KVH, ctx = 256, 8, 2, 32
    w = synth.make_attention(3, H, QH, KVH)
    plan = moe.AttnPlan(H, QH, KVH, 2, ctx)
    plan.load_weights({k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
                       for k, v in w.items()})
    x = torch.from_numpy(synth.f32_to_bf16_bits(np.ones((2, H))).view(np.int16)).cuda()
    out = torch.empty((2, H), dtype=torch.float32, device="cuda")
    plan.decode(x, torch.tensor([ctx, 4], dtype=torch.int32, device="cuda"), out)
    torch.cuda.synchronize()
    kc = plan.k_cache.cpu().numpy()
    assert not kc[0].any()                      # sequence 0 untouched
    assert kc[1, 4].any() and not kc[1, :4].any() and not kc[1, 5:].any()
    plan.close()


def test_repeated_steps_are_bitwise_identical():
    """The same step three times on one plan (the cache row it appends is
    rewritten with the same values): identical outputs, so the projections'
    cross-CTA partial sums are added in a fixed order and their tickets come
    back to zero after every launch.  Shapes whose tiles are shared by two,
    three and four CTAs."""
    import torch
    for H, QH, KVH, B in [(2880, 64, 8, 16), (512, 16, 4, 5), (256, 8, 2, 32)]:
        w = synth.make_attention(21, H, QH, KVH)
        kh, vh = synth.make_kv_history(21, B, 300, KVH)
        plan = moe.AttnPlan(H, QH, KVH, B, 300, sliding_window=0)
        plan.load_weights({k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
                           for k, v in w.items()})
        plan.k_cache.copy_(torch.from_numpy(kh))
        plan.v_cache.copy_(torch.from_numpy(vh))
        x = torch.from_numpy(synth.f32_to_bf16_bits(np.random.default_rng(2).normal(0, 1, (B, H))).view(np.int16)).cuda()
        pos = torch.tensor([(37 * i) % 300 for i in range(B)], dtype=torch.int32, device="cuda")
        outs = []
        for _ in range(3):
            out = torch.empty((B, H), dtype=torch.float32, device="cuda")
            plan.decode(x, pos, out)
            outs.append(out.cpu().numpy())
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
        plan.close()



@pytest.mark.parametrize("window,prefill_rows", [(0, 0), (16, 0), (16, 64), (0, 33)])
def test_prefill_matches_the_oracle(window, prefill_rows):
    """Prefill (goosedump gpt_oss.rs prefill_attention_layer): 40 new tokens
    of sequence 1 in blocks of the plan's 16 rows (or 64 or 33: one block, a
    ragged one; the projections then take the tokens 32 at a time on their
    grid's second axis), after 300 cached tokens
    (across the first 256-token chunk's end), then 9 more from position 340;
    and a first prompt of 5 tokens into the empty sequence 2.  Outputs within the block tolerance; the new cache rows
    within one fp16 rounding; every other cache row unchanged."""
    import torch
    H, QH, KVH, S, ctx = 512, 16, 4, 16, 600
    w = synth.make_attention(51 + window, H, QH, KVH)
    kh, vh = synth.make_kv_history(51, S, ctx, KVH)
    dev = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda() for k, v in w.items()}
    plan = moe.AttnPlan(H, QH, KVH, S, ctx, sliding_window=window, prefill_rows=prefill_rows)
    plan.load_weights(dev)
    plan.k_cache.copy_(torch.from_numpy(kh))
    plan.v_cache.copy_(torch.from_numpy(vh))
    wts = dict(gamma=w["gamma"], wq=_as64(w["wq"]), wk=_as64(w["wk"]), wv=_as64(w["wv"]), wo=_as64(w["wo"]),
               bq=w["bq"].astype(np.float64), bk=w["bk"].astype(np.float64), bv=w["bv"].astype(np.float64),
               bo=w["bo"].astype(np.float64), sinks=w["sinks"].astype(np.float64))
    kref, vref = kh.astype(np.float64), vh.astype(np.float64)
    rng = np.random.default_rng(4)
    for seq, pos0, n in [(1, 300, 40), (1, 340, 9), (2, 0, 5)]:
        x = synth.f32_to_bf16_bits(rng.normal(0.0, 1.0, (n, H)))
        out = torch.empty((n, H), dtype=torch.float32, device="cuda")
        plan.prefill(torch.from_numpy(x.view(np.int16)).cuda(), seq, pos0, out)
        torch.cuda.synchronize()
        kseq, vseq = kref[seq, :pos0 + n].copy(), vref[seq, :pos0 + n].copy()
        ref = A.prefill(wts, x, kseq, vseq, pos0, q_heads=QH, kv_heads=KVH, head_dim=64, sliding=window > 0,
                        window=window or 1, eps=1e-5)
        check_close(out.cpu().numpy(), ref, x, what=f"prefill seq {seq} from {pos0}")
        kc, vc = plan.k_cache.cpu().numpy(), plan.v_cache.cpu().numpy()
        for got_c, ref_rows in ((kc, kseq), (vc, vseq)):
            g = got_c[seq, pos0:pos0 + n].astype(np.float64)
            r = ref_rows[pos0:pos0 + n]
            assert np.all(np.abs(g - r) <= 2.0 ** -10 * np.abs(r) + 1e-5 * np.abs(r).max())
        assert plan.device_status() == 0
        # the oracle continues from the GPU's appended rows; nothing else moved
        kref[seq, pos0:pos0 + n] = kc[seq, pos0:pos0 + n]
        vref[seq, pos0:pos0 + n] = vc[seq, pos0:pos0 + n]
        assert np.array_equal(kc, kref.astype(np.float16)) and np.array_equal(vc, vref.astype(np.float16))
    plan.close()


@pytest.mark.parametrize("pos0,n", [(100, 150), (0, 400)])
def test_prefill_gpt_oss_shape_tensor_core_projections(pos0, n):
    """Prompts at gpt-oss shapes in one block, the projections as tensor-core
    GEMMs: 150 tokens after 100 cached ones (two 128-token tiles, 128-row
    weight tiles), and 400 tokens into an empty cache (four token tiles: the
    Q/K/V GEMM takes 256-row weight tiles), on a sliding layer: every output
    row within the block tolerance."""
    import torch
    a = synth.ATTN_GPT_OSS
    H, QH, KVH, S, ctx = a["hidden"], a["q_heads"], a["kv_heads"], 2, 512
    w = synth.make_attention(61, H, QH, KVH)
    kh, vh = synth.make_kv_history(61, S, ctx, KVH)
    dev = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda() for k, v in w.items()}
    plan = moe.AttnPlan(H, QH, KVH, S, ctx, sliding_window=a["window"], prefill_rows=n)
    plan.load_weights(dev)
    plan.k_cache.copy_(torch.from_numpy(kh))
    plan.v_cache.copy_(torch.from_numpy(vh))
    x = synth.f32_to_bf16_bits(np.random.default_rng(8).normal(0.0, 1.0, (n, H)))
    out = torch.empty((n, H), dtype=torch.float32, device="cuda")
    plan.prefill(torch.from_numpy(x.view(np.int16)).cuda(), 1, pos0, out)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    wts = dict(gamma=w["gamma"], wq=_as64(w["wq"]), wk=_as64(w["wk"]), wv=_as64(w["wv"]), wo=_as64(w["wo"]),
               bq=w["bq"].astype(np.float64), bk=w["bk"].astype(np.float64), bv=w["bv"].astype(np.float64),
               bo=w["bo"].astype(np.float64), sinks=w["sinks"].astype(np.float64))
    kseq, vseq = kh[1, :pos0 + n].astype(np.float64), vh[1, :pos0 + n].astype(np.float64)
    ref = A.prefill(wts, x, kseq, vseq, pos0, q_heads=QH, kv_heads=KVH, head_dim=64, sliding=True,
                    window=a["window"], eps=1e-5)
    check_close(out.cpu().numpy(), ref, x, what="prefill at gpt-oss shapes")
    plan.close()


@pytest.mark.parametrize("window", [0, 128])
def test_prefill_at_the_benchmark_size(window):
    """The benchmark's own launch: one 512-token prompt into the empty cache
    of one of 32 sequences (4096 rows each), in one block of 512 rows, full
    and sliding: every output row within the block tolerance, the appended
    rows within one fp16 rounding."""
    import torch
    a = synth.ATTN_GPT_OSS
    H, QH, KVH, S, ctx, n = a["hidden"], a["q_heads"], a["kv_heads"], 32, 4096, 512
    w = synth.make_attention(71 + window, H, QH, KVH)
    dev = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda() for k, v in w.items()}
    plan = moe.AttnPlan(H, QH, KVH, S, ctx, sliding_window=window, prefill_rows=n)
    plan.load_weights(dev)
    plan.k_cache.zero_()
    plan.v_cache.zero_()
    x = synth.f32_to_bf16_bits(np.random.default_rng(9).normal(0.0, 1.0, (n, H)))
    out = torch.empty((n, H), dtype=torch.float32, device="cuda")
    plan.prefill(torch.from_numpy(x.view(np.int16)).cuda(), 0, 0, out)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    wts = dict(gamma=w["gamma"], wq=_as64(w["wq"]), wk=_as64(w["wk"]), wv=_as64(w["wv"]), wo=_as64(w["wo"]),
               bq=w["bq"].astype(np.float64), bk=w["bk"].astype(np.float64), bv=w["bv"].astype(np.float64),
               bo=w["bo"].astype(np.float64), sinks=w["sinks"].astype(np.float64))
    kseq, vseq = np.zeros((n, KVH, 64)), np.zeros((n, KVH, 64))
    ref = A.prefill(wts, x, kseq, vseq, 0, q_heads=QH, kv_heads=KVH, head_dim=64, sliding=window > 0,
                    window=window or 1, eps=1e-5)
    check_close(out.cpu().numpy(), ref, x, what=f"prefill at the benchmark size (window {window})")
    kc, vc = plan.k_cache[0, :n].cpu().numpy(), plan.v_cache[0, :n].cpu().numpy()
    for got_c, r in ((kc, kseq), (vc, vseq)):
        g = got_c.astype(np.float64)
        assert np.all(np.abs(g - r) <= 2.0 ** -10 * np.abs(r) + 1e-5 * np.abs(r).max())
    plan.close()


def test_prefill_sixteen_query_heads_per_kv_head():
    """16 query heads on one kv head (the flash kernel's 512-thread form):
    a 40-token prompt after 20 cached tokens, full and sliding (24)."""
    import torch
    H, QH, KVH, S, ctx, pos0, n = 256, 16, 1, 2, 96, 20, 40
    for window in (0, 24):
        w = synth.make_attention(71 + window, H, QH, KVH)
        kh, vh = synth.make_kv_history(71, S, ctx, KVH)
        dev = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda() for k, v in w.items()}
        plan = moe.AttnPlan(H, QH, KVH, S, ctx, sliding_window=window, prefill_rows=64)
        plan.load_weights(dev)
        plan.k_cache.copy_(torch.from_numpy(kh))
        plan.v_cache.copy_(torch.from_numpy(vh))
        x = synth.f32_to_bf16_bits(np.random.default_rng(9).normal(0.0, 1.0, (n, H)))
        out = torch.empty((n, H), dtype=torch.float32, device="cuda")
        plan.prefill(torch.from_numpy(x.view(np.int16)).cuda(), 0, pos0, out)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        wts = dict(gamma=w["gamma"], wq=_as64(w["wq"]), wk=_as64(w["wk"]), wv=_as64(w["wv"]), wo=_as64(w["wo"]),
                   bq=w["bq"].astype(np.float64), bk=w["bk"].astype(np.float64), bv=w["bv"].astype(np.float64),
                   bo=w["bo"].astype(np.float64), sinks=w["sinks"].astype(np.float64))
        ref = A.prefill(wts, x, kh[0, :pos0 + n].astype(np.float64), vh[0, :pos0 + n].astype(np.float64), pos0,
                        q_heads=QH, kv_heads=KVH, head_dim=64, sliding=window > 0, window=window or 1, eps=1e-5)
        check_close(out.cpu().numpy(), ref, x, what=f"prefill, 16 heads per kv head, window {window}")
        plan.close()


def test_bad_arguments_are_refused_before_anything_runs():
    """Sequence index and positions outside the plan, a prompt that runs past
    the cache, too many sequences, overlapping x and out: refused with
    MOE_EINVAL and a message, the caches untouched."""
    import torch
    H, QH, KVH, S, ctx = 256, 8, 2, 2, 64
    w = synth.make_attention(81, H, QH, KVH)
    plan = moe.AttnPlan(H, QH, KVH, S, ctx)
    plan.load_weights({k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
                       for k, v in w.items()})
    x = torch.zeros((4, H), dtype=torch.int16, device="cuda")
    out = torch.empty((4, H), dtype=torch.float32, device="cuda")
    for call in (lambda: plan.prefill(x, S, 0, out),            # no sequence S
                 lambda: plan.prefill(x, -1, 0, out),
                 lambda: plan.prefill(x, 0, ctx - 3, out),      # rows ctx - 3 .. ctx: one past the cache
                 lambda: plan.prefill(x, 0, -1, out),
                 lambda: plan.decode(x[:3], torch.zeros(3, dtype=torch.int32, device="cuda"), out),  # 3 > max_seqs
                 lambda: plan.decode(x[:2], torch.zeros(2, dtype=torch.int32, device="cuda"), x[:2])):  # out == x
        with pytest.raises(moe.MoeError) as ei:
            call()
        assert ei.value.status == moe.MOE_EINVAL, ei.value
    torch.cuda.synchronize()
    assert not plan.k_cache.any() and not plan.v_cache.any()
    plan.close()
