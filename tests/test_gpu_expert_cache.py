"""GPU tests of the expert cache (plan option expert_cache_slots): the expert
matrices in pinned host memory (the store), C device slots, slots chosen and
missing experts copied on the device after the routing (antirez ds4 ds4.c, the
expert cache beside `ds4_expert_profile_record`; goosedump gpt_oss.rs
`ExpertStore`).

* Outputs and routes equal those of a plan whose weights are resident in HBM,
  bit for bit, over a sequence of forwards that hit and miss; one forward is
  also checked against the oracle at the block tolerance.
* The slot table after every forward equals the policy's own statement, run
  here on the host from the forward's routed experts: resident experts hit;
  each missing expert, in ascending order, takes the least recently used slot
  the forward does not use (the lowest slot on a tie; empty slots first).
* Calls the cache cannot serve are refused before anything runs."""
import numpy as np
import pytest

import oracle
from mxfp4_mixture_experts_rms_gb300 import moe, synth

from gpu_helpers import check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    moe.load()


class PolicyModel:
    """The cache policy, restated on the host."""

    def __init__(self, n_experts, slots):
        self.slot_of = np.full(n_experts, -1, np.int64)
        self.expert_of = [-1] * slots
        self.stamp = [-1] * slots
        self.fwd = 0
        self.hits = self.misses = 0

    def step(self, used):
        now = self.fwd + 1
        for e in used:
            if self.slot_of[e] >= 0:
                self.stamp[self.slot_of[e]] = now
                self.hits += 1
        for e in used:
            if self.slot_of[e] < 0:
                free = [s for s in range(len(self.stamp)) if self.stamp[s] != now]
                s = min(free, key=lambda q: (self.stamp[q], q))
                if self.expert_of[s] >= 0:
                    self.slot_of[self.expert_of[s]] = -1
                self.expert_of[s] = e
                self.slot_of[e] = s
                self.stamp[s] = now
                self.misses += 1
        self.fwd = now


def _run_sequence(shape, blk, config, slots, token_counts, check_oracle_at=None):
    import torch
    T_max = max(token_counts)
    ref = moe.Plan(shape, max_tokens=T_max).alloc_workspace().load_weights(moe.DeviceBlock(blk))
    cached = moe.Plan(shape, max_tokens=T_max, expert_cache_slots=slots).alloc_workspace()
    cached.load_weights(moe.HostStoreBlock(blk))
    model = PolicyModel(shape.n_experts, slots)
    for i, T in enumerate(token_counts):
        x_bits = synth.make_tokens(config, T, shape.hidden, sub=100 + i)
        x = torch.from_numpy(x_bits.view(np.int16)).cuda()
        outs, idss = [], []
        for plan in (ref, cached):
            out = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
            ids = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
            plan.forward(x, out, ids)
            torch.cuda.synchronize()
            outs.append(out.cpu().numpy())
            idss.append(ids.cpu().numpy())
        assert np.array_equal(idss[0], idss[1]), f"forward {i}: routes differ"
        assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32)), f"forward {i}: outputs differ"
        assert cached.device_status() == 0
        model.step(sorted(set(idss[1].ravel().tolist())))
        slot_of, hits, misses, fwds = cached.cache_state()
        assert np.array_equal(slot_of, model.slot_of), f"forward {i}: slot table"
        assert (hits, misses, fwds) == (model.hits, model.misses, i + 1)
        if check_oracle_at == i:
            r = oracle.moe_forward(blk, x_bits)
            assert np.array_equal(idss[1], r["ids"])
            check_close(outs[1], r["out"], x_bits, what="cached block against the oracle")
    ref.close()
    cached.close()
    return model


def test_gpt_oss_block_through_a_12_slot_cache():
    """gpt-oss shape (32 experts, top-4), 12 slots, 1-3 tokens per forward:
    the early forwards miss, later ones evict and hit."""
    blk = synth.make_block(0)
    model = _run_sequence(blk["shape"], blk, 0, 12, [1, 3, 2, 1, 3, 3, 1, 2, 3, 1], check_oracle_at=4)
    assert model.hits > 0 and model.misses > 12  # the sequence both reuses and evicts


def test_the_benchmark_launch_4_tokens_16_slots():
    """The benchmark's own configuration: 4 tokens a step through 16 slots of
    the gpt-oss block's 32 experts, fresh tokens every step."""
    blk = synth.make_block(0)
    model = _run_sequence(blk["shape"], blk, 0, 16, [4] * 8)
    assert model.misses > 16


def test_shared_expert_and_a_cache_of_every_expert():
    """A small shape with an always-on shared expert (kept on the device, not
    cached): 4 slots for 16 experts at top-2, then a cache as large as the
    expert count (after the first touch of each expert, only hits)."""
    shape = synth.BlockShape(256, 128, 16, 2, n_shared=1)
    blk = synth.make_block(0, shape=shape)
    _run_sequence(shape, blk, 0, 4, [1, 2, 1, 2, 2, 1, 2])
    model = _run_sequence(shape, blk, 0, 16, [8, 8, 8, 8])
    assert model.misses <= 16


def test_256_experts_top_8_with_a_shared_expert():
    """Many experts (the assignment walks them in eight groups of 32; the
    routing uses its 16-CTA clusters): a small 256-expert, top-8 shape with a
    shared expert through 24 slots, 1-3 tokens per forward."""
    shape = synth.BlockShape(256, 128, 256, 8, n_shared=1)
    blk = synth.make_block(0, shape=shape)
    model = _run_sequence(shape, blk, 0, 24, [3, 1, 2, 3, 3, 2, 1, 3])
    assert model.misses > 24


def test_calls_the_cache_cannot_serve_are_refused():
    import torch
    blk = synth.make_block(0)
    shape = blk["shape"]
    plan = moe.Plan(shape, max_tokens=64, expert_cache_slots=8).alloc_workspace()
    plan.load_weights(moe.HostStoreBlock(blk))
    x = torch.from_numpy(synth.make_tokens(0, 3, shape.hidden).view(np.int16)).cuda()
    out = torch.empty((3, shape.hidden), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:          # 3 tokens x top-4 can reach 12 experts > 8 slots
        plan.forward(x, out)
    assert ei.value.status == moe.MOE_ESHAPE
    plan.forward(x[:2], out[:2])                     # 2 x 4 = 8: served
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    plan.close()
    # pageable host memory: refused where the device cannot read it; where it
    # can (a coherent CPU-GPU link), served like pinned memory
    dev = moe.DeviceBlock(blk)
    dev.mats = {m: tuple(t.cpu() for t in v) for m, v in dev.mats.items()}
    plan = moe.Plan(shape, max_tokens=4, expert_cache_slots=8).alloc_workspace()
    try:
        plan.load_weights(dev)
    except moe.MoeError as err:
        assert err.status == moe.MOE_EINVAL
    else:
        ref = moe.Plan(shape, max_tokens=4).alloc_workspace().load_weights(moe.DeviceBlock(blk))
        got, want = (torch.empty((2, shape.hidden), dtype=torch.float32, device="cuda") for _ in range(2))
        plan.forward(x[:2], got)
        ref.forward(x[:2], want)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
        ref.close()
    plan.close()
    # FP4 activations take the grouped GEMM, which the cache does not serve
    plan = moe.Plan(shape, max_tokens=4, expert_cache_slots=8, act_fp4=1).alloc_workspace()
    with pytest.raises(moe.MoeError) as ei:
        plan.load_weights(moe.HostStoreBlock(blk))
    assert ei.value.status == moe.MOE_EINVAL
    plan.close()
