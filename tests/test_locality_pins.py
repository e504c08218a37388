"""Pins of the oracle's expert-locality statistics (ds4.c expert locality
profiler; goosedump gpt_oss.rs ExpertRouteProfile) against definitions that
are not its own code: closed forms of constructed traces, least-recently-used
membership by brute force over the access history, and hand-counted
overlaps.  Each planted mistake at the end (a first-in-first-out list, the
miss inserted at the back, the union not reduced by the intersection,
adjacency without the position test, invalid experts counted) must fail one of them."""

import numpy as np
import pytest

from oracle.locality import Locality


def _trace(rng, T, E, k):
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return ids, w


def _lru_hits_brute(accesses, cap):
    """Hit iff the expert is among the `cap` distinct experts used most
    recently before this access (the definition of a least-recently-used
    cache of capacity cap), by scanning the history backwards."""
    hits = []
    for i, e in enumerate(accesses):
        seen = []
        for prev in reversed(accesses[:i]):
            if prev not in seen:
                seen.append(prev)
            if len(seen) == cap:
                break
        hits.append(e in seen)
    return hits


def _check_lru(L, ids, w, caps, il=0):
    acc = [int(e) for e in ids.reshape(-1)]
    ws = [float(x) for x in w.reshape(-1)]
    for ci, cap in enumerate(caps):
        h = _lru_hits_brute(acc, cap)
        assert L.cache_hits[ci][il] == sum(h), (cap, L.cache_hits[ci][il], sum(h))
        want_w = 0.0
        for hit, x in zip(h, ws):
            if hit:
                want_w += x
        assert L.cache_weight_hits[ci][il] == pytest.approx(want_w, rel=1e-12)


def test_repeating_selection_closed_form():
    """The same k experts every token at consecutive positions: every count is
    T, each adjacent pair overlaps fully, caches of at least k entries hit on
    every selection after the first token, smaller ones never (they cycle)."""
    T, E, k = 20, 16, 4
    sel = np.array([3, 9, 0, 12], np.int32)
    w = np.array([0.5, 0.25, 0.125, 0.125], np.float32)
    L = Locality(1, E, k, [2, 3, 4, 8])
    for t in range(T):
        L.record(0, 100 + t, sel, w)
    assert L.layer_records[0] == T and L.total_selections == T * k
    assert [L.hist[0][e] for e in sel] == [T] * k and L.selections() == T * k
    assert L.unique_layer_experts() == k and L.layer_unique_counts() == [k]
    assert L.adjacent_pairs[0] == T - 1
    assert L.adjacent_overlap_sum[0] == T - 1 and L.adjacent_jaccard_sum[0] == T - 1
    assert L.cache_hits[0][0] == 0 and L.cache_hits[1][0] == 0          # capacities 2, 3 < k
    assert L.cache_hits[2][0] == (T - 1) * k and L.cache_hits[3][0] == (T - 1) * k
    assert L.cache_weight_hits[2][0] == pytest.approx((T - 1) * 1.0)
    s = L.cache_summary()
    assert s[2]["hit_rate"] == pytest.approx((T - 1) / T)
    assert s[2]["weighted_hit_rate"] == pytest.approx((T - 1) / T)
    assert L.weight_hist[0][3] == pytest.approx(T * 0.5) and L.total_weight == pytest.approx(T * 1.0)


@pytest.mark.parametrize("seed,E,k,T", [(1, 8, 2, 60), (2, 16, 4, 50), (3, 32, 4, 40), (4, 12, 6, 30)])
def test_cache_hits_are_least_recently_used_membership(seed, E, k, T):
    rng = np.random.default_rng(seed)
    ids, w = _trace(rng, T, E, k)
    caps = [1, 2, k, k + 1, E // 2, E]
    L = Locality(1, E, k, caps)
    L.record_batch(0, 0, ids, w)
    _check_lru(L, ids, w, L.caps)


def test_adjacent_overlap_counts():
    """Hand-counted: {0,1,2,3} then {2,3,4,5}: intersection 2, union 6; then
    {6,7,8,9} (disjoint); then a gap in positions (no pair); then {9,8,7,6}
    (the same set in another order, full overlap)."""
    L = Locality(1, 16, 4, [4])
    w = np.ones(4, np.float32)
    L.record(0, 0, [0, 1, 2, 3], w)
    L.record(0, 1, [2, 3, 4, 5], w)
    assert L.adjacent_pairs[0] == 1
    assert L.adjacent_overlap_sum[0] == pytest.approx(0.5) and L.adjacent_jaccard_sum[0] == pytest.approx(1 / 3)
    L.record(0, 2, [6, 7, 8, 9], w)
    assert L.adjacent_pairs[0] == 2 and L.adjacent_overlap_sum[0] == pytest.approx(0.5)
    L.record(0, 5, [10, 11, 12, 13], w)                 # not the position after 2
    assert L.adjacent_pairs[0] == 2
    L.record(0, 6, [13, 12, 11, 10], w)
    assert L.adjacent_pairs[0] == 3
    assert L.adjacent_overlap_sum[0] == pytest.approx(1.5)
    assert L.adjacent_jaccard_sum[0] == pytest.approx(1 / 3 + 1.0)


def test_layers_are_independent_and_invalid_experts_skipped():
    L = Locality(3, 8, 2, [2])
    w = np.array([0.5, 0.5], np.float32)
    L.record(0, 0, [1, 2], w)
    L.record(2, 1, [1, 2], w)                             # another layer: no adjacency with layer 0
    assert L.adjacent_pairs == [0, 0, 0]
    L.record(2, 2, [-1, 2], w)                            # expert -1 skipped, still part of the overlap
    assert L.hist[2][2] == 2 and L.hist[2][1] == 1 and L.total_selections == 5
    assert L.adjacent_pairs[2] == 1 and L.adjacent_overlap_sum[2] == pytest.approx(0.5)
    L.record(5, 0, [1, 2], w)                             # layer out of range: ignored
    assert L.total_records == 3
    assert L.layer_unique_counts() == [2, 0, 2]


# ------------------------------------------------------- planted mistakes
class _Fifo(Locality):
    def _cache_use(self, ci, il, expert, weight):  # a hit does not move to the front
        entries = self.cache_entries[ci][il]
        if expert in entries:
            self.cache_hits[ci][il] += 1
            self.cache_weight_hits[ci][il] += weight
            return
        entries.insert(0, expert)
        if len(entries) > self.caps[ci]:
            entries.pop()


class _MissAtBack(Locality):
    def _cache_use(self, ci, il, expert, weight):  # a miss goes to the back
        entries = self.cache_entries[ci][il]
        if expert in entries:
            self.cache_hits[ci][il] += 1
            self.cache_weight_hits[ci][il] += weight
            entries.remove(expert)
            entries.insert(0, expert)
            return
        if len(entries) < self.caps[ci]:
            entries.append(expert)
        else:
            entries[-1] = expert


class _UnionNoSubtract(Locality):
    def record(self, il, pos, selected, weights):  # the union taken as 2k, the intersection not subtracted
        j0 = self.adjacent_jaccard_sum[il]
        adj = self.prev_valid[il] and self.prev_pos[il] + 1 == pos
        inter = sum(1 for a in self.prev_selected[il] if a in [int(e) for e in selected]) if adj else 0
        super().record(il, pos, selected, weights)
        if adj:
            self.adjacent_jaccard_sum[il] = j0 + inter / (2 * self.k)


class _NoPositionTest(Locality):
    def record(self, il, pos, selected, weights):  # any previous token counts as adjacent
        if self.prev_valid[il]:
            pos = self.prev_pos[il] + 1
        super().record(il, pos, selected, weights)


class _CountsInvalid(Locality):
    def record(self, il, pos, selected, weights):  # an invalid expert lands in expert 0
        super().record(il, pos, [e if 0 <= e < self.E else 0 for e in selected], weights)


def _pins_pass(cls):
    try:
        rng = np.random.default_rng(7)
        ids, w = _trace(rng, 40, 16, 4)
        L = cls(1, 16, 4, [2, 4, 5, 8])
        L.record_batch(0, 0, ids, w)
        _check_lru(L, ids, w, L.caps)
        M = cls(1, 16, 4, [4])
        one = np.ones(4, np.float32)
        for pos, sel in [(0, [0, 1, 2, 3]), (1, [2, 3, 4, 5]), (2, [6, 7, 8, 9]), (5, [10, 11, 12, 13]),
                         (6, [13, 12, 11, 10])]:
            M.record(0, pos, sel, one)
        assert M.adjacent_pairs[0] == 3 and M.adjacent_overlap_sum[0] == pytest.approx(1.5)
        assert M.adjacent_jaccard_sum[0] == pytest.approx(1 / 3 + 1.0)
        N = cls(3, 8, 2, [2])
        N.record(0, 0, [1, 2], np.ones(2, np.float32))
        N.record(0, 1, [-1, 2], np.ones(2, np.float32))
        assert N.hist[0][0] == 0 and N.total_selections == 3
        return True
    except AssertionError:
        return False


def test_the_pins_pass_on_the_oracle():
    assert _pins_pass(Locality)


@pytest.mark.parametrize("cls", [_Fifo, _MissAtBack, _UnionNoSubtract, _NoPositionTest, _CountsInvalid])
def test_each_planted_mistake_fails_a_pin(cls):
    assert not _pins_pass(cls)
