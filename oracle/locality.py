"""Expert-locality statistics of a routing trace, written plainly from the
pages (TEST INFRASTRUCTURE ONLY, like the rest of this folder: the tests are
its only users; the CUDA library never imports it and it never imports the
library).

Follows antirez ds4, ds4.c, the Metal expert locality profiler
(`ds4_expert_profile_record`, `ds4_expert_profile_cache_use`,
`ds4_expert_profile_write_cache_summary`), whose per-layer histogram is also
goosedump gpt_oss.rs `ExpertRouteProfile` (`record`, `selections`,
`unique_layer_experts`, `layer_unique_counts`).  For every recorded token of a
layer, in the page's order:

* the layer's record count goes up by one;
* if the layer's previous recorded token sat at the position just before this
  one, the two selected sets are compared: the intersection counts each
  previous selection found among the current ones, the union is 2k minus it;
  the adjacent-pair count, the sum of intersection / k and the sum of
  intersection / union go up;
* the token becomes the layer's previous one;
* each selected expert (slot order) adds one to its count and its route
  weight to its weight total (experts outside [0, E) are skipped), and is
  looked up in one most-recently-used list per cache capacity: found, it
  counts a hit (and its weight a weighted hit) and moves to the front; not
  found, it goes in front and the list drops its last entry if it would exceed
  the capacity.

Plain Python loops over plain lists: sizes of a few thousand selections.
"""
from __future__ import annotations

import numpy as np


class Locality:
    def __init__(self, n_layer: int, n_expert: int, k: int, caps):
        self.L, self.E, self.k = n_layer, n_expert, k
        self.caps = [int(c) for c in caps if 0 < int(c) <= n_expert]
        self.layer_records = [0] * n_layer
        self.total_records = 0
        self.prev_valid = [False] * n_layer
        self.prev_pos = [0] * n_layer
        self.prev_selected = [[0] * k for _ in range(n_layer)]
        self.adjacent_pairs = [0] * n_layer
        self.adjacent_overlap_sum = [0.0] * n_layer
        self.adjacent_jaccard_sum = [0.0] * n_layer
        self.hist = [[0] * n_expert for _ in range(n_layer)]
        self.weight_hist = [[0.0] * n_expert for _ in range(n_layer)]
        self.total_selections = 0
        self.total_weight = 0.0
        self.cache_entries = [[[] for _ in range(n_layer)] for _ in self.caps]
        self.cache_hits = [[0] * n_layer for _ in self.caps]
        self.cache_weight_hits = [[0.0] * n_layer for _ in self.caps]

    def _cache_use(self, ci: int, il: int, expert: int, weight: float):
        cap = self.caps[ci]
        entries = self.cache_entries[ci][il]
        if expert in entries:
            self.cache_hits[ci][il] += 1
            self.cache_weight_hits[ci][il] += float(weight)
            entries.remove(expert)
            entries.insert(0, expert)
            return
        entries.insert(0, expert)
        if len(entries) > cap:
            entries.pop()

    def record(self, il: int, pos: int, selected, weights):
        """One token of layer il at sequence position pos: its k selected
        experts (slot order) and their route weights."""
        if il < 0 or il >= self.L:
            return
        k = self.k
        self.layer_records[il] += 1
        self.total_records += 1
        if self.prev_valid[il] and self.prev_pos[il] + 1 == pos:
            inter = 0
            for a in range(k):
                for b in range(k):
                    if self.prev_selected[il][a] == int(selected[b]):
                        inter += 1
                        break
            union = 2 * k - inter
            self.adjacent_pairs[il] += 1
            self.adjacent_overlap_sum[il] += inter / k
            if union != 0:
                self.adjacent_jaccard_sum[il] += inter / union
        self.prev_valid[il] = True
        self.prev_pos[il] = pos
        for s in range(k):
            e, w = int(selected[s]), float(np.float32(weights[s]))
            self.prev_selected[il][s] = e
            if e < 0 or e >= self.E:
                continue
            self.hist[il][e] += 1
            self.weight_hist[il][e] += w
            self.total_selections += 1
            self.total_weight += w
            for ci in range(len(self.caps)):
                self._cache_use(ci, il, e, w)

    def record_batch(self, il: int, first_pos: int, ids, weights):
        """Tokens t = 0..T-1 of one forward at positions first_pos + t."""
        for t in range(ids.shape[0]):
            self.record(il, first_pos + t, ids[t], weights[t])

    # ---- the summaries the pages derive from the counts
    def selections(self) -> int:
        return int(sum(sum(r) for r in self.hist))

    def unique_layer_experts(self) -> int:
        return int(sum(1 for r in self.hist for c in r if c))

    def layer_unique_counts(self):
        return [sum(1 for c in r if c) for r in self.hist]

    def cache_summary(self):
        """Per capacity: hits, selections, hit rate, weighted hit rate."""
        out = []
        for ci, cap in enumerate(self.caps):
            hits = sum(self.cache_hits[ci])
            wh = sum(self.cache_weight_hits[ci])
            out.append(dict(n=cap, hits=hits, selections=self.total_selections,
                            hit_rate=hits / self.total_selections if self.total_selections else 0.0,
                            weighted_hit_rate=wh / self.total_weight if self.total_weight > 0 else 0.0))
        return out
