"""The GPU block cache's bookkeeping, written out plainly: which (page, kv head) blocks a call
uses, which of them are hits, and which slots the misses take.

TEST INFRASTRUCTURE (see the package docstring). Pure Python: the cache of a test holds a
few hundred slots.

Sources: InfiniteHiP article (163.com), section "实现 7.24 倍的端到端解码加速" (the GPU keeps a
cache of recently used KV blocks, least recently used first out, the rest of the KV cache in
host memory); HCAttention excerpt, contribution list (dynamic, reversible eviction of the
least important KV pairs from the GPU cache by a cumulative-magnitude criterion).

Readings (the pages give the policies' names only):
  * a call's blocks are its segments in the attention's order: for every (sequence b, kv
    head h) in ascending order, the sink pages, the window pages, then the kept blocks
    (clipped to the candidate region; a kept block without a candidate token is no segment);
  * the cache unit is a (page, kv head) block, key = page * hkv + h; a block that is two
    segments of one call (a partial sink or window page that is also kept) is looked up once;
  * "least recently used" is exact: every slot carries the number of the last call that used
    it; a hit refreshes it; the misses, in call order, take the slots this call does not use
    with the oldest stamps, ties to the lower slot, assigned in ascending slot order;
  * the cumulative-magnitude policy takes free slots first (lower slot first), then the slots
    whose blocks have the least cumulative attention mass (ties: the lower slot);
  * the page holding a sequence's last token may have changed since it was cached (the
    append writes it): a hit on it is copied again ("refresh").
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np


@dataclasses.dataclass
class CacheState:
    """slot_of[key] = slot + 1 (0: not cached); key_of[slot] = key + 1 (0: free);
    stamp[slot] = last call that used the slot (0: never); step = calls so far."""
    slot_of: np.ndarray
    key_of: np.ndarray
    stamp: np.ndarray
    step: int = 0

    @classmethod
    def empty(cls, num_keys: int, capacity: int) -> "CacheState":
        return cls(np.zeros(num_keys, np.int64), np.zeros(capacity, np.int64),
                   np.zeros(capacity, np.int64), 0)

    def copy(self) -> "CacheState":
        return CacheState(self.slot_of.copy(), self.key_of.copy(), self.stamp.copy(), self.step)


def call_segments(n: int, sink: int, window: int, k2: int, block_idx: Sequence[int],
                  n_blocks: int, block: int = 16) -> List[Optional[int]]:
    """Segments of one (sequence, kv head) in the attention's order: the block of each, or
    None for an unused entry. n: the context; block_idx / n_blocks: the kept blocks."""
    sink_end = min(sink, n)
    n_sink = -(-sink_end // block)
    cand_hi = n - window
    n_sel_max = k2 if cand_hi > sink else 0
    w0 = max(n - window, sink_end)
    n_win = -(-n // block) - w0 // block if w0 < n else 0
    segs: List[Optional[int]] = [i for i in range(n_sink)]
    segs += [w0 // block + i for i in range(n_win)]
    for r in range(n_sel_max):
        k = None
        if r < min(max(int(n_blocks), 0), n_sel_max):
            kk = int(block_idx[r])
            if 0 <= kk < -(-n // block) and max(kk * block, sink) < min(kk * block + block, cand_hi):
                k = kk
        segs.append(k)
    return segs


def cache_plan(state: CacheState, calls: Sequence[Tuple[Tuple[int, int], Sequence[Optional[int]],
                                                       int]],
               page_table: np.ndarray, hkv: int, policy: int = 0,
               mass: Optional[np.ndarray] = None) -> Dict[str, list]:
    """One call of the cache, in place on `state`. calls: ((b, h), segments, last_block) for
    every (sequence, kv head) in order (segments as call_segments returns them; last_block:
    the block holding the sequence's last token). policy 0: least recently used; policy 1:
    least cumulative mass, mass[key] the masses before this call. Returns the hits (slots),
    the misses (keys, call order), the victims (slots, ascending, one per miss), the evicted
    keys and the refreshes ((slot, key) of hits on a last-token page)."""
    state.step += 1
    step = state.step
    seen, hits, misses, refresh = set(), [], [], []
    for (b, h), segs, last_block in calls:
        for k in segs:
            if k is None:
                continue
            key = int(page_table[b, k]) * hkv + h
            if key in seen:  # a block that is two segments of the call: one lookup
                continue
            seen.add(key)
            s = int(state.slot_of[key]) - 1
            if s >= 0:
                state.stamp[s] = step
                hits.append(s)
                if k == last_block:
                    refresh.append((s, key))
            else:
                misses.append(key)
    unused = [s for s in range(len(state.key_of)) if state.stamp[s] < step]
    if policy == 0:
        order = sorted(unused, key=lambda s: (int(state.stamp[s]), s))
    else:
        def rank(s):
            k = int(state.key_of[s]) - 1
            return (0, 0.0, s) if k < 0 else (1, float(mass[k]), s)
        order = sorted(unused, key=rank)
    if len(misses) > len(order):
        raise ValueError("the cache cannot hold one call's blocks")
    victims = sorted(order[:len(misses)])
    evicted = []
    for v in victims:
        old = int(state.key_of[v]) - 1
        if old >= 0:
            state.slot_of[old] = 0
            evicted.append(old)
    for v, key in zip(victims, misses):
        state.slot_of[key] = v + 1
        state.key_of[v] = key + 1
        state.stamp[v] = step
    return {"hits": hits, "misses": misses, "victims": victims, "evicted": evicted,
            "refresh": refresh}
