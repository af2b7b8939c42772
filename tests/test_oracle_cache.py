"""Pins of the block cache's bookkeeping in the oracle (oracle/cache.py): a hand-worked call
sequence under both policies (tests/golden/block_cache_policies.txt: a tie to the lower slot,
a block that is two segments of a call, the last token's page refreshed on a hit, a tie of
cumulative masses), the segment list of a call worked by hand, and invariants of random
call sequences."""
import numpy as np
import pytest

from conftest import read_golden

import oracle

MASS = {10: 0.5, 11: 0.2, 12: 0.2, 13: 0.1, 14: 0.9}


def _ints(text):
    return [] if text == "" else [int(x) for x in text.split(",")]


@pytest.mark.parametrize("policy", [0, 1])
def test_cache_policies_worked_example(policy):
    cases = [c for c in read_golden("block_cache_policies.txt")["cases"]
             if int(c["policy"]) == policy]
    assert [int(c["call"]) for c in cases] == [1, 2, 3, 4]
    pt = np.arange(32, dtype=np.int32)[None, :]  # identity page table: key = block
    st = oracle.CacheState.empty(32, 4)
    mass = np.array([MASS.get(k, 0.0) for k in range(32)])
    for c in cases:
        res = oracle.cache_plan(st, [((0, 0), _ints(c["segs"]), int(c["last"]))], pt, 1,
                                policy=policy, mass=mass)
        assert res["victims"] == _ints(c["victims"])
        keys = [int(k) - 1 if k > 0 else None for k in st.key_of]
        assert keys == [None if x == "-" else int(x) for x in c["keys"].split(",")]
        assert st.stamp.tolist() == _ints(c["stamps"])
        assert [s for s, _ in res["refresh"]] == _ints(c["refresh"])
        for s, k in enumerate(st.key_of):  # slot_of is key_of's inverse
            if k > 0:
                assert st.slot_of[k - 1] == s + 1
        assert (st.slot_of > 0).sum() == (st.key_of > 0).sum()


def test_call_segments_worked_example():
    # n = 100, sink 20 (blocks 0, 1 partly), window 30 ([70, 100): blocks 4, 5, 6), k2 = 3:
    # kept 2 and 3 lie in [20, 70); kept 5 = [80, 96) has no candidate token
    assert oracle.call_segments(100, 20, 30, 3, [2, 3, 5], 3) == [0, 1, 4, 5, 6, 2, 3, None]
    # only n_blocks entries count; -1 padding is no segment
    assert oracle.call_segments(100, 20, 30, 3, [2, -1, -1], 1) == [0, 1, 4, 5, 6, 2, None, None]
    # a context inside sink + window: no candidate region, no kept entries
    assert oracle.call_segments(40, 20, 30, 3, [0, 1, 2], 3) == [0, 1, 1, 2]
    # the block straddling the sink's end is a sink page and, when kept, a segment again
    assert oracle.call_segments(200, 40, 16, 2, [2, 9], 2) == [0, 1, 2, 11, 12, 2, 9]


@pytest.mark.parametrize("policy", [0, 1])
def test_cache_plan_invariants_random(policy):
    rng = np.random.default_rng(40 + policy)
    hkv, pages, cap = 2, 60, 24
    pt = rng.permutation(pages).astype(np.int32)[None, :]
    st = oracle.CacheState.empty(pages * hkv, cap)
    mass = rng.random(pages * hkv)
    for call in range(1, 30):
        calls = []
        for h in range(hkv):
            segs = [int(x) for x in rng.choice(pages, size=int(rng.integers(1, 7)))]
            calls.append(((0, h), segs + [None], segs[-1]))
        before = st.copy()
        res = oracle.cache_plan(st, calls, pt, hkv, policy=policy, mass=mass)
        keys = {int(pt[0, k]) * hkv + h for (_, h), segs, _ in calls for k in segs if k is not None}
        assert len(res["victims"]) == len(res["misses"]) == len(keys) - len(res["hits"])
        assert not set(res["victims"]) & set(res["hits"])
        for k in keys:  # every block of the call is cached, stamped with this call
            s = st.slot_of[k] - 1
            assert s >= 0 and st.key_of[s] == k + 1 and st.stamp[s] == call
        unused = [s for s in range(cap) if before.stamp[s] < call and s not in res["hits"]]
        kept = sorted(set(unused) - set(res["victims"]))
        for v in res["victims"]:  # no better candidate was left out
            for r in kept:
                if policy == 0:
                    assert (before.stamp[v], v) < (before.stamp[r], r)
                else:
                    kv, kr = before.key_of[v] - 1, before.key_of[r] - 1
                    rv = (0, 0.0, v) if kv < 0 else (1, mass[kv], v)
                    rr = (0, 0.0, r) if kr < 0 else (1, mass[kr], r)
                    assert rv < rr
