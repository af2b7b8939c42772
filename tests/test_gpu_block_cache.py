"""The GPU block cache in front of K/V in host memory: attention through the cache against
the oracle, the cache's state after every call against the oracle's cache plan
(oracle.cache_plan: hits refresh a block's stamp; misses take the slots used longest ago,
lower slot first; the page holding a sequence's last token is copied again), and the cached
blocks' bytes against the host K/V. Under the cumulative-mass policy: every block's
accumulated attention mass against the oracle's per-call block masses, and the cache's state
after every call against the oracle's plan under that policy given the masses the GPU held
before the call (free slots, then least cumulative mass, lower slot first)."""
import dataclasses

import numpy as np
import pytest
import torch

import harness as H
import oracle
from kv_cache_int8_gb300 import hsa
from kv_cache_int8_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _up(x):
    return (x + 255) // 256 * 256


def _calls(lens, cfg, bidx, nb, B, Hkv):
    """The oracle cache plan's view of one call: ((b, h), segments, last block) in order."""
    return [((b, hh), oracle.call_segments(int(lens[b]), cfg.sink, cfg.window, cfg.k2,
                                            bidx[b, hh], nb[b, hh]), (int(lens[b]) - 1) // 16)
            for b in range(B) for hh in range(Hkv)]


@pytest.mark.parametrize("sink,window", [(32, 64), (40, 72)])
def test_block_cache_lru_and_attention(sink, window):
    """With a sink and window that end inside a page, calls 0 and 4 keep the blocks that
    straddle them: one block is two segments of the call, looked up and filled once."""
    cfg = dataclasses.replace(W.CONFIGS["llama3-8b-128k"], context=None, context_range=(2000, 4000),
                              batch=2, hq=8, hkv=2, k1=20, k2=12, sink=sink, window=window,
                              paged_permuted=True)
    wl = W.make_workload(cfg, seed=91, host_pinned=True)
    hd, od = H.dims_pair(wl)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
    stride = (cfg.sink + 15) // 16 + (cfg.window + 15) // 16 + 1 + cfg.k2
    capacity = B * Hkv * stride + 9  # little room beyond one call: evictions every call
    assert hsa.load().hsa_block_cache_bytes(hd.c(), B * Hkv * stride - 1) == 0
    cache = hsa.block_cache(hd, capacity)
    ws = hsa.workspace(hd, hsa.HSA_OP_CACHED)
    h = H.host_arrays(wl)
    pt, lens = h["pt"], h["lens"]
    model = oracle.CacheState.empty(wl["num_pages"] * Hkv, capacity)
    gen = np.random.default_rng(5)
    q = dwl["q"]
    for call in range(6):
        # kept blocks: a different random draw each call (some repeats of earlier ones)
        n_cand = [((int(n) - cfg.window + 15) // 16) for n in lens]
        bidx = np.full((B, Hkv, cfg.k2), -1, dtype=np.int32)
        nb = np.zeros((B, Hkv), dtype=np.int32)
        for b in range(B):
            for hh in range(Hkv):
                pool = np.arange(cfg.sink // 16, n_cand[b])
                if call % 2:
                    pool = pool[: len(pool) // 3]  # overlap with earlier calls
                pick = gen.choice(pool, size=cfg.k2, replace=False)
                if call % 4 == 0:  # the blocks that straddle the sink's end and the window's start
                    pick[:2] = [cfg.sink // 16, n_cand[b] - 1]
                    pick = np.unique(pick)
                    while len(pick) < cfg.k2:
                        pick = np.unique(np.append(pick, gen.choice(pool)))
                bidx[b, hh] = np.sort(pick)
                nb[b, hh] = cfg.k2 - (call % 3) if call % 4 else cfg.k2
                bidx[b, hh, nb[b, hh]:] = -1
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        hsa.hsa_attend_cached(hd, q, dwl["k_cache"], dwl["v_cache"], dwl["page_table"],
                              dwl["seq_lens"], torch.from_numpy(bidx).to(dev),
                              torch.from_numpy(nb).to(dev), cache, capacity, out, lse, ws)
        torch.cuda.synchronize()
        assert hsa.hsa_read_device_error(ws) == 0
        out_o, lse_o = oracle.attend(od, h["q"], h["k"], h["v"], pt, lens, bidx, nb)
        H.assert_close(out.cpu().numpy(), out_o, f"call {call} output")
        np.testing.assert_allclose(lse.cpu().numpy(), lse_o, atol=2e-4, rtol=1e-5)
        # the cache's state against the oracle's plan
        oracle.cache_plan(model, _calls(lens, cfg, bidx, nb, B, Hkv), pt, Hkv, policy=0)
        raw = cache.cpu().numpy()
        off_of = 256
        off_key = off_of + _up(wl["num_pages"] * Hkv * 4)
        off_stamp = off_key + _up(capacity * 4)
        off_mass = off_stamp + _up(capacity * 4)
        off_data = off_mass + _up(wl["num_pages"] * Hkv * 4)
        as_i32 = lambda o, n: raw[o:o + 4 * n].view(np.int32)
        assert int(raw[:4].view(np.int32)[0]) == model.step
        np.testing.assert_array_equal(as_i32(off_of, wl["num_pages"] * Hkv), model.slot_of)
        np.testing.assert_array_equal(as_i32(off_key, capacity), model.key_of)
        np.testing.assert_array_equal(as_i32(off_stamp, capacity), model.stamp)
        assert not raw[off_mass:off_data].any()  # no masses under the LRU policy
        data = raw[off_data:off_data + capacity * 8192].view(np.uint16).reshape(capacity, 2, 16, 128)
        for v in np.nonzero(model.key_of)[0]:
            key = int(model.key_of[v]) - 1
            page, hh = key // Hkv, key % Hkv
            np.testing.assert_array_equal(data[v, 0], h["k"][page, hh])
            np.testing.assert_array_equal(data[v, 1], h["v"][page, hh])


@pytest.mark.parametrize("policy", [0, 1])
def test_cached_decode_step_matches_the_uncached_one(policy):
    """Whole steps with host K/V, through the cache and without it: same selection, same
    outputs within rounding; the new token reaches the cached page (copied again). Under the
    cumulative-mass policy the masses of all blocks add up to one per query head and step."""
    cfg = dataclasses.replace(W.CONFIGS["llama3-8b-128k"], context=None, context_range=(3000, 5000),
                              batch=2, hq=8, hkv=2, k1=10, k2=8, sink=32, window=64,
                              paged_permuted=True)
    wl = W.make_workload(cfg, seed=17, host_pinned=True)
    hd, od = H.dims_pair(wl)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
    stride = (cfg.sink + 15) // 16 + (cfg.window + 15) // 16 + 1 + cfg.k2
    capacity = 2 * B * Hkv * stride
    hc = dataclasses.replace(hd, cache_policy=policy)
    cache = hsa.block_cache(hc, capacity)
    kq = torch.zeros(dwl["k_cache"].shape, dtype=torch.int8, device=dev)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    gen = torch.Generator(device="cpu").manual_seed(3)
    ws1, ws2 = hsa.workspace(hc, hsa.HSA_OP_STEP), hsa.workspace(hd, hsa.HSA_OP_STEP)
    for step in range(3):
        k_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16).to(dev)
        v_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16).to(dev)
        res = []
        for cached, ws in ((True, ws1), (False, ws2)):
            out = torch.zeros((B, Hq, 128), dtype=torch.float32, device=dev)
            lse = torch.zeros((B, Hq), dtype=torch.float32, device=dev)
            bidx = torch.full((B, Hkv, cfg.k2), -7, dtype=torch.int32, device=dev)
            nb = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev)
            args = (hd, dwl["q"], k_new, v_new, out, lse, dwl["k_cache"], dwl["v_cache"], kq,
                    k_scale, dwl["page_table"], dwl["seq_lens"], bidx, nb)
            if cached:
                hsa.hsa_decode_step_cached(hc, *args[1:], cache, capacity, ws)
            else:
                hsa.hsa_decode_step(*args, ws)
            torch.cuda.synchronize()
            assert hsa.hsa_read_device_error(ws) == 0
            res.append((out.cpu().numpy(), lse.cpu().numpy(), bidx.cpu().numpy(), nb.cpu().numpy()))
        np.testing.assert_array_equal(res[0][2], res[1][2])
        np.testing.assert_array_equal(res[0][3], res[1][3])
        np.testing.assert_allclose(res[0][0], res[1][0], atol=1e-4, rtol=0)
        np.testing.assert_allclose(res[0][1], res[1][1], atol=1e-4, rtol=0)
    total = float(hsa.block_cache_mass(hc, cache, capacity).double().sum())
    if policy == 1:
        assert abs(total - 3 * B * Hq) < 1e-3
    else:
        assert total == 0.0


@pytest.mark.parametrize("sink,window,hq", [(32, 64, 8), (40, 72, 8), (40, 72, 2), (40, 72, 4),
                                            (40, 72, 16)])
def test_block_cache_cumulative_mass_policy(sink, window, hq):
    """HCAttention's reversible eviction read as a cache policy: the blocks with the least
    cumulative attention mass leave the cache first and stay in host memory. With a sink and
    window that end inside a page, some calls keep the two blocks that straddle them, so one
    block is two segments of a call (its masses must add up)."""
    cfg = dataclasses.replace(W.CONFIGS["llama3-8b-128k"], context=None, context_range=(2000, 4000),
                              batch=2, hq=hq, hkv=2, k1=20, k2=12, sink=sink, window=window,
                              paged_permuted=True)
    wl = W.make_workload(cfg, seed=93, host_pinned=True)
    hd, od = H.dims_pair(wl)
    hd = dataclasses.replace(hd, cache_policy=1)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
    G = Hq // Hkv
    stride = (cfg.sink + 15) // 16 + (cfg.window + 15) // 16 + 1 + cfg.k2
    capacity = B * Hkv * stride + 9
    cache = hsa.block_cache(hd, capacity)
    ws = hsa.workspace(hd, hsa.HSA_OP_CACHED)
    mass_view = hsa.block_cache_mass(hd, cache, capacity)
    h = H.host_arrays(wl)
    pt, lens = h["pt"], h["lens"]
    num_pages = wl["num_pages"]
    want_mass = np.zeros(num_pages * Hkv)
    model = oracle.CacheState.empty(num_pages * Hkv, capacity)
    gen = np.random.default_rng(7)
    qgen = torch.Generator(device="cpu").manual_seed(11)
    raw_i32 = lambda raw, o, n: raw[o:o + 4 * n].view(np.int32).astype(np.int64)
    off_of = 256
    off_key = off_of + _up(num_pages * Hkv * 4)
    off_stamp = off_key + _up(capacity * 4)
    for call in range(1, 9):
        q = torch.randn((B, Hq, 128), generator=qgen).to(torch.bfloat16)
        n_cand = [((int(n) - cfg.window + 15) // 16) for n in lens]
        bidx = np.full((B, Hkv, cfg.k2), -1, dtype=np.int32)
        nb = np.zeros((B, Hkv), dtype=np.int32)
        for b in range(B):
            for hh in range(Hkv):
                pool = np.arange(cfg.sink // 16, n_cand[b])
                if call % 2:
                    pool = pool[: len(pool) // 3]
                pick = gen.choice(pool, size=cfg.k2, replace=False)
                if call % 4 == 0:  # the blocks that straddle the sink's end and the window's start
                    pick[:2] = [cfg.sink // 16, n_cand[b] - 1]
                    pick = np.unique(pick)
                    while len(pick) < cfg.k2:
                        pick = np.unique(np.append(pick, gen.choice(pool)))
                bidx[b, hh] = np.sort(pick)
                nb[b, hh] = cfg.k2 - (call % 3) if call % 4 else cfg.k2
                bidx[b, hh, nb[b, hh]:] = -1
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        gpu_mass = mass_view.cpu().numpy().reshape(-1).astype(np.float64)  # before the call
        hsa.hsa_attend_cached(hd, q.to(dev), dwl["k_cache"], dwl["v_cache"], dwl["page_table"],
                              dwl["seq_lens"], torch.from_numpy(bidx).to(dev),
                              torch.from_numpy(nb).to(dev), cache, capacity, out, lse, ws)
        torch.cuda.synchronize()
        assert hsa.hsa_read_device_error(ws) == 0
        qb = W.to_numpy_bits(q)
        out_o, lse_o = oracle.attend(od, qb, h["k"], h["v"], pt, lens, bidx, nb)
        H.assert_close(out.cpu().numpy(), out_o, f"call {call} output")
        # the cache's state against the oracle's plan under this policy, given the masses the
        # GPU held before the call (fp32, as the GPU ranks them)
        oracle.cache_plan(model, _calls(lens, cfg, bidx, nb, B, Hkv), pt, Hkv, policy=1,
                          mass=gpu_mass)
        raw = cache.cpu().numpy()
        assert int(raw[:4].view(np.int32)[0]) == model.step
        np.testing.assert_array_equal(raw_i32(raw, off_of, num_pages * Hkv), model.slot_of)
        np.testing.assert_array_equal(raw_i32(raw, off_key, capacity), model.key_of)
        np.testing.assert_array_equal(raw_i32(raw, off_stamp, capacity), model.stamp)
        # this call's attention mass of every block, summed over each kv head's query heads
        m = oracle.block_mass(od, qb, h["k"], pt, lens, bidx, nb)        # [B][Hq][blocks]
        for b in range(B):
            for hh in range(Hkv):
                mk = m[b, hh * G:(hh + 1) * G].sum(axis=0)
                for k in np.nonzero(mk)[0]:
                    want_mass[int(pt[b, k]) * Hkv + hh] += mk[k]
        got = mass_view.cpu().numpy().reshape(-1).astype(np.float64)
        np.testing.assert_allclose(got, want_mass, rtol=1e-4, atol=1e-7)
        assert abs(got.sum() - call * B * Hq) < 1e-3 * call  # every head's probabilities sum to 1
