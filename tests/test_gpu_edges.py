"""GPU parity on edge cases: ragged and tiny contexts, empty candidate regions, zero and
all-covering budgets, other chunk sizes and group sizes, mixed batches, the decode-step
append and whole-step entry points, and the device-side bounds checks."""
import dataclasses

import numpy as np
import pytest
import torch

import harness as H
import oracle
from kv_cache_int8_gb300 import hsa
from kv_cache_int8_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BASE = W.CONFIGS["llama3-8b-128k"]


def _cfg(**kw):
    return dataclasses.replace(BASE, **kw)


def _check(wl, dense=True, **over):
    hd, od = H.dims_pair(wl, **over)
    h = H.host_arrays(wl)
    g = H.gpu_step(H.to_cuda(wl), hd, dense=dense)
    o = H.oracle_step(h, od, dense=dense)
    pairs = [(b, hh) for b in range(od.batch) for hh in range(od.hkv)]
    H.compare_step(g, o, h, od, pairs, dense=dense)
    return g, o


@pytest.mark.parametrize("n", [1, 7, 16, 17, 63, 64, 65, 1000, 1153, 1154, 5003])
def test_ragged_context_lengths(n):
    wl = W.make_workload(_cfg(context=n, batch=1, hq=8, hkv=2, k1=8, k2=6, sink=20, window=100),
                         seed=n)
    g, _ = _check(wl)
    if n <= 120:
        assert (g["n_blocks"] == 0).all()


def test_mixed_batch_permuted_pages():
    cfg = _cfg(context=None, context_range=(1, 9000), batch=12, hq=16, hkv=4, k1=9, k2=13,
               sink=33, window=77, paged_permuted=True)
    wl = W.make_workload(cfg, seed=5)
    _check(wl)


@pytest.mark.parametrize("batch", [33, 300])
def test_large_batch_of_short_sequences(batch):
    """Many sequences (the scorer's per-CTA length and tile-prefix tables span several warp
    passes; one prune CTA and a split-K grid per sequence and kv head), some of length 0."""
    cfg = _cfg(context=None, context_range=(0, 900), batch=batch, hq=8, hkv=2, k1=4, k2=5,
               sink=16, window=48, paged_permuted=True)
    wl = W.make_workload(cfg, seed=batch)
    for i in (3, batch - 1):
        wl["seq_lens"][i] = 0
        wl["lens"][i] = 0
    g, _ = _check(wl, dense=False)
    assert (g["n_blocks"][3] == 0).all() and (g["n_blocks"][batch - 1] == 0).all()


def test_empty_sequence_in_a_batch():
    """A sequence of length 0 beside others: zero scales and codes, nothing selected, output
    0 and lse -inf for its heads; the other sequences as usual (dense decode too)."""
    cfg = _cfg(context=None, context_range=(600, 3000), batch=3, hq=8, hkv=2, k1=6, k2=7,
               sink=20, window=50, paged_permuted=True)
    wl = W.make_workload(cfg, seed=13)
    wl["seq_lens"][1] = 0
    wl["lens"][1] = 0
    g, o = _check(wl)
    assert (g["n_blocks"][1] == 0).all() and (g["k_scale"][1] == 0).all()
    assert (g["out"][1] == 0).all() and np.isneginf(g["lse"][1]).all()
    assert (g["out_dense"][1] == 0).all() and np.isneginf(g["lse_dense"][1]).all()


@pytest.mark.parametrize("k1,k2", [(0, 0), (0, 5), (5, 0), (1, 1), (3, 40)])
def test_small_and_zero_budgets(k1, k2):
    wl = W.make_workload(_cfg(context=4099, batch=2, hq=8, hkv=2), seed=11)
    _check(wl, k1=k1, k2=k2, sink=16, window=64)


def test_budget_covering_everything_equals_dense():
    wl = W.make_workload(_cfg(context=3001, batch=2, hq=8, hkv=2), seed=12)
    g, o = _check(wl, k1=10000, k2=10000, sink=5, window=9)
    H.assert_close(g["out"], o["out_dense"], "sparse with every block vs dense oracle")
    np.testing.assert_allclose(g["out"], g["out_dense"], atol=5e-6, rtol=0)


@pytest.mark.parametrize("chunk", [16, 32, 128, 256])
def test_other_chunk_sizes(chunk):
    wl = W.make_workload(_cfg(context=20000, batch=1, hq=8, hkv=2), seed=chunk)
    _check(wl, chunk=chunk, k1=40, k2=30, sink=64, window=128)


@pytest.mark.parametrize("hq,hkv,key_bits", [(8, 8, 8), (8, 4, 8), (4, 1, 8), (16, 2, 8),
                                              (8, 1, 8), (16, 2, 4), (8, 4, 4), (8, 8, 4)])
def test_group_sizes(hq, hkv, key_bits):
    wl = W.make_workload(_cfg(context=12345, batch=2, hq=hq, hkv=hkv, k1=20, k2=17,
                              key_bits=key_bits), seed=hq + hkv)
    _check(wl, sink=40, window=200)


@pytest.mark.parametrize("hq,hkv,key_bits,chunk", [(8, 2, 8, 64), (16, 2, 8, 64), (8, 2, 4, 64),
                                                    (4, 1, 8, 32), (8, 8, 8, 64)])
def test_per_head_selection(hq, hkv, key_bits, chunk):
    """Every query head selects its own chunks and blocks: per-head block and tile maxima,
    one selection row per query head, each head's attention over its own row."""
    wl = W.make_workload(_cfg(context=None, context_range=(900, 7000), batch=2, hq=hq, hkv=hkv,
                              paged_permuted=True, key_bits=key_bits), seed=60 + hq + key_bits)
    g, o = _check(wl, per_head=1, chunk=chunk, k1=12, k2=10, sink=24, window=150)
    # the heads of a group do not all keep the same blocks
    if hq // hkv > 1:
        assert any(not np.array_equal(g["block_idx"][b, 0], g["block_idx"][b, 1])
                   for b in range(2))


@pytest.mark.parametrize("hq,hkv,per_head", [(8, 2, 0), (16, 2, 0), (4, 1, 0), (8, 2, 1)])
def test_fp8_keys(hq, hkv, per_head):
    """FP8 E4M3 key codes: scales amax / 448 and codes bit-exact against the oracle; the
    fp32 block maxima (as ordered integers) within the fp32 bound of the exact scores, the
    selection valid within that bound, the whole step's selection equal to hsa_select's, and
    outputs within tolerance of the oracle's attention over the GPU's selection."""
    wl = W.make_workload(_cfg(context=None, context_range=(900, 7000), batch=2, hq=hq, hkv=hkv,
                              paged_permuted=True, key_fp8=1), seed=80 + hq + per_head)
    g, o = _check(wl, per_head=per_head, k1=12, k2=10, sink=24, window=150)
    codes = g["kq"].view(np.uint8)
    assert (codes & 0x7F).max() == 0x7E  # the channel maxima code as +-448


@pytest.mark.parametrize("scale_exp", [11, 16])
def test_fp8_keys_large_query(scale_exp):
    """FP8 keys with the query scaled by 2^11 and 2^16 (folded query values past 2^7, fp32
    scores in the tens of thousands): block maxima within the fp32 bound of the exact scores,
    the selection valid within it, and the whole step's selection equal to hsa_select's.
    (Logits that large leave the fp32 attention itself outside the output tolerance, so
    outputs are not compared here.)"""
    wl = W.make_workload(_cfg(context=None, context_range=(900, 7000), batch=2, hq=8, hkv=2,
                              paged_permuted=True, key_fp8=1), seed=90 + scale_exp)
    wl["q"] = (wl["q"].float() * 2.0 ** scale_exp).to(torch.bfloat16)
    hd, od = H.dims_pair(wl, k1=12, k2=10, sink=24, window=150)
    h = H.host_arrays(wl)
    g = H.gpu_step(H.to_cuda(wl), hd, dense=False)
    o = H.oracle_step(h, od, dense=False)
    pairs = [(b, hh) for b in range(od.batch) for hh in range(od.hkv)]
    H.fp8_validity(g, o, h, od, pairs)
    np.testing.assert_array_equal(g["step_block_idx"], g["block_idx"])
    np.testing.assert_array_equal(g["step_n_blocks"], g["n_blocks"])
    B, hkv = od.batch, od.hkv
    q = wl["q"].float().view(B, hkv, od.hq // hkv, 128)
    q_fold = (q * torch.from_numpy(g["k_scale"]).view(B, hkv, 1, 128)).abs().amax()
    assert q_fold >= 2.0 ** 7


def test_unaligned_sink_and_window():
    wl = W.make_workload(_cfg(context=7777, batch=3, hq=8, hkv=2), seed=21)
    _check(wl, k1=11, k2=19, sink=37, window=101)


def test_window_only_and_sink_only():
    wl = W.make_workload(_cfg(context=2222, batch=1, hq=4, hkv=1), seed=22)
    _check(wl, k1=4, k2=4, sink=0, window=0)
    _check(wl, k1=4, k2=4, sink=0, window=300)
    _check(wl, k1=4, k2=4, sink=300, window=0)


def test_many_ties_lower_index_wins():
    """Constant keys make every chunk and block tie: the lowest indices must be kept."""
    wl = W.make_workload(_cfg(context=5000, batch=1, hq=4, hkv=1), seed=23)
    wl["k_cache"][:] = 0.5
    g, o = _check(wl, k1=6, k2=9, sink=64, window=128)
    assert g["block_idx"][0, 0].tolist() == list(range(4, 13))


@pytest.mark.parametrize("run,k1,k2", [(64, 20, 17), (16, 20, 17), (64, 12, 5),
                                         (16, 40, 40), (1, 30, 23)])
def test_selection_with_runs_of_equal_keys(run, k1, k2):
    """Keys constant over runs of `run` tokens, the runs' keys random (K1 >= K2, as in the
    128K configurations, where the whole step keeps the blocks at or above the K2-th chunk
    maximum). Runs of 64: the four blocks of a chunk tie, so about 4 K2 blocks reach that
    maximum and many are dropped, equal maxima ranked by index; runs of 16: every block has
    its own maximum and a few are dropped. Selection bit-exact against the oracle."""
    wl = W.make_workload(_cfg(context=30000, batch=2, hq=8, hkv=2, k1=k1, k2=k2, sink=64,
                              window=256, paged_permuted=True), seed=71 + run + k2)
    pt = wl["page_table"].long()
    gen = torch.Generator(device="cpu").manual_seed(5 + run)
    for b, n in enumerate(wl["lens"]):
        vecs = (torch.randn(((n + run - 1) // run, 2, 128), generator=gen) * 2).to(torch.bfloat16)
        t = torch.arange(n)
        wl["k_cache"][pt[b, t // 16], :, t % 16] = vecs[t // run]
    _check(wl)


def test_tied_top_chunks_beyond_the_candidate_room():
    """Eight chunks of each kv head hold, in every token, the key of its first query head's
    direction, so their maxima tie at the top: with K2 = 5 the blocks at or above the K2-th
    chunk maximum number 32, more than the 4 K2 the whole step's short path takes (it then
    runs the general modules). Lowest indices win the ties."""
    wl = W.make_workload(_cfg(context=20000, batch=1, hq=8, hkv=2, k1=12, k2=5, sink=64,
                              window=256), seed=37)
    pt = wl["page_table"].long()
    n = wl["lens"][0]
    chunks = [40, 41, 77, 90, 120, 121, 200, 250]
    for h in range(2):
        vec = (wl["q"][0, h * 4].float() * 3).to(torch.bfloat16)
        for c in chunks:
            t = torch.arange(c * 64, min(n, c * 64 + 64))
            wl["k_cache"][pt[0, t // 16], h, t % 16] = vec
    g, o = _check(wl)
    for h in range(2):
        assert g["block_idx"][0, h].tolist() == [160, 161, 162, 163, 164]


def test_all_equal_keys_with_k1_at_least_k2():
    """Every chunk and block maximum equal (the K2-th chunk maximum's bin holds them all):
    the lowest indices are kept."""
    wl = W.make_workload(_cfg(context=5000, batch=1, hq=4, hkv=1), seed=29)
    wl["k_cache"][:] = 0.5
    g, o = _check(wl, k1=12, k2=9, sink=64, window=128)
    assert g["block_idx"][0, 0].tolist() == list(range(4, 13))


def test_append_then_step_matches_oracle():
    """hsa_append_kv writes the new token and its codes with the stored scales; the whole
    step entry point gives the same result as the separate calls (selection, cache and codes
    bit for bit; outputs up to the order of the split-K sums)."""
    cfg = _cfg(context=None, context_range=(3000, 9000), batch=3, hq=8, hkv=2, k1=12, k2=10,
               sink=32, window=96, paged_permuted=True)
    wl = W.make_workload(cfg, seed=31)
    hd, od = H.dims_pair(wl)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hkv = cfg.batch, cfg.hkv
    gen = torch.Generator(device="cpu").manual_seed(99)
    k_new = (torch.randn((B, Hkv, 128), generator=gen) * 9).to(torch.bfloat16)
    v_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16)
    kq = torch.zeros(dwl["k_cache"].shape, dtype=torch.int8, device=dev)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    kc2, vc2, kq2 = dwl["k_cache"].clone(), dwl["v_cache"].clone(), kq.clone()
    hsa.hsa_append_kv(hd, k_new.cuda(), v_new.cuda(), kc2, vc2, kq2, k_scale, dwl["page_table"],
                      dwl["seq_lens"])
    torch.cuda.synchronize()
    # oracle: write the token into a host copy, codes with the stored scales
    kh = wl["k_cache"].clone()
    vh = wl["v_cache"].clone()
    pt = wl["page_table"].numpy()
    for b, n in enumerate(wl["lens"]):
        kh[pt[b, (n - 1) // 16], :, (n - 1) % 16] = k_new[b]
        vh[pt[b, (n - 1) // 16], :, (n - 1) % 16] = v_new[b]
    np.testing.assert_array_equal(kc2.cpu().view(torch.int16).numpy(), kh.view(torch.int16).numpy())
    np.testing.assert_array_equal(vc2.cpu().view(torch.int16).numpy(), vh.view(torch.int16).numpy())
    # the oracle's own scales and codes of the cache before the append
    kq_full, sc_o = oracle.quantize_keys(od, W.to_numpy_bits(wl["k_cache"]), pt,
                                         wl["seq_lens"].numpy())
    np.testing.assert_array_equal(k_scale.cpu().numpy(), sc_o)
    kq_o = oracle.quantize_append(od, W.to_numpy_bits(kh), pt, wl["seq_lens"].numpy(), -1,
                                  sc_o, kq_full)
    np.testing.assert_array_equal(kq2.cpu().numpy(), kq_o)
    # the APPEND mode of hsa_quantize_keys agrees
    kq3 = kq.clone()
    hsa.hsa_quantize_keys(hd, kc2, dwl["page_table"], dwl["seq_lens"], 1, -1, kq3, k_scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kq3.cpu().numpy(), kq_o)

    # whole step (device io) == separate calls
    out_a = torch.zeros((B, cfg.hq, 128), dtype=torch.float32, device=dev)
    lse_a = torch.zeros((B, cfg.hq), dtype=torch.float32, device=dev)
    bidx = torch.zeros((B, Hkv, cfg.k2), dtype=torch.int32, device=dev)
    nb = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    wst = hsa.workspace(hd, hsa.HSA_OP_STEP)
    kc4, vc4, kq4 = dwl["k_cache"].clone(), dwl["v_cache"].clone(), kq.clone()
    hsa.hsa_decode_step(hd, dwl["q"], k_new.cuda(), v_new.cuda(), out_a, lse_a, kc4, vc4, kq4,
                        k_scale, dwl["page_table"], dwl["seq_lens"], bidx, nb, wst)
    ws = hsa.workspace(hd, hsa.HSA_OP_SELECT)
    ci = torch.zeros((B, Hkv, cfg.k1), dtype=torch.int32, device=dev)
    nc = torch.zeros((B, Hkv), dtype=torch.int32, device=dev)
    bidx2 = torch.zeros_like(bidx)
    nb2 = torch.zeros_like(nb)
    hsa.hsa_select(hd, dwl["q"], kq2, k_scale, dwl["page_table"], dwl["seq_lens"], ci, nc, bidx2,
                   nb2, ws)
    out_b = torch.zeros_like(out_a)
    lse_b = torch.zeros_like(lse_a)
    hsa.hsa_attend(hd, dwl["q"], kc2, vc2, dwl["page_table"], dwl["seq_lens"], bidx2, nb2, out_b,
                   lse_b, hsa.workspace(hd, hsa.HSA_OP_ATTEND))
    torch.cuda.synchronize()
    assert torch.equal(bidx, bidx2) and torch.equal(nb, nb2)
    # the step's attention may split and merge its partials differently: the same sums in
    # another order
    torch.testing.assert_close(out_a, out_b, rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(lse_a, lse_b, rtol=1e-5, atol=1e-5)
    assert torch.equal(kq4, kq2) and torch.equal(kc4, kc2)
    # whole step with pinned host io
    q_h = wl["q"].pin_memory()
    out_h = torch.zeros((B, cfg.hq, 128), dtype=torch.float32).pin_memory()
    lse_h = torch.zeros((B, cfg.hq), dtype=torch.float32).pin_memory()
    kc5, vc5, kq5 = dwl["k_cache"].clone(), dwl["v_cache"].clone(), kq.clone()
    hsa.hsa_decode_step(hd, q_h, k_new.pin_memory(), v_new.pin_memory(), out_h, lse_h, kc5, vc5,
                        kq5, k_scale, dwl["page_table"], dwl["seq_lens"], None, None, wst,
                        io_on_host=True)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_a.cpu()) and torch.equal(lse_h, lse_a.cpu())
    assert hsa.hsa_read_device_error(wst) == 0


def test_device_bounds_checks_report_without_faulting():
    """A page-table entry past the pool and a sequence longer than its table are caught by
    the kernels' own checks: the error word reports them and no access goes out of range."""
    wl = W.make_workload(_cfg(context=4000, batch=2, hq=8, hkv=2, k1=8, k2=8, sink=16,
                              window=64), seed=41)
    hd, _ = H.dims_pair(wl)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    kq = torch.zeros(dwl["k_cache"].shape, dtype=torch.int8, device=dev)
    k_scale = torch.zeros((2, 2, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    bad_pt = dwl["page_table"].clone()
    bad_pt[1, 100] = hd.num_pages + 5
    bidx = torch.zeros((2, 2, 8), dtype=torch.int32, device=dev)
    nb = torch.zeros((2, 2), dtype=torch.int32, device=dev)
    ws = hsa.workspace(hd, hsa.HSA_OP_SELECT)
    hsa.hsa_select(hd, dwl["q"], kq, k_scale, bad_pt, dwl["seq_lens"], None, None, bidx, nb, ws)
    assert hsa.hsa_read_device_error(ws) == hsa.HSA_ERR_DEVICE_CHECK
    assert hsa.hsa_read_device_error(ws) == 0  # cleared by the read
    long_lens = dwl["seq_lens"].clone()
    long_lens[0] = hd.max_pages_per_seq * 16 + 1
    out = torch.zeros((2, 8, 128), dtype=torch.float32, device=dev)
    wa = hsa.workspace(hd, hsa.HSA_OP_ATTEND)
    hsa.hsa_attend(hd, dwl["q"], dwl["k_cache"], dwl["v_cache"], dwl["page_table"], long_lens,
                   bidx, nb, out, None, wa)
    assert hsa.hsa_read_device_error(wa) == hsa.HSA_ERR_DEVICE_CHECK
    # the context is still usable
    hsa.hsa_select(hd, dwl["q"], kq, k_scale, dwl["page_table"], dwl["seq_lens"], None, None,
                   bidx, nb, ws)
    assert hsa.hsa_read_device_error(ws) == 0


def _clone(t):
    """A copy on the same side: device, or pinned host for an offloaded cache."""
    return t.clone().pin_memory() if t.device.type == "cpu" else t.clone()


@pytest.mark.parametrize("window,k1,k2,on_host,hq,per_head", [
    (0, 6, 9, False, 8, 0), (1, 6, 9, False, 8, 0), (5, 3, 0, False, 8, 0),
    (300, 8, 8, False, 8, 0), (0, 6, 9, True, 8, 0), (300, 8, 8, True, 8, 0),
    (300, 8, 8, False, 16, 0), (40, 8, 8, True, 16, 0),
    (0, 6, 9, False, 8, 1), (300, 8, 8, False, 8, 1), (40, 8, 8, True, 16, 1)])
def test_decode_step_matches_separate_calls_and_oracle(window, k1, k2, on_host, hq, per_head):
    """The whole step (append ordered before or beside the scorer, the selection run inside
    the attention or by the pruning kernel, the sink and window pages fetched early) equals
    the separate calls (selection and cache bit for bit, outputs up to the order of the
    split-K sums), and the oracle on the appended cache; also with K/V in mapped pinned host
    memory, with groups of 8 query heads, and with per-head selection."""
    cfg = _cfg(context=None, context_range=(700, 5000), batch=3, hq=hq, hkv=2, k1=k1, k2=k2,
               sink=20, window=window, paged_permuted=True)
    wl = W.make_workload(cfg, seed=40 + window, host_pinned=on_host)
    hd, od = H.dims_pair(wl, per_head=per_head)
    assert bool(hd.kv_on_host) == on_host
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hkv = cfg.batch, cfg.hkv
    R = cfg.hq if per_head else Hkv  # selection rows per sequence
    gen = torch.Generator(device="cpu").manual_seed(7 + window)
    k_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16)
    v_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16)
    kq = torch.zeros(dwl["k_cache"].shape, dtype=torch.int8, device=dev)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    # whole step
    kc1, vc1, kq1 = _clone(dwl["k_cache"]), _clone(dwl["v_cache"]), kq.clone()
    out1 = torch.zeros((B, cfg.hq, 128), dtype=torch.float32, device=dev)
    lse1 = torch.zeros((B, cfg.hq), dtype=torch.float32, device=dev)
    bidx1 = torch.full((B, R, max(k2, 1)), -7, dtype=torch.int32, device=dev)
    nb1 = torch.full((B, R), -7, dtype=torch.int32, device=dev)
    wst = hsa.workspace(hd, hsa.HSA_OP_STEP)
    for _ in range(2):  # the second call finds the first call's workspace contents
        hsa.hsa_decode_step(hd, dwl["q"], k_new.cuda(), v_new.cuda(), out1, lse1, kc1, vc1, kq1,
                            k_scale, dwl["page_table"], dwl["seq_lens"], bidx1, nb1, wst)
    # separate calls
    kc2, vc2, kq2 = _clone(dwl["k_cache"]), _clone(dwl["v_cache"]), kq.clone()
    hsa.hsa_append_kv(hd, k_new.cuda(), v_new.cuda(), kc2, vc2, kq2, k_scale, dwl["page_table"],
                      dwl["seq_lens"])
    bidx2 = torch.full_like(bidx1, -7)
    nb2 = torch.full_like(nb1, -7)
    hsa.hsa_select(hd, dwl["q"], kq2, k_scale, dwl["page_table"], dwl["seq_lens"], None, None,
                   bidx2, nb2, hsa.workspace(hd, hsa.HSA_OP_SELECT))
    out2 = torch.zeros_like(out1)
    lse2 = torch.zeros_like(lse1)
    hsa.hsa_attend(hd, dwl["q"], kc2, vc2, dwl["page_table"], dwl["seq_lens"], bidx2, nb2, out2,
                   lse2, hsa.workspace(hd, hsa.HSA_OP_ATTEND))
    torch.cuda.synchronize()
    assert hsa.hsa_read_device_error(wst) == 0
    assert torch.equal(kq1, kq2) and torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert torch.equal(nb1, nb2) and torch.equal(bidx1, bidx2)
    # the step may split the attention over another number of CTAs than hsa_attend (it needs
    # no SMs for a pruning kernel): the same sums in another order
    torch.testing.assert_close(out1, out2, rtol=1e-5, atol=1e-5)
    torch.testing.assert_close(lse1, lse2, rtol=1e-5, atol=1e-5)
    # oracle on the appended cache
    kh, vh = kc2.cpu(), vc2.cpu()
    h = {"q": W.to_numpy_bits(wl["q"]), "k": W.to_numpy_bits(kh), "v": W.to_numpy_bits(vh),
         "pt": wl["page_table"].numpy(), "lens": wl["seq_lens"].numpy()}
    kq_o, sc_o = oracle.quantize_keys(od, W.to_numpy_bits(wl["k_cache"]), h["pt"], h["lens"])
    kq_o = oracle.quantize_append(od, h["k"], h["pt"], h["lens"], -1, sc_o, kq_o)
    np.testing.assert_array_equal(kq1.cpu().numpy(), kq_o)
    sel = oracle.select(od, h["q"], sc_o, kq_o, h["pt"], h["lens"])
    np.testing.assert_array_equal(nb1.cpu().numpy(), sel["n_blocks"])
    np.testing.assert_array_equal(bidx1.cpu().numpy()[..., :k2], sel["block_idx"])
    out_o, lse_o = oracle.attend(od, h["q"], h["k"], h["v"], h["pt"], h["lens"], sel["block_idx"],
                                 sel["n_blocks"])
    H.assert_close(out1.cpu().numpy(), out_o, "whole-step output")
    np.testing.assert_allclose(lse1.cpu().numpy(), lse_o, atol=2e-4, rtol=1e-5)


def _prune_reference(row, n, chunk, k1, k2, sink, window):
    """Both modules by their definition on one row of block maxima: chunk score = max of its
    candidate blocks' maxima; keep the top K1 chunks, then the top K2 of their candidate
    blocks, by (score descending, index ascending); both lists returned ascending."""
    P = chunk // 16
    lo, hi = sink, n - window
    if hi <= lo:
        return [], []
    k_lo, k_hi = lo // 16, (hi + 15) // 16
    c_lo = k_lo // P
    c_hi = (k_hi + P - 1) // P
    score = {c: max(int(row[k]) for k in range(max(c * P, k_lo), min(c * P + P, k_hi)))
             for c in range(c_lo, c_hi)}
    kept = sorted(sorted(score, key=lambda c: (-score[c], c))[:k1])
    blocks = [k for c in kept for k in range(c * P, c * P + P) if k_lo <= k < k_hi]
    return kept, sorted(sorted(blocks, key=lambda k: (-int(row[k]), k))[:k2])


@pytest.mark.parametrize("max_pages,chunk,with_tiles", [
    (16384, 64, True), (16384, 128, False), (40000, 64, True), (40000, 64, False),
    (40000, 32, True)])
@pytest.mark.parametrize("dist", ["spread", "ties", "const", "wide"])
def test_prune_on_synthetic_maxima(max_pages, chunk, with_tiles, dist):
    """hsa_prune alone on seeded block maxima: the whole row staged in shared memory (up to
    16384 blocks) or the 64-token tile maxima or a gather from global memory; large chunk
    counts (the threshold digit's keys compacted); many ties at the threshold. Entries
    outside the candidate region hold values that would win if they were read."""
    B, Hkv, sink, window = 2, 2, 128, 2048
    gen = np.random.default_rng(max_pages + chunk + len(dist) + int(with_tiles))
    lens = [max_pages * 16, max_pages * 16 - 12345]
    if dist == "spread":
        bm = gen.integers(-2_000_000, 2_000_000, size=(B, Hkv, max_pages))
    elif dist == "ties":
        levels = gen.integers(-1_000_000, 1_000_000, size=200)
        bm = levels[gen.integers(0, 200, size=(B, Hkv, max_pages))]
    elif dist == "wide":  # nearly the whole int32 range (INT_MIN is the placeholder)
        bm = gen.integers(-(2 ** 31) + 1, 2 ** 31, size=(B, Hkv, max_pages))
    else:
        bm = np.full((B, Hkv, max_pages), 777)
    bm = bm.astype(np.int32)
    n_tiles = (max_pages + 3) // 4
    tm = np.full((B, Hkv, n_tiles), 2_000_000_000, dtype=np.int32)
    for b, n in enumerate(lens):
        k_lo, k_hi = sink // 16, (n - window + 15) // 16
        bm[b, :, :k_lo] = 2_000_000_000            # never a candidate
        bm[b, :, k_hi:] = 2_000_000_000
        for t in range(k_lo // 4, (k_hi + 3) // 4):
            tm[b, :, t] = bm[b, :, max(4 * t, k_lo):min(4 * t + 4, k_hi)].max(axis=-1)
    k1, k2 = 512, 256
    d = hsa.Dims(batch=B, hq=Hkv * 4, hkv=Hkv, max_pages_per_seq=max_pages, num_pages=B * max_pages,
                 chunk=chunk, k1=k1, k2=k2, sink=sink, window=window)
    dev = torch.device("cuda")
    bm_d = torch.from_numpy(bm).to(dev)
    tm_d = torch.from_numpy(tm).to(dev) if with_tiles else None
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    ci = torch.full((B, Hkv, k1), -7, dtype=torch.int32, device=dev)
    nc = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev)
    bi = torch.full((B, Hkv, k2), -7, dtype=torch.int32, device=dev)
    nb = torch.full((B, Hkv), -7, dtype=torch.int32, device=dev)
    hsa.hsa_prune(d, lens_d, bm_d, tm_d, ci, nc, bi, nb)
    torch.cuda.synchronize()
    ci, nc, bi, nb = (x.cpu().numpy() for x in (ci, nc, bi, nb))
    for b, n in enumerate(lens):
        for h in range(Hkv):
            chunks, blocks = _prune_reference(bm[b, h], n, chunk, k1, k2, sink, window)
            assert nc[b, h] == len(chunks) and nb[b, h] == len(blocks)
            np.testing.assert_array_equal(ci[b, h], chunks + [-1] * (k1 - len(chunks)))
            np.testing.assert_array_equal(bi[b, h], blocks + [-1] * (k2 - len(blocks)))


@pytest.mark.parametrize("chunk,chunk0,k0,k1,k2", [(64, 256, 6, 20, 15), (32, 128, 3, 10, 40),
                                                   (64, 64, 40, 10, 10), (64, 512, 2, 8, 8),
                                                   (64, 256, 100, 20, 15)])
def test_three_stacked_modules(chunk, chunk0, k0, k1, k2):
    """A first module on coarse chunks in front of the two others (and K0 >= all coarse
    chunks, where it keeps everything)."""
    wl = W.make_workload(_cfg(context=30000, batch=2, hq=8, hkv=2), seed=chunk0 + k0)
    _check(wl, chunk=chunk, chunk0=chunk0, k0=k0, k1=k1, k2=k2, sink=64, window=128)
