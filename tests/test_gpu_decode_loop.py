"""A decode loop over several steps: a whole step (scoring and both pruning modules) every
`refresh` steps, and between them steps that reuse that selection (append + attend only),
as the InfiniteHiP article's decoding reuses its pruning results for several steps. Every
step is checked against the oracle on the cache as it stands after that step's append:
codes and selections bit-exact, outputs within the tolerance of the attention tests."""
import dataclasses

import numpy as np
import pytest
import torch

import harness as H
import oracle
from kv_cache_int8_gb300 import hsa
from kv_cache_int8_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _clone(t):
    return t.clone().pin_memory() if t.device.type == "cpu" else t.clone()


def test_prepared_decode_step_equals_the_plain_call():
    """hsa.DecodeStep (arguments marshalled once), and the same replayed from a CUDA graph,
    give the same bits as hsa_decode_step, with host I/O, over several steps whose inputs
    change in place. The plain calls after the first replay the library's own recording of
    the step; the captured graph holds the kernels launched one by one (a stream that is
    being captured is not recorded again), so the two launch paths are compared."""
    cfg = dataclasses.replace(W.CONFIGS["llama3-8b-128k"], context=None,
                              context_range=(2000, 4000), batch=2, hq=8, hkv=2, k1=10, k2=8,
                              sink=32, window=64, paged_permuted=True)
    wl = W.make_workload(cfg, seed=5)
    hd, _ = H.dims_pair(wl)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
    kq = H.kq_like(dwl["k_cache"], hd)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    gen = torch.Generator(device="cpu").manual_seed(9)
    res = []
    for mode in ("plain", "prepared", "graph"):
        kc, vc, kqc = dwl["k_cache"].clone(), dwl["v_cache"].clone(), kq.clone()
        q = torch.zeros((B, Hq, 128), dtype=torch.bfloat16).pin_memory()
        kn = torch.zeros((B, Hkv, 128), dtype=torch.bfloat16).pin_memory()
        vn = torch.zeros((B, Hkv, 128), dtype=torch.bfloat16).pin_memory()
        out = torch.zeros((B, Hq, 128), dtype=torch.float32).pin_memory()
        lse = torch.zeros((B, Hq), dtype=torch.float32).pin_memory()
        lens = dwl["seq_lens"].clone()
        ws = hsa.workspace(hd, hsa.HSA_OP_STEP)
        args = (hd, q, kn, vn, out, lse, kc, vc, kqc, k_scale, dwl["page_table"], lens, None,
                None, ws)
        step = (hsa.DecodeStep(*args, io_on_host=True, graph=mode == "graph")
                if mode != "plain" else None)
        gen.manual_seed(9)
        outs = []
        for i in range(3):
            q.copy_(torch.randn((B, Hq, 128), generator=gen).to(torch.bfloat16))
            kn.copy_(torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16))
            vn.copy_(torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16))
            if i:
                lens.sub_(1)  # the step before: one token shorter, same buffers
            if step is not None:
                step()
            else:
                hsa.hsa_decode_step(*args, io_on_host=True)
            torch.cuda.synchronize()
            assert hsa.hsa_read_device_error(ws) == 0
            outs.append((out.clone(), lse.clone()))
        res.append((outs, kc, vc, kqc))
    for other in res[1:]:
        for (o1, l1), (o2, l2) in zip(res[0][0], other[0]):
            assert torch.equal(o1, o2) and torch.equal(l1, l2)
        for a, b in zip(res[0][1:], other[1:]):
            assert torch.equal(a, b)


def test_recorded_steps_beyond_the_kept_sets():
    """hsa_decode_step keeps the recordings of its 64 most recently used argument sets: 70
    calls with 70 output buffers (70 sets) on the same inputs, then the first set again
    (recorded anew after its eviction), all give the bits of the first call; an argument
    error is still returned before anything is recorded or launched."""
    cfg = dataclasses.replace(W.CONFIGS["llama3-8b-128k"], context=None,
                              context_range=(2000, 4000), batch=2, hq=8, hkv=2, k1=10, k2=8,
                              sink=32, window=64, paged_permuted=True)
    wl = W.make_workload(cfg, seed=6)
    hd, _ = H.dims_pair(wl)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
    kq = H.kq_like(dwl["k_cache"], hd)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    lens = dwl["seq_lens"]
    n = lens.long() - 1
    pages = dwl["page_table"].long().gather(1, (n // 16).unsqueeze(1)).squeeze(1)
    k_new = dwl["k_cache"][pages, :, n % 16, :].contiguous()  # re-append the last token
    v_new = dwl["v_cache"][pages, :, n % 16, :].contiguous()
    ws = hsa.workspace(hd, hsa.HSA_OP_STEP)

    def call(out, lse):
        hsa.hsa_decode_step(hd, dwl["q"], k_new, v_new, out, lse, dwl["k_cache"], dwl["v_cache"],
                            kq, k_scale, dwl["page_table"], lens, None, None, ws)

    outs = [(torch.full((B, Hq, 128), float("nan"), device=dev),
             torch.full((B, Hq), float("nan"), device=dev)) for _ in range(70)]
    for o, l in outs:
        call(o, l)
    o0, l0 = outs[0]
    o0.fill_(float("nan"))
    call(o0, l0)  # the first set, evicted by the 69 after it
    torch.cuda.synchronize()
    assert hsa.hsa_read_device_error(ws) == 0
    for o, l in outs[1:]:
        assert torch.equal(o, o0) and torch.equal(l, l0)
    with pytest.raises(hsa.HsaError):
        hsa.hsa_decode_step(hd, dwl["q"], k_new, v_new, o0, l0, dwl["k_cache"], dwl["v_cache"],
                            kq, k_scale, dwl["page_table"], lens, None, None, ws[:64])


@pytest.mark.parametrize("refresh,on_host,key_bits,per_head,fp8", [
    (3, False, 8, 0, 0), (2, True, 8, 0, 0), (1, False, 8, 0, 0), (2, False, 4, 0, 0),
    (2, False, 8, 1, 0), (2, False, 8, 0, 1)])
def test_decode_loop_with_selection_reuse(refresh, on_host, key_bits, per_head, fp8):
    steps = 6
    cfg = dataclasses.replace(W.CONFIGS["llama3-8b-128k"], context=None,
                              context_range=(3000, 6000), batch=2, hq=8, hkv=2, k1=12, k2=10,
                              sink=32, window=96, paged_permuted=True, key_bits=key_bits,
                              key_fp8=fp8)
    wl = W.make_workload(cfg, seed=77 + refresh, host_pinned=on_host)
    hd, od = H.dims_pair(wl, per_head=per_head)
    dwl = H.to_cuda(wl)
    dev = torch.device("cuda")
    B, Hq, Hkv = cfg.batch, cfg.hq, cfg.hkv
    # the caches are sized for the final lengths; the loop starts `steps` tokens earlier
    start = wl["seq_lens"] - steps
    pt = wl["page_table"].numpy()
    kc, vc = _clone(dwl["k_cache"]), _clone(dwl["v_cache"])
    kq = H.kq_like(kc, hd)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(hd, kc, dwl["page_table"], start.to(dev), 0, 0, kq, k_scale,
                          hsa.workspace(hd, hsa.HSA_OP_QUANTIZE))
    k_host = W.to_numpy_bits(wl["k_cache"]).copy()
    v_host = W.to_numpy_bits(wl["v_cache"]).copy()
    kq_o, sc_o = oracle.quantize_keys(od, k_host, pt, start.numpy())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(k_scale.cpu().numpy(), sc_o)

    gen = torch.Generator(device="cpu").manual_seed(1234 + refresh)
    ws = hsa.workspace(hd, hsa.HSA_OP_STEP)
    R = Hq if per_head else Hkv  # selection rows per sequence
    bidx = torch.full((B, R, cfg.k2), -7, dtype=torch.int32, device=dev)
    nb = torch.full((B, R), -7, dtype=torch.int32, device=dev)
    sel = None
    for i in range(steps):
        lens = start + 1 + i
        q = torch.randn((B, Hq, 128), generator=gen).to(torch.bfloat16)
        k_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16)
        v_new = torch.randn((B, Hkv, 128), generator=gen).to(torch.bfloat16)
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        args = (hd, q.to(dev), k_new.to(dev), v_new.to(dev), out, lse, kc, vc, kq, k_scale,
                dwl["page_table"], lens.to(dev), bidx, nb, ws)
        full = i % refresh == 0
        (hsa.hsa_decode_step if full else hsa.hsa_decode_step_reuse)(*args)
        torch.cuda.synchronize()
        assert hsa.hsa_read_device_error(ws) == 0
        # oracle: the same append on a host copy, codes with the stored scales
        kb, vb = W.to_numpy_bits(k_new), W.to_numpy_bits(v_new)
        for b in range(B):
            n = int(lens[b])
            k_host[pt[b, (n - 1) // 16], :, (n - 1) % 16] = kb[b]
            v_host[pt[b, (n - 1) // 16], :, (n - 1) % 16] = vb[b]
        np.testing.assert_array_equal(W.to_numpy_bits(kc.cpu()), k_host)
        np.testing.assert_array_equal(W.to_numpy_bits(vc.cpu()), v_host)
        kq_o = oracle.quantize_append(od, k_host, pt, lens.numpy(), -1, sc_o, kq_o)
        np.testing.assert_array_equal(H.unpack_codes(kq.cpu().numpy(), key_bits), kq_o)
        qb = W.to_numpy_bits(q)
        if full and fp8:
            # FP8 scores have no fixed fp32 order: the step's selection equals hsa_select's on
            # the same state (the same scorer), which must be valid within the fp32 bound
            ci2 = torch.full((B, R, cfg.k1), -7, dtype=torch.int32, device=dev)
            nc2 = torch.full((B, R), -7, dtype=torch.int32, device=dev)
            bi2, nb2 = torch.full_like(bidx, -7), torch.full_like(nb, -7)
            hsa.hsa_select(hd, q.to(dev), kq, k_scale, dwl["page_table"], lens.to(dev), ci2, nc2,
                           bi2, nb2, hsa.workspace(hd, hsa.HSA_OP_SELECT))
            torch.cuda.synchronize()
            assert torch.equal(bi2, bidx) and torch.equal(nb2, nb)
            score, bound = oracle.fp8_block_scores(od, qb, sc_o, kq_o, pt, lens.numpy())
            bad = oracle.selection_within_bounds(od, lens.numpy(), score, bound,
                                                 ci2.cpu().numpy(), nc2.cpu().numpy(),
                                                 bidx.cpu().numpy(), nb.cpu().numpy())
            assert not bad, bad[:4]
            sel = {"block_idx": bidx.cpu().numpy(), "n_blocks": nb.cpu().numpy()}
        elif full:
            sel = oracle.select(od, qb, sc_o, kq_o, pt, lens.numpy())
            np.testing.assert_array_equal(nb.cpu().numpy(), sel["n_blocks"])
            np.testing.assert_array_equal(bidx.cpu().numpy(), sel["block_idx"])
        out_o, lse_o = oracle.attend(od, qb, k_host, v_host, pt, lens.numpy(), sel["block_idx"],
                                     sel["n_blocks"])
        H.assert_close(out.cpu().numpy(), out_o, f"step {i} output")
        np.testing.assert_allclose(lse.cpu().numpy(), lse_o, atol=2e-4, rtol=1e-5)
