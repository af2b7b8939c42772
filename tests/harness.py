"""Shared helpers of the parity tests: run one decode step through the C ABI and through
the CPU oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kv_cache_int8_gb300 import hsa
from kv_cache_int8_gb300 import workloads as W

INT32_MIN = np.iinfo(np.int32).min

# Output tolerance of the sparse and dense attention against the fp64 oracle.
MAX_ABS_ERR = 1e-2
MAX_REL_L2 = 5e-3


def dims_pair(wl: dict, **over):
    """(hsa.Dims, oracle.Dims) for a workload, with optional overrides of k1, k2, sink,
    window, chunk, chunk0, k0, key_bits, per_head."""
    cfg = wl["config"]
    p = dict(k1=cfg.k1, k2=cfg.k2, sink=cfg.sink, window=cfg.window, chunk=cfg.chunk,
             chunk0=cfg.chunk0, k0=cfg.k0, key_bits=cfg.key_bits, per_head=0,
             key_fp8=cfg.key_fp8)
    p.update(over)
    hd = hsa.Dims(batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, max_pages_per_seq=wl["max_pages"],
                  num_pages=wl["num_pages"], chunk=p["chunk"], k1=p["k1"], k2=p["k2"],
                  sink=p["sink"], window=p["window"],
                  kv_on_host=wl["k_cache"].device.type == "cpu" and wl["k_cache"].is_pinned(),
                  chunk0=p["chunk0"], k0=p["k0"], key_bits=p["key_bits"],
                  per_head=p["per_head"], key_fp8=p["key_fp8"])
    od = oracle.Dims(batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, head_dim=W.HEAD_DIM,
                     page_size=W.PAGE, max_pages_per_seq=wl["max_pages"],
                     num_pages=wl["num_pages"], chunk=p["chunk"], block=16, k1=p["k1"],
                     k2=p["k2"], sink=p["sink"], window=p["window"], chunk0=p["chunk0"],
                     k0=p["k0"], key_bits=p["key_bits"], per_head=p["per_head"],
                     key_fp8=p["key_fp8"])
    return hd, od


def kq_like(k_cache: torch.Tensor, d: hsa.Dims) -> torch.Tensor:
    """A zeroed device key-code cache for a bf16 cache of shape [P][Hkv][16][128]: int8
    codes of the same shape, or with 4-bit codes [P][Hkv][16][64] bytes."""
    shape = list(k_cache.shape)
    if d.key_bits == 4:
        shape[-1] //= 2
    return torch.zeros(shape, dtype=torch.int8, device="cuda")


def unpack_codes(kq: np.ndarray, key_bits: int) -> np.ndarray:
    """The codes of a key-code cache as int8 [..][128]: 8-bit codes as they are; 4-bit ones
    from their two's-complement nibbles (channel 2i in the low nibble of byte i)."""
    if key_bits != 4:
        return kq
    u = kq.view(np.uint8).astype(np.int16)
    lo = ((u & 0xF) ^ 8) - 8
    hi = ((u >> 4) ^ 8) - 8
    return np.stack([lo, hi], axis=-1).reshape(*kq.shape[:-1], 2 * kq.shape[-1]).astype(np.int8)


def to_cuda(wl: dict) -> dict:
    out = dict(wl)
    for key in ("q", "page_table", "seq_lens"):
        out[key] = wl[key].cuda()
    for key in ("k_cache", "v_cache"):
        t = wl[key]
        out[key] = t if (t.device.type == "cpu" and t.is_pinned()) else t.cuda()
    return out


def gpu_step(wl: dict, d: hsa.Dims, dense: bool = True) -> dict:
    """Quantise the keys, score, prune, attend (and dense decode) through the C ABI."""
    dev = torch.device("cuda")
    B, Hq, Hkv = d.batch, d.hq, d.hkv
    R = Hq if d.per_head else Hkv  # selection rows per sequence
    kq = kq_like(wl["k_cache"], d)
    k_scale = torch.zeros((B, Hkv, 128), dtype=torch.float32, device=dev)
    wq = hsa.workspace(d, hsa.HSA_OP_QUANTIZE)
    hsa.hsa_quantize_keys(d, wl["k_cache"], wl["page_table"], wl["seq_lens"], 0, 0, kq, k_scale, wq)
    bm = torch.full((B, R, d.max_pages_per_seq), INT32_MIN, dtype=torch.int32, device=dev)
    hsa.hsa_score_blocks(d, wl["q"], kq, k_scale, wl["page_table"], wl["seq_lens"], bm)
    chunk_idx = torch.full((B, R, max(d.k1, 1)), -7, dtype=torch.int32, device=dev)
    n_chunks = torch.full((B, R), -7, dtype=torch.int32, device=dev)
    block_idx = torch.full((B, R, max(d.k2, 1)), -7, dtype=torch.int32, device=dev)
    n_blocks = torch.full((B, R), -7, dtype=torch.int32, device=dev)
    ws = hsa.workspace(d, hsa.HSA_OP_SELECT)
    hsa.hsa_select(d, wl["q"], kq, k_scale, wl["page_table"], wl["seq_lens"], chunk_idx, n_chunks,
                   block_idx, n_blocks, ws)
    # the split entry points (score with per-tile maxima, then prune) agree with hsa_select
    bm2 = torch.full_like(bm, INT32_MIN)
    tm = torch.full((B, R, (d.max_pages_per_seq + 3) // 4), INT32_MIN, dtype=torch.int32,
                    device=dev)
    hsa.hsa_score_blocks(d, wl["q"], kq, k_scale, wl["page_table"], wl["seq_lens"], bm2, tm)
    bi2 = torch.full_like(block_idx, -7)
    nb2 = torch.full_like(n_blocks, -7)
    ci2 = torch.full_like(chunk_idx, -7)
    hsa.hsa_prune(d, wl["seq_lens"], bm2, tm, ci2, None, bi2, nb2)
    # without chunk outputs (K1 >= K2: module 2 ranks only the blocks at or above module 1's
    # threshold) the kept blocks are the same
    bi3 = torch.full_like(block_idx, -7)
    nb3 = torch.full_like(n_blocks, -7)
    hsa.hsa_prune(d, wl["seq_lens"], bm2, tm, None, None, bi3, nb3)
    torch.cuda.synchronize()
    assert torch.equal(bi3, block_idx) and torch.equal(nb3, n_blocks)
    assert torch.equal(bm2, bm)
    k_tiles = tm.shape[-1]
    pad = torch.full((B, R, 4 * k_tiles - bm.shape[-1]), INT32_MIN, dtype=torch.int32, device=dev)
    assert torch.equal(tm, torch.cat([bm, pad], dim=-1).view(B, R, k_tiles, 4).amax(-1))
    assert torch.equal(bi2, block_idx) and torch.equal(nb2, n_blocks)
    assert torch.equal(ci2, chunk_idx)
    wa = hsa.workspace(d, hsa.HSA_OP_ATTEND)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
    hsa.hsa_attend(d, wl["q"], wl["k_cache"], wl["v_cache"], wl["page_table"], wl["seq_lens"],
                   block_idx, n_blocks, out, lse, wa)
    res = {"kq": kq, "k_scale": k_scale, "block_max": bm, "chunk_idx": chunk_idx[..., :d.k1],
           "n_chunks": n_chunks, "block_idx": block_idx[..., :d.k2], "n_blocks": n_blocks,
           "out": out, "lse": lse}
    if dense:
        wd = hsa.workspace(d, hsa.HSA_OP_DENSE)
        out_d = torch.full_like(out, float("nan"))
        lse_d = torch.full_like(lse, float("nan"))
        hsa.dense_decode(d, wl["q"], wl["k_cache"], wl["v_cache"], wl["page_table"],
                         wl["seq_lens"], out_d, lse_d, wd)
        res["out_dense"], res["lse_dense"] = out_d, lse_d
    res.update(step_by_reappend(wl, d, kq, k_scale))
    torch.cuda.synchronize()
    for name, w in (("quantize", wq), ("select", ws), ("attend", wa)):
        assert hsa.hsa_read_device_error(w) == 0, f"device error word set by {name}"
    res = {k: v.cpu().numpy() for k, v in res.items()}
    res["kq"] = unpack_codes(res["kq"], d.key_bits)
    return res


def step_by_reappend(wl: dict, d: hsa.Dims, kq: torch.Tensor, k_scale: torch.Tensor) -> dict:
    """The whole decode step (hsa_decode_step: append, scorer, both modules, attention, in
    the launch configuration the benchmark times) on the same inputs: every sequence's token
    at slot N_b - 1 is appended again with its own K/V bits, whose codes come out the same
    from the stored scales, so the cache is unchanged and the step's selection and output
    are those of the separate calls. Returns step_block_idx / step_n_blocks / step_out /
    step_lse, or nothing when a sequence is empty (there is no token to append)."""
    lens = wl["seq_lens"]
    if int(lens.min()) < 1:
        return {}
    dev = torch.device("cuda")
    B, Hq = d.batch, d.hq
    R = Hq if d.per_head else d.hkv
    n = lens.long() - 1
    pages = wl["page_table"].long().gather(1, (n // 16).unsqueeze(1)).squeeze(1)
    kc, vc = wl["k_cache"], wl["v_cache"]
    idx_p, idx_s = pages.to(kc.device), (n % 16).to(kc.device)
    k_new = kc[idx_p, :, idx_s, :].to(dev).contiguous()
    v_new = vc[idx_p, :, idx_s, :].to(dev).contiguous()
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
    bidx = torch.full((B, R, max(d.k2, 1)), -7, dtype=torch.int32, device=dev)
    nb = torch.full((B, R), -7, dtype=torch.int32, device=dev)
    wst = hsa.workspace(d, hsa.HSA_OP_STEP)
    hsa.hsa_decode_step(d, wl["q"], k_new, v_new, out, lse, kc, vc, kq, k_scale,
                        wl["page_table"], lens, bidx, nb, wst)
    torch.cuda.synchronize()
    assert hsa.hsa_read_device_error(wst) == 0, "device error word set by the decode step"
    return {"step_block_idx": bidx[..., :d.k2], "step_n_blocks": nb, "step_out": out,
            "step_lse": lse}


def host_arrays(wl: dict) -> dict:
    return {
        "q": W.to_numpy_bits(wl["q"]),
        "k": W.to_numpy_bits(wl["k_cache"]),
        "v": W.to_numpy_bits(wl["v_cache"]),
        "pt": wl["page_table"].cpu().numpy(),
        "lens": wl["seq_lens"].cpu().numpy(),
    }


def oracle_step(h: dict, od: oracle.Dims, bh_mask=None, qh_mask=None, dense: bool = True) -> dict:
    kq, sc = oracle.quantize_keys(od, h["k"], h["pt"], h["lens"], bh_mask=bh_mask)
    sel = oracle.select(od, h["q"], sc, kq, h["pt"], h["lens"], bh_mask=bh_mask,
                        want_block_max=True)
    out, lse = oracle.attend(od, h["q"], h["k"], h["v"], h["pt"], h["lens"], sel["block_idx"],
                             sel["n_blocks"], qh_mask=qh_mask)
    res = dict(sel, kq=kq, k_scale=sc, out=out, lse=lse)
    if od.key_fp8:  # exact block scores and the fp32 bound around them
        res["fp8_score"], res["fp8_bound"] = oracle.fp8_block_scores(
            od, h["q"], sc, kq, h["pt"], h["lens"], bh_mask=bh_mask)
    if dense:
        res["out_dense"], res["lse_dense"] = oracle.dense(od, h["q"], h["k"], h["v"], h["pt"],
                                                          h["lens"], qh_mask=qh_mask)
    return res


def err_stats(got: np.ndarray, want: np.ndarray):
    got = got.astype(np.float64)
    diff = got - want
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, want, what: str):
    max_abs, rel = err_stats(got, want)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert max_abs <= MAX_ABS_ERR and rel <= MAX_REL_L2, (
        f"{what}: max|err| {max_abs:.3e} (bound {MAX_ABS_ERR}), rel L2 {rel:.3e} "
        f"(bound {MAX_REL_L2})")
    return max_abs, rel


def logical_rows(arr: np.ndarray, pt: np.ndarray, lens, b: int, h: int) -> np.ndarray:
    """[N_b][128] rows of (b, h) from a paged [P][Hkv][16][128] array."""
    n = int(lens[b])
    pages = pt[b, : (n + 15) // 16]
    rows = arr[pages, h].reshape(-1, arr.shape[-1])
    return rows[:n]


def ordered_to_float(keys) -> np.ndarray:
    """fp32 values of the order-preserving integers that FP8 block maxima are kept as."""
    k = np.asarray(keys, dtype=np.int64)
    bits = np.where(k >= 0, k, k ^ 0x7FFFFFFF).astype(np.int64) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def fp8_rows(od: oracle.Dims, bh_pairs):
    """The selection rows of the (b, kv head) pairs: the kv head's row, or with per-head
    selection the rows of its query heads."""
    G = od.hq // od.hkv
    return [(b, r) for b, hh in bh_pairs
            for r in (range(hh * G, hh * G + G) if od.per_head else (hh,))]


def fp8_validity(g: dict, o: dict, h: dict, od: oracle.Dims, bh_pairs):
    """FP8 keys, whose fp32 scores the pages fix in no order: the GPU's block maxima within
    the fp32 bound of the exact ones and its selection valid for scores known to that bound
    (oracle.selection_within_bounds)."""
    rows = fp8_rows(od, bh_pairs)
    for b, r in rows:
        valid = np.isfinite(o["fp8_score"][b, r])
        bm = g["block_max"][b, r]
        assert (bm[~valid] == INT32_MIN).all()
        err = np.abs(ordered_to_float(bm[valid]).astype(np.float64) - o["fp8_score"][b, r][valid])
        assert (err <= o["fp8_bound"][b, r][valid]).all(), "FP8 block maxima outside the bound"
    bad = oracle.selection_within_bounds(od, h["lens"], o["fp8_score"], o["fp8_bound"],
                                         g["chunk_idx"], g["n_chunks"], g["block_idx"],
                                         g["n_blocks"], rows)
    assert not bad, f"FP8 selection not valid within the fp32 bound: {bad[:4]}"


def fp8_reference(g: dict, o: dict, h: dict, od: oracle.Dims, bh_pairs):
    """fp8_validity, then the oracle's attention over the GPU's own selection, which the
    outputs are then compared with. Returns (out, lse)."""
    G = od.hq // od.hkv
    fp8_validity(g, o, h, od, bh_pairs)
    qh_mask = np.zeros((od.batch, od.hq), dtype=np.int32)
    for b, hh in bh_pairs:
        qh_mask[b, hh * G:(hh + 1) * G] = 1
    return oracle.attend(od, h["q"], h["k"], h["v"], h["pt"], h["lens"], g["block_idx"],
                         g["n_blocks"], qh_mask=qh_mask)


def compare_step(g: dict, o: dict, h: dict, od: oracle.Dims, bh_pairs, dense: bool = True):
    """Bit-exact integer outputs and toleranced float outputs on the (b, h) pairs given
    (with per-head selection, the selection rows of every query head of kv head h). FP8
    keys: the selection is checked for validity within the fp32 bound instead
    (fp8_reference) and the outputs against the oracle's attention over it."""
    G = od.hq // od.hkv
    stats = []
    fp8 = bool(od.key_fp8)
    if fp8:
        o = dict(o)
        o["out"], o["lse"] = fp8_reference(g, o, h, od, bh_pairs)
    for b, hh in bh_pairs:
        np.testing.assert_array_equal(g["k_scale"][b, hh], o["k_scale"][b, hh])
        np.testing.assert_array_equal(logical_rows(g["kq"], h["pt"], h["lens"], b, hh),
                                      logical_rows(o["kq"], h["pt"], h["lens"], b, hh))
        for r in (range(hh * G, hh * G + G) if od.per_head else (hh,)):
            # FP8: the selection was validated above; the step's must be the same one (the
            # same fp32 scorer and exact selection on its maxima)
            want = g if fp8 else o
            if not fp8:
                np.testing.assert_array_equal(g["block_max"][b, r], o["block_max"][b, r])
                np.testing.assert_array_equal(g["chunk_idx"][b, r], o["chunk_idx"][b, r])
                np.testing.assert_array_equal(g["n_chunks"][b, r], o["n_chunks"][b, r])
                np.testing.assert_array_equal(g["block_idx"][b, r], o["block_idx"][b, r])
                np.testing.assert_array_equal(g["n_blocks"][b, r], o["n_blocks"][b, r])
            if "step_block_idx" in g:  # the whole decode step's own selection
                np.testing.assert_array_equal(g["step_block_idx"][b, r], want["block_idx"][b, r])
                np.testing.assert_array_equal(g["step_n_blocks"][b, r], want["n_blocks"][b, r])
        rows = slice(hh * G, (hh + 1) * G)
        stats.append(assert_close(g["out"][b, rows], o["out"][b, rows], f"sparse out b{b} h{hh}"))
        np.testing.assert_allclose(g["lse"][b, rows], o["lse"][b, rows], atol=2e-4, rtol=1e-5)
        if "step_out" in g:
            stats.append(assert_close(g["step_out"][b, rows], o["out"][b, rows],
                                      f"decode-step out b{b} h{hh}"))
            np.testing.assert_allclose(g["step_lse"][b, rows], o["lse"][b, rows], atol=2e-4,
                                       rtol=1e-5)
        if dense:
            stats.append(assert_close(g["out_dense"][b, rows], o["out_dense"][b, rows],
                                      f"dense out b{b} h{hh}"))
            np.testing.assert_allclose(g["lse_dense"][b, rows], o["lse_dense"][b, rows],
                                       atol=2e-4, rtol=1e-5)
    return stats
