"""ctypes front end of the C oracle (``oracle.c``); numpy in, numpy out.

TEST INFRASTRUCTURE (see the package docstring). bf16 tensors travel as their raw
16-bit patterns (``numpy.uint16``); the C side widens them exactly.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import numpy as np

from . import build as _build

_LIB = None


class _CDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "hq", "hkv", "head_dim", "page_size", "max_pages_per_seq", "num_pages",
        "chunk", "block", "k1", "k2", "sink", "window")] + [("sm_scale", ctypes.c_double),
                                                            ("chunk0", ctypes.c_int32),
                                                            ("k0", ctypes.c_int32),
                                                            ("key_bits", ctypes.c_int32),
                                                            ("per_head", ctypes.c_int32),
                                                            ("key_fp8", ctypes.c_int32)]


@dataclasses.dataclass
class Dims:
    """Problem sizes; the same fields as the CUDA library's descriptor, kept separately."""
    batch: int
    hq: int
    hkv: int
    head_dim: int
    page_size: int
    max_pages_per_seq: int
    num_pages: int
    chunk: int
    block: int
    k1: int
    k2: int
    sink: int
    window: int
    sm_scale: float = 0.0
    chunk0: int = 0  # k0 > 0: a first module keeps the top-k0 chunks of chunk0 tokens
    k0: int = 0
    key_bits: int = 0  # 4: 4-bit key codes (levels +-7); 0 or 8: 8-bit
    per_head: int = 0  # 1: every query head selects its own chunks and blocks
    key_fp8: int = 0  # 1: FP8 E4M3 key codes (int8 arrays hold their bits), fp32 scores

    def c(self) -> _CDims:
        return _CDims(*[int(getattr(self, f[0])) for f in _CDims._fields_[:13]],
                      float(self.sm_scale), int(self.chunk0), int(self.k0),
                      int(self.key_bits), int(self.per_head), int(self.key_fp8))

    @property
    def sel_rows(self) -> int:
        """Selection rows per sequence: kv heads, or query heads with per-head selection."""
        return self.hq if self.per_head else self.hkv

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def max_blocks(self) -> int:
        return -(-self.max_pages_per_seq * self.page_size // self.block)


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        D = ctypes.POINTER(_CDims)
        sigs = {
            "oracle_quantize_keys": [D, P, P, P, P, P, P],
            "oracle_quantize_append": [D, P, P, P, ctypes.c_int32, P, P],
            "oracle_query_codes": [D, P, P, P, P],
            "oracle_select": [D, P, P, P, P, P, P, P, P, P, P, P],
            "oracle_attend": [D, P, P, P, P, P, P, P, P, P, P],
            "oracle_dense": [D, P, P, P, P, P, P, P, P],
            "oracle_recall": [D, P, P, P, P, P, P, P, P],
            "oracle_block_mass": [D, P, P, P, P, P, P, P],
            "oracle_fp8_block_scores": [D, P, P, P, P, P, P, P, P],
        }
        for name, args in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _LIB = lib
    return _LIB


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 tensors are passed as raw uint16 bit patterns"
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (code {rc})")


def num_threads() -> int:
    return int(_lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """The threads later oracle calls may use (n >= 1)."""
    _lib().oracle_set_num_threads(int(n))


def quantize_keys(d: Dims, k: np.ndarray, page_table, seq_lens, bh_mask=None):
    """Full key quantisation: returns (kq int8 same shape as k, k_scale f32 [B][Hkv][D])."""
    k = _u16(k)
    kq = np.zeros(k.shape, dtype=np.int8)
    scale = np.zeros((d.batch, d.hkv, d.head_dim), dtype=np.float32)
    cd = d.c()
    _check(_lib().oracle_quantize_keys(ctypes.byref(cd), _ptr(k), _ptr(_i32(page_table)),
                                       _ptr(_i32(seq_lens)),
                                       _ptr(None if bh_mask is None else _i32(bh_mask)),
                                       _ptr(kq), _ptr(scale)), "oracle_quantize_keys")
    return kq, scale


def quantize_append(d: Dims, k: np.ndarray, page_table, seq_lens, start: int,
                    k_scale: np.ndarray, kq: np.ndarray) -> np.ndarray:
    """Codes of tokens [start, N_b) (start < 0: each sequence's last token) with the
    stored scales; returns an updated copy of ``kq``."""
    kq = np.array(kq, dtype=np.int8, copy=True, order="C")
    cd = d.c()
    _check(_lib().oracle_quantize_append(ctypes.byref(cd), _ptr(_u16(k)), _ptr(_i32(page_table)),
                                         _ptr(_i32(seq_lens)), int(start),
                                         _ptr(np.ascontiguousarray(k_scale, dtype=np.float32)),
                                         _ptr(kq)), "oracle_quantize_append")
    return kq


def query_codes(d: Dims, q: np.ndarray, k_scale: np.ndarray):
    """Query codes qq [B][Hkv][G][D] int8 and the group scales sq [B][Hkv] f32."""
    qq = np.zeros((d.batch, d.hkv, d.group, d.head_dim), dtype=np.int8)
    sq = np.zeros((d.batch, d.hkv), dtype=np.float32)
    cd = d.c()
    _check(_lib().oracle_query_codes(ctypes.byref(cd), _ptr(_u16(q)),
                                     _ptr(np.ascontiguousarray(k_scale, dtype=np.float32)),
                                     _ptr(qq), _ptr(sq)), "oracle_query_codes")
    return qq, sq


def select(d: Dims, q: np.ndarray, k_scale: np.ndarray, kq: np.ndarray, page_table, seq_lens,
           bh_mask=None, want_block_max: bool = False):
    """The two pruning modules. Returns a dict with chunk_idx [B][R][K1],
    n_chunks [B][R], block_idx [B][R][K2], n_blocks [B][R] and, on request,
    block_max [B][R][max_blocks] (INT32_MIN where a block has no candidate token); R is
    Hkv, or Hq with per-head selection. bh_mask [B][Hkv] selects kv heads (all rows of a
    selected kv head are computed)."""
    B, H = d.batch, d.sel_rows
    out = {
        "chunk_idx": np.full((B, H, max(d.k1, 0)), -1, dtype=np.int32),
        "n_chunks": np.zeros((B, H), dtype=np.int32),
        "block_idx": np.full((B, H, max(d.k2, 0)), -1, dtype=np.int32),
        "n_blocks": np.zeros((B, H), dtype=np.int32),
    }
    bm = np.zeros((B, H, d.max_blocks), dtype=np.int32) if want_block_max else None
    cd = d.c()
    kq = np.ascontiguousarray(kq)
    assert kq.dtype == np.int8
    _check(_lib().oracle_select(ctypes.byref(cd), _ptr(_u16(q)),
                                _ptr(np.ascontiguousarray(k_scale, dtype=np.float32)), _ptr(kq),
                                _ptr(_i32(page_table)), _ptr(_i32(seq_lens)),
                                _ptr(None if bh_mask is None else _i32(bh_mask)), _ptr(bm),
                                _ptr(out["chunk_idx"]), _ptr(out["n_chunks"]),
                                _ptr(out["block_idx"]), _ptr(out["n_blocks"])), "oracle_select")
    if want_block_max:
        out["block_max"] = bm
    return out


def fp8_block_scores(d: Dims, q: np.ndarray, k_scale: np.ndarray, kq: np.ndarray, page_table,
                     seq_lens, bh_mask=None):
    """FP8 keys: (score, bound), both f64 [B][R][max_blocks]. score = the exact block score
    (max over the block's candidate tokens and the row's query heads of the dot of the folded
    fp32 query with the E4M3 values; -inf where the block has no candidate token); bound =
    Higham's gamma_128 times the largest sum |q' x| among those: any fp32 evaluation of the
    dots with one rounding per term gives block maxima within `bound` of `score`."""
    assert d.key_fp8 == 1
    B, H = d.batch, d.sel_rows
    score = np.zeros((B, H, d.max_blocks), dtype=np.float64)
    bound = np.zeros((B, H, d.max_blocks), dtype=np.float64)
    cd = d.c()
    kq = np.ascontiguousarray(kq)
    assert kq.dtype == np.int8
    _check(_lib().oracle_fp8_block_scores(
        ctypes.byref(cd), _ptr(_u16(q)), _ptr(np.ascontiguousarray(k_scale, dtype=np.float32)),
        _ptr(kq), _ptr(_i32(page_table)), _ptr(_i32(seq_lens)),
        _ptr(None if bh_mask is None else _i32(bh_mask)), _ptr(score), _ptr(bound)),
        "oracle_fp8_block_scores")
    return score, bound


def selection_within_bounds(d: Dims, seq_lens, score: np.ndarray, bound: np.ndarray,
                            chunk_idx, n_chunks, block_idx, n_blocks, rows=None):
    """Whether a selection is one of the two modules' results for block scores known only to
    within `bound` of `score` (fp8_block_scores): per row, the counts are min(K1, #valid
    chunks) and min(K2, #candidate blocks of the kept chunks), the lists ascending and -1
    padded, and no dropped chunk (block) beats a kept one by more than their two bounds. A
    chunk's score is the max of its blocks' scores, its bound the max of their bounds.
    Returns a list of violations (empty: valid). rows: (b, r) pairs to check (all if None)."""
    P = d.chunk // d.block
    bad = []
    B, R = score.shape[:2]
    for b, r in (rows if rows is not None else [(b, r) for b in range(B) for r in range(R)]):
        valid = np.isfinite(score[b, r])
        n_ch = -(-score.shape[2] // P)
        cs = np.full(n_ch, -np.inf)
        cb = np.zeros(n_ch)
        for k in np.nonzero(valid)[0]:
            cs[k // P] = max(cs[k // P], score[b, r, k])
            cb[k // P] = max(cb[k // P], bound[b, r, k])
        cvalid = np.nonzero(np.isfinite(cs))[0]
        nc = int(n_chunks[b, r])
        kept_c = [int(c) for c in chunk_idx[b, r][:nc]]
        if nc != min(d.k1, cvalid.size):
            bad.append((b, r, "chunk count", nc, min(d.k1, cvalid.size)))
        if any(c < 0 for c in kept_c) or kept_c != sorted(set(kept_c)) or \
                any(int(c) != -1 for c in chunk_idx[b, r][nc:]):
            bad.append((b, r, "chunk list", kept_c))
            continue
        if any(not np.isfinite(cs[c]) for c in kept_c):
            bad.append((b, r, "invalid chunk kept"))
            continue
        dropped_c = np.setdiff1d(cvalid, kept_c)
        if dropped_c.size and kept_c:
            worst_kept = min(kept_c, key=lambda c: cs[c] + cb[c])
            best_drop = dropped_c[np.argmax(cs[dropped_c] - cb[dropped_c])]
            if cs[best_drop] - cb[best_drop] > cs[worst_kept] + cb[worst_kept]:
                bad.append((b, r, "chunk order", int(best_drop), worst_kept))
        cand = [k for c in kept_c for k in range(c * P, c * P + P) if k < valid.size and valid[k]]
        nb = int(n_blocks[b, r])
        kept_b = [int(k) for k in block_idx[b, r][:nb]]
        if nb != min(d.k2, len(cand)):
            bad.append((b, r, "block count", nb, min(d.k2, len(cand))))
        if kept_b != sorted(set(kept_b)) or any(int(k) != -1 for k in block_idx[b, r][nb:]) \
                or not set(kept_b) <= set(cand):
            bad.append((b, r, "block list", kept_b))
            continue
        dropped_b = np.array(sorted(set(cand) - set(kept_b)), dtype=np.int64)
        if dropped_b.size and kept_b:
            s_, e_ = score[b, r], bound[b, r]
            worst_kept = min(kept_b, key=lambda k: s_[k] + e_[k])
            best_drop = dropped_b[np.argmax(s_[dropped_b] - e_[dropped_b])]
            if s_[best_drop] - e_[best_drop] > s_[worst_kept] + e_[worst_kept]:
                bad.append((b, r, "block order", int(best_drop), worst_kept))
    return bad


def attend(d: Dims, q, k, v, page_table, seq_lens, block_idx, n_blocks, qh_mask=None):
    """Sparse decode attention: returns (out f64 [B][Hq][D], lse f64 [B][Hq])."""
    out = np.zeros((d.batch, d.hq, d.head_dim), dtype=np.float64)
    lse = np.zeros((d.batch, d.hq), dtype=np.float64)
    cd = d.c()
    _check(_lib().oracle_attend(ctypes.byref(cd), _ptr(_u16(q)), _ptr(_u16(k)), _ptr(_u16(v)),
                                _ptr(_i32(page_table)), _ptr(_i32(seq_lens)),
                                _ptr(_i32(block_idx)), _ptr(_i32(n_blocks)),
                                _ptr(None if qh_mask is None else _i32(qh_mask)),
                                _ptr(out), _ptr(lse)), "oracle_attend")
    return out, lse


def dense(d: Dims, q, k, v, page_table, seq_lens, qh_mask=None):
    """Dense decode attention over [0, N): returns (out f64 [B][Hq][D], lse f64 [B][Hq])."""
    out = np.zeros((d.batch, d.hq, d.head_dim), dtype=np.float64)
    lse = np.zeros((d.batch, d.hq), dtype=np.float64)
    cd = d.c()
    _check(_lib().oracle_dense(ctypes.byref(cd), _ptr(_u16(q)), _ptr(_u16(k)), _ptr(_u16(v)),
                               _ptr(_i32(page_table)), _ptr(_i32(seq_lens)),
                               _ptr(None if qh_mask is None else _i32(qh_mask)),
                               _ptr(out), _ptr(lse)), "oracle_dense")
    return out, lse


def recall(d: Dims, q, k, page_table, seq_lens, block_idx, n_blocks, qh_mask=None):
    """Attention-mass recall of the attended set against dense attention, [B][Hq]."""
    r = np.zeros((d.batch, d.hq), dtype=np.float64)
    cd = d.c()
    _check(_lib().oracle_recall(ctypes.byref(cd), _ptr(_u16(q)), _ptr(_u16(k)),
                                _ptr(_i32(page_table)), _ptr(_i32(seq_lens)),
                                _ptr(_i32(block_idx)), _ptr(_i32(n_blocks)),
                                _ptr(None if qh_mask is None else _i32(qh_mask)), _ptr(r)),
           "oracle_recall")
    return r


def block_mass(d: Dims, q, k, page_table, seq_lens, block_idx, n_blocks):
    """Attention mass of every block under one call's sparse attention, [B][Hq][max_blocks]:
    the softmax probability over the attended set that the block's attended tokens receive
    from each query head. Summed over a kv head's query heads and accumulated over calls it
    is the block cache's cumulative-magnitude eviction key."""
    m = np.zeros((d.batch, d.hq, d.max_blocks), dtype=np.float64)
    cd = d.c()
    _check(_lib().oracle_block_mass(ctypes.byref(cd), _ptr(_u16(q)), _ptr(_u16(k)),
                                    _ptr(_i32(page_table)), _ptr(_i32(seq_lens)),
                                    _ptr(_i32(block_idx)), _ptr(_i32(n_blocks)), _ptr(m)),
           "oracle_block_mass")
    return m
