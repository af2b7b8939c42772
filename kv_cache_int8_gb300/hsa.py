"""Thin ctypes binding of libhsa (``include/hsa.h``), same names as the C ABI.

Arguments are marshalled only: torch tensors become raw pointers, the current torch
stream becomes the ``void* stream`` argument, and a nonzero status raises ``HsaError``.
Every step of the decode path runs in the CUDA library; nothing here computes. When the
library is missing or fails to load, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libhsa.so")

HSA_OK = 0
HSA_ERR_INVALID_ARG = 1
HSA_ERR_UNSUPPORTED = 2
HSA_ERR_CUDA = 3
HSA_ERR_TIMEOUT = 4
HSA_ERR_WORKSPACE_TOO_SMALL = 5
HSA_ERR_DEVICE_CHECK = 6

HSA_OP_QUANTIZE = 0
HSA_OP_SELECT = 1
HSA_OP_ATTEND = 2
HSA_OP_DENSE = 3
HSA_OP_STEP = 4
HSA_OP_CACHED = 5

# Every entry point declared in include/hsa.h.
EXPORTS = (
    "hsa_workspace_bytes", "hsa_status_string", "hsa_quantize_keys", "hsa_append_kv",
    "hsa_score_blocks", "hsa_prune", "hsa_select", "hsa_attend", "dense_decode",
    "hsa_decode_step", "hsa_decode_step_reuse", "hsa_read_device_error", "hsa_select_noalloc",
    "hsa_decode_step_kernels",
    "hsa_block_cache_bytes", "hsa_block_cache_mass", "hsa_attend_cached",
    "hsa_decode_step_cached",
)


class HsaError(RuntimeError):
    def __init__(self, name: str, code: int, text: str):
        super().__init__(f"{name} failed: {text} (status {code})")
        self.code = code


class hsa_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "hq", "hkv", "head_dim", "page_size", "max_pages_per_seq", "num_pages",
        "chunk", "block", "k1", "k2", "sink", "window")] + [
        ("sm_scale", ctypes.c_float), ("kv_on_host", ctypes.c_int32),
        ("chunk0", ctypes.c_int32), ("k0", ctypes.c_int32), ("key_bits", ctypes.c_int32),
        ("per_head", ctypes.c_int32), ("key_fp8", ctypes.c_int32),
        ("cache_policy", ctypes.c_int32)]


class hsa_step_io(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("io_on_host", ctypes.c_int32)]


_DIMS_CACHE: dict = {}  # field values -> their C struct (read-only to the library)


@dataclasses.dataclass
class Dims:
    batch: int
    hq: int
    hkv: int
    max_pages_per_seq: int
    num_pages: int
    chunk: int = 64
    k1: int = 16
    k2: int = 16
    sink: int = 64
    window: int = 256
    head_dim: int = 128
    page_size: int = 16
    block: int = 16
    sm_scale: float = 0.0
    kv_on_host: bool = False
    chunk0: int = 0  # k0 > 0: module 0 keeps the top-k0 chunks of chunk0 tokens
    k0: int = 0
    key_bits: int = 0  # 4: 4-bit key codes, two per byte; 0 or 8: 8-bit
    per_head: int = 0  # 1: every query head selects its own blocks (rows = hq)
    key_fp8: int = 0  # 1: FP8 E4M3 key codes (8-bit layout), fp32 scores
    cache_policy: int = 0  # block cache victims: 0 least recently used, 1 least cumulative mass

    def c(self) -> hsa_dims:
        """The C struct, built once per set of field values (every call of a step passes it)."""
        key = (self.batch, self.hq, self.hkv, self.head_dim, self.page_size,
               self.max_pages_per_seq, self.num_pages, self.chunk, self.block, self.k1,
               self.k2, self.sink, self.window, float(self.sm_scale),
               1 if self.kv_on_host else 0, self.chunk0, self.k0, self.key_bits, self.per_head,
               self.key_fp8, self.cache_policy)
        c = _DIMS_CACHE.get(key)
        if c is None:
            if len(_DIMS_CACHE) > 256:
                _DIMS_CACHE.clear()
            c = _DIMS_CACHE[key] = hsa_dims(*key)
        return c


_LIB = None


def load(path: Optional[str] = None):
    """Load libhsa.so (once). Raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libhsa.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(hsa_dims)
    sig = {
        "hsa_workspace_bytes": (SZ, [D, I32]),
        "hsa_status_string": (ctypes.c_char_p, [I32]),
        "hsa_quantize_keys": (I32, [D, P, P, P, I32, I32, P, P, P, SZ, P]),
        "hsa_append_kv": (I32, [D, P, P, P, P, P, P, P, P, P]),
        "hsa_score_blocks": (I32, [D, P, P, P, P, P, P, P, P]),
        "hsa_prune": (I32, [D, P, P, P, P, P, P, P, P]),
        "hsa_select": (I32, [D, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "hsa_attend": (I32, [D, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "dense_decode": (I32, [D, P, P, P, P, P, P, P, P, SZ, P]),
        "hsa_decode_step": (I32, [D, ctypes.POINTER(hsa_step_io), P, P, P, P, P, P, P, P, P,
                                  SZ, P]),
        "hsa_decode_step_reuse": (I32, [D, ctypes.POINTER(hsa_step_io), P, P, P, P, P, P, P, P,
                                        P, SZ, P]),
        "hsa_block_cache_bytes": (SZ, [D, I32]),
        "hsa_block_cache_mass": (P, [D, P, I32]),
        "hsa_attend_cached": (I32, [D, P, P, P, P, P, P, P, P, I32, P, P, P, SZ, P]),
        "hsa_decode_step_cached": (I32, [D, ctypes.POINTER(hsa_step_io), P, P, P, P, P, P, P, P,
                                         P, I32, P, SZ, P]),
        "hsa_read_device_error": (I32, [P, P, ctypes.POINTER(I32)]),
        "hsa_select_noalloc": (I32, [D, P, P, P, P, P, P, P, P, P, P]),
        "hsa_decode_step_kernels": (I32, [D]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None) -> int:
    if stream is None:
        if _RAW_STREAM is not None:  # the current stream's handle without a Stream object
            return _RAW_STREAM(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(name: str, rc: int) -> None:
    if rc != HSA_OK:
        raise HsaError(name, rc, load().hsa_status_string(rc).decode())


def hsa_status_string(code: int) -> str:
    return load().hsa_status_string(code).decode()


def hsa_workspace_bytes(d: Dims, op: int) -> int:
    cd = d.c()
    return int(load().hsa_workspace_bytes(ctypes.byref(cd), op))


def workspace(d: Dims, op: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace tensor of the size `op` needs (256-byte aligned storage)."""
    n = hsa_workspace_bytes(d, op)
    if n == 0:
        raise HsaError("hsa_workspace_bytes", HSA_ERR_INVALID_ARG, "invalid descriptor")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def hsa_quantize_keys(d: Dims, k_cache, page_table, seq_lens, mode: int, append_from: int, kq,
                      k_scale, ws=None, stream=None) -> None:
    cd = d.c()
    _check("hsa_quantize_keys", load().hsa_quantize_keys(
        ctypes.byref(cd), _p(k_cache), _p(page_table), _p(seq_lens), mode, append_from, _p(kq),
        _p(k_scale), _p(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def hsa_append_kv(d: Dims, k_new, v_new, k_cache, v_cache, kq, k_scale, page_table, seq_lens,
                  stream=None) -> None:
    cd = d.c()
    _check("hsa_append_kv", load().hsa_append_kv(
        ctypes.byref(cd), _p(k_new), _p(v_new), _p(k_cache), _p(v_cache), _p(kq), _p(k_scale),
        _p(page_table), _p(seq_lens), _stream(stream)))


def hsa_score_blocks(d: Dims, q, kq, k_scale, page_table, seq_lens, block_max, tile_max=None,
                     stream=None) -> None:
    cd = d.c()
    _check("hsa_score_blocks", load().hsa_score_blocks(
        ctypes.byref(cd), _p(q), _p(kq), _p(k_scale), _p(page_table), _p(seq_lens),
        _p(block_max), _p(tile_max), _stream(stream)))


def hsa_prune(d: Dims, seq_lens, block_max, tile_max, chunk_idx, n_chunks, block_idx, n_blocks,
              stream=None) -> None:
    cd = d.c()
    _check("hsa_prune", load().hsa_prune(
        ctypes.byref(cd), _p(seq_lens), _p(block_max), _p(tile_max), _p(chunk_idx),
        _p(n_chunks), _p(block_idx), _p(n_blocks), _stream(stream)))


def hsa_select(d: Dims, q, kq, k_scale, page_table, seq_lens, chunk_idx, n_chunks, block_idx,
               n_blocks, ws, stream=None) -> None:
    cd = d.c()
    _check("hsa_select", load().hsa_select(
        ctypes.byref(cd), _p(q), _p(kq), _p(k_scale), _p(page_table), _p(seq_lens),
        _p(chunk_idx), _p(n_chunks), _p(block_idx), _p(n_blocks), _p(ws), ws.numel(),
        _stream(stream)))


def hsa_select_noalloc(d: Dims, q, kq, k_scale, page_table, seq_lens, chunk_idx, n_chunks,
                       block_idx, n_blocks, stream=None) -> None:
    """hsa_select for callers that cannot allocate device memory: the scratch is a fixed
    4 MiB array inside the library (see include/hsa.h for the size limit and the sharing
    rules)."""
    cd = d.c()
    _check("hsa_select_noalloc", load().hsa_select_noalloc(
        ctypes.byref(cd), _p(q), _p(kq), _p(k_scale), _p(page_table), _p(seq_lens),
        _p(chunk_idx), _p(n_chunks), _p(block_idx), _p(n_blocks), _stream(stream)))


def hsa_attend(d: Dims, q, k_cache, v_cache, page_table, seq_lens, block_idx, n_blocks, out,
               lse, ws, stream=None) -> None:
    cd = d.c()
    _check("hsa_attend", load().hsa_attend(
        ctypes.byref(cd), _p(q), _p(k_cache), _p(v_cache), _p(page_table), _p(seq_lens),
        _p(block_idx), _p(n_blocks), _p(out), _p(lse), _p(ws), ws.numel(), _stream(stream)))


def dense_decode(d: Dims, q, k_cache, v_cache, page_table, seq_lens, out, lse, ws,
                 stream=None) -> None:
    cd = d.c()
    _check("dense_decode", load().dense_decode(
        ctypes.byref(cd), _p(q), _p(k_cache), _p(v_cache), _p(page_table), _p(seq_lens),
        _p(out), _p(lse), _p(ws), ws.numel(), _stream(stream)))


def hsa_decode_step(d: Dims, q, k_new, v_new, out, lse, k_cache, v_cache, kq, k_scale,
                    page_table, seq_lens, block_idx, n_blocks, ws, io_on_host: bool = False,
                    stream=None) -> None:
    cd = d.c()
    io = hsa_step_io(_p(q), _p(k_new), _p(v_new), _p(out), _p(lse), 1 if io_on_host else 0)
    _check("hsa_decode_step", load().hsa_decode_step(
        ctypes.byref(cd), ctypes.byref(io), _p(k_cache), _p(v_cache), _p(kq), _p(k_scale),
        _p(page_table), _p(seq_lens), _p(block_idx), _p(n_blocks), _p(ws), ws.numel(),
        _stream(stream)))


class DecodeStep:
    """hsa_decode_step over a fixed set of buffers, for a decode loop that calls it every
    step: the C arguments are marshalled once, so a call costs the C call alone. The
    buffers' contents may change between calls (new q / k_new / v_new, longer seq_lens);
    the buffers themselves must stay alive and in place.

    graph=True: the first call runs the step and then records it into a CUDA graph; every
    later call replays the graph on the current stream (one launch instead of one per
    kernel). The kernels read every input from its buffer, so replays see new contents; the
    descriptor and the buffers are those of the recording."""

    def __init__(self, d: Dims, q, k_new, v_new, out, lse, k_cache, v_cache, kq, k_scale,
                 page_table, seq_lens, block_idx, n_blocks, ws, io_on_host: bool = False,
                 stream=None, graph: bool = False):
        self._keep = (q, k_new, v_new, out, lse, k_cache, v_cache, kq, k_scale, page_table,
                      seq_lens, block_idx, n_blocks, ws)
        self._cd = d.c()
        self._io = hsa_step_io(_p(q), _p(k_new), _p(v_new), _p(out), _p(lse),
                               1 if io_on_host else 0)
        self._fn = load().hsa_decode_step
        self._head = (ctypes.byref(self._cd), ctypes.byref(self._io), _p(k_cache), _p(v_cache),
                      _p(kq), _p(k_scale), _p(page_table), _p(seq_lens), _p(block_idx),
                      _p(n_blocks), _p(ws), ws.numel())
        self._args = self._head + (_stream(stream),)
        self._use_graph = graph
        self._graph = None

    def _run(self, args) -> None:
        rc = self._fn(*args)
        if rc != HSA_OK:
            _check("hsa_decode_step", rc)

    def __call__(self) -> None:
        if self._graph is not None:
            self._graph.replay()
            return
        self._run(self._args)
        if self._use_graph:
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):  # the step's launches, on the recording stream
                self._run(self._head + (_stream(None),))
            self._graph = g


def hsa_decode_step_reuse(d: Dims, q, k_new, v_new, out, lse, k_cache, v_cache, kq, k_scale,
                          page_table, seq_lens, block_idx, n_blocks, ws, io_on_host: bool = False,
                          stream=None) -> None:
    """Append + attend with the selection block_idx / n_blocks of an earlier step."""
    cd = d.c()
    io = hsa_step_io(_p(q), _p(k_new), _p(v_new), _p(out), _p(lse), 1 if io_on_host else 0)
    _check("hsa_decode_step_reuse", load().hsa_decode_step_reuse(
        ctypes.byref(cd), ctypes.byref(io), _p(k_cache), _p(v_cache), _p(kq), _p(k_scale),
        _p(page_table), _p(seq_lens), _p(block_idx), _p(n_blocks), _p(ws), ws.numel(),
        _stream(stream)))


def block_cache(d: Dims, capacity: int):
    """A zeroed device buffer for the GPU block cache (see hsa_block_cache_bytes)."""
    n = load().hsa_block_cache_bytes(ctypes.byref(d.c()), capacity)
    if n == 0:
        raise HsaError("hsa_block_cache_bytes", HSA_ERR_INVALID_ARG, "capacity or shape rejected")
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def block_cache_mass(d: Dims, cache, capacity: int):
    """The block cache's cumulative attention masses: a float32 [num_pages][hkv] view into
    `cache` (see hsa_block_cache_mass)."""
    ptr = load().hsa_block_cache_mass(ctypes.byref(d.c()), _p(cache), capacity)
    if not ptr:
        raise HsaError("hsa_block_cache_mass", HSA_ERR_INVALID_ARG, "shape or capacity rejected")
    off = ptr - cache.data_ptr()
    n = d.num_pages * d.hkv
    return cache[off: off + 4 * n].view(torch.float32).view(d.num_pages, d.hkv)


def hsa_attend_cached(d: Dims, q, k_cache, v_cache, page_table, seq_lens, block_idx, n_blocks,
                      cache, capacity: int, out, lse, ws, stream=None) -> None:
    cd = d.c()
    _check("hsa_attend_cached", load().hsa_attend_cached(
        ctypes.byref(cd), _p(q), _p(k_cache), _p(v_cache), _p(page_table), _p(seq_lens),
        _p(block_idx), _p(n_blocks), _p(cache), capacity, _p(out), _p(lse), _p(ws), ws.numel(),
        _stream(stream)))


def hsa_decode_step_cached(d: Dims, q, k_new, v_new, out, lse, k_cache, v_cache, kq, k_scale,
                           page_table, seq_lens, block_idx, n_blocks, cache, capacity: int, ws,
                           io_on_host: bool = False, stream=None) -> None:
    cd = d.c()
    io = hsa_step_io(_p(q), _p(k_new), _p(v_new), _p(out), _p(lse), 1 if io_on_host else 0)
    _check("hsa_decode_step_cached", load().hsa_decode_step_cached(
        ctypes.byref(cd), ctypes.byref(io), _p(k_cache), _p(v_cache), _p(kq), _p(k_scale),
        _p(page_table), _p(seq_lens), _p(block_idx), _p(n_blocks), _p(cache), capacity, _p(ws),
        ws.numel(), _stream(stream)))


def hsa_decode_step_kernels(d: Dims) -> int:
    """Kernels that hsa_decode_step launches for d (device I/O)."""
    return int(load().hsa_decode_step_kernels(ctypes.byref(d.c())))


def hsa_read_device_error(ws, stream=None) -> int:
    """Reads and clears a workspace's device error word (ws None: the error word of
    hsa_select_noalloc's fixed scratch array)."""
    code = ctypes.c_int32(0)
    _check("hsa_read_device_error", load().hsa_read_device_error(
        _p(ws), _stream(stream), ctypes.byref(code)))
    return int(code.value)
