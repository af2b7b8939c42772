"""Seeded synthetic decode-step workloads.

This module draws random inputs only; it holds none of the method's arithmetic, so both
the CUDA path and the CPU oracle can consume what it makes. It stands in for the
long-context benchmarks the pages evaluate on (InfiniteHiP article: InfiniteBench
multiple-choice and a passkey-retrieval sample; HCAttention: LongBench), none of which
is used here.

Recipe (all seeded; one torch.Generator on the requested device):
  * q ~ N(0, 1) per element, rounded to bf16 (the configurations give only K/V);
  * K, V ~ N(0, 1), bf16, in 16-token pages laid out [page][kv head][slot][channel];
  * per (sequence, kv head) 4 of the 128 key channels, drawn without replacement, are
    multiplied by 8 over every token (outlier channels);
  * per (sequence, kv head) `planted` token positions, drawn uniformly without
    replacement from [0, N_b), get the key 3*u + N(0, 0.3^2) with u the unit vector
    of the mean of the group's fp32 query vectors (written after the outlier scaling);
    the 1M-token configuration adds 64 more such "needle" positions;
  * page table: the identity for single-sequence configurations; for the batched
    configuration the pool of sum_b ceil(N_b / 16) pages is randomly permuted; unused
    table entries are -1; the slots of a last page past N_b hold random keys (they are
    outside the sequence and must be ignored).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch

PAGE = 16
HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    batch: int
    hq: int
    hkv: int
    context: Optional[int]          # fixed context (tokens, including the current one)
    context_range: Optional[tuple]  # (lo, hi) inclusive, per sequence, when batched
    k1: int
    k2: int
    sink: int
    window: int
    chunk: int = 64
    block: int = 16
    paged_permuted: bool = False
    planted: int = 8
    needles: int = 0
    kv_on_host: bool = False
    chunk0: int = 0  # k0 > 0: a pruning module on chunks of chunk0 tokens in front
    k0: int = 0
    key_bits: int = 8  # key codes: 8-bit, or 4-bit (two per byte)
    per_head: int = 0  # 1: every query head selects its own blocks
    key_fp8: int = 0  # 1: FP8 E4M3 key codes


CONFIGS: Dict[str, Config] = {
    # tiny decode step: batch 1, 4 query heads sharing 1 kv head, 8192 tokens
    "tiny-8k": Config("tiny-8k", 1, 4, 1, 8192, None, k1=16, k2=16, sink=64, window=256),
    # Llama-3-8B-shaped single layer at 128K tokens
    "llama3-8b-128k": Config("llama3-8b-128k", 1, 32, 8, 131072, None,
                             k1=256, k2=128, sink=128, window=1024),
    # batched paged decode, 8 sequences of 32K..128K tokens, permuted page pool
    "paged-b8-32k-128k": Config("paged-b8-32k-128k", 8, 32, 8, None, (32768, 131072),
                                k1=16, k2=16, sink=64, window=256, paged_permuted=True),
    # the same batch with the 128K configuration's pruning budget
    "paged-b8-32k-128k-wide": Config("paged-b8-32k-128k-wide", 8, 32, 8, None, (32768, 131072),
                                     k1=256, k2=128, sink=128, window=1024,
                                     paged_permuted=True),
    # 1M tokens with 64 extra needles per kv head
    "llama3-8b-1m": Config("llama3-8b-1m", 1, 32, 8, 1048576, None,
                           k1=512, k2=256, sink=128, window=2048, needles=64),
    # the same with three stacked modules: top-256 chunks of 256 tokens, then top-512 of
    # their 64-token chunks, then top-256 blocks
    "llama3-8b-1m-3mod": Config("llama3-8b-1m-3mod", 1, 32, 8, 1048576, None,
                                k1=512, k2=256, sink=128, window=2048, needles=64,
                                chunk0=256, k0=256),
    # a 128K step with groups of 8 query heads (Llama-3-70B-shaped attention layer)
    "llama3-70b-128k": Config("llama3-70b-128k", 1, 64, 8, 131072, None,
                              k1=256, k2=128, sink=128, window=1024),
    # the 128K step with per-head selection (every query head keeps its own 128 blocks)
    "llama3-8b-128k-perhead": Config("llama3-8b-128k-perhead", 1, 32, 8, 131072, None,
                                     k1=256, k2=128, sink=128, window=1024, per_head=1),
    # the 128K step with FP8 E4M3 key codes (fp32 scores)
    "llama3-8b-128k-fp8": Config("llama3-8b-128k-fp8", 1, 32, 8, 131072, None,
                                 k1=256, k2=128, sink=128, window=1024, key_fp8=1),
    # the 128K and 1M steps with 4-bit key codes (half the bytes the scorer reads)
    "llama3-8b-128k-int4": Config("llama3-8b-128k-int4", 1, 32, 8, 131072, None,
                                  k1=256, k2=128, sink=128, window=1024, key_bits=4),
    "llama3-8b-1m-int4": Config("llama3-8b-1m-int4", 1, 32, 8, 1048576, None,
                                k1=512, k2=256, sink=128, window=2048, needles=64, key_bits=4),
    # 3M tokens, bf16 K/V in pinned host memory, int8 keys in HBM
    "llama3-8b-3m-offload": Config("llama3-8b-3m-offload", 1, 32, 8, 3145728, None,
                                   k1=512, k2=256, sink=128, window=2048, kv_on_host=True),
    # the offloaded step at 1M tokens: the same attended set (K2, sink, window), so the same
    # bytes over the host link per step, with a third of the scan (profiler captures)
    "llama3-8b-1m-offload": Config("llama3-8b-1m-offload", 1, 32, 8, 1048576, None,
                                   k1=512, k2=256, sink=128, window=2048, kv_on_host=True),
}

ORDER: List[str] = ["tiny-8k", "llama3-8b-128k", "paged-b8-32k-128k", "llama3-8b-1m",
                    "llama3-8b-3m-offload"]


def with_context(cfg: Config, context: int, **changes) -> Config:
    """A copy of ``cfg`` at another (fixed) context length, for smaller test cases."""
    return dataclasses.replace(cfg, context=context, context_range=None, **changes)


def seq_lengths(cfg: Config, seed: int) -> List[int]:
    if cfg.context is not None:
        return [int(cfg.context)] * cfg.batch
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)
    lo, hi = cfg.context_range
    return [int(x) for x in torch.randint(lo, hi + 1, (cfg.batch,), generator=g)]


def _randn(shape, gen, device, chunk_rows: int = 1 << 20):
    """Standard normals in fp32, drawn in row slabs so that huge tensors never need a
    full fp32 copy; returned as bf16."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def make_workload(cfg: Config, seed: int = 0, device: str = "cpu",
                  host_pinned: bool = False) -> dict:
    """Build one decode step's inputs. Returns a dict of torch tensors:
    q [B][Hq][D] bf16, k_cache / v_cache [P][Hkv][16][D] bf16, page_table [B][maxP]
    int32, seq_lens [B] int32, plus 'config', 'lens', 'outlier_channels' and
    'planted' (per (b, h) the planted positions) for reporting.

    ``device`` is where the random numbers are drawn; with ``host_pinned`` the K/V
    caches are moved to pinned host memory afterwards (page slabs at a time)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    lens = seq_lengths(cfg, seed)
    B, Hq, Hkv, D = cfg.batch, cfg.hq, cfg.hkv, HEAD_DIM
    G = Hq // Hkv
    pages_per_seq = [-(-n // PAGE) for n in lens]
    max_pages = max(pages_per_seq)
    num_pages = sum(pages_per_seq)

    # page table
    if cfg.paged_permuted:
        gp = torch.Generator(device="cpu").manual_seed(seed + 104729)
        pool = torch.randperm(num_pages, generator=gp).to(torch.int32)
    else:
        pool = torch.arange(num_pages, dtype=torch.int32)
    page_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    owner = torch.empty(num_pages, dtype=torch.int64)
    off = 0
    for b, npg in enumerate(pages_per_seq):
        page_table[b, :npg] = pool[off:off + npg]
        owner[pool[off:off + npg].long()] = b
        off += npg

    q = torch.randn((B, Hq, D), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    k_cache = _randn((num_pages, Hkv, PAGE, D), gen, dev, chunk_rows=1 << 14)
    v_cache = _randn((num_pages, Hkv, PAGE, D), gen, dev, chunk_rows=1 << 14)

    # outlier channels: x8 over every token of (b, h)
    outliers = torch.stack([torch.stack([torch.randperm(D, generator=gen, device=dev)[:4]
                                         for _ in range(Hkv)]) for _ in range(B)])  # [B][Hkv][4]
    chan_scale = torch.ones((B, Hkv, D), device=dev, dtype=torch.float32)
    for b in range(B):
        for h in range(Hkv):
            chan_scale[b, h, outliers[b, h]] = 8.0
    owner_dev = owner.to(dev)
    slab = 1 << 14
    for p0 in range(0, num_pages, slab):
        p1 = min(num_pages, p0 + slab)
        s = chan_scale[owner_dev[p0:p1]]  # [pages][Hkv][D]
        k_cache[p0:p1] = (k_cache[p0:p1].float() * s[:, :, None, :]).to(torch.bfloat16)

    # planted tokens (and needles): k = 3 u + N(0, 0.3^2)
    planted = {}
    n_plant = cfg.planted + cfg.needles
    qf = q.float()
    for b in range(B):
        for h in range(Hkv):
            u = qf[b, h * G:(h + 1) * G].mean(dim=0)
            u = u / u.norm()
            pos = torch.randperm(lens[b], generator=gen, device=dev)[:n_plant]
            noise = torch.randn((pos.numel(), D), generator=gen, device=dev, dtype=torch.float32)
            keys = (3.0 * u[None, :] + 0.3 * noise).to(torch.bfloat16)
            pos_cpu = pos.cpu().long()
            pages = page_table[b, (pos_cpu // PAGE)].long().to(dev)
            slots = (pos_cpu % PAGE).to(dev)
            k_cache[pages, h, slots] = keys
            planted[(b, h)] = sorted(int(x) for x in pos_cpu)

    if host_pinned:
        k_cache = _to_pinned(k_cache)
        v_cache = _to_pinned(v_cache)

    return {
        "config": cfg,
        "lens": lens,
        "q": q,
        "k_cache": k_cache,
        "v_cache": v_cache,
        "page_table": page_table.to(dev),
        "seq_lens": torch.tensor(lens, dtype=torch.int32, device=dev),
        "num_pages": num_pages,
        "max_pages": max_pages,
        "outlier_channels": outliers.cpu(),
        "planted": planted,
    }


def _to_pinned(t: torch.Tensor, slab: int = 1 << 14) -> torch.Tensor:
    out = torch.empty(t.shape, dtype=t.dtype, device="cpu", pin_memory=True)
    for p0 in range(0, t.shape[0], slab):
        p1 = min(t.shape[0], p0 + slab)
        out[p0:p1].copy_(t[p0:p1])
    return out


def to_numpy_bits(t: torch.Tensor):
    """Raw 16-bit patterns of a bf16 tensor as a numpy uint16 array (CPU)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
