"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded
inputs. Integer outputs (key codes and scales, block maxima, kept chunk and block indices
and counts) must match bit for bit; attention outputs must satisfy max|err| <= 1e-2 and
relative L2 <= 5e-3 against the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import harness as H
from kv_cache_int8_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(wl, bh_pairs=None, qh_mask=None, dense=True, **over):
    hd, od = H.dims_pair(wl, **over)
    h = H.host_arrays(wl)
    g = H.gpu_step(H.to_cuda(wl), hd, dense=dense)
    bh_mask = None
    if bh_pairs is not None:
        bh_mask = np.zeros((od.batch, od.hkv), dtype=np.int32)
        for b, hh in bh_pairs:
            bh_mask[b, hh] = 1
        G = od.hq // od.hkv
        qh_mask = np.zeros((od.batch, od.hq), dtype=np.int32)
        for b, hh in bh_pairs:
            qh_mask[b, hh * G:(hh + 1) * G] = 1
    else:
        bh_pairs = [(b, hh) for b in range(od.batch) for hh in range(od.hkv)]
    o = H.oracle_step(h, od, bh_mask=bh_mask, qh_mask=qh_mask, dense=dense)
    return H.compare_step(g, o, h, od, bh_pairs, dense=dense), g, o


def test_tiny_8k_full():
    wl = W.make_workload(W.CONFIGS["tiny-8k"], seed=0)
    stats, g, o = _run(wl)
    assert g["n_blocks"][0, 0] == 16


def test_llama3_8b_128k_full():
    wl = W.make_workload(W.CONFIGS["llama3-8b-128k"], seed=0, device="cuda")
    _run(wl)


@pytest.mark.parametrize("name", ["paged-b8-32k-128k", "paged-b8-32k-128k-wide"])
def test_paged_batch_full(name):
    wl = W.make_workload(W.CONFIGS[name], seed=0, device="cuda")
    _run(wl)


def test_llama3_8b_1m_full():
    """1M tokens, all 8 kv heads: codes, scales, block maxima, both modules' index sets and
    the whole step's selection bit-exact; outputs within tolerance."""
    wl = W.make_workload(W.CONFIGS["llama3-8b-1m"], seed=0, device="cuda")
    _run(wl)


def test_llama3_8b_1m_three_modules_full():
    wl = W.make_workload(W.CONFIGS["llama3-8b-1m-3mod"], seed=0, device="cuda")
    _run(wl)


def test_llama3_70b_shaped_128k_groups_of_8_sampled_heads():
    """64 query heads over 8 kv heads: the scorer's max over 8 heads, the attention of 8
    heads per kv head."""
    wl = W.make_workload(W.CONFIGS["llama3-70b-128k"], seed=0, device="cuda")
    _run(wl, bh_pairs=[(0, 0), (0, 7)])


def test_llama3_8b_128k_per_head_selection_sampled_heads():
    """Per-head selection at 128K: the 4 query heads of kv heads 1 and 6, each on its own
    selection row."""
    wl = W.make_workload(W.CONFIGS["llama3-8b-128k"], seed=0, device="cuda")
    _run(wl, bh_pairs=[(0, 1), (0, 6)], per_head=1)


def test_llama3_8b_128k_fp8_keys_full():
    wl = W.make_workload(W.CONFIGS["llama3-8b-128k-fp8"], seed=0, device="cuda")
    _run(wl)


def test_tiny_8k_four_bit_keys():
    """4-bit key codes: codes (unpacked from their nibbles), scales amax / 7, block maxima
    and selections bit-exact against the oracle's 4-bit format; outputs within tolerance."""
    wl = W.make_workload(W.CONFIGS["tiny-8k"], seed=4)
    stats, g, o = _run(wl, key_bits=4)
    assert np.abs(g["kq"]).max() == 7


def test_paged_batch_four_bit_keys():
    """Ragged lengths, a permuted page pool and last pages past N_b with 4-bit codes."""
    cfg = dataclasses.replace(W.CONFIGS["paged-b8-32k-128k"], context_range=(1000, 9000),
                              batch=3, key_bits=4)
    wl = W.make_workload(cfg, seed=8)
    _run(wl)


def test_llama3_8b_128k_four_bit_keys_full():
    wl = W.make_workload(W.CONFIGS["llama3-8b-128k-int4"], seed=0, device="cuda")
    _run(wl)


def test_llama3_8b_1m_four_bit_keys_full():
    wl = W.make_workload(W.CONFIGS["llama3-8b-1m-int4"], seed=0, device="cuda")
    _run(wl)


def test_llama3_8b_3m_offloaded_four_heads():
    """3M tokens with K/V in pinned host memory: kv heads 0, 3, 5 and 7."""
    torch.cuda.empty_cache()
    wl = W.make_workload(W.CONFIGS["llama3-8b-3m-offload"], seed=0, device="cuda",
                         host_pinned=True)
    assert wl["k_cache"].is_pinned() and wl["v_cache"].is_pinned()
    _run(wl, bh_pairs=[(0, 0), (0, 3), (0, 5), (0, 7)], dense=False)


def test_deterministic_repeat():
    wl = W.make_workload(W.with_context(W.CONFIGS["llama3-8b-128k"], 20000), seed=3)
    hd, _ = H.dims_pair(wl)
    a = H.gpu_step(H.to_cuda(wl), hd)
    b = H.gpu_step(H.to_cuda(wl), hd)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
