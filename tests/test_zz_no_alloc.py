"""hsa_select_noalloc: the selection for callers that cannot allocate device memory (code
living inside a host program that owns every device allocation through its own pool, or
on a latency-critical path where cudaMalloc and its implicit device synchronisation are
not allowed). It keeps its scratch in a fixed 4 MiB array inside the library instead of a
caller workspace. This file is collected last on purpose, so that a run stopping at the
first failure has already run every other test."""
import pytest
import torch

import harness as H
from kv_cache_int8_gb300 import hsa
from kv_cache_int8_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(wl, d):
    dev = torch.device("cuda")
    dwl = H.to_cuda(wl)
    kq = torch.zeros(dwl["k_cache"].shape, dtype=torch.int8, device=dev)
    k_scale = torch.zeros((d.batch, d.hkv, 128), dtype=torch.float32, device=dev)
    hsa.hsa_quantize_keys(d, dwl["k_cache"], dwl["page_table"], dwl["seq_lens"], 0, 0, kq,
                          k_scale, hsa.workspace(d, hsa.HSA_OP_QUANTIZE))
    return dwl, kq, k_scale


def _outputs(d):
    dev = torch.device("cuda")
    rows = d.hq if d.per_head else d.hkv  # selection rows per sequence
    return (torch.full((d.batch, rows, d.k1), -7, dtype=torch.int32, device=dev),
            torch.full((d.batch, rows), -7, dtype=torch.int32, device=dev),
            torch.full((d.batch, rows, d.k2), -7, dtype=torch.int32, device=dev),
            torch.full((d.batch, rows), -7, dtype=torch.int32, device=dev))


def test_noalloc_select_matches_workspace_select_twice():
    """Calls in a row on different shapes (each one finds the previous one's data in the
    shared array), with shared and per-head selection, give exactly the index sets and
    counts of hsa_select, and leave the array's error word clear."""
    cases = [
        (W.make_workload(W.with_context(W.CONFIGS["llama3-8b-128k"], 50001), seed=3,
                         device="cuda"), 0),
        (W.make_workload(W.CONFIGS["paged-b8-32k-128k"], seed=4, device="cuda"), 0),
        (W.make_workload(W.with_context(W.CONFIGS["llama3-8b-128k"], 30000), seed=5,
                         device="cuda"), 1),
    ]
    assert hsa.hsa_read_device_error(None) == 0
    for wl, per_head in cases:
        d, _ = H.dims_pair(wl, per_head=per_head)
        dwl, kq, k_scale = _inputs(wl, d)
        ref = _outputs(d)
        hsa.hsa_select(d, dwl["q"], kq, k_scale, dwl["page_table"], dwl["seq_lens"], *ref,
                       hsa.workspace(d, hsa.HSA_OP_SELECT))
        got = _outputs(d)
        hsa.hsa_select_noalloc(d, dwl["q"], kq, k_scale, dwl["page_table"], dwl["seq_lens"],
                               *got)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert int(got[3].min()) > 0
        assert hsa.hsa_read_device_error(None) == 0


def test_noalloc_select_rejects_shapes_beyond_its_scratch():
    wl = W.make_workload(W.with_context(W.CONFIGS["llama3-8b-128k"], 4096), seed=5,
                         device="cuda")
    d, _ = H.dims_pair(wl)
    dwl, kq, k_scale = _inputs(wl, d)
    # 4 x 8 x 60000 blocks need 7.7 MB of block maxima: more than the 4 MiB array
    big = hsa.Dims(**{**d.__dict__, "batch": 4, "max_pages_per_seq": 60000, "num_pages": 60000})
    with pytest.raises(hsa.HsaError) as e:
        hsa.hsa_select_noalloc(big, dwl["q"], kq, k_scale, dwl["page_table"], dwl["seq_lens"],
                               *_outputs(big))
    assert e.value.code == hsa.HSA_ERR_WORKSPACE_TOO_SMALL
