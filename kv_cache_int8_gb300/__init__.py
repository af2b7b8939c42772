"""kv_cache_int8_gb300 — one decode step of hierarchically pruned, block-sparse attention
over an int8-keyed paged KV cache, as hand-written CUDA for GB300 (sm_103a).

The compute path lives in the C-ABI library ``libhsa.so`` (``include/hsa.h``);
``kv_cache_int8_gb300.hsa`` is its thin ctypes binding. ``workloads`` draws the seeded
synthetic inputs. Importing the package does not load the CUDA library; the first call
into ``hsa`` does, and fails loudly if it is missing.
"""
__all__ = ["hsa", "workloads"]
