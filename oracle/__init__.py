"""CPU oracle for one decode step of hierarchically pruned, block-sparse attention over
an int8-keyed paged KV cache.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package. It shares no code with the CUDA library.
Every function is pinned by the tests in ``tests/test_oracle_*.py`` (worked examples,
brute force, closed forms and special cases); none is "parity unpinned".
"""
from .cache import CacheState, cache_plan, call_segments  # noqa: F401
from .oracle import (  # noqa: F401
    Dims,
    attend,
    block_mass,
    dense,
    fp8_block_scores,
    num_threads,
    quantize_append,
    quantize_keys,
    query_codes,
    recall,
    select,
    selection_within_bounds,
    set_num_threads,
)
