"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every entry point
include/hsa.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "hsa.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc is needed to build libhsa.so")


@pytest.fixture(scope="module")
def lib():
    from kv_cache_int8_gb300 import build, hsa
    build.build()
    return hsa


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_binding_exports():
    from kv_cache_int8_gb300 import hsa
    assert declared_functions() == sorted(hsa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    path = lib.LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"not exported: {missing}"
    handle = ctypes.CDLL(path)
    for n in declared_functions():
        assert getattr(handle, n) is not None


def _dims(lib, **kw):
    base = dict(batch=1, hq=32, hkv=8, max_pages_per_seq=8192, num_pages=8192, chunk=64, k1=256,
                k2=128, sink=128, window=1024)
    base.update(kw)
    return lib.Dims(**base)


def test_status_strings(lib):
    assert lib.hsa_status_string(0) == "ok"
    assert "workspace" in lib.hsa_status_string(lib.HSA_ERR_WORKSPACE_TOO_SMALL)
    assert lib.hsa_status_string(999) == "unknown status"


def test_workspace_sizes(lib):
    d = _dims(lib)
    for op in range(5):
        assert lib.hsa_workspace_bytes(d, op) > 0
    assert lib.hsa_workspace_bytes(d, 9) == 0
    # block maxima of every (b, h, page) plus the error word
    assert lib.hsa_workspace_bytes(d, lib.HSA_OP_SELECT) >= 8 * 8192 * 4 + 256
    assert lib.hsa_workspace_bytes(_dims(lib, head_dim=64), 0) == 0
    assert lib.hsa_workspace_bytes(_dims(lib, hq=12, hkv=8), 0) == 0
    # groups of 1, 2, 4 and 8 query heads per kv head; 4-bit and 8-bit key codes
    for hq in (8, 16, 32, 64):
        assert lib.hsa_workspace_bytes(_dims(lib, hq=hq, hkv=8), 0) > 0
    assert lib.hsa_workspace_bytes(_dims(lib, hq=48, hkv=8), 0) == 0
    for bits in (0, 4, 8):
        assert lib.hsa_workspace_bytes(_dims(lib, key_bits=bits), 0) > 0
    assert lib.hsa_workspace_bytes(_dims(lib, key_bits=2), 0) == 0
    # per-head selection: one selection row per query head (4x the block maxima here)
    sel = lib.hsa_workspace_bytes(_dims(lib), lib.HSA_OP_SELECT)
    sel_ph = lib.hsa_workspace_bytes(_dims(lib, per_head=1), lib.HSA_OP_SELECT)
    assert sel_ph >= 4 * (sel - 256)
    assert lib.hsa_workspace_bytes(_dims(lib, per_head=2), 0) == 0
    # FP8 keys: 8-bit layout only
    assert lib.hsa_workspace_bytes(_dims(lib, key_fp8=1), 0) > 0
    assert lib.hsa_workspace_bytes(_dims(lib, key_fp8=1, key_bits=4), 0) == 0
    assert lib.hsa_workspace_bytes(_dims(lib, key_fp8=2), 0) == 0
    # the block cache plan works per kv head: no cache with per-head selection
    host = dict(kv_on_host=True, k2=16, sink=64, window=256)
    assert lib.load().hsa_block_cache_bytes(_dims(lib, **host).c(), 4096) > 0
    assert lib.load().hsa_block_cache_bytes(_dims(lib, per_head=1, **host).c(), 4096) == 0
    # cache policies: 0 least recently used, 1 least cumulative attention mass; the buffer
    # holds the masses under both, and the cached workspace grows by the per-segment sums
    lru, mass = _dims(lib, **host), _dims(lib, cache_policy=1, **host)
    cache = lib.load().hsa_block_cache_bytes(lru.c(), 4096)
    assert lib.load().hsa_block_cache_bytes(mass.c(), 4096) == cache
    assert cache >= 4096 * 8192 + 2 * 8 * 8192 * 4  # data + slot_of + masses (8192 pages)
    assert (lib.hsa_workspace_bytes(mass, lib.HSA_OP_CACHED) >
            lib.hsa_workspace_bytes(lru, lib.HSA_OP_CACHED))
    assert lib.hsa_workspace_bytes(_dims(lib, cache_policy=2, **host), lib.HSA_OP_CACHED) == 0
    assert lib.load().hsa_block_cache_mass(mass.c(), None, 4096) is None  # null buffer
    base = 1 << 20
    off = lib.load().hsa_block_cache_mass(mass.c(), base, 4096) - base
    assert 0 < off and off % 16 == 0 and off + 8 * 8192 * 4 <= cache


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), 2), (dict(page_size=32), 2), (dict(block=32), 2), (dict(hq=24), 2),
    (dict(hq=128), 2), (dict(key_bits=6), 2),
    (dict(hq=30), 1), (dict(batch=0), 1), (dict(k1=-1), 1), (dict(window=-3), 1),
    (dict(chunk=40), 1), (dict(chunk=0), 1), (dict(batch=2000), 2),
])
def test_select_rejects_bad_descriptors(lib, kw, code):
    d = _dims(lib, **kw)
    fake = 1 << 20  # never dereferenced: validation fails first
    with pytest.raises(lib.HsaError) as e:
        lib.hsa_select(d, fake, fake, fake, fake, fake, None, None, fake, fake,
                       _FakeWs(fake, 1 << 40), stream=0)
    assert e.value.code == code


class _FakeWs:
    def __init__(self, ptr, n):
        self.ptr, self.n = ptr, n

    def data_ptr(self):
        return self.ptr

    def numel(self):
        return self.n


def test_null_and_misaligned_pointers(lib):
    d = _dims(lib)
    ok = 1 << 20
    with pytest.raises(lib.HsaError) as e:
        lib.hsa_select(d, None, ok, ok, ok, ok, None, None, ok, ok, _FakeWs(ok, 1 << 40), stream=0)
    assert e.value.code == lib.HSA_ERR_INVALID_ARG
    with pytest.raises(lib.HsaError) as e:
        lib.hsa_select(d, ok + 4, ok, ok, ok, ok, None, None, ok, ok, _FakeWs(ok, 1 << 40),
                       stream=0)
    assert e.value.code == lib.HSA_ERR_INVALID_ARG
    with pytest.raises(lib.HsaError) as e:
        lib.hsa_attend(d, ok, ok + 8, ok, ok, ok, ok, ok, ok, None, _FakeWs(ok, 1 << 40), stream=0)
    assert e.value.code == lib.HSA_ERR_INVALID_ARG
    with pytest.raises(lib.HsaError) as e:  # workspace not 256-byte aligned
        lib.hsa_attend(d, ok, ok, ok, ok, ok, ok, ok, ok, None, _FakeWs(ok + 16, 1 << 40),
                       stream=0)
    assert e.value.code == lib.HSA_ERR_INVALID_ARG


def test_workspace_too_small(lib):
    d = _dims(lib)
    ok = 1 << 20
    need = lib.hsa_workspace_bytes(d, lib.HSA_OP_SELECT)
    with pytest.raises(lib.HsaError) as e:
        lib.hsa_select(d, ok, ok, ok, ok, ok, None, None, ok, ok, _FakeWs(ok, need - 1), stream=0)
    assert e.value.code == lib.HSA_ERR_WORKSPACE_TOO_SMALL
    need = lib.hsa_workspace_bytes(d, lib.HSA_OP_DENSE)
    with pytest.raises(lib.HsaError) as e:
        lib.dense_decode(d, ok, ok, ok, ok, ok, ok, None, _FakeWs(ok, need - 1), stream=0)
    assert e.value.code == lib.HSA_ERR_WORKSPACE_TOO_SMALL


def test_prune_rejects_too_many_chunks(lib):
    d = _dims(lib, max_pages_per_seq=60000 * 4, num_pages=60000 * 4)
    ok = 1 << 20
    with pytest.raises(lib.HsaError) as e:
        lib.hsa_prune(d, ok, ok, None, None, None, ok, ok, stream=0)
    assert e.value.code == lib.HSA_ERR_UNSUPPORTED


def _header_struct_fields(name):
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef struct %s \{(.*?)\} %s;" % (name, name), text, flags=re.S).group(1)
    fields = re.finditer(r"(?:const\s+)?(int32_t|float|void)\s*(\*?)\s*(\w+);", body)
    return [("ptr" if m.group(2) else m.group(1), m.group(3)) for m in fields]


@pytest.mark.parametrize("struct", ["hsa_dims", "hsa_step_io"])
def test_binding_structs_match_the_header(struct):
    """The ctypes structures of the binding declare the header's fields, in order, with
    the same C types (a field added on one side only would shift every later one)."""
    from kv_cache_int8_gb300 import hsa
    ctype = {"int32_t": ctypes.c_int32, "float": ctypes.c_float, "ptr": ctypes.c_void_p}
    want = _header_struct_fields(struct)
    got = getattr(hsa, struct)._fields_
    assert [n for n, _ in got] == [n for _, n in want]
    for (gn, gt), (wt, wn) in zip(got, want):
        assert gt is ctype[wt], gn
