import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def bf16_bits(x) -> np.ndarray:
    """Raw bf16 bit patterns of values that bf16 represents exactly (asserted)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, f), "value not exactly representable in bf16"
    return bits


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def read_golden(name: str):
    """Parse a golden fixture: '#' lines are comments; a line with one word starts a
    matrix section; 'key value...' lines are scalars or vectors."""
    path = os.path.join(GOLDEN, name)
    data, section = {}, None
    with open(path, encoding="utf-8") as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if len(parts) == 1 and not _is_number(parts[0]):
                section = parts[0]
                data[section] = []
                continue
            if _is_number(parts[0]) and section is not None:
                data[section].append([float(p) for p in parts])
                continue
            section = None
            if parts[0] == "case":
                data.setdefault("cases", []).append(dict(p.split("=") for p in parts[1:]))
            else:
                vals = [float(p) if _is_number(p) else p for p in parts[1:]]
                data[parts[0]] = vals[0] if len(vals) == 1 else vals
    return data


def _is_number(s: str) -> bool:
    try:
        float(s)
        return True
    except ValueError:
        return False


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    return oracle
