import importlib.util
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def _build_library():
    # Load the build script by path: importing the package itself requires the
    # library to exist already.
    path = os.path.join(ROOT, "quantized_weight_block_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_ndq_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


_build_library()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name: str) -> list[list[str]]:
    """Rows of whitespace-separated fields; '#' starts a comment."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


# ---- bitwise comparison of decoded outputs --------------------------------
_INT_VIEW = {"float32": np.uint32, "float64": np.uint64, "float16": np.uint16, "bfloat16": np.uint16}


def nan_mask(bits: np.ndarray, out_dtype: str) -> np.ndarray:
    if out_dtype == "float32":
        return (bits & 0x7F800000 == 0x7F800000) & (bits & 0x007FFFFF != 0)
    if out_dtype == "float64":
        return (bits & 0x7FF0000000000000 == 0x7FF0000000000000) & (bits & 0x000FFFFFFFFFFFFF != 0)
    if out_dtype == "float16":
        return (bits & 0x7C00 == 0x7C00) & (bits & 0x03FF != 0)
    return (bits & 0x7F80 == 0x7F80) & (bits & 0x007F != 0)


def as_bits(a: np.ndarray, out_dtype: str) -> np.ndarray:
    return np.ascontiguousarray(a).reshape(-1).view(_INT_VIEW[out_dtype])


def assert_bit_exact(got: np.ndarray, want: np.ndarray, out_dtype: str, what: str = ""):
    """0-ULP parity: identical bits everywhere except that NaN only needs to be NaN."""
    g, w = as_bits(got, out_dtype), as_bits(want, out_dtype)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    if np.array_equal(g, w):  # identical bits (the usual case; cheap on large outputs)
        return
    gn, wn = nan_mask(g, out_dtype), nan_mask(w, out_dtype)
    bad = (gn != wn) | (~wn & (g != w))
    if bad.any():
        idx = np.flatnonzero(bad)
        raise AssertionError(f"{what}: {idx.size} mismatches, first at {idx[:8].tolist()}: "
                             f"got {g[idx[:8]].tolist()} want {w[idx[:8]].tolist()}")
