import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def read_golden(name):
    """Rows of a golden fixture, comments stripped, split on whitespace."""
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
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def bruteforce():
    """The brute-force encoder checker, compiled from tests/pins/bruteforce.c."""
    import ctypes
    import subprocess
    src = os.path.join(ROOT, "tests", "pins", "bruteforce.c")
    out_dir = os.path.join(ROOT, "tests", "pins", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libbruteforce.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", so + ".tmp",
                        src, "-lm"], check=True)
        os.replace(so + ".tmp", so)
    L = ctypes.CDLL(so)
    L.bf_e2m1.restype = ctypes.c_uint8
    L.bf_e2m1.argtypes = [ctypes.c_float]
    L.bf_e4m3.restype = ctypes.c_uint8
    L.bf_e4m3.argtypes = [ctypes.c_float]
    L.bf_compare.restype = ctypes.c_int64
    L.bf_compare.argtypes = [ctypes.c_int, ctypes.c_uint32, ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint8),
                             ctypes.POINTER(ctypes.c_uint32)]
    return L
