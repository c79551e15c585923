import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def pin_lib():
    """The independent rounding formulation (tests/pins/rounding_pin.c), compiled."""
    import ctypes
    src = os.path.join(ROOT, "tests", "pins", "rounding_pin.c")
    out_dir = os.path.join(ROOT, "tests", "pins", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "rounding_pin.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        tmp = so + ".tmp%d" % os.getpid()
        base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fvisibility=hidden", src,
                "-o", tmp]
        try:
            subprocess.run(base + ["-fopenmp"], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True)
        os.replace(tmp, so)
    lib = ctypes.CDLL(so)
    for nm in ("pin_sweep_e2m1", "pin_sweep_e4m3"):
        f = getattr(lib, nm)
        f.restype = ctypes.c_int64
        f.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                      ctypes.POINTER(ctypes.c_uint32)]
    for nm in ("pin_e2m1_from_bits", "pin_e4m3_from_bits"):
        f = getattr(lib, nm)
        f.restype = ctypes.c_uint32
        f.argtypes = [ctypes.c_uint32]
    return lib


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_ok():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
