import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: longer CPU test")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def capi():
    """The product binding with its CUDA library loaded (built in-tree if needed)."""
    from lattice_boltzmann_cfd_gb300 import capi as c
    c.load()
    return c


@pytest.fixture(scope="session")
def emu_lib():
    """Host build of tests/aa_emulation.cu: the library's per-cell functions run on the
    CPU with a NaN-filled write buffer per step."""
    import ctypes
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = os.path.join(ROOT, "tests", "aa_emulation.cu")
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libaa_emulation.so")
    deps = [src] + [os.path.join(ROOT, "lattice_boltzmann_cfd_gb300", "csrc", n)
                    for n in os.listdir(os.path.join(ROOT, "lattice_boltzmann_cfd_gb300", "csrc"))]
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(d) for d in deps):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc, "-std=c++17", "-O2", "-Xcompiler", "-fPIC", "-shared",
                               "-I", os.path.join(ROOT, "include"),
                               "-I", os.path.join(ROOT, "lattice_boltzmann_cfd_gb300", "csrc"),
                               "-o", tmp, src])
        os.replace(tmp, lib)
    return ctypes.CDLL(lib)
