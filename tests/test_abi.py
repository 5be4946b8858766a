"""The C-ABI library: it loads, exports every entry point include/lbm.h declares, and
rejects bad configurations on the host before touching the GPU.  CPU only."""
import ctypes
import dataclasses
import os
import re

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W
from lattice_boltzmann_cfd_gb300.solver import make_config

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "lbm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lbm_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(capi):
    lib = ctypes.CDLL(capi.library_path())
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/lbm.h but not exported"
    assert {s[0] for s in capi.SIGNATURES} == set(names)


def test_version_string(capi):
    assert "sm_103a" in capi.lbm_version()


def test_null_context_calls_fail_cleanly(capi):
    lib = capi.load()
    assert lib.lbm_step(None, 1) == capi.LBM_ERR_ARG
    assert lib.lbm_init_equilibrium(None, None, None, None) == capi.LBM_ERR_ARG
    assert lib.lbm_macroscopic(None, None, None, None) == capi.LBM_ERR_ARG
    assert lib.lbm_parity(None) == -1
    assert lib.lbm_steps_taken(None) == -1
    assert "ctx is NULL" in capi.lbm_last_error(None)
    lib.lbm_destroy(None)


def _bytes(capi, w, **overrides):
    cfg, keep = make_config(w)
    for k, v in overrides.items():
        if isinstance(v, (list, tuple)):
            arr = getattr(cfg, k)
            for i, x in enumerate(v):
                arr[i] = x
        else:
            setattr(cfg, k, v)
    return capi.lbm_workspace_bytes(cfg)


def test_workspace_size_matches_layout(capi):
    w = W.cavity3d(shape=(40, 30, 20))
    n = 40 * 30 * 20
    S = (n + 63) // 64 * 64
    need = _bytes(capi, w)
    # 19 + 7 population planes and the link mask at least
    assert need >= (19 + 7) * S * 4 + S * 4
    assert need % 256 == 0
    # fully periodic, no solid: no mask
    p = W.random_periodic(shape=(40, 30, 20))
    assert _bytes(capi, p) < 19 * S * 4 + S * 4 + (1 << 20)


@pytest.mark.parametrize("field,value,status", [
    ("nx", 0, 1), ("nz", 3, 1),                      # 2-D lattice needs nz == 1
    ("tau", 0.5, 1), ("collision", 7, 1), ("lattice", 15, 1),
    ("thermal", 7, 2),                               # D2Q9 with D3Q7
    ("up_axis", 2, 1),                               # 2-D: z is not an axis
])
def test_bad_2d_configs_rejected(capi, field, value, status):
    w = W.cavity2d(shape=(16, 12, 1))
    w = dataclasses.replace(w, collision="bgk")
    with pytest.raises(capi.LbmError) as e:
        _bytes(capi, w, **{field: value})
    assert e.value.status == status


@pytest.mark.parametrize("overrides,status,text", [
    ({"s": [0, 2.0]}, 1, "rates"),                  # s_e = 2 is out of [0, 2)
    ({"s_T": [0, -0.1]}, 1, "thermal rates"),
    ({"a_T": 1.0}, 1, "a_T"),
    ({"face_flow": [1, 0]}, 2, "same flow kind"),   # wall on -x, periodic on +x
    ({"face_T": [5]}, 1, "face_T"),
    ({"g_body": [float("nan")]}, 1, "finite"),
])
def test_bad_3d_configs_rejected(capi, overrides, status, text):
    w = W.cavity3d(shape=(16, 12, 10))
    with pytest.raises(capi.LbmError) as e:
        _bytes(capi, w, **overrides)
    assert e.value.status == status
    assert text in str(e.value)


@pytest.mark.parametrize("lattice,faces,extra,text", [
    (19, [0, 0, 0, 0, 0, 2], {}, "same flow kind"),           # periodic paired with HALO
    (19, [0, 2, 0, 0, 0, 0], {}, "same flow kind"),           # the same on x
    (19, [0, 0, 0, 0, 2, 2], {"streaming": 1}, "AA layout"),  # PULL layout
    (19, [2, 2, 0, 0, 0, 0], {"streaming": 2}, "AA layout"),
    (19, [0, 0, 0, 0, 2, 2], {"ib_max_samples": 4}, "immersed"),
    (19, [0, 0, 0, 0, 2, 2], {"nz": 2}, "owned plane"),      # ghosts only
    (19, [2, 2, 0, 0, 0, 0], {"nx": 2}, "owned plane"),
    (19, [1, 2, 2, 2, 0, 0], {"ny": 2}, "owned plane"),
    (9, [1, 1, 2, 1, 0, 0], {"ny": 1}, "owned plane"),
    (9, [2, 2, 1, 1, 0, 0], {"nx": 2}, "owned plane"),
])
def test_halo_faces_validated(capi, lattice, faces, extra, text):
    """HALO faces (on any axis): never paired with a wrap, AA layout only, no immersed
    samples, and at least one owned plane besides the ghosts."""
    w = (W.random_periodic(shape=(8, 6, 5)) if lattice == 19
         else W.random_periodic(shape=(8, 6, 1), lattice=9))
    with pytest.raises(capi.LbmError, match=text):
        _bytes(capi, w, face_flow=faces, **extra)


def test_halo_faces_accepted(capi):
    w = W.random_periodic(shape=(8, 6, 5))
    assert _bytes(capi, w, face_flow=[0, 0, 0, 0, 2, 2]) > 0
    assert _bytes(capi, w, face_flow=[1, 1, 0, 0, 1, 2], nz=2) > 0
    w2 = W.cavity2d(shape=(8, 6, 1))
    assert _bytes(capi, w2, face_flow=[1, 1, 2, 1, 0, 0]) > 0
    # the z faces of a 2-D problem are not read, whatever they hold
    assert _bytes(capi, w2, face_flow=[1, 1, 1, 1, 2, 2]) > 0
    # blocks: HALO faces on several axes, mixed with walls
    assert _bytes(capi, w, face_flow=[2, 2, 2, 1, 2, 2]) > 0
    assert _bytes(capi, w, face_flow=[1, 2, 0, 0, 2, 1], nx=2) > 0
    assert _bytes(capi, w2, face_flow=[2, 2, 2, 2, 0, 0]) > 0


def test_buoyancy_needs_thermal(capi):
    w = dataclasses.replace(W.random_periodic(shape=(8, 8, 8)), gbeta=1e-3)
    with pytest.raises(capi.LbmError, match="buoyancy"):
        _bytes(capi, w)


def test_too_many_cells_rejected(capi):
    w = W.random_periodic(shape=(8, 8, 8))
    with pytest.raises(capi.LbmError, match="2\\^31"):
        _bytes(capi, w, nx=2048, ny=1024, nz=1024)


def test_create_rejects_bad_workspace_before_cuda(capi):
    w = W.random_periodic(shape=(8, 8, 8))
    cfg, _ = make_config(w)
    n = capi.lbm_workspace_bytes(cfg)
    with pytest.raises(capi.LbmError) as e:
        capi.lbm_create(cfg, None, n, 0)
    assert e.value.status == capi.LBM_ERR_WORKSPACE
    with pytest.raises(capi.LbmError) as e:
        capi.lbm_create(cfg, 256 * 1000 + 16, n, 0)     # misaligned
    assert e.value.status == capi.LBM_ERR_WORKSPACE
    with pytest.raises(capi.LbmError) as e:
        capi.lbm_create(cfg, 256 * 1000, n - 256, 0)    # too small
    assert e.value.status == capi.LBM_ERR_WORKSPACE


def test_binding_rejects_noncontiguous_tensor(capi):
    torch = pytest.importorskip("torch")
    t = torch.zeros(4, 4)[:, ::2]
    with pytest.raises(ValueError):
        capi._addr(t)


def test_product_package_does_not_import_oracle():
    """The product path never touches the oracle."""
    root = os.path.join(os.path.dirname(os.path.dirname(__file__)), "lattice_boltzmann_cfd_gb300")
    for dirpath, _, files in os.walk(root):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "lbm_oracle" not in src, fn


@pytest.mark.parametrize("overrides,status,text", [
    ({"collision": 1}, 2, "D3Q27 goes with LBM_CM"),        # D3Q27 with MRT
    ({"cm_rates": [2.0]}, 1, "central-moment rates"),
    ({"cm_rates": [1.0, 0.0]}, 1, "central-moment rates"),
    ({"tau": 0.5}, 1, "tau"),
    ({"thermal": 7}, 2, "thermal"),
    ({"streaming": 1}, 2, "AA layout"),
])
def test_d3q27_configs_validated(capi, overrides, status, text):
    """D3Q27 takes the central-moment collision only, rates in (0, 2), no thermal lattice
    and the AA layout only (immersed-boundary samples are accepted)."""
    w = W.random_periodic(shape=(8, 6, 5), lattice=27)
    assert _bytes(capi, w) > 0
    assert _bytes(capi, w, ib_max_samples=8) > _bytes(capi, w)
    with pytest.raises(capi.LbmError) as e:
        _bytes(capi, w, **overrides)
    assert e.value.status == status
    assert text in str(e.value)


def test_central_moments_only_on_d3q27(capi):
    with pytest.raises(capi.LbmError, match="LBM_CM with D3Q27 only"):
        _bytes(capi, W.random_periodic(shape=(8, 6, 5)), collision=2)


def test_d3q27_workspace_holds_27_planes(capi):
    w = W.random_periodic(shape=(40, 30, 20), lattice=27)
    S = (40 * 30 * 20 + 63) // 64 * 64
    assert _bytes(capi, w) >= 27 * S * 4
    # slab halos of D3Q27 move the 9 populations with c_z = +-1
    assert _bytes(capi, w, face_flow=[0, 0, 0, 0, 2, 2]) > 0


def test_launch_grid_limits(capi):
    """The launch grid's y extent (ny over the rows per block) and z extent (nz) stay within
    65535: rows of 64 cells take one y row per block, rows of 32 or fewer two."""
    w = W.random_periodic(shape=(8, 8, 8))
    assert _bytes(capi, w, nx=64, ny=65535, nz=1) > 0
    with pytest.raises(capi.LbmError, match="ny too large"):
        _bytes(capi, w, nx=64, ny=65536, nz=1)
    assert _bytes(capi, w, nx=32, ny=131070, nz=1) > 0
    with pytest.raises(capi.LbmError, match="ny too large"):
        _bytes(capi, w, nx=32, ny=131071, nz=1)
    with pytest.raises(capi.LbmError, match="nz must be"):
        _bytes(capi, w, nx=4, ny=4, nz=65536)
