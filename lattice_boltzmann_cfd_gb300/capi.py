"""ctypes binding of the C ABI in include/lbm.h (argument marshalling only).

Every function here has the name of the C entry point it wraps and does nothing but
convert arguments (torch tensors or raw addresses) and raise on a non-OK status; all
device work happens in liblbm_gb300.so.  There is no fallback: if the library is missing
and cannot be built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

LBM_OK, LBM_ERR_ARG, LBM_ERR_UNSUPPORTED, LBM_ERR_WORKSPACE = 0, 1, 2, 3
LBM_ERR_CUDA, LBM_ERR_NONFINITE, LBM_ERR_STATE = 4, 5, 6
STATUS_NAMES = {0: "LBM_OK", 1: "LBM_ERR_ARG", 2: "LBM_ERR_UNSUPPORTED",
                3: "LBM_ERR_WORKSPACE", 4: "LBM_ERR_CUDA", 5: "LBM_ERR_NONFINITE",
                6: "LBM_ERR_STATE"}
LBM_D2Q9, LBM_D3Q19, LBM_D3Q27 = 9, 19, 27
LBM_THERMAL_NONE, LBM_D2Q5, LBM_D3Q7 = 0, 5, 7
LBM_BGK, LBM_MRT, LBM_CM = 0, 1, 2
LBM_FACE_PERIODIC, LBM_FACE_WALL, LBM_FACE_HALO = 0, 1, 2
LBM_HALO_FILL, LBM_HALO_DRAIN = 0, 1
LBM_TFACE_ADIABATIC, LBM_TFACE_DIRICHLET = 0, 1
LBM_STREAM_AA, LBM_STREAM_PULL, LBM_STREAM_SPLIT = 0, 1, 2
STREAMING = {"aa": LBM_STREAM_AA, "pull": LBM_STREAM_PULL, "split": LBM_STREAM_SPLIT}


class LbmError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class lbm_config(ctypes.Structure):
    _fields_ = [
        ("nx", ctypes.c_int), ("ny", ctypes.c_int), ("nz", ctypes.c_int),
        ("lattice", ctypes.c_int), ("thermal", ctypes.c_int), ("collision", ctypes.c_int),
        ("tau", ctypes.c_double), ("s", ctypes.c_double * 19), ("s_T", ctypes.c_double * 7),
        ("cm_rates", ctypes.c_double * 5),
        ("a_T", ctypes.c_double), ("g_body", ctypes.c_double * 3),
        ("gbeta", ctypes.c_double), ("T0", ctypes.c_double), ("up_axis", ctypes.c_int),
        ("face_flow", ctypes.c_int * 6), ("face_T", ctypes.c_int * 6),
        ("T_wall", ctypes.c_double * 6), ("solid_mask", ctypes.POINTER(ctypes.c_uint8)),
        ("streaming", ctypes.c_int), ("ib_max_samples", ctypes.c_int),
        ("ib_block", ctypes.c_int),
    ]


class lbm_diag(ctypes.Structure):
    _fields_ = [
        ("mass", ctypes.c_double), ("momentum", ctypes.c_double * 3),
        ("force", ctypes.c_double * 3), ("heat", ctypes.c_double * 6),
        ("nu_hot", ctypes.c_double), ("nu_cold", ctypes.c_double),
        ("fluid_cells", ctypes.c_longlong), ("steps", ctypes.c_longlong),
        ("finite", ctypes.c_int), ("ib_samples", ctypes.c_int),
        ("ib_force", ctypes.c_double * 3), ("ib_torque", ctypes.c_double * 3),
        ("uT", ctypes.c_double * 3), ("nu_volume", ctypes.c_double),
        ("ib_dropped", ctypes.c_int),
    ]


# (name, restype, argtypes) of every exported entry point, in header order.
_VP, _D = ctypes.c_void_p, ctypes.POINTER(ctypes.c_double)
SIGNATURES = [
    ("lbm_workspace_bytes", ctypes.c_int, [ctypes.POINTER(lbm_config),
                                           ctypes.POINTER(ctypes.c_size_t)]),
    ("lbm_create", ctypes.c_int, [ctypes.POINTER(lbm_config), _VP, ctypes.c_size_t, _VP,
                                  ctypes.POINTER(_VP)]),
    ("lbm_init_equilibrium", ctypes.c_int, [_VP, _VP, _VP, _VP]),
    ("lbm_step", ctypes.c_int, [_VP, ctypes.c_int]),
    ("lbm_step_planes", ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int]),
    ("lbm_step_box", ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    ("lbm_macroscopic", ctypes.c_int, [_VP, _VP, _VP, _VP]),
    ("lbm_solid_force", ctypes.c_int, [_VP, _D]),
    ("lbm_diagnostics", ctypes.c_int, [_VP, ctypes.POINTER(lbm_diag)]),
    ("lbm_get_populations", ctypes.c_int, [_VP, _VP, _VP]),
    ("lbm_set_populations", ctypes.c_int, [_VP, _VP, _VP]),
    ("lbm_get_link_mask", ctypes.c_int, [_VP, _VP]),
    ("lbm_set_ib_samples", ctypes.c_int, [_VP, ctypes.c_int, _VP, _VP, _VP]),
    ("lbm_set_ib_samples_device", ctypes.c_int, [_VP, ctypes.c_int, _VP, _VP, _VP,
                                                  ctypes.c_int]),
    ("lbm_halo_bytes", ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_size_t)]),
    ("lbm_halo_pack", ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, _VP]),
    ("lbm_halo_unpack", ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, _VP]),
    ("lbm_halo_axis_bytes", ctypes.c_int, [_VP, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]),
    ("lbm_halo_axis_pack", ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, ctypes.c_int, _VP]),
    ("lbm_halo_axis_unpack", ctypes.c_int, [_VP, ctypes.c_int, ctypes.c_int, ctypes.c_int, _VP]),
    ("lbm_halo_axis_swap", ctypes.c_int, [_VP, _VP, ctypes.c_int, ctypes.c_int]),
    ("lbm_halo_axis_swap_many", ctypes.c_int,
     [ctypes.POINTER(_VP), ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    ("lbm_set_stream", ctypes.c_int, [_VP, _VP]),
    ("lbm_reduce_populations_static", ctypes.c_int,
     [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _VP, _VP, _VP,
      _VP]),
    ("lbm_parity", ctypes.c_int, [_VP]),
    ("lbm_steps_taken", ctypes.c_longlong, [_VP]),
    ("lbm_last_error", ctypes.c_char_p, [_VP]),
    ("lbm_version", ctypes.c_char_p, []),
    ("lbm_destroy", None, [_VP]),
]

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load():
    """Load liblbm_gb300.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing")
            lib = ctypes.CDLL(path)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status, ctx=None):
    if status != LBM_OK:
        msg = load().lbm_last_error(ctx)
        raise LbmError(status, msg.decode() if msg else "")
    return status


def _addr(x):
    """Address of a tensor's storage (float32/uint32, contiguous) or a raw int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if isinstance(x, torch.Tensor):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        if x.dtype not in (torch.float32, torch.float64, torch.int32, torch.uint8):
            raise ValueError(f"unsupported dtype {x.dtype}")
        return x.data_ptr()
    raise TypeError(f"expected a tensor, an int address or None, got {type(x)}")


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------- entry points ---------

def lbm_workspace_bytes(cfg: lbm_config) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lbm_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def lbm_create(cfg: lbm_config, workspace, workspace_bytes: int, stream=None):
    ctx = _VP()
    _check(load().lbm_create(ctypes.byref(cfg), _addr(workspace), workspace_bytes,
                             _stream_handle(stream), ctypes.byref(ctx)))
    return ctx


def lbm_init_equilibrium(ctx, rho, u, T=None):
    _check(load().lbm_init_equilibrium(ctx, _addr(rho), _addr(u), _addr(T)), ctx)


def lbm_step(ctx, n: int):
    _check(load().lbm_step(ctx, int(n)), ctx)


def lbm_step_planes(ctx, lo: int, hi: int):
    _check(load().lbm_step_planes(ctx, int(lo), int(hi)), ctx)


def lbm_step_box(ctx, lo, hi):
    """The current step on the cells [lo, hi) (3 ints each: x, y, z)."""
    a = (ctypes.c_int * 3)(*[int(v) for v in lo])
    b = (ctypes.c_int * 3)(*[int(v) for v in hi])
    _check(load().lbm_step_box(ctx, a, b), ctx)


def lbm_macroscopic(ctx, rho=None, u=None, T=None):
    _check(load().lbm_macroscopic(ctx, _addr(rho), _addr(u), _addr(T)), ctx)


def lbm_solid_force(ctx):
    F = (ctypes.c_double * 3)()
    _check(load().lbm_solid_force(ctx, F), ctx)
    return [F[0], F[1], F[2]]


def lbm_diagnostics(ctx, allow_nonfinite: bool = False) -> dict:
    d = lbm_diag()
    st = load().lbm_diagnostics(ctx, ctypes.byref(d))
    if not (allow_nonfinite and st == LBM_ERR_NONFINITE):
        _check(st, ctx)
    return {"mass": d.mass, "momentum": list(d.momentum), "force": list(d.force),
            "heat": list(d.heat), "nu_hot": d.nu_hot, "nu_cold": d.nu_cold,
            "fluid_cells": d.fluid_cells, "steps": d.steps, "finite": bool(d.finite),
            "ib_samples": d.ib_samples, "ib_force": list(d.ib_force),
            "ib_torque": list(d.ib_torque), "uT": list(d.uT), "nu_volume": d.nu_volume,
            "ib_dropped": d.ib_dropped, "status": st}


def lbm_get_populations(ctx, f, g=None):
    _check(load().lbm_get_populations(ctx, _addr(f), _addr(g)), ctx)


def lbm_set_populations(ctx, f, g=None):
    _check(load().lbm_set_populations(ctx, _addr(f), _addr(g)), ctx)


def lbm_get_link_mask(ctx, mask):
    _check(load().lbm_get_link_mask(ctx, _addr(mask)), ctx)


def lbm_set_ib_samples(ctx, xyz, ub=None, weight=None):
    """Immersed-boundary samples from host arrays: xyz (n, 3), ub (n, 3), weight (n,)."""
    import numpy as np
    x = np.ascontiguousarray(xyz, dtype=np.float32).reshape(-1, 3)
    n = x.shape[0]
    u = None if ub is None else np.ascontiguousarray(ub, dtype=np.float32).reshape(n, 3)
    w = None if weight is None else np.ascontiguousarray(weight, dtype=np.float32).reshape(n)
    ptr = lambda a: None if a is None else a.ctypes.data
    _check(load().lbm_set_ib_samples(ctx, n, ptr(x), ptr(u), ptr(w)), ctx)


def lbm_set_ib_samples_device(ctx, n: int, xyz, ub=None, weight=None, reorder=True):
    """Immersed-boundary samples from device (or page-locked host) tensors: xyz (n, 3)
    float32, ub (n, 3) or None, weight (n,) or None; sorted on the device (reorder) or
    placed in the stored order of the last sort."""
    _check(load().lbm_set_ib_samples_device(ctx, int(n), _addr(xyz), _addr(ub),
                                            _addr(weight), int(bool(reorder))), ctx)


def lbm_halo_bytes(ctx) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lbm_halo_bytes(ctx, ctypes.byref(n)), ctx)
    return n.value


def lbm_halo_pack(ctx, side: int, phase: int, buf):
    _check(load().lbm_halo_pack(ctx, int(side), int(phase), _addr(buf)), ctx)


def lbm_halo_unpack(ctx, side: int, phase: int, buf):
    _check(load().lbm_halo_unpack(ctx, int(side), int(phase), _addr(buf)), ctx)


def lbm_halo_axis_bytes(ctx, axis: int) -> int:
    n = ctypes.c_size_t()
    _check(load().lbm_halo_axis_bytes(ctx, int(axis), ctypes.byref(n)), ctx)
    return n.value


def lbm_halo_axis_pack(ctx, axis: int, side: int, phase: int, buf):
    _check(load().lbm_halo_axis_pack(ctx, int(axis), int(side), int(phase), _addr(buf)), ctx)


def lbm_halo_axis_unpack(ctx, axis: int, side: int, phase: int, buf):
    _check(load().lbm_halo_axis_unpack(ctx, int(axis), int(side), int(phase), _addr(buf)), ctx)


def lbm_halo_axis_swap(lo, hi, axis: int, phase: int):
    _check(load().lbm_halo_axis_swap(lo, hi, int(axis), int(phase)), lo)


def lbm_halo_axis_swap_many(lo, hi, axis: int, phase: int):
    """Face swaps of pairs (lo[p], hi[p]) of one axis in one launch."""
    n = len(lo)
    a = (_VP * n)(*lo)
    b = (_VP * n)(*hi)
    _check(load().lbm_halo_axis_swap_many(a, b, n, int(axis), int(phase)),
           lo[0] if 1 <= n <= 32 else None)


def lbm_set_stream(ctx, stream):
    _check(load().lbm_set_stream(ctx, _stream_handle(stream)), ctx)


def lbm_reduce_populations_static(lattice, thermal, nx, ny, nz, f, g, out, stream=None):
    """Allocation-free sums (mass, momentum, thermal energy, non-finite cells) of
    caller-held populations into ``out`` (6 doubles, device or page-locked host)."""
    _check(load().lbm_reduce_populations_static(int(lattice), int(thermal), int(nx), int(ny),
                                                int(nz), _addr(f), _addr(g), _addr(out),
                                                _stream_handle(stream)))


def lbm_parity(ctx) -> int:
    return load().lbm_parity(ctx)


def lbm_steps_taken(ctx) -> int:
    return load().lbm_steps_taken(ctx)


def lbm_last_error(ctx=None) -> str:
    m = load().lbm_last_error(ctx)
    return m.decode() if m else ""


def lbm_version() -> str:
    return load().lbm_version().decode()


def lbm_destroy(ctx):
    load().lbm_destroy(ctx)
