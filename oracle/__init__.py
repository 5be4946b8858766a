"""fp64 CPU oracle of the lattice-Boltzmann collide-and-stream step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The product path (the CUDA library and its
binding) never does, and this package imports nothing from it.

The arithmetic lives in ``lbm_oracle.c`` (plain C, fp64, two buffers, pull streaming,
literal moment-matrix products).  This wrapper only marshals numpy arrays and maps a
workload description (physical parameters) onto the oracle's own problem struct; the one
piece of method arithmetic here is the relation between transport coefficients and
relaxation rates:

* momentum: nu = (1/s_nu - 1/2) / 3, i.e. s_nu = 1 / (3 nu + 1/2) and tau = 3 nu + 1/2
  (BGK), with the lattice sound speed c_s^2 = 1/3;
* thermal: kappa = c_sT^2 (1/s_kappa - 1/2) with c_sT^2 = omega, the anti-bounce-back
  weight the multi-GPU thermal LBM page prints ((4 + a_T)/10 on D2Q5, (6 + a_T)/21 on D3Q7).

Array shapes: populations (Q, wz, wy, wx) float64; rho, T (wz, wy, wx); u (dim, wz, wy, wx).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lbm_oracle.c")
_LIB = os.path.join(_HERE, "liblbm_oracle.so")
_lock = threading.Lock()
_lib = None

PERIODIC, WALL = 0, 1
ADIABATIC, DIRICHLET = 0, 1
BGK, MRT, CM = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile liblbm_oracle.so next to its source (gcc, OpenMP, -O3)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "lbm_oracle.h")))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-fopenmp", "-std=c11", "-shared", "-fPIC",
                               "-o", tmp, _SRC, "-lm"], cwd=_HERE)
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("lattice", ctypes.c_int), ("thermal", ctypes.c_int), ("collision", ctypes.c_int),
        ("tau", ctypes.c_double), ("s", ctypes.c_double * 19), ("s_T", ctypes.c_double * 7),
        ("cm_rates", ctypes.c_double * 5),
        ("a_T", ctypes.c_double), ("g_body", ctypes.c_double * 3), ("gbeta", ctypes.c_double),
        ("T0", ctypes.c_double), ("up_axis", ctypes.c_int), ("face_flow", ctypes.c_int * 6),
        ("face_T", ctypes.c_int * 6), ("T_wall", ctypes.c_double * 6),
        ("nx", ctypes.c_int), ("ny", ctypes.c_int), ("nz", ctypes.c_int),
        ("x0", ctypes.c_int), ("y0", ctypes.c_int), ("z0", ctypes.c_int),
        ("wx", ctypes.c_int), ("wy", ctypes.c_int), ("wz", ctypes.c_int),
        ("solid", ctypes.POINTER(ctypes.c_ubyte)),
        ("ib_n", ctypes.c_int), ("ib_x", ctypes.POINTER(ctypes.c_double)),
        ("ib_ub", ctypes.POINTER(ctypes.c_double)), ("ib_w", ctypes.POINTER(ctypes.c_double)),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            D = ctypes.POINTER(ctypes.c_double)
            lib.oracle_check.argtypes = [P]
            lib.oracle_init_equilibrium.argtypes = [P, D, D, D, D, D]
            lib.oracle_step.argtypes = [P, D, D, D, D, D, D]
            lib.oracle_run.argtypes = [P, D, D, ctypes.c_int, D, D]
            lib.oracle_ib_forces.argtypes = [P, D, D, D, D]
            lib.oracle_macroscopic.argtypes = [P, D, D, D, D, D]
            lib.oracle_diagnostics.argtypes = [P, D, D, D]
            lib.oracle_lattice.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                           ctypes.POINTER(ctypes.c_int), D, D]
            lib.oracle_max_threads.argtypes = []
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            for fn in ("oracle_check", "oracle_init_equilibrium", "oracle_step", "oracle_run",
                       "oracle_macroscopic", "oracle_diagnostics", "oracle_lattice",
                       "oracle_max_threads", "oracle_ib_forces", "oracle_set_threads"):
                getattr(lib, fn).restype = ctypes.c_int
            _lib = lib
    return _lib


def _dptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# Moment-row groups of each basis: which rows a named rate applies to.
_ROWS = {
    19: {"e": [1], "eps": [2], "q": [4, 6, 8], "nu": [9, 11, 13, 14, 15], "pi": [10, 12],
         "m": [16, 17, 18]},
    9: {"e": [1], "eps": [2], "q": [4, 6], "nu": [7, 8]},
    7: {"kappa": [1, 2, 3], "e": [4], "v": [5, 6]},
    5: {"kappa": [1, 2], "e": [3], "v": [4]},
}

# D3Q27 central-moment rates by name: trace of the second-order moments, then one per order
# (the shear rate comes from nu).
CM_RATE_NAMES = ("bulk", "r3", "r4", "r5", "r6")


class Problem:
    """The oracle's view of a workload, optionally restricted to a window of the domain.

    ``spec`` is a workload description (``lattice_boltzmann_cfd_gb300.workloads.Workload``
    or any object with the same attributes).  ``window`` = ((x0, y0, z0), (wx, wy, wz)).
    """

    def __init__(self, spec, window=None):
        nx, ny, nz = spec.shape
        if window is None:
            window = ((0, 0, 0), (nx, ny, nz))
        (x0, y0, z0), (wx, wy, wz) = window
        p = _Problem()
        p.lattice = spec.lattice
        p.thermal = spec.thermal
        p.collision = {"bgk": BGK, "mrt": MRT, "cm": CM}[spec.collision]
        p.tau = 3.0 * spec.nu + 0.5
        s = [0.0] * 19
        rates = dict(spec.rates)
        rates["nu"] = 1.0 / (3.0 * spec.nu + 0.5)
        if spec.lattice == 27:
            p.cm_rates = (ctypes.c_double * 5)(*[rates[n] for n in CM_RATE_NAMES])
        else:
            for name, rows in _ROWS[spec.lattice].items():
                for k in rows:
                    s[k] = rates[name]
        p.s = (ctypes.c_double * 19)(*s)
        sT = [0.0] * 7
        if spec.thermal:
            omega = (4.0 + spec.a_T) / 10.0 if spec.thermal == 5 else (6.0 + spec.a_T) / 21.0
            trates = dict(spec.thermal_rates)
            trates["kappa"] = 1.0 / (spec.kappa / omega + 0.5)
            for name, rows in _ROWS[spec.thermal].items():
                for k in rows:
                    sT[k] = trates[name]
        p.s_T = (ctypes.c_double * 7)(*sT)
        p.a_T = spec.a_T
        p.g_body = (ctypes.c_double * 3)(*spec.g_body)
        p.gbeta = spec.gbeta
        p.T0 = spec.T0
        p.up_axis = spec.up_axis
        p.face_flow = (ctypes.c_int * 6)(*[{"periodic": PERIODIC, "wall": WALL}[k]
                                           for k in spec.face_flow])
        p.face_T = (ctypes.c_int * 6)(*[{"adiabatic": ADIABATIC, "dirichlet": DIRICHLET}[k]
                                        for k in spec.face_T])
        p.T_wall = (ctypes.c_double * 6)(*spec.T_wall)
        p.nx, p.ny, p.nz = nx, ny, nz
        p.x0, p.y0, p.z0 = x0, y0, z0
        p.wx, p.wy, p.wz = wx, wy, wz
        self._solid = None
        if spec.solid is not None:
            sol = np.ascontiguousarray(
                spec.solid[z0:z0 + wz, y0:y0 + wy, x0:x0 + wx], dtype=np.uint8)
            self._solid = sol
            p.solid = sol.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))
        self._ib = []
        ib_x = getattr(spec, "ib_x", None)
        if ib_x is not None and len(ib_x):
            x = np.ascontiguousarray(ib_x, dtype=np.float64).reshape(-1, 3)
            n = x.shape[0]
            ub = getattr(spec, "ib_ub", None)
            ub = (np.zeros((n, 3)) if ub is None else
                  np.ascontiguousarray(ub, dtype=np.float64).reshape(n, 3))
            wt = getattr(spec, "ib_w", None)
            wt = np.ones(n) if wt is None else np.ascontiguousarray(wt, dtype=np.float64)
            self._ib = [x, ub, wt]
            p.ib_n = n
            p.ib_x, p.ib_ub, p.ib_w = (_dptr(a) for a in self._ib)
        self.last_ib = np.zeros(6)
        self.p = p
        self.Q = spec.lattice
        self.QT = spec.thermal
        self.dim = 2 if spec.lattice == 9 else 3
        self.wshape = (wz, wy, wx)
        self.window = window
        _check(_load().oracle_check(ctypes.byref(p)), "check")

    @property
    def solid(self):
        return self._solid

    def zeros_f(self):
        return np.zeros((self.Q,) + self.wshape)

    def zeros_g(self):
        return np.zeros((max(self.QT, 1),) + self.wshape)


def _window_of(prob: Problem, a, lead=()):
    """The window's part of a field given on the whole domain (or already windowed)."""
    a = np.asarray(a)
    if a.size == int(np.prod(lead + prob.wshape)):
        return np.ascontiguousarray(a, dtype=np.float64).reshape(lead + prob.wshape)
    (x0, y0, z0), (wx, wy, wz) = prob.window
    a = a.reshape(lead + (prob.p.nz, prob.p.ny, prob.p.nx))
    sub = a[(Ellipsis, slice(z0, z0 + wz), slice(y0, y0 + wy), slice(x0, x0 + wx))]
    return np.ascontiguousarray(sub, dtype=np.float64)


def init_equilibrium(prob: Problem, rho, u, T=None):
    """f = f_eq(rho, u), g = g_eq(T, u) from (fp32 or fp64) fields, widened to fp64.
    Fields may cover the window or the whole domain (then the window's part is used)."""
    rho = _window_of(prob, rho)
    u = _window_of(prob, u, (prob.dim,))
    Td = None if T is None else _window_of(prob, T)
    f, g = prob.zeros_f(), prob.zeros_g()
    _check(_load().oracle_init_equilibrium(ctypes.byref(prob.p), _dptr(rho), _dptr(u),
                                           _dptr(Td), _dptr(f), _dptr(g)), "init")
    return f, g


def run(prob: Problem, f, g, steps: int):
    """Advance (f, g) in place by ``steps`` steps; returns the last step's solid force
    (the immersed boundary's reaction force and torque go to ``prob.last_ib``)."""
    force = np.zeros(3)
    ib = np.zeros(6)
    _check(_load().oracle_run(ctypes.byref(prob.p), _dptr(f), _dptr(g), int(steps),
                              _dptr(force), _dptr(ib)), "run")
    prob.last_ib = ib
    return force


def ib_forces(prob: Problem, f, g):
    """(per-cell immersed-boundary force (3, wz, wy, wx), ib[6]) of the state (f, g)."""
    F = np.zeros((3,) + prob.wshape)
    ib = np.zeros(6)
    _check(_load().oracle_ib_forces(ctypes.byref(prob.p), _dptr(f), _dptr(g), _dptr(F),
                                    _dptr(ib)), "ib_forces")
    return F, ib


def macroscopic(prob: Problem, f, g):
    rho = np.zeros(prob.wshape)
    u = np.zeros((prob.dim,) + prob.wshape)
    T = np.zeros(prob.wshape)
    _check(_load().oracle_macroscopic(ctypes.byref(prob.p), _dptr(f), _dptr(g), _dptr(rho),
                                      _dptr(u), _dptr(T)), "macroscopic")
    return rho, u, (T if prob.QT else None)


def diagnostics(prob: Problem, f, g):
    out = np.zeros(13)
    _check(_load().oracle_diagnostics(ctypes.byref(prob.p), _dptr(f), _dptr(g), _dptr(out)),
           "diagnostics")
    return {"mass": out[0], "momentum": out[1:4].copy(), "heat": out[4:10].copy(),
            "uT": out[10:13].copy()}


def lattice(kind: int):
    """(c[Q,3], w[Q] or None, M[Q,Q]) as the oracle builds them for kind 27, 19, 9, 7 or 5
    (M is zero for 27, whose central-moment matrix depends on u)."""
    Q = ctypes.c_int(0)
    c = (ctypes.c_int * 81)()
    w = np.zeros(27)
    M = np.zeros(27 * 27)
    _check(_load().oracle_lattice(kind, ctypes.byref(Q), c, _dptr(w), _dptr(M)), "lattice")
    q = Q.value
    cc = np.array(c[:3 * q], dtype=np.int64).reshape(q, 3)
    return cc, (w[:q].copy() if kind in (9, 19, 27) else None), M[:q * q].reshape(q, q).copy()


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> int:
    """Threads of the following oracle calls; returns the previous count."""
    return int(_load().oracle_set_threads(int(n)))
