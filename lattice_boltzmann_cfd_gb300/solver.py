"""Problem set-up and a small handle class over the C ABI.

``make_config`` turns a problem description (grid, lattice, transport coefficients,
forcing, faces, solid mask) into the library's ``lbm_config``: relaxation rates follow
from the transport coefficients as nu = (1/s_nu - 1/2)/3 (c_s^2 = 1/3; BGK tau = 3 nu + 1/2)
and kappa = omega (1/s_kappa - 1/2), omega being the anti-bounce-back weight of the
thermal lattice ((4 + a_T)/10 on D2Q5, (6 + a_T)/21 on D3Q7), which is also its c_sT^2.

``Simulation`` owns the device workspace (a torch tensor) and the library context; each
method is one C-ABI call.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import capi

# Moment rows each named rate applies to (row order of include/lbm.h).
RATE_ROWS = {
    19: {"e": [1], "eps": [2], "q": [4, 6, 8], "nu": [9, 11, 13, 14, 15], "pi": [10, 12],
         "m": [16, 17, 18]},
    9: {"e": [1], "eps": [2], "q": [4, 6], "nu": [7, 8]},
    7: {"kappa": [1, 2, 3], "e": [4], "v": [5, 6]},
    5: {"kappa": [1, 2], "e": [3], "v": [4]},
}
# D3Q27 central moments: rates by name, in lbm_config.cm_rates order (the shear rate is
# 1/tau).
CM_RATES = ("bulk", "r3", "r4", "r5", "r6")
_FLOW = {"periodic": capi.LBM_FACE_PERIODIC, "wall": capi.LBM_FACE_WALL,
         "halo": capi.LBM_FACE_HALO}
_TFACE = {"adiabatic": capi.LBM_TFACE_ADIABATIC, "dirichlet": capi.LBM_TFACE_DIRICHLET}


def anti_bounce_back_weight(thermal: int, a_T: float) -> float:
    return (4.0 + a_T) / 10.0 if thermal == 5 else (6.0 + a_T) / 21.0


def make_config(w, streaming: str = "aa"):
    """lbm_config for a problem description; returns (cfg, keep-alive objects).
    ``streaming``: "aa" (in place), "pull" or "split" (two buffers)."""
    cfg = capi.lbm_config()
    cfg.streaming = capi.STREAMING[streaming]
    cfg.nx, cfg.ny, cfg.nz = (int(v) for v in w.shape)
    cfg.lattice = int(w.lattice)
    cfg.thermal = int(w.thermal)
    cfg.collision = {"bgk": capi.LBM_BGK, "mrt": capi.LBM_MRT, "cm": capi.LBM_CM}[w.collision]
    cfg.tau = 3.0 * w.nu + 0.5
    rates = dict(w.rates)
    rates["nu"] = 1.0 / cfg.tau
    s = [0.0] * 19
    if cfg.lattice == capi.LBM_D3Q27:
        cfg.cm_rates = (ctypes.c_double * 5)(*[float(rates[n]) for n in CM_RATES])
    else:
        for name, rows in RATE_ROWS[cfg.lattice].items():
            for k in rows:
                s[k] = float(rates[name])
    cfg.s = (ctypes.c_double * 19)(*s)
    sT = [0.0] * 7
    if cfg.thermal:
        omega = anti_bounce_back_weight(cfg.thermal, w.a_T)
        trates = dict(w.thermal_rates)
        trates["kappa"] = 1.0 / (w.kappa / omega + 0.5)
        for name, rows in RATE_ROWS[cfg.thermal].items():
            for k in rows:
                sT[k] = float(trates[name])
    cfg.s_T = (ctypes.c_double * 7)(*sT)
    cfg.a_T = float(w.a_T)
    cfg.g_body = (ctypes.c_double * 3)(*[float(v) for v in w.g_body])
    cfg.gbeta = float(w.gbeta)
    cfg.T0 = float(w.T0)
    cfg.up_axis = int(w.up_axis)
    cfg.face_flow = (ctypes.c_int * 6)(*[_FLOW[k] for k in w.face_flow])
    cfg.face_T = (ctypes.c_int * 6)(*[_TFACE[k] for k in w.face_T])
    cfg.T_wall = (ctypes.c_double * 6)(*[float(v) for v in w.T_wall])
    ib_x = getattr(w, "ib_x", None)
    cfg.ib_max_samples = 0 if ib_x is None else int(len(ib_x))
    keep = []
    if w.solid is not None:
        solid = np.ascontiguousarray(w.solid, dtype=np.uint8)
        keep.append(solid)
        cfg.solid_mask = solid.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))
    return cfg, keep


class Simulation:
    """A lattice-Boltzmann state on one GPU: workspace + context (one C-ABI call per
    method).  Fields are torch tensors shaped (nz, ny, nx), velocity (dim, nz, ny, nx),
    populations (Q, nz, ny, nx); they may live on the device or in page-locked host
    memory."""

    def __init__(self, w, device=None, stream=None, edit=None, streaming: str = "aa"):
        """``edit``, if given, is called with the ``lbm_config`` before it is used (to set
        raw fields such as individual rates).  ``streaming``: "aa", "pull" or "split"."""
        import torch
        self.device = torch.device(device if device is not None else "cuda")
        self.cfg, self._keep = make_config(w, streaming)
        if edit is not None:
            edit(self.cfg)
        self.nbytes = capi.lbm_workspace_bytes(self.cfg)
        self.workspace = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
        self.ctx = capi.lbm_create(self.cfg, self.workspace, self.nbytes, stream)
        self.shape = tuple(w.shape)
        self.grid = (self.cfg.nz, self.cfg.ny, self.cfg.nx)
        self.Q, self.QT = self.cfg.lattice, self.cfg.thermal
        self.dim = 2 if self.Q == 9 else 3
        self.cells = self.cfg.nx * self.cfg.ny * self.cfg.nz
        if getattr(w, "ib_x", None) is not None and len(w.ib_x):
            self.set_ib_samples(w.ib_x, w.ib_ub, w.ib_w)

    # -- state ---------------------------------------------------------------------
    def init_equilibrium(self, rho, u, T=None):
        capi.lbm_init_equilibrium(self.ctx, rho, u, T)

    def step(self, n: int = 1):
        capi.lbm_step(self.ctx, n)

    def step_planes(self, lo: int, hi: int):
        """The current step on outer-axis planes [lo, hi) only (see lbm_step_planes)."""
        capi.lbm_step_planes(self.ctx, lo, hi)

    def step_box(self, lo, hi):
        """The current step on the cells [lo, hi) only, (x, y, z) each (see lbm_step_box)."""
        capi.lbm_step_box(self.ctx, lo, hi)

    def macroscopic(self, rho=None, u=None, T=None):
        import torch
        rho = rho if rho is not None else torch.empty(self.grid, device=self.device)
        u = u if u is not None else torch.empty((self.dim,) + self.grid, device=self.device)
        if self.QT and T is None:
            T = torch.empty(self.grid, device=self.device)
        capi.lbm_macroscopic(self.ctx, rho, u, T if self.QT else None)
        return rho, u, (T if self.QT else None)

    def populations(self):
        import torch
        f = torch.empty((self.Q,) + self.grid, device=self.device)
        g = torch.empty((self.QT,) + self.grid, device=self.device) if self.QT else None
        capi.lbm_get_populations(self.ctx, f, g)
        return f, g

    def set_populations(self, f, g=None):
        capi.lbm_set_populations(self.ctx, f, g)

    def link_mask(self):
        import torch
        m = torch.empty(self.grid, dtype=torch.int32, device=self.device)
        capi.lbm_get_link_mask(self.ctx, m)
        return m

    def set_ib_samples(self, xyz, ub=None, weight=None):
        capi.lbm_set_ib_samples(self.ctx, xyz, ub, weight)

    def set_ib_samples_device(self, xyz, ub=None, weight=None, reorder=True):
        """Samples as device tensors (float32, xyz and ub (n, 3), weight (n,)), sorted on
        the device (reorder) or placed in the order of the last sort; nothing waits for the
        stream."""
        capi.lbm_set_ib_samples_device(self.ctx, int(xyz.shape[0]), xyz, ub, weight, reorder)

    def diagnostics(self, allow_nonfinite: bool = False) -> dict:
        return capi.lbm_diagnostics(self.ctx, allow_nonfinite)

    def solid_force(self):
        return capi.lbm_solid_force(self.ctx)

    @property
    def parity(self) -> int:
        return capi.lbm_parity(self.ctx)

    @property
    def steps_taken(self) -> int:
        return capi.lbm_steps_taken(self.ctx)

    def set_stream(self, stream):
        capi.lbm_set_stream(self.ctx, stream)

    def close(self):
        if getattr(self, "ctx", None) is not None:
            capi.lbm_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
