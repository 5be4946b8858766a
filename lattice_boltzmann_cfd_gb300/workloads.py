"""Seeded synthetic workloads for the lattice-Boltzmann step.

This module only describes problems and draws their inputs: grid, lattice, physical
parameters (viscosity, diffusivity, forcing, wall temperatures), boundary kinds, solid
mask and initial macroscopic fields.  It holds none of the method's arithmetic: neither
the CUDA library's binding nor the oracle takes relaxation rates from here; each maps the
physical parameters onto its own rates.  Both sides draw their inputs from here, so that
they see the same fp32 fields.

The five workloads follow the shapes of the pages' test problems:

* ``taylor_green``   -- D3Q19 BGK, periodic 32^3, 3-D Taylor-Green field (u0 = 0.05,
  k = 2 pi / 32), nu = 0.1 (tau = 0.8), rho = 1, 200 steps.
* ``random_periodic`` -- D3Q19 MRT, periodic 128^3 (also 512^3), rho = 1 + N(0, 1e-3),
  each velocity component U(-0.02, 0.02) i.i.d., nu = 0.01, other rates 1.2, 1000 steps.
  Stands in for the streaming-layout page's "periodic 128^3" case.
* ``channel_sphere``  -- D3Q19 MRT, 128^3, periodic in x, no-slip walls in y and z, a
  bounce-back sphere of radius 16 at (40, 64, 64), body acceleration g_x = 1e-6,
  nu = 0.02, rest start, 2000 steps.  Stands in for that page's "sphere 128^3" case.
* ``cavity2d``        -- D2Q9 MRT + D2Q5 MRT, 4096^2 side-heated square cavity
  (Ra = 1e8, Pr = 0.71, U_ff = 0.1), left wall T = +0.5, right wall T = -0.5, top and
  bottom adiabatic, all no-slip, buoyancy along +y, 20000 steps.
* ``cavity3d``        -- D3Q19 MRT + D3Q7 MRT, 512^3 cube (Ra = 1e7, Pr = 0.71,
  U_ff = 0.1), hot x = 0 and cold x = L walls, four adiabatic walls, all no-slip,
  buoyancy along +z, 5000 steps.
  The two cavities stand in for the side-heated cells of the multi-GPU thermal LBM page
  (8193^2 and 385^3 there).

Lattice units for the cavities: H = N cells (half-way walls at -1/2 and N - 1/2),
Delta T = 1, T0 = 0, nu = U_ff H sqrt(Pr / Ra), kappa = nu / Pr, g beta = U_ff^2 / H
(from Ra = g beta dT H^3 / (nu kappa), Pr = nu / kappa and the free-fall velocity
U_ff = sqrt(g beta dT H)).

Array conventions: x fastest; scalar fields have shape (nz, ny, nx); velocity (dim, nz,
ny, nx); the solid mask is uint8 (nz, ny, nx) with 1 = solid.  Fields are float32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np


@dataclasses.dataclass
class Workload:
    name: str
    lattice: int                     # 19 (D3Q19) or 9 (D2Q9)
    thermal: int                     # 0, 7 (D3Q7) or 5 (D2Q5)
    collision: str                   # "bgk" or "mrt"
    shape: tuple                     # (nx, ny, nz)
    nu: float                        # kinematic viscosity (lattice units)
    rates: dict                      # non-hydrodynamic momentum rates by moment group
    kappa: float = 0.0               # thermal diffusivity
    thermal_rates: dict = dataclasses.field(default_factory=dict)
    a_T: float = 0.0
    g_body: tuple = (0.0, 0.0, 0.0)  # body acceleration
    gbeta: float = 0.0               # g * beta_T
    T0: float = 0.0
    up_axis: int = 2
    face_flow: tuple = ("periodic",) * 6   # faces -x, +x, -y, +y, -z, +z
    face_T: tuple = ("adiabatic",) * 6
    T_wall: tuple = (0.0,) * 6
    solid: Optional[np.ndarray] = None
    rho0: Optional[np.ndarray] = None
    u0: Optional[np.ndarray] = None
    T_init: Optional[np.ndarray] = None
    steps: int = 0
    # immersed-boundary samples: positions (n, 3) in cell units (cell centres at integers),
    # boundary velocities (n, 3), weights (n,); all float32
    ib_x: Optional[np.ndarray] = None
    ib_ub: Optional[np.ndarray] = None
    ib_w: Optional[np.ndarray] = None

    @property
    def dim(self) -> int:
        return 2 if self.lattice == 9 else 3

    @property
    def cells(self) -> int:
        nx, ny, nz = self.shape
        return nx * ny * nz

    @property
    def grid(self) -> tuple:
        """(nz, ny, nx): the numpy shape of a scalar field."""
        nx, ny, nz = self.shape
        return (nz, ny, nx)

    def fluid_cells(self) -> int:
        return self.cells - (0 if self.solid is None else int(self.solid.sum()))

    def describe(self) -> str:
        return self.name


_OTHER = 1.2   # rate of every non-hydrodynamic moment in the workloads


def _momentum_rates(lattice):
    if lattice == 27:   # central moments: trace of the second order, then orders 3-6
        return {"bulk": _OTHER, "r3": _OTHER, "r4": _OTHER, "r5": _OTHER, "r6": _OTHER}
    if lattice == 19:
        return {"e": _OTHER, "eps": _OTHER, "q": _OTHER, "pi": _OTHER, "m": _OTHER}
    return {"e": _OTHER, "eps": _OTHER, "q": _OTHER}


def _thermal_rates():
    return {"e": _OTHER, "v": _OTHER}


def _rest(shape, dim):
    nx, ny, nz = shape
    return (np.ones((nz, ny, nx), np.float32), np.zeros((dim, nz, ny, nx), np.float32))


def taylor_green(n: int = 32, u0: float = 0.05, nu: float = 0.1, shape=None) -> Workload:
    nx, ny, nz = shape or (n, n, n)
    k = 2.0 * math.pi / n
    z, y, x = np.meshgrid(np.arange(nz, dtype=np.float64), np.arange(ny, dtype=np.float64),
                          np.arange(nx, dtype=np.float64), indexing="ij")
    u = np.zeros((3, nz, ny, nx))
    u[0] = u0 * np.sin(k * x) * np.cos(k * y) * np.cos(k * z)
    u[1] = -u0 * np.cos(k * x) * np.sin(k * y) * np.cos(k * z)
    return Workload(
        name=f"D3Q19 BGK periodic {nx}x{ny}x{nz} Taylor-Green", lattice=19, thermal=0,
        collision="bgk", shape=(nx, ny, nz), nu=nu, rates=_momentum_rates(19),
        rho0=np.ones((nz, ny, nx), np.float32), u0=u.astype(np.float32), steps=200)


def random_periodic(n: int = 128, seed: int = 2, nu: float = 0.01, shape=None,
                    collision: str = "mrt", lattice: int = 19) -> Workload:
    nx, ny, nz = shape or ((n, n, 1) if lattice == 9 else (n, n, n))
    dim = 2 if lattice == 9 else 3
    if lattice == 27:
        collision = "cm"
    rng = np.random.default_rng(seed)
    rho = (1.0 + rng.normal(0.0, 1e-3, size=(nz, ny, nx))).astype(np.float32)
    u = rng.uniform(-0.02, 0.02, size=(dim, nz, ny, nx)).astype(np.float32)
    name = f"D{dim}Q{lattice} {collision.upper()} periodic {nx}x{ny}x{nz} random"
    return Workload(name=name, lattice=lattice, thermal=0, collision=collision,
                    shape=(nx, ny, nz), nu=nu, rates=_momentum_rates(lattice), rho0=rho,
                    u0=u, up_axis=dim - 1, steps=1000)


def sphere_mask(shape, center, radius) -> np.ndarray:
    """Cells whose integer (0-based) index lies within ``radius`` of ``center``."""
    nx, ny, nz = shape
    z, y, x = np.meshgrid(np.arange(nz), np.arange(ny), np.arange(nx), indexing="ij")
    cx, cy, cz = center
    d2 = (x - cx) ** 2 + (y - cy) ** 2 + (z - cz) ** 2
    return (d2 <= radius * radius).astype(np.uint8)


def channel_sphere(n: int = 128, radius: float = 16, center=(40, 64, 64), gx: float = 1e-6,
                   nu: float = 0.02, shape=None, lattice: int = 19) -> Workload:
    """Body-force-driven channel (walls in y and z, periodic in x) around a solid sphere;
    lattice 19 with MRT or 27 with central moments."""
    shape = shape or (n, n, n)
    rho, u = _rest(shape, 3)
    nx, ny, nz = shape
    coll = "cm" if lattice == 27 else "mrt"
    return Workload(
        name=f"D3Q{lattice} {coll.upper()} channel {nx}x{ny}x{nz} + sphere r={radius:g}",
        lattice=lattice, thermal=0, collision=coll, shape=shape, nu=nu,
        rates=_momentum_rates(lattice),
        g_body=(gx, 0.0, 0.0),
        face_flow=("periodic", "periodic", "wall", "wall", "wall", "wall"),
        solid=sphere_mask(shape, center, radius), rho0=rho, u0=u, steps=2000)


def sphere_samples(center, radius: float, n: int, seed: int = 0) -> np.ndarray:
    """n points spread evenly over a sphere (Fibonacci lattice, randomly rotated by a seeded
    rotation), float32 (n, 3).  A stand-in for Poisson-disk surface sampling."""
    k = np.arange(n) + 0.5
    phi = np.arccos(1.0 - 2.0 * k / n)
    theta = math.pi * (1.0 + 5.0 ** 0.5) * k
    pts = np.stack([np.cos(theta) * np.sin(phi), np.sin(theta) * np.sin(phi), np.cos(phi)], 1)
    q, _ = np.linalg.qr(np.random.default_rng(seed).standard_normal((3, 3)))
    return (np.asarray(center, np.float64) + radius * pts @ q.T).astype(np.float32)


def channel_ib_sphere(n: int = 128, radius: float = 16, center=(40, 64, 64),
                      gx: float = 1e-6, nu: float = 0.02, samples_per_area: float = 4.0,
                      shape=None, lattice: int = 19) -> Workload:
    """Config 3's channel with the sphere represented by immersed-boundary samples instead
    of bounce-back cells: samples_per_area samples per unit area, each weighted by the area
    it represents, at rest."""
    w = channel_sphere(n=n, radius=radius, center=center, gx=gx, nu=nu, shape=shape,
                       lattice=lattice)
    area = 4.0 * math.pi * radius * radius
    ns = max(4, int(round(samples_per_area * area)))
    x = sphere_samples(center, radius, ns)
    return dataclasses.replace(
        w, name=w.name.replace("+ sphere", "+ IB sphere") + f" ({ns} samples)", solid=None,
        ib_x=x, ib_ub=np.zeros_like(x), ib_w=np.full(ns, area / ns, np.float32))


def cavity_parameters(H: float, Ra: float, Pr: float, Uff: float, dT: float = 1.0):
    """(nu, kappa, g*beta) in lattice units for a side-heated cavity of height H."""
    nu = Uff * H * math.sqrt(Pr / Ra)
    kappa = nu / Pr
    gbeta = Uff * Uff / (dT * H)
    return nu, kappa, gbeta


def cavity2d(n: int = 4096, Ra: float = 1e8, Pr: float = 0.71, Uff: float = 0.1,
             shape=None, T_hot: float = 0.5, T_cold: float = -0.5) -> Workload:
    nx, ny, _ = shape or (n, n, 1)
    nu, kappa, gbeta = cavity_parameters(float(nx), Ra, Pr, Uff, T_hot - T_cold)
    rho, u = _rest((nx, ny, 1), 2)
    return Workload(
        name=f"D2Q9 MRT + D2Q5 MRT cavity {nx}x{ny} Ra={Ra:g}", lattice=9, thermal=5,
        collision="mrt", shape=(nx, ny, 1), nu=nu, rates=_momentum_rates(9), kappa=kappa,
        thermal_rates=_thermal_rates(), a_T=0.0, gbeta=gbeta, T0=0.0, up_axis=1,
        face_flow=("wall", "wall", "wall", "wall", "periodic", "periodic"),
        face_T=("dirichlet", "dirichlet", "adiabatic", "adiabatic", "adiabatic", "adiabatic"),
        T_wall=(T_hot, T_cold, 0.0, 0.0, 0.0, 0.0),
        rho0=rho, u0=u, T_init=np.zeros((1, ny, nx), np.float32), steps=20000)


def cavity3d(n: int = 512, Ra: float = 1e7, Pr: float = 0.71, Uff: float = 0.1,
             shape=None, T_hot: float = 0.5, T_cold: float = -0.5) -> Workload:
    nx, ny, nz = shape or (n, n, n)
    nu, kappa, gbeta = cavity_parameters(float(nx), Ra, Pr, Uff, T_hot - T_cold)
    rho, u = _rest((nx, ny, nz), 3)
    return Workload(
        name=f"D3Q19 MRT + D3Q7 MRT cavity {nx}x{ny}x{nz} Ra={Ra:g}", lattice=19, thermal=7,
        collision="mrt", shape=(nx, ny, nz), nu=nu, rates=_momentum_rates(19), kappa=kappa,
        thermal_rates=_thermal_rates(), a_T=0.0, gbeta=gbeta, T0=0.0, up_axis=2,
        face_flow=("wall",) * 6,
        face_T=("dirichlet", "dirichlet", "adiabatic", "adiabatic", "adiabatic", "adiabatic"),
        T_wall=(T_hot, T_cold, 0.0, 0.0, 0.0, 0.0),
        rho0=rho, u0=u, T_init=np.zeros((nz, ny, nx), np.float32), steps=5000)


def perturbed(w: Workload, seed: int = 7, drho: float = 1e-3, du: float = 0.02,
              dT: float = 0.2) -> Workload:
    """The same problem started from a seeded random state (every cell active), for parity
    coverage: rho = 1 + N(0, drho), u ~ U(-du, du), T ~ U(-dT, dT)."""
    rng = np.random.default_rng(seed)
    grid = w.grid
    rho = (1.0 + rng.normal(0.0, drho, size=grid)).astype(np.float32)
    u = rng.uniform(-du, du, size=(w.dim,) + grid).astype(np.float32)
    T = rng.uniform(-dT, dT, size=grid).astype(np.float32) if w.thermal else None
    return dataclasses.replace(w, name=w.name + f" perturbed(seed={seed})", rho0=rho, u0=u,
                               T_init=T)


def by_name(name: str, **kw) -> Workload:
    table = {"taylor_green": taylor_green, "random_periodic": random_periodic,
             "channel_sphere": channel_sphere, "cavity2d": cavity2d, "cavity3d": cavity3d}
    return table[name](**kw)
