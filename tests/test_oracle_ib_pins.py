"""Pins of the oracle's immersed boundary ("GPU Optimization for High-Quality Kinetic Fluid
Simulation", Sec. 3.1, Eq. 6-8) against closed forms and conservation (CPU)."""
import dataclasses
import itertools

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W


def _box(shape=(12, 10, 8), lattice=19, **kw):
    if lattice == 27:
        rates, coll = {"bulk": 1.2, "r3": 1.2, "r4": 1.2, "r5": 1.2, "r6": 1.2}, "cm"
    elif lattice == 19:
        rates, coll = {"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}, "mrt"
    else:
        rates, coll = {"e": 1.2, "eps": 1.2, "q": 1.2}, "mrt"
    w = W.Workload(name="ib", lattice=lattice, thermal=0, collision=coll, shape=shape, nu=0.1,
                   rates=rates, up_axis=1 if lattice == 9 else 2, **kw)
    dim = w.dim
    if w.rho0 is None:
        w.rho0 = np.ones(w.grid, np.float32)
    if w.u0 is None:
        w.u0 = np.zeros((dim,) + w.grid, np.float32)
    return w


def _samples(rng, n, lo, hi, dim):
    x = rng.uniform(lo, hi, size=(n, 3)).astype(np.float32)
    if dim == 2:
        x[:, 2] = 0.0
    return x


@pytest.mark.parametrize("lattice", [19, 9, 27])
def test_linear_field_interpolation_and_momentum_balance(oracle_mod, lattice):
    """With rho = 1 and a velocity field linear in x, y, z the trilinear kernel interpolates
    exactly, so the penalty of each sample is w (u_b - u(x_s)) in closed form; the spread
    conserves it (the kernel weights sum to 1), so the fluid momentum grows by exactly
    sum_s w (u_b - u(x_s)) in one step, and the reported reaction is minus that."""
    rng = np.random.default_rng(3)
    shape = (12, 10, 1) if lattice == 9 else (12, 10, 8)
    w = _box(shape, lattice)
    dim = w.dim
    nz, ny, nx = w.grid
    z, y, x = np.meshgrid(np.arange(nz), np.arange(ny), np.arange(nx), indexing="ij")
    a = np.array([0.01, -0.02, 0.015])[:dim]
    B = np.array([[1e-3, -2e-3, 5e-4], [3e-4, 1e-3, -1e-3], [-6e-4, 2e-4, 8e-4]])[:dim, :dim]
    coords = [x, y, z][:dim]
    u = np.stack([a[i] + sum(B[i, k] * coords[k] for k in range(dim)) for i in range(dim)])
    w.u0 = u.astype(np.float32)
    n = 9
    lo, hi = 2.0, min(shape[:dim]) - 3.0
    xs = _samples(rng, n, lo, hi, dim)
    ub = rng.uniform(-0.02, 0.02, size=(n, 3)).astype(np.float32)
    wt = rng.uniform(0.5, 1.5, size=n).astype(np.float32)
    if dim == 2:
        ub[:, 2] = 0.0
    w = dataclasses.replace(w, ib_x=xs, ib_ub=ub, ib_w=wt)
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    # analytic velocity at the samples (the fp32-rounded field is still linear to 1e-9)
    xs64 = xs.astype(np.float64)
    u_at = np.stack([a[i] + xs64[:, :dim] @ B[i] for i in range(dim)], axis=1)
    expect = np.zeros(3)
    expect[:dim] = (wt[:, None] * (ub[:, :dim].astype(np.float64) - u_at)).sum(axis=0)
    d0 = oracle_mod.diagnostics(p, f, g)
    oracle_mod.run(p, f, g, 1)
    d1 = oracle_mod.diagnostics(p, f, g)
    assert np.allclose(d1["momentum"] - d0["momentum"], expect, rtol=1e-6, atol=1e-9)
    assert np.allclose(p.last_ib[:3], -expect, rtol=1e-6, atol=1e-9)


def test_scatter_equals_gather(oracle_mod):
    """The per-cell force the oracle scatters from each sample (Eq. 8 as 'scattering') equals
    a brute-force gather over all samples for each cell (the 'gathering' form of the same
    sum): for every cell, sum_s K(x_s, x_f) g_s."""
    rng = np.random.default_rng(5)
    w = dataclasses.replace(W.perturbed(_box((10, 9, 8)), seed=2), ib_x=None)
    n = 40
    xs = _samples(rng, n, 1.0, 7.0, 3)
    ub = rng.uniform(-0.01, 0.01, size=(n, 3)).astype(np.float32)
    w = dataclasses.replace(w, ib_x=xs, ib_ub=ub, ib_w=np.ones(n, np.float32))
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    F, ib = oracle_mod.ib_forces(p, f, g)
    rho, u, _ = oracle_mod.macroscopic(p, f, g)
    nz, ny, nx = w.grid
    # penalty of each sample from the interpolated fields
    gs = np.zeros((n, 3))
    stencils = []
    for s in range(n):
        base = np.floor(xs[s].astype(np.float64)).astype(int)
        fr = xs[s].astype(np.float64) - base
        st = []
        r_s, u_s = 0.0, np.zeros(3)
        for d in itertools.product((0, 1), repeat=3):
            K = np.prod([fr[k] if d[k] else 1 - fr[k] for k in range(3)])
            i, j, k = (base + np.array(d)) % np.array([nx, ny, nz])
            st.append((K, (k, j, i)))
            r_s += K * rho[k, j, i]
            u_s += K * u[:, k, j, i]
        gs[s] = r_s * (ub[s] - u_s)
        stencils.append(st)
    gather = np.zeros_like(F)
    for k in range(nz):
        for j in range(ny):
            for i in range(nx):
                for s in range(n):
                    for K, node in stencils[s]:
                        if node == (k, j, i):
                            gather[:, k, j, i] += K * gs[s]
    assert np.allclose(F, gather, rtol=1e-12, atol=1e-15)
    assert np.allclose(ib[:3], -gs.sum(axis=0), rtol=1e-12, atol=1e-15)


def test_matched_boundary_velocity_is_a_fixed_point(oracle_mod):
    """A uniform flow with every sample's boundary velocity equal to it feels no force and
    stays unchanged."""
    rng = np.random.default_rng(8)
    w = _box((10, 8, 6))
    u0 = np.array([0.03, -0.01, 0.02], np.float32)
    w.u0 = np.broadcast_to(u0[:, None, None, None], (3,) + w.grid).astype(np.float32).copy()
    xs = _samples(rng, 25, 1.0, 5.0, 3)
    w = dataclasses.replace(w, ib_x=xs, ib_ub=np.broadcast_to(u0, xs.shape).copy())
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    f0 = f.copy()
    oracle_mod.run(p, f, g, 4)
    assert np.allclose(f, f0, rtol=0, atol=1e-15)
    assert np.all(np.abs(p.last_ib) < 1e-14)


def test_steady_force_balance_with_body_force(oracle_mod):
    """Periodic box, body acceleration g, an immersed sphere at rest: at steady state the
    momentum balance gives a reaction force on the sphere equal to the total body force."""
    shape = (16, 12, 12)
    w = dataclasses.replace(W.channel_ib_sphere(shape=shape, center=(7.3, 5.6, 6.2), radius=3.0,
                                                gx=2e-5, nu=0.1),
                            face_flow=("periodic",) * 6)
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    oracle_mod.run(p, f, g, 3000)
    d = oracle_mod.diagnostics(p, f, g)
    total_body = d["mass"] * w.g_body[0]
    assert abs(p.last_ib[0] / total_body - 1) < 1e-3
    assert abs(p.last_ib[1]) < 1e-3 * total_body and abs(p.last_ib[2]) < 1e-3 * total_body


@pytest.mark.parametrize("lattice", [19, 9, 27])
def test_samples_moving_with_a_uniform_flow_exert_no_force(oracle_mod, lattice):
    """A uniform flow u0 on a periodic box is a fixed point.  Samples that move with it
    (displaced by u0 every step, boundary velocity u0) see u(x_s) = u0 wherever they sit
    between the cells, since the kernel weights sum to 1, so their penalty
    w rho (u_b - u) vanishes: every step's reaction force is zero and the state stays
    uniform, while the samples sweep through new stencils."""
    rng = np.random.default_rng(11)
    shape = (10, 8, 1) if lattice == 9 else (10, 8, 6)
    w = _box(shape, lattice)
    dim = w.dim
    u0 = np.array([0.03, -0.02, 0.01], np.float32)
    w.u0 = np.broadcast_to(u0[:dim].reshape((dim,) + (1,) * 3), (dim,) + w.grid).astype(np.float32)
    xs0 = _samples(rng, 7, 1.0, min(shape[:dim]) - 2.0, dim).astype(np.float64)
    v = np.zeros(3)
    v[:dim] = u0[:dim]
    ub = np.tile(v.astype(np.float32), (len(xs0), 1))
    ext = np.array(shape, np.float64)
    f, g = oracle_mod.init_equilibrium(oracle_mod.Problem(w), w.rho0, w.u0)
    for k in range(6):
        xk = xs0 + k * v
        xk[:, :dim] = np.mod(xk[:, :dim], ext[:dim])
        p = oracle_mod.Problem(dataclasses.replace(w, ib_x=xk.astype(np.float32), ib_ub=ub))
        oracle_mod.run(p, f, g, 1)
        assert np.abs(p.last_ib[:3]).max() < 1e-13, k
    rho, u, _ = oracle_mod.macroscopic(p, f, g)
    assert np.abs(rho - 1.0).max() < 1e-13
    for a in range(dim):
        assert np.abs(u[a] - float(u0[a])).max() < 1e-13
