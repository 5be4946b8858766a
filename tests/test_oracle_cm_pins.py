"""Pins of the oracle's D3Q27 central-moment MRT ("GPU Optimization for High-Quality Kinetic
Fluid Simulation", Sec. 3.1: the D3Q27 lattice of Fig. 2, Omega = -M^-1 D (m - m_eq) of
Eq. 5 with central moments) against closed forms and the mathematics of the method (CPU).

The reading pinned here: the moments are the central moments prod_a (c_a - u_a)^e_a,
e in {0,1,2}^3, with the second-order normal ones recombined as xx - yy, xx - zz (shear
rate 1/tau) and xx + yy + zz (bulk rate); orders 3 to 6 relax at one fixed rate each; the
equilibrium central moments are those of a Maxwellian, rho prod_a (1, 0, 1/3)[e_a]; the
force source is (F/rho) . d f_eq / du, relaxed with (I - D/2), with u = (j + F/2)/rho."""
import dataclasses
import itertools
import math

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W

MU = (1.0, 0.0, 1.0 / 3.0)      # central moments of order 0, 1, 2 of the 1-D Maxwellian

# the basis as the reading states it (rows 7, 8, 9 are the recombined normal moments)
EXP = [(0, 0, 0), (1, 0, 0), (0, 1, 0), (0, 0, 1), (1, 1, 0), (1, 0, 1), (0, 1, 1),
       None, None, None,
       (1, 2, 0), (1, 0, 2), (2, 1, 0), (0, 1, 2), (2, 0, 1), (0, 2, 1), (1, 1, 1),
       (2, 2, 0), (2, 0, 2), (0, 2, 2), (2, 1, 1), (1, 2, 1), (1, 1, 2),
       (2, 2, 1), (2, 1, 2), (1, 2, 2), (2, 2, 2)]


def _central(f, c, u, e):
    return float(np.sum(f * np.prod((c - u) ** np.array(e), axis=1)))


def _moments(f, c, u):
    """The 27 basis moments of populations f (27,) about u, by definition."""
    out = []
    for k in range(27):
        if k == 7:
            out.append(_central(f, c, u, (2, 0, 0)) - _central(f, c, u, (0, 2, 0)))
        elif k == 8:
            out.append(_central(f, c, u, (2, 0, 0)) - _central(f, c, u, (0, 0, 2)))
        elif k == 9:
            out.append(sum(_central(f, c, u, e) for e in ((2, 0, 0), (0, 2, 0), (0, 0, 2))))
        else:
            out.append(_central(f, c, u, EXP[k]))
    return np.array(out)


def _matrix(c, u):
    return np.stack([_moments(np.eye(27)[i], c, u) for i in range(27)], axis=1)


def _maxwell(rho, e):
    return rho * MU[e[0]] * MU[e[1]] * MU[e[2]]


def _eq_moments(rho):
    out = []
    for k in range(27):
        if k == 7 or k == 8:
            out.append(0.0)
        elif k == 9:
            out.append(rho)
        else:
            out.append(_maxwell(rho, EXP[k]))
    return np.array(out)


def _cube(shape=(1, 1, 1), **kw):
    rates = kw.pop("rates", {"bulk": 1.1, "r3": 1.3, "r4": 1.5, "r5": 1.7, "r6": 0.9})
    w = W.Workload(name="cm", lattice=27, thermal=0, collision="cm", shape=shape,
                   nu=kw.pop("nu", 0.1), rates=rates, **kw)
    nz, ny, nx = w.grid
    if w.rho0 is None:
        w.rho0 = np.ones(w.grid)
    if w.u0 is None:
        w.u0 = np.zeros((3,) + w.grid)
    return w


def _cell(f):
    return np.ascontiguousarray(f.reshape(27, 1, 1, 1), dtype=np.float64)


def test_d3q27_lattice(oracle_mod):
    c, w, _ = oracle_mod.lattice(27)
    c19, _, _ = oracle_mod.lattice(19)
    assert sorted(map(tuple, c)) == sorted(itertools.product((-1, 0, 1), repeat=3))
    assert np.array_equal(c[:19], c19)                # D3Q19's order first
    assert abs(w.sum() - 1) < 1e-15
    for a in range(3):
        for b in range(3):
            assert abs(np.sum(w * c[:, a] * c[:, b]) - (a == b) / 3) < 1e-15
        assert abs(np.sum(w * c[:, a] ** 4) - 1 / 3) < 1e-15
    assert abs(np.sum(w * c[:, 0] ** 2 * c[:, 1] ** 2) - 1 / 9) < 1e-15
    assert abs(np.sum(w * c[:, 0] ** 2 * c[:, 1] ** 2 * c[:, 2] ** 2) - 1 / 27) < 1e-15


def test_equilibrium_has_maxwellian_central_moments(oracle_mod):
    """f_eq(rho, u) of the oracle: every central moment prod (c - u)^e equals
    rho prod (1, 0, 1/3)[e_a], for all 27 exponent triples."""
    c, _, _ = oracle_mod.lattice(27)
    rng = np.random.default_rng(1)
    for _ in range(5):
        rho = rng.uniform(0.8, 1.2)
        u = rng.uniform(-0.2, 0.2, 3)
        w = _cube(rho0=np.full((1, 1, 1), rho), u0=u.reshape(3, 1, 1, 1))
        f, _ = oracle_mod.init_equilibrium(oracle_mod.Problem(w), w.rho0, w.u0)
        f = f.reshape(27)
        for e in itertools.product((0, 1, 2), repeat=3):
            assert abs(_central(f, c, u, e) - _maxwell(rho, e)) < 1e-14, e


def test_uniform_rates_are_bgk_with_the_product_equilibrium(oracle_mod):
    """With every rate equal to omega = 1/tau and no force, the collision is BGK toward the
    product-form equilibrium; one step is that, then pull streaming."""
    c, _, _ = oracle_mod.lattice(27)
    tau = 0.8
    om = 1 / tau
    w = W.perturbed(_cube((5, 4, 3), nu=(tau - 0.5) / 3,
                          rates={k: om for k in ("bulk", "r3", "r4", "r5", "r6")}),
                    seed=2, du=0.05)
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    rng = np.random.default_rng(3)
    f *= 1.0 + 0.01 * rng.standard_normal(f.shape)     # leave equilibrium
    f0 = f.copy()
    oracle_mod.run(p, f, g, 1)
    rho = f0.sum(axis=0)
    u = np.einsum("qa,qzyx->azyx", c.astype(float), f0) / rho

    def phi(ci, ua):
        return np.where(ci == 0, 2 / 3 - ua ** 2, 0.5 * (1 / 3 + ua ** 2 + ci * ua))
    feq = np.stack([rho * phi(c[q, 0], u[0]) * phi(c[q, 1], u[1]) * phi(c[q, 2], u[2])
                    for q in range(27)])
    post = f0 - om * (f0 - feq)
    expect = np.stack([np.roll(post[q], shift=(c[q, 2], c[q, 1], c[q, 0]), axis=(0, 1, 2))
                       for q in range(27)])
    assert np.abs(f - expect).max() < 1e-14


@pytest.mark.parametrize("row", range(4, 27))
def test_each_moment_relaxes_at_its_own_rate(oracle_mod, row):
    """On one periodic cell (streaming is the identity), a state off equilibrium in one basis
    moment only: after a step that moment has relaxed by (1 - s_row), every other moment
    stays at equilibrium, and rho and j are unchanged."""
    c, _, _ = oracle_mod.lattice(27)
    tau = 0.8
    rates = {"bulk": 1.1, "r3": 1.3, "r4": 1.5, "r5": 1.7, "r6": 0.9}
    s = [0.0] * 4 + [1 / tau] * 5 + [rates["bulk"]] + [rates["r3"]] * 7 + \
        [rates["r4"]] * 6 + [rates["r5"]] * 3 + [rates["r6"]]
    rho, u = 1.02, np.array([0.03, -0.02, 0.01])
    w = _cube(nu=(tau - 0.5) / 3, rates=rates, rho0=np.full((1, 1, 1), rho),
              u0=u.reshape(3, 1, 1, 1))
    p = oracle_mod.Problem(w)
    feq, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    M = _matrix(c, u)
    eps = 1e-3
    f = _cell(feq.reshape(27) + np.linalg.solve(M, eps * np.eye(27)[row]))
    oracle_mod.run(p, f, g, 1)
    m = M @ f.reshape(27)
    meq = _eq_moments(rho)
    want = meq.copy()
    want[row] += (1 - s[row]) * eps
    assert np.abs(m - want).max() < 1e-14


def test_force_central_moments(oracle_mod):
    """All rates 1 (tau = 1) and a body force: the collision leaves the central moments about
    u = (j + F/2)/rho at m_eq + R/2, where R, the source's central moments, is
    F_a prod_{b != a} (1, 0, 1/3)[e_b] when e_a = 1 (zero otherwise), and the first-order
    central moments at F/2 (momentum grows by exactly F)."""
    c, _, _ = oracle_mod.lattice(27)
    g_body = np.array([2e-3, -1e-3, 1.5e-3])
    w = _cube(nu=0.5 / 3, rates={k: 1.0 for k in ("bulk", "r3", "r4", "r5", "r6")},
              g_body=tuple(g_body))
    p = oracle_mod.Problem(w)
    rng = np.random.default_rng(4)
    f = _cell(rng.uniform(0.02, 0.08, 27))
    f0 = f.reshape(27).copy()
    rho = f0.sum()
    F = rho * g_body
    u = (c.T.astype(float) @ f0 + F / 2) / rho
    oracle_mod.run(p, f, np.zeros((1, 1, 1, 1)), 1)
    m = _matrix(c, u) @ f.reshape(27)

    def R(e):
        return sum(F[a] * np.prod([MU[e[b]] for b in range(3) if b != a])
                   for a in range(3) if e[a] == 1)
    want = _eq_moments(rho)
    for k in range(27):
        if k in (7, 8, 9):
            continue                       # second-order normal moments: R = 0
        want[k] += R(EXP[k]) / 2
    want[1:4] = F / 2
    assert np.abs(m - want).max() < 1e-15
    assert np.abs(c.T.astype(float) @ f.reshape(27) - (c.T.astype(float) @ f0 + F)).max() < 1e-15


def _shear_wave(oracle_mod, background, n=32, tau=0.65, amp=1e-3, t0=20, t1=220):
    nu = (tau - 0.5) / 3
    k = 2 * math.pi / n
    z = np.arange(n)
    u0 = np.zeros((3, n, 1, 1))
    u0[0, :, 0, 0] = amp * np.sin(k * z)
    u0[1] = background
    w = _cube((1, 1, n), nu=nu, rho0=np.ones((n, 1, 1)), u0=u0)
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    amps = []
    for steps in (t0, t1 - t0):
        oracle_mod.run(p, f, g, steps)
        _, u, _ = oracle_mod.macroscopic(p, f, g)
        amps.append(2 / n * np.sum(u[0, :, 0, 0] * np.sin(k * z)))
    nu_fit = -math.log(amps[1] / amps[0]) / (k * k * (t1 - t0))
    return nu_fit / nu


def test_shear_wave_decays_at_the_viscosity(oracle_mod):
    """A small shear wave u_x = A sin(k z) decays as exp(-nu k^2 t) with nu = (tau - 1/2)/3
    (to the lattice's O(k^2) dispersion, 0.25 % at 32 cells per wavelength), and a uniform
    background flow across it leaves the decay unchanged: the central moments make the
    relaxation Galilean invariant, where raw moments would not."""
    still = _shear_wave(oracle_mod, 0.0)
    moving = _shear_wave(oracle_mod, 0.08)
    assert abs(still - 1) < 5e-3
    assert abs(moving - still) < 1e-9


def test_poiseuille_between_walls(oracle_mod):
    """Body-force-driven flow between half-way bounce-back walls at z = -1/2 and N - 1/2
    reaches the parabola u = g (z + 1/2)(N - z - 1/2) / (2 nu)."""
    n, nu, gx = 12, 1 / 6, 1e-5
    w = _cube((1, 1, n), nu=nu, rho0=np.ones((n, 1, 1)), u0=np.zeros((3, n, 1, 1)),
              g_body=(gx, 0.0, 0.0),
              face_flow=("periodic",) * 4 + ("wall", "wall"))
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    oracle_mod.run(p, f, g, 4000)
    _, u, _ = oracle_mod.macroscopic(p, f, g)
    z = np.arange(n) + 0.5
    exact = gx * z * (n - z) / (2 * nu)
    assert np.abs(u[0, :, 0, 0] - exact).max() < 5e-3 * exact.max()
    assert np.abs(u[1:]).max() < 1e-12


# ------------------------------------- streaming, walls, conservation on D3Q27 -------

_FROZEN = {"bulk": 1e-300, "r3": 1e-300, "r4": 1e-300, "r5": 1e-300, "r6": 1e-300}


def _frozen(shape, **kw):
    """No relaxation: every central-moment rate 1e-300 and the shear rate 1/tau ~ 3e-13
    (nu = 1e12), so a step is streaming (with the wall rules) to ~1e-12."""
    return _cube(shape, rates=dict(_FROZEN), nu=1e12, **kw)


def _opp(c):
    return [int(np.nonzero((c == -c[q]).all(axis=1))[0][0]) for q in range(27)]


def test_d3q27_streaming_is_the_lattice_permutation(oracle_mod):
    """Without relaxation a D3Q27 step is the pull permutation f_q(x) <- f_q(x - c_q) on
    the periodic grid, for all 27 velocities (brute force with np.roll)."""
    shape = (5, 4, 3)
    w = _frozen(shape)
    p = oracle_mod.Problem(w)
    f = np.random.default_rng(21).random((27,) + w.grid)
    g = np.zeros((1,) + w.grid)
    c, _, _ = oracle_mod.lattice(27)
    expect = np.stack([np.roll(f[q], shift=(c[q, 2], c[q, 1], c[q, 0]), axis=(0, 1, 2))
                       for q in range(27)])
    oracle_mod.run(p, f, g, 1)
    assert np.allclose(f, expect, rtol=0, atol=1e-10)


def test_d3q27_bounce_back_links_brute_force(oracle_mod):
    """Without relaxation, with walls on y and z and a solid cell, each D3Q27 wall link
    (corner links included) returns the cell's own opposite population."""
    shape = (5, 4, 3)
    solid = np.zeros(shape[::-1], np.uint8)
    solid[1, 2, 2] = 1
    w = _frozen(shape, face_flow=("periodic", "periodic", "wall", "wall", "wall", "wall"),
                solid=solid)
    p = oracle_mod.Problem(w)
    f = np.random.default_rng(22).random((27,) + w.grid)
    f[:, solid == 1] = 0.0
    g = np.zeros((1,) + w.grid)
    f_old = f.copy()
    oracle_mod.run(p, f, g, 1)
    c, _, _ = oracle_mod.lattice(27)
    opp = _opp(c)
    nx, ny, nz = shape
    for z, y, x in itertools.product(range(nz), range(ny), range(nx)):
        if solid[z, y, x]:
            continue
        for q in range(27):
            sx, sy, sz = (x - c[q, 0]) % nx, y - c[q, 1], z - c[q, 2]
            wall = not (0 <= sy < ny and 0 <= sz < nz) or solid[sz, sy, sx]
            want = f_old[opp[q], z, y, x] if wall else f_old[q, sz, sy, sx]
            assert abs(f[q, z, y, x] - want) < 1e-10


def test_d3q27_mass_momentum_and_forcing(oracle_mod):
    """Periodic D3Q27 with the fixed central-moment rates: mass is conserved to 1e-12 and
    the total momentum grows by exactly sum(rho) g per step."""
    w = W.random_periodic(shape=(6, 5, 4), seed=23, lattice=27, nu=0.05)
    w = dataclasses.replace(w, g_body=(2e-4, -1e-4, 5e-5))
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    for _ in range(4):
        d0 = oracle_mod.diagnostics(p, f, g)
        oracle_mod.run(p, f, g, 1)
        d1 = oracle_mod.diagnostics(p, f, g)
        assert abs(d1["mass"] - d0["mass"]) <= 1e-12 * d0["mass"]
        expect = d0["mass"] * np.array(w.g_body)
        assert np.allclose(d1["momentum"] - d0["momentum"], expect, rtol=1e-10, atol=1e-15)


def test_d3q27_momentum_exchange_balances_momentum(oracle_mod):
    """Periodic D3Q27 box with a solid obstacle and a body force: per step the fluid's
    momentum change equals the body force minus the momentum exchanged with the solid."""
    shape = (10, 8, 7)
    solid = W.sphere_mask(shape, (4, 4, 3), 2.0)
    base = W.perturbed(W.channel_sphere(shape=shape, lattice=27), seed=24)
    w = dataclasses.replace(base, face_flow=("periodic",) * 6, solid=solid,
                            g_body=(1e-4, 3e-5, -2e-5))
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0)
    for _ in range(3):
        d0 = oracle_mod.diagnostics(p, f, g)
        F = oracle_mod.run(p, f, g, 1)
        d1 = oracle_mod.diagnostics(p, f, g)
        body = d0["mass"] * np.array(w.g_body)
        assert np.allclose(d1["momentum"] - d0["momentum"], body - F, rtol=0, atol=1e-13)
        assert np.linalg.norm(F) > 1e-6
