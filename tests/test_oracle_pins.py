"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each checks a textbook value, a closed
form, a conservation law, an exact fixed point, a brute-force permutation, or a value the
pages print.  CPU only.
"""
import dataclasses
import itertools
import json
import math
import os

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spec(**kw):
    """A small problem description with defaults (periodic, MRT, rest)."""
    base = dict(name="test", lattice=19, thermal=0, collision="mrt", shape=(4, 4, 4), nu=0.1,
                rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2})
    base.update(kw)
    w = W.Workload(**base)
    if w.rho0 is None:
        w.rho0 = np.ones(w.grid, np.float32)
    if w.u0 is None:
        w.u0 = np.zeros((w.dim,) + w.grid, np.float32)
    if w.thermal and w.T_init is None:
        w.T_init = np.zeros(w.grid, np.float32)
    return w


def _start(oracle, w, window=None):
    p = oracle.Problem(w, window)
    f, g = oracle.init_equilibrium(p, w.rho0, w.u0, w.T_init)
    return p, f, g


# ------------------------------------------------------------------ lattices ------

@pytest.mark.parametrize("kind,dim", [(19, 3), (9, 2)])
def test_velocity_set_isotropy(oracle_mod, kind, dim):
    """Weights and velocities give the isotropic moments of a c_s^2 = 1/3 lattice up to
    fourth order: sum w = 1, sum w c = 0, sum w c_a c_b = d_ab/3,
    sum w c_a c_b c_c c_d = (d_ab d_cd + d_ac d_bd + d_ad d_bc)/9."""
    c, w, _ = oracle_mod.lattice(kind)
    c = c[:, :dim].astype(float)
    assert math.isclose(w.sum(), 1.0, abs_tol=1e-15)
    assert np.allclose(np.einsum("q,qa->a", w, c), 0, atol=1e-15)
    I = np.eye(dim)
    assert np.allclose(np.einsum("q,qa,qb->ab", w, c, c), I / 3, atol=1e-15)
    iso = (np.einsum("ab,cd->abcd", I, I) + np.einsum("ac,bd->abcd", I, I)
           + np.einsum("ad,bc->abcd", I, I)) / 9
    assert np.allclose(np.einsum("q,qa,qb,qc,qd->abcd", w, c, c, c, c), iso, atol=1e-15)
    assert len({tuple(v) for v in c}) == kind


def test_d2q9_d2q5_order_matches_halo_description(oracle_mod):
    """The thermal multi-GPU page sends f2, f5, f6 and g2 to the top neighbour and f4, f7,
    f8 and g4 to the bottom one: those are exactly the populations with c_y = +1 / -1."""
    c9, _, _ = oracle_mod.lattice(9)
    c5, _, _ = oracle_mod.lattice(5)
    assert sorted(np.nonzero(c9[:, 1] == 1)[0].tolist()) == [2, 5, 6]
    assert sorted(np.nonzero(c9[:, 1] == -1)[0].tolist()) == [4, 7, 8]
    assert np.nonzero(c5[:, 1] == 1)[0].tolist() == [2]
    assert np.nonzero(c5[:, 1] == -1)[0].tolist() == [4]


@pytest.mark.parametrize("kind", [19, 9, 7, 5])
def test_moment_basis_orthogonal(oracle_mod, kind):
    """Rows of each basis are mutually orthogonal, row 0 is the density (all ones) and
    the first-order rows are the velocity components."""
    c, _, M = oracle_mod.lattice(kind)
    G = M @ M.T
    assert np.allclose(G - np.diag(np.diag(G)), 0)
    assert np.all(M[0] == 1)
    jrows = {19: [3, 5, 7], 9: [3, 5], 7: [1, 2, 3], 5: [1, 2]}[kind]
    for a, r in enumerate(jrows):
        assert np.array_equal(M[r], c[:, a])


@pytest.mark.parametrize("kind", [19, 9])
def test_equilibrium_moments_textbook(oracle_mod, kind):
    """m_eq = M f_eq reproduces the published equilibrium moments of the d'Humieres D3Q19
    and the Lallemand-Luo D2Q9 models (golden fixture, with citation)."""
    gold = json.load(open(os.path.join(GOLDEN, "mrt_equilibrium_moments.json")))
    gold = gold["D3Q19" if kind == 19 else "D2Q9"]
    _, _, M = oracle_mod.lattice(kind)
    rng = np.random.default_rng(0)
    for _ in range(5):
        rho = 1.0 + 0.1 * rng.standard_normal()
        dim = 3 if kind == 19 else 2
        u = 0.05 * rng.standard_normal(dim)
        w = _spec(lattice=kind, shape=(1, 1, 1),
                  rho0=np.full((1, 1, 1), rho, np.float32),
                  u0=u.reshape(dim, 1, 1, 1).astype(np.float32))
        rho32, u32 = float(w.rho0.ravel()[0]), w.u0.reshape(dim).astype(float)
        _, f, _ = _start(oracle_mod, w)
        m = M @ f.reshape(kind)
        u2 = float(u32 @ u32)
        j = rho32 * u32
        assert math.isclose(m[0], rho32, rel_tol=1e-13)
        assert math.isclose(m[1], gold["e"]["rho"] * rho32 + gold["e"]["rho_u2"] * rho32 * u2,
                            rel_tol=1e-12, abs_tol=1e-13)
        assert math.isclose(m[2], gold["eps"]["rho"] * rho32 + gold["eps"]["rho_u2"] * rho32 * u2,
                            rel_tol=1e-12, abs_tol=1e-13)
        if kind == 19:
            jrows, qrows = [3, 5, 7], [4, 6, 8]
            p = {9: rho32 * (2 * u32[0] ** 2 - u32[1] ** 2 - u32[2] ** 2),
                 11: rho32 * (u32[1] ** 2 - u32[2] ** 2), 13: rho32 * u32[0] * u32[1],
                 14: rho32 * u32[1] * u32[2], 15: rho32 * u32[0] * u32[2]}
            for r, v in p.items():
                assert math.isclose(m[r], v, abs_tol=1e-14)
            assert math.isclose(m[10], gold["pi_over_p"] * p[9], abs_tol=1e-14)
            assert math.isclose(m[12], gold["pi_over_p"] * p[11], abs_tol=1e-14)
            assert np.allclose(m[16:19], gold["m"], atol=1e-14)
        else:
            jrows, qrows = [3, 5], [4, 6]
            assert math.isclose(m[7], rho32 * (u32[0] ** 2 - u32[1] ** 2), abs_tol=1e-14)
            assert math.isclose(m[8], rho32 * u32[0] * u32[1], abs_tol=1e-14)
        for a in range(dim):
            assert math.isclose(m[jrows[a]], j[a], rel_tol=1e-12, abs_tol=1e-15)
            assert math.isclose(m[qrows[a]], gold["q_over_j"] * j[a], rel_tol=1e-12,
                                abs_tol=1e-15)


# --------------------------------------------------------------- fixed points -----

@pytest.mark.parametrize("lattice,thermal", [(19, 0), (19, 7), (9, 5)])
@pytest.mark.parametrize("collision", ["bgk", "mrt"])
def test_rest_state_is_fixed_point(oracle_mod, lattice, thermal, collision):
    """A uniform rest state (rho = 1, u = 0, T = T_w = T0) is an exact fixed point under
    walls, solids, Dirichlet and adiabatic faces, buoyancy and every collision."""
    shape = (6, 5, 4) if lattice == 19 else (6, 5, 1)
    solid = np.zeros(shape[::-1], np.uint8)
    solid[..., 2, 3] = 1
    Tw = 0.25
    w = _spec(lattice=lattice, thermal=thermal, collision=collision, shape=shape,
              rates={"e": 1.3, "eps": 1.1, "q": 1.4, "pi": 1.5, "m": 1.6} if lattice == 19
              else {"e": 1.3, "eps": 1.1, "q": 1.4},
              kappa=0.05, thermal_rates={"e": 1.1, "v": 1.3}, a_T=0.2,
              gbeta=1e-3 if thermal else 0.0, T0=Tw, up_axis=1,
              face_flow=("wall", "wall", "wall", "wall", "periodic", "periodic"),
              face_T=("dirichlet", "dirichlet", "adiabatic", "adiabatic", "adiabatic",
                      "adiabatic"),
              T_wall=(Tw, Tw, 0, 0, 0, 0), solid=solid)
    if thermal:
        w.T_init = np.full(w.grid, Tw, np.float32)
    p, f, g = _start(oracle_mod, w)
    f0, g0 = f.copy(), g.copy()
    oracle_mod.run(p, f, g, 7)
    assert np.allclose(f, f0, rtol=0, atol=1e-15)
    assert np.allclose(g, g0, rtol=0, atol=1e-15)


def test_uniform_flow_is_fixed_point(oracle_mod):
    """A uniform moving equilibrium on a periodic domain is an exact fixed point."""
    w = _spec(shape=(5, 4, 3))
    w.u0 = np.empty((3,) + w.grid, np.float32)
    for a, v in enumerate((0.03, -0.02, 0.01)):
        w.u0[a] = v
    p, f, g = _start(oracle_mod, w)
    f0 = f.copy()
    oracle_mod.run(p, f, g, 5)
    assert np.allclose(f, f0, rtol=0, atol=1e-15)


# ------------------------------------------------------------ conservation -------

@pytest.mark.parametrize("collision", ["bgk", "mrt"])
def test_mass_and_momentum_conserved_periodic(oracle_mod, collision):
    """Periodic and unforced: mass and momentum are conserved to 1e-12 relative."""
    w = W.random_periodic(shape=(12, 10, 8), seed=3, collision=collision)
    p, f, g = _start(oracle_mod, w)
    d0 = oracle_mod.diagnostics(p, f, g)
    oracle_mod.run(p, f, g, 150)
    d1 = oracle_mod.diagnostics(p, f, g)
    assert abs(d1["mass"] - d0["mass"]) <= 1e-12 * d0["mass"]
    assert np.all(np.abs(d1["momentum"] - d0["momentum"]) <= 1e-12 * d0["mass"])


def test_thermal_energy_conserved_periodic_and_adiabatic(oracle_mod):
    """sum T is conserved with periodic faces and with adiabatic walls and solids."""
    base = W.perturbed(W.cavity3d(shape=(10, 8, 6)), seed=4)
    for faces_T in (("adiabatic",) * 6,):
        w = dataclasses.replace(base, face_T=faces_T)
        solid = np.zeros(w.grid, np.uint8)
        solid[2:4, 3:5, 4:6] = 1
        w.solid = solid
        p, f, g = _start(oracle_mod, w)
        T0 = oracle_mod.macroscopic(p, f, g)[2].sum()
        oracle_mod.run(p, f, g, 60)
        T1 = oracle_mod.macroscopic(p, f, g)[2].sum()
        assert abs(T1 - T0) <= 1e-12 * np.abs(w.T_init).sum()


def test_guo_forcing_momentum_increment(oracle_mod):
    """Periodic domain, uniform body acceleration g: total momentum grows by exactly
    sum(rho) g per step (Guo forcing adds F to the momentum in every collision)."""
    w = dataclasses.replace(W.random_periodic(shape=(8, 6, 5), seed=5),
                            g_body=(2e-4, -1e-4, 5e-5))
    p, f, g = _start(oracle_mod, w)
    for _ in range(3):
        d0 = oracle_mod.diagnostics(p, f, g)
        oracle_mod.run(p, f, g, 1)
        d1 = oracle_mod.diagnostics(p, f, g)
        expect = d0["mass"] * np.array(w.g_body)
        assert np.allclose(d1["momentum"] - d0["momentum"], expect, rtol=1e-10, atol=1e-15)


# ---------------------------------------------------------------- streaming ------

_FROZEN_RATES = {19: ("e", "eps", "q", "pi", "m"), 9: ("e", "eps", "q")}


@pytest.mark.parametrize("lattice,shape", [(19, (4, 4, 4)), (19, (5, 4, 3)), (9, (5, 4, 1))])
def test_streaming_is_the_lattice_permutation(oracle_mod, lattice, shape):
    """With no relaxation (every rate 0, no force) a step is pure streaming: the new
    f_q(x) is f_q(x - c_q) on the periodic grid (brute force with np.roll)."""
    # the viscous rate follows from nu: a huge nu makes it ~3e-13
    w = _spec(lattice=lattice, shape=shape, nu=1e12,
              rates={k: 0.0 for k in _FROZEN_RATES[lattice]})
    p = oracle_mod.Problem(w)
    rng = np.random.default_rng(1)
    Q = lattice
    f = rng.random((Q,) + w.grid)
    g = np.zeros((1,) + w.grid)
    c, _, _ = oracle_mod.lattice(Q)
    expect = np.stack([np.roll(f[q], shift=(c[q, 2], c[q, 1], c[q, 0]), axis=(0, 1, 2))
                       for q in range(Q)])
    oracle_mod.run(p, f, g, 1)
    assert np.allclose(f, expect, rtol=0, atol=1e-11)


@pytest.mark.parametrize("lattice", [19, 9])
def test_bounce_back_links_brute_force(oracle_mod, lattice):
    """With no relaxation, on a grid with walls and a solid cell, each wall link returns
    the cell's own opposite population (brute force over every cell and direction)."""
    shape = (5, 4, 3) if lattice == 19 else (6, 5, 1)
    solid = np.zeros(shape[::-1], np.uint8)
    solid[(1, 2, 2) if lattice == 19 else (0, 2, 2)] = 1
    # x periodic, every other axis walled (z is unused in 2-D: c_z = 0)
    faces = ("periodic", "periodic", "wall", "wall", "wall", "wall")
    w = _spec(lattice=lattice, shape=shape, nu=1e12,
              rates={k: 0.0 for k in _FROZEN_RATES[lattice]}, face_flow=faces, solid=solid)
    p = oracle_mod.Problem(w)
    rng = np.random.default_rng(2)
    Q = lattice
    f = rng.random((Q,) + w.grid)
    f[:, solid == 1] = 0.0
    g = np.zeros((1,) + w.grid)
    f_old = f.copy()
    oracle_mod.run(p, f, g, 1)
    c, _, _ = oracle_mod.lattice(Q)
    opp = [int(np.nonzero((c == -c[q]).all(axis=1))[0][0]) for q in range(Q)]
    nx, ny, nz = shape
    for z in range(nz):
        for y in range(ny):
            for x in range(nx):
                if solid[z, y, x]:
                    continue
                for q in range(Q):
                    sx, sy, sz = (x - c[q, 0]) % nx, y - c[q, 1], z - c[q, 2]
                    wall = not (0 <= sy < ny and 0 <= sz < nz) or solid[sz, sy, sx]
                    want = f_old[opp[q], z, y, x] if wall else f_old[q, sz, sy, sx]
                    assert abs(f[q, z, y, x] - want) < 1e-11


@pytest.mark.parametrize("lattice,thermal", [(19, 7), (9, 5)])
def test_thermal_wall_links_brute_force(oracle_mod, lattice, thermal):
    """Without relaxation (flow and thermal rates ~0), one step on a cavity with Dirichlet
    x faces, adiabatic walls elsewhere and a solid cell, checked link by link: a thermal
    link through a Dirichlet face returns -g_opp(x) + omega T_w with the page's omega,
    (4 + a_T)/10 on D2Q5 and (6 + a_T)/21 on D3Q7 ("Multi-GPU thermal lattice Boltzmann
    simulations using OpenACC and MPI", Sec. 2); a link through an adiabatic wall or into
    the solid returns g_opp(x); every other link streams, g_k(x) = g_k(x - c_k)."""
    shape = (5, 4, 3) if lattice == 19 else (6, 5, 1)
    base = W.cavity3d(shape=shape) if lattice == 19 else W.cavity2d(shape=shape)
    solid = np.zeros(base.grid, np.uint8)
    solid[(0, 2, 2) if lattice == 9 else (1, 2, 2)] = 1
    frozen = ({k: 0.0 for k in ("e", "eps", "q", "pi", "m")} if lattice == 19
              else {k: 0.0 for k in ("e", "eps", "q")})
    a_T = 0.3
    w = dataclasses.replace(base, solid=solid, nu=1e12, rates=frozen, kappa=1e12,
                            thermal_rates={"e": 0.0, "v": 0.0}, a_T=a_T, gbeta=0.0,
                            T_wall=(0.7, -0.4, 0.0, 0.0, 0.0, 0.0))
    omega = (4.0 + a_T) / 10.0 if thermal == 5 else (6.0 + a_T) / 21.0
    p = oracle_mod.Problem(w)
    rng = np.random.default_rng(9)
    f = 0.05 + 0.01 * rng.random((lattice,) + w.grid)
    g = rng.uniform(-0.2, 0.2, size=(thermal,) + w.grid)
    g_old = g.copy()
    oracle_mod.run(p, f, g, 1)
    c, _, _ = oracle_mod.lattice(thermal)
    opp = [int(np.nonzero((c == -c[k]).all(axis=1))[0][0]) for k in range(thermal)]
    nz, ny, nx = w.grid
    n = (nx, ny, nz)
    checked = 0
    for z, y, x in itertools.product(range(nz), range(ny), range(nx)):
        if solid[z, y, x]:
            continue
        for k in range(thermal):
            src = [x - c[k, 0], y - c[k, 1], z - c[k, 2]]
            face = None
            for a in range(3):
                if src[a] < 0:
                    face = 2 * a
                elif src[a] >= n[a]:
                    face = 2 * a + 1
            if face is not None:
                if w.face_T[face] == "dirichlet":
                    want = -g_old[opp[k], z, y, x] + omega * w.T_wall[face]
                else:
                    want = g_old[opp[k], z, y, x]
            elif solid[src[2], src[1], src[0]]:
                want = g_old[opp[k], z, y, x]
            else:
                want = g_old[k, src[2], src[1], src[0]]
            assert abs(g[k, z, y, x] - want) < 1e-10, (x, y, z, k)
            checked += 1
    assert checked == thermal * (nx * ny * nz - 1)


# -------------------------------------------------------------------- MRT --------

def test_mrt_with_equal_rates_is_bgk(oracle_mod):
    """Every non-conserved rate equal to 1/tau makes the MRT operator (with its moment
    space forcing) identical to BGK with Guo forcing."""
    tau = 0.8
    base = dataclasses.replace(W.perturbed(W.cavity3d(shape=(7, 6, 5)), seed=9),
                               g_body=(1e-4, 2e-4, 0.0), gbeta=3e-3)
    s = 1.0 / tau
    w_mrt = dataclasses.replace(base, collision="mrt", nu=(tau - 0.5) / 3,
                                rates={k: s for k in ("e", "eps", "q", "pi", "m")})
    w_bgk = dataclasses.replace(w_mrt, collision="bgk")
    out = []
    for w in (w_mrt, w_bgk):
        p, f, g = _start(oracle_mod, w)
        oracle_mod.run(p, f, g, 12)
        out.append((f, g))
    assert np.allclose(out[0][0], out[1][0], rtol=0, atol=1e-13)
    assert np.allclose(out[0][1], out[1][1], rtol=0, atol=1e-13)


def _fit_rate(ts, amps):
    return -np.polyfit(np.asarray(ts, float), np.log(np.asarray(amps)), 1)[0]


def test_taylor_green_decay_rate():
    """3-D Taylor-Green, 32^3, BGK tau = 0.8: after the initial acoustic transient the
    projection on the initial mode decays as exp(-3 nu k^2 t); the fitted rate over
    t in [50, 200] is within 1%."""
    import oracle
    w = W.taylor_green()
    p, f, g = _start(oracle, w)
    n = 32
    k = 2 * math.pi / n
    z, y, x = np.meshgrid(np.arange(n), np.arange(n), np.arange(n), indexing="ij")
    mode = np.sin(k * x) * np.cos(k * y) * np.cos(k * z)
    ts, amps = [], []
    oracle.run(p, f, g, 50)
    for t in range(50, 201, 25):
        if t > 50:
            oracle.run(p, f, g, 25)
        u = oracle.macroscopic(p, f, g)[1]
        ts.append(t)
        amps.append((u[0] * mode).sum() / (mode * mode).sum())
    rate = _fit_rate(ts, amps)
    assert abs(rate / (3 * w.nu * k * k) - 1) < 0.01


@pytest.mark.parametrize("lattice,collision", [(19, "mrt"), (19, "bgk"), (9, "mrt")])
def test_shear_wave_second_order(oracle_mod, lattice, collision):
    """A shear wave u_x = u0 sin(k y) decays as exp(-nu k^2 t); the error of the fitted
    rate falls ~4x when the wavelength doubles (second-order accuracy), < 0.5% at 64."""
    errs = []
    for n in (32, 64):
        shape = (1, n, 1)
        k = 2 * math.pi / n
        y = np.arange(n)
        w = _spec(lattice=lattice, collision=collision, shape=shape, nu=0.05,
                  rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}
                  if lattice == 19 else {"e": 1.2, "eps": 1.2, "q": 1.2})
        u = np.zeros((w.dim,) + w.grid, np.float32)
        u[0, 0, :, 0] = 0.01 * np.sin(k * y)
        w.u0 = u
        p, f, g = _start(oracle_mod, w)
        steps = int(round(1.0 / (w.nu * k * k)))   # one e-folding
        ts, amps = [], []
        oracle_mod.run(p, f, g, steps // 4)
        for i in range(5):
            if i:
                oracle_mod.run(p, f, g, steps // 4)
            uu = oracle_mod.macroscopic(p, f, g)[1][0, 0, :, 0]
            ts.append(i)
            amps.append((uu * np.sin(k * y)).sum() / (np.sin(k * y) ** 2).sum())
        rate = _fit_rate(np.array(ts) * (steps // 4), amps)
        errs.append(abs(rate / (w.nu * k * k) - 1))
    assert errs[1] < 0.005
    assert errs[1] < errs[0] / 3


@pytest.mark.parametrize("lattice,collision", [(19, "mrt"), (9, "mrt"), (19, "bgk")])
def test_poiseuille_profile(oracle_mod, lattice, collision):
    """Body-force driven flow between two half-way bounce-back walls: the steady profile
    is g (y + 1/2)(H - 1/2 - y) / (2 nu) with the walls at -1/2 and H - 1/2; within 0.5%
    at H = 32."""
    H, nu, gx = 32, 0.1, 1e-6
    shape = (1, H, 1)
    w = _spec(lattice=lattice, collision=collision, shape=shape, nu=nu, g_body=(gx, 0, 0),
              rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}
              if lattice == 19 else {"e": 1.2, "eps": 1.2, "q": 1.2},
              face_flow=("periodic", "periodic", "wall", "wall", "periodic", "periodic"))
    p, f, g = _start(oracle_mod, w)
    oracle_mod.run(p, f, g, int(8 * H * H / nu))
    ux = oracle_mod.macroscopic(p, f, g)[1][0, 0, :, 0]
    y = np.arange(H)
    exact = gx * (y + 0.5) * (H - 0.5 - y) / (2 * nu)
    assert np.max(np.abs(ux - exact)) < 0.005 * exact.max()


# ------------------------------------------------------------------ thermal -------

@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "thermal_abb_weight.json")))["cases"])
def test_anti_bounce_back_weight_matches_page(oracle_mod, case):
    """From g = 0 (T = 0, u = 0) a Dirichlet wall at T_w returns omega T_w on its link
    after one step; omega must be the page's (4 + a_T)/10 or (6 + a_T)/21."""
    lattice, thermal = (9, 5) if case["lattice"] == "D2Q5" else (19, 7)
    shape = (1, 1, 1)
    Tw = 0.7
    w = _spec(lattice=lattice, thermal=thermal, shape=shape, kappa=0.1,
              thermal_rates={"e": 1.2, "v": 1.2}, a_T=case["a_T"],
              rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}
              if lattice == 19 else {"e": 1.2, "eps": 1.2, "q": 1.2},
              face_flow=("wall", "wall") + ("periodic",) * 4,
              face_T=("dirichlet", "adiabatic") + ("adiabatic",) * 4, T_wall=(Tw,) + (0,) * 5)
    p, f, g = _start(oracle_mod, w)
    oracle_mod.run(p, f, g, 1)
    c, _, _ = oracle_mod.lattice(thermal)
    plus_x = int(np.nonzero((c == [1, 0, 0]).all(axis=1))[0][0])
    assert math.isclose(g[plus_x].ravel()[0] / Tw, case["omega"], rel_tol=1e-14)


@pytest.mark.parametrize("lattice,thermal", [(19, 7), (9, 5)])
@pytest.mark.parametrize("a_T", [0.0, 0.4, -0.3])
def test_dirichlet_uniform_temperature_fixed_point(oracle_mod, lattice, thermal, a_T):
    """Uniform T = T_w at rest between Dirichlet walls at T_w is an exact fixed point: the
    anti-bounce-back weight is consistent with the thermal equilibrium's weights.
    (T_w = 0.375 is exact in fp32, the precision of the initial fields.)"""
    Tw = 0.375
    shape = (4, 3, 3) if lattice == 19 else (4, 3, 1)
    w = _spec(lattice=lattice, thermal=thermal, shape=shape, kappa=0.1,
              thermal_rates={"e": 1.3, "v": 1.1}, a_T=a_T,
              rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}
              if lattice == 19 else {"e": 1.2, "eps": 1.2, "q": 1.2},
              face_flow=("wall",) * 6, face_T=("dirichlet",) * 6, T_wall=(Tw,) * 6,
              T_init=np.full(shape[::-1], Tw, np.float32))
    p, f, g = _start(oracle_mod, w)
    g0 = g.copy()
    oracle_mod.run(p, f, g, 5)
    assert np.allclose(g, g0, rtol=0, atol=1e-15)


@pytest.mark.parametrize("lattice,thermal", [(19, 7), (9, 5)])
def test_conduction_profile_and_unit_nusselt(oracle_mod, lattice, thermal):
    """Pure conduction between Dirichlet faces T_h (x = -1/2) and T_c (x = N - 1/2): the
    steady profile is T_h - (T_h - T_c)(x + 1/2)/N, and the wall heat flux gives Nu = 1."""
    N, Th, Tc = 16, 0.5, -0.5
    shape = (N, 2, 2) if lattice == 19 else (N, 2, 1)
    w = _spec(lattice=lattice, thermal=thermal, shape=shape, kappa=0.2,
              thermal_rates={"e": 1.2, "v": 1.2},
              rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}
              if lattice == 19 else {"e": 1.2, "eps": 1.2, "q": 1.2},
              face_flow=("wall", "wall") + ("periodic",) * 4,
              face_T=("dirichlet", "dirichlet") + ("adiabatic",) * 4,
              T_wall=(Th, Tc) + (0,) * 4)
    p, f, g = _start(oracle_mod, w)
    oracle_mod.run(p, f, g, int(12 * N * N / w.kappa))
    T = oracle_mod.macroscopic(p, f, g)[2]
    x = np.arange(N)
    exact = Th - (Th - Tc) * (x + 0.5) / N
    assert np.allclose(T, exact[None, None, :], rtol=0, atol=1e-9)
    d = oracle_mod.diagnostics(p, f, g)
    area = shape[1] * shape[2]
    nu_hot = d["heat"][0] * N / ((Th - Tc) * area)
    nu_cold = -d["heat"][1] * N / ((Th - Tc) * area)
    assert math.isclose(nu_hot, 1.0, rel_tol=1e-8)
    assert math.isclose(nu_cold, 1.0, rel_tol=1e-8)


@pytest.mark.parametrize("lattice,thermal", [(19, 7), (9, 5)])
def test_thermal_diffusion_rate(oracle_mod, lattice, thermal):
    """A temperature sine mode at rest decays as exp(-kappa k^2 t) (periodic), which pins
    the diffusivity of the thermal MRT and its rate mapping (< 0.5% at wavelength 64)."""
    n = 64
    k = 2 * math.pi / n
    shape = (n, 1, 1)
    x = np.arange(n)
    w = _spec(lattice=lattice, thermal=thermal, shape=shape, kappa=0.05,
              thermal_rates={"e": 1.2, "v": 1.2}, a_T=0.2,
              rates={"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2}
              if lattice == 19 else {"e": 1.2, "eps": 1.2, "q": 1.2},
              T_init=(0.1 * np.sin(k * x)).reshape(1, 1, n).astype(np.float32))
    p, f, g = _start(oracle_mod, w)
    steps = int(round(1.0 / (w.kappa * k * k)))
    ts, amps = [], []
    for i in range(5):
        if i:
            oracle_mod.run(p, f, g, steps // 4)
        T = oracle_mod.macroscopic(p, f, g)[2].ravel()
        ts.append(i * (steps // 4))
        amps.append((T * np.sin(k * x)).sum() / (np.sin(k * x) ** 2).sum())
    assert abs(_fit_rate(ts, amps) / (w.kappa * k * k) - 1) < 0.005


def test_thermal_advection_speed(oracle_mod):
    """In a uniform flow u0 a temperature mode is carried at u0: its phase moves by
    k u0 t (pins the advective moment u T of the thermal equilibrium)."""
    n, u0 = 64, 0.05
    k = 2 * math.pi / n
    x = np.arange(n)
    w = _spec(lattice=9, thermal=5, shape=(n, 1, 1), kappa=0.02,
              rates={"e": 1.2, "eps": 1.2, "q": 1.2}, thermal_rates={"e": 1.2, "v": 1.2},
              T_init=(0.1 * np.sin(k * x)).reshape(1, 1, n).astype(np.float32))
    uu = np.zeros((2, 1, 1, n), np.float32)
    uu[0] = u0
    w.u0 = uu
    p, f, g = _start(oracle_mod, w)
    t = 400
    oracle_mod.run(p, f, g, t)
    T = oracle_mod.macroscopic(p, f, g)[2].ravel()
    phase = math.atan2(-(T * np.cos(k * x)).sum(), (T * np.sin(k * x)).sum())
    assert abs(phase - k * np.float32(u0) * t) < 0.01 * k * u0 * t


# -------------------------------------------------------- momentum exchange -------

def test_momentum_exchange_balances_momentum(oracle_mod):
    """Periodic box with a solid obstacle and a body force: per step the fluid's momentum
    change equals the body force minus the momentum exchanged with the solid, exactly.
    Pins the sign and factor 2 of the solid force."""
    shape = (12, 9, 8)
    solid = W.sphere_mask(shape, (5, 4, 4), 2.5)
    base = W.perturbed(W.channel_sphere(shape=shape), seed=11)
    w = dataclasses.replace(base, face_flow=("periodic",) * 6, solid=solid,
                            g_body=(1e-4, 3e-5, -2e-5))
    p, f, g = _start(oracle_mod, w)
    for _ in range(4):
        d0 = oracle_mod.diagnostics(p, f, g)
        F = oracle_mod.run(p, f, g, 1)
        d1 = oracle_mod.diagnostics(p, f, g)
        body = d0["mass"] * np.array(w.g_body)
        assert np.allclose(d1["momentum"] - d0["momentum"], body - F, rtol=0, atol=1e-13)
        assert np.linalg.norm(F) > 1e-6


def test_closed_body_at_rest_feels_no_force(oracle_mod):
    """At rest (f = w) the exchanged momentum over any closed solid is zero (each link's
    2 w_q c_q cancels its mirror link; only summation rounding of ~1e3 terms remains)."""
    w = W.channel_sphere(shape=(24, 20, 20), center=(10, 9, 9), radius=5)
    p, f, g = _start(oracle_mod, dataclasses.replace(w, g_body=(0, 0, 0)))
    F = oracle_mod.run(p, f, g, 1)
    assert np.all(np.abs(F) < 1e-13)


def test_symmetric_body_has_no_transverse_force(oracle_mod):
    """A sphere centred between symmetric walls feels no force across the flow."""
    n = 17
    w = W.channel_sphere(shape=(20, n, n), center=(8, 8, 8), radius=4, gx=1e-5)
    p, f, g = _start(oracle_mod, w)
    F = oracle_mod.run(p, f, g, 40)
    assert F[0] > 0
    assert abs(F[1]) < 1e-12 * abs(F[0]) + 1e-18
    assert abs(F[2]) < 1e-12 * abs(F[0]) + 1e-18


# ------------------------------------------------------------------ windows ------

def test_window_run_matches_full_run(oracle_mod):
    """A run on a window of the domain reproduces the full run exactly at cells further
    than the step count from the window's cut faces, and marks the rest unknown (NaN)."""
    w = W.perturbed(W.cavity3d(shape=(14, 12, 10)), seed=13)
    solid = np.zeros(w.grid, np.uint8)
    solid[4:6, 5:7, 1:3] = 1
    w.solid = solid
    steps = 3
    p, f, g = _start(oracle_mod, w)
    oracle_mod.run(p, f, g, steps)
    org, ext = (0, 2, 1), (9, 8, 8)
    pw, fw, gw = _start(oracle_mod, w, (org, ext))
    oracle_mod.run(pw, fw, gw, steps)
    # valid region: cut faces are x = 9 (high side), y = 2 and 9, z = 1 and 8 -> shrink
    lo = [0, steps, steps]
    hi = [ext[0] - steps, ext[1] - steps, ext[2] - steps]
    sl_w = (slice(None), slice(lo[2], hi[2]), slice(lo[1], hi[1]), slice(lo[0], hi[0]))
    sl_f = (slice(None), slice(org[2] + lo[2], org[2] + hi[2]),
            slice(org[1] + lo[1], org[1] + hi[1]), slice(org[0] + lo[0], org[0] + hi[0]))
    assert np.array_equal(fw[sl_w], f[sl_f])
    assert np.array_equal(gw[sl_w], g[sl_f])
    assert np.isnan(fw).any()


@pytest.mark.parametrize("lattice,walls", [(19, "y"), (19, "z"), (9, "y")])
def test_poiseuille_exact_in_two_rate_limit(oracle_mod, lattice, walls):
    """With every odd non-conserved moment (q, m) relaxed at s_odd and every even one at
    s_nu, half-way bounce-back Poiseuille flow is exact when
    Lambda = (1/s_nu - 1/2)(1/s_odd - 1/2) = 3/16 (Ginzburg and d'Humieres' two-relaxation-
    time result; not on the pages).  Exactness to 1e-9 pins which rows each rate acts on,
    the half-way wall position and the forcing."""
    H, nu, gx = 16, 0.1, 1e-6
    s_nu = 1.0 / (3 * nu + 0.5)
    s_odd = 1.0 / ((3.0 / 16.0) / (1.0 / s_nu - 0.5) + 0.5)
    rates = ({"e": s_nu, "eps": s_nu, "q": s_odd, "pi": s_nu, "m": s_odd} if lattice == 19
             else {"e": s_nu, "eps": s_nu, "q": s_odd})
    if walls == "y":
        shape, faces = (1, H, 1), ("periodic", "periodic", "wall", "wall", "periodic", "periodic")
    else:
        shape, faces = (1, 1, H), ("periodic", "periodic", "periodic", "periodic", "wall", "wall")
    w = _spec(lattice=lattice, shape=shape, nu=nu, g_body=(gx, 0, 0), rates=rates,
              face_flow=faces)
    p, f, g = _start(oracle_mod, w)
    oracle_mod.run(p, f, g, int(20 * H * H / nu))
    ux = oracle_mod.macroscopic(p, f, g)[1][0].ravel()
    y = np.arange(H)
    exact = gx * (y + 0.5) * (H - 0.5 - y) / (2 * nu)
    assert np.max(np.abs(ux - exact)) < 1e-9 * exact.max()


def test_buoyancy_momentum_increment(oracle_mod):
    """Periodic domain with a random temperature field: per step the momentum along the
    vertical axis grows by exactly sum rho g beta (T - T0) (Boussinesq force of the thermal
    multi-GPU page, taken at the pre-collision state), the other components not at all."""
    base = W.perturbed(W.cavity3d(shape=(6, 5, 4)), seed=1)
    for up in (0, 1, 2):
        w = dataclasses.replace(base, face_flow=("periodic",) * 6, gbeta=0.05, T0=0.1,
                                up_axis=up)
        p, f, g = _start(oracle_mod, w)
        for _ in range(2):
            d0 = oracle_mod.diagnostics(p, f, g)
            rho, _, T = oracle_mod.macroscopic(p, f, g)
            oracle_mod.run(p, f, g, 1)
            d1 = oracle_mod.diagnostics(p, f, g)
            want = np.zeros(3)
            want[up] = (rho * w.gbeta * (T - w.T0)).sum()
            assert np.allclose(d1["momentum"] - d0["momentum"], want, rtol=1e-10, atol=1e-14)


@pytest.mark.parametrize("lattice,thermal", [(19, 7), (9, 5)])
def test_convective_transport_sum_closed_form(oracle_mod, lattice, thermal):
    """A uniform state in a periodic box with buoyancy stays uniform, and its momentum grows
    by F = rho gbeta (T - T0) e_up per step, so after n steps the diagnostics' sum of u_a T
    with u = (j + F/2)/rho is N T (u0 + (n + 1/2) gbeta (T - T0) e_up) in closed form."""
    dim = 3 if lattice == 19 else 2
    shape = (5, 4, 3) if dim == 3 else (5, 4, 1)
    up = dim - 1
    rates = ({"e": 1.2, "eps": 1.2, "q": 1.2, "pi": 1.2, "m": 1.2} if lattice == 19
             else {"e": 1.2, "eps": 1.2, "q": 1.2})
    w = W.Workload(name="uT", lattice=lattice, thermal=thermal, collision="mrt", shape=shape,
                   nu=0.05, rates=rates, kappa=0.05, thermal_rates={"e": 1.2, "v": 1.2},
                   gbeta=2e-3, T0=0.1, up_axis=up)
    N = int(np.prod(shape))
    u0 = np.array([0.02, -0.01, 0.015])[:dim]
    T, rho = 0.35, 1.0
    w.rho0 = np.full(w.grid, rho)
    w.u0 = np.broadcast_to(u0.reshape((dim,) + (1,) * 3), (dim,) + w.grid).copy()
    w.T_init = np.full(w.grid, T)
    p = oracle_mod.Problem(w)
    f, g = oracle_mod.init_equilibrium(p, w.rho0, w.u0, w.T_init)
    acc = w.gbeta * (T - w.T0)
    for n in (0, 1, 4):
        if n:
            oracle_mod.run(p, f, g, n - (0 if n == 1 else 1))
        want = np.zeros(3)
        want[:dim] = N * T * u0
        want[up] += N * T * (n + 0.5) * acc
        d = oracle_mod.diagnostics(p, f, g)
        assert np.allclose(d["uT"], want, rtol=1e-12, atol=1e-15), n
