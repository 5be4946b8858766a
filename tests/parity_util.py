"""Helpers shared by the parity tests: run a workload through the oracle, through the
CUDA library (GPU) or through the host emulation of its kernels, and compare."""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np

from lattice_boltzmann_cfd_gb300 import workloads as W
from lattice_boltzmann_cfd_gb300.solver import make_config

# parity tolerances: fp32 GPU against the fp64 oracle after 200 steps
TOL_FIELDS = 2e-5      # max-abs on rho, u, T
TOL_FORCE_REL = 1e-4   # relative on the solid force


def fluid_of(w):
    return np.ones(w.grid, bool) if w.solid is None else (w.solid == 0)


def oracle_states(oracle, w, checkpoints, window=None):
    """{steps: dict(f, g, rho, u, T, force, diag)} from the fp64 oracle."""
    p = oracle.Problem(w, window)
    f, g = oracle.init_equilibrium(p, w.rho0, w.u0, w.T_init)
    out, done = {}, 0
    for n in sorted(checkpoints):
        force = oracle.run(p, f, g, n - done)
        done = n
        rho, u, T = oracle.macroscopic(p, f, g)
        out[n] = dict(f=f.copy(), g=g.copy(), rho=rho, u=u, T=T, force=force,
                      ib=p.last_ib.copy(),
                      diag=oracle.diagnostics(p, f, g) if window is None else None)
    return out


def mask_brute_force(w) -> np.ndarray:
    """The link mask from its definition (numpy, independent of the library): bit q when
    the neighbour along c_q is outside through a WALL face or solid; bit 19+k when thermal
    axis link k leaves through a Dirichlet face; bit 31 for a solid cell."""
    c = {19: [(0, 0, 0), (1, 0, 0), (-1, 0, 0), (0, 1, 0), (0, -1, 0), (0, 0, 1), (0, 0, -1),
              (1, 1, 0), (-1, 1, 0), (1, -1, 0), (-1, -1, 0), (1, 0, 1), (-1, 0, 1), (1, 0, -1),
              (-1, 0, -1), (0, 1, 1), (0, -1, 1), (0, 1, -1), (0, -1, -1)],
         9: [(0, 0, 0), (1, 0, 0), (0, 1, 0), (-1, 0, 0), (0, -1, 0), (1, 1, 0), (-1, 1, 0),
             (-1, -1, 0), (1, -1, 0)]}
    c[27] = c[19] + [(1, 1, 1), (-1, 1, 1), (1, -1, 1), (-1, -1, 1), (1, 1, -1), (-1, 1, -1),
                     (1, -1, -1), (-1, -1, -1)]
    c = c[w.lattice]
    nz, ny, nx = w.grid
    solid = np.zeros(w.grid, bool) if w.solid is None else w.solid.astype(bool)
    z, y, x = np.meshgrid(np.arange(nz), np.arange(ny), np.arange(nx), indexing="ij")
    m = np.zeros(w.grid, np.uint64)
    wall_face = [k == "wall" for k in w.face_flow]
    dirichlet = [bool(w.face_flow[i] == "wall" and w.face_T[i] == "dirichlet" and w.thermal)
                 for i in range(6)]
    for q in range(1, w.lattice):
        cx, cy, cz = c[q]
        wall = np.zeros(w.grid, bool)
        dir_hit = np.zeros(w.grid, bool)
        coords = []
        for a, (pos, d, n) in enumerate(((x, cx, nx), (y, cy, ny), (z, cz, nz))):
            s = pos + d
            lo, hi = s < 0, s >= n
            if wall_face[2 * a]:
                wall |= lo
                dir_hit |= lo & dirichlet[2 * a]
            if wall_face[2 * a + 1]:
                wall |= hi
                dir_hit |= hi & dirichlet[2 * a + 1]
            coords.append(np.mod(s, n))
        wall |= ~wall & solid[coords[2], coords[1], coords[0]]
        m |= wall.astype(np.uint64) << np.uint64(q)
        if w.thermal and q < w.thermal:
            m |= dir_hit.astype(np.uint64) << np.uint64(19 + q)
    # bit 30: the cell lies in the 2^dim stencil of an immersed-boundary sample
    if getattr(w, "ib_x", None) is not None:
        ext = np.array([nx, ny, nz])
        for xs in np.asarray(w.ib_x, np.float32):
            base = np.floor(xs[:w.dim]).astype(int)
            for corner in range(1 << w.dim):
                q = [0, 0, 0]
                for a in range(w.dim):
                    q[a] = (base[a] + ((corner >> a) & 1)) % ext[a]
                m[q[2], q[1], q[0]] |= np.uint64(1 << 30)
    m = np.where(solid, np.uint64(1 << 31), m)
    return m.astype(np.uint32)


def emulate(emu_lib, w, steps, narrow=True, streaming="aa"):
    """(f, g, mask) after ``steps`` steps of the host emulation of the CUDA kernels."""
    cfg, keep = make_config(w, streaming)
    N = w.cells
    fo = np.zeros((w.lattice, N), np.float32)
    go = np.zeros((max(w.thermal, 1), N), np.float32)
    mo = np.zeros(N, np.uint32)
    rho = np.ascontiguousarray(w.rho0, np.float32)
    u = np.ascontiguousarray(w.u0, np.float32)
    T = np.ascontiguousarray(w.T_init, np.float32) if w.thermal else None
    vp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    ib = [None, None, None]
    n_ib = 0
    if getattr(w, "ib_x", None) is not None:
        n_ib = len(w.ib_x)
        ib = [np.ascontiguousarray(a, np.float32) if a is not None else None
              for a in (w.ib_x, w.ib_ub, w.ib_w)]
    rc = emu_lib.emu_run(ctypes.byref(cfg), vp(rho), vp(u), vp(T), int(steps), vp(fo), vp(go),
                         vp(mo), int(bool(narrow)), n_ib, vp(ib[0]), vp(ib[1]), vp(ib[2]))
    assert rc == 0
    return (fo.reshape((w.lattice,) + w.grid), go.reshape((max(w.thermal, 1),) + w.grid),
            mo.reshape(w.grid))


def emulate_slabs(emu_lib, w, steps, nslabs):
    """(f, g) of the whole domain after ``steps`` steps of the host emulation run as
    ``nslabs`` slabs along the outer axis with the library's halo exchange."""
    from lattice_boltzmann_cfd_gb300.slabs import split_ranges
    cfg, keep = make_config(w, "aa")
    N = w.cells
    fo = np.full((w.lattice, N), np.nan, np.float32)
    go = np.full((max(w.thermal, 1), N), np.nan, np.float32)
    rho = np.ascontiguousarray(w.rho0, np.float32)
    u = np.ascontiguousarray(w.u0, np.float32)
    T = np.ascontiguousarray(w.T_init, np.float32) if w.thermal else None
    ranges = split_ranges(w.shape[w.dim - 1], nslabs)
    edges = np.array([r[0] for r in ranges] + [ranges[-1][1]], np.int32)
    vp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = emu_lib.emu_run_slabs(ctypes.byref(cfg), vp(rho), vp(u), vp(T), int(steps),
                               int(nslabs), vp(edges), vp(fo), vp(go))
    assert rc == 0, rc
    return fo.reshape((w.lattice,) + w.grid), go.reshape((max(w.thermal, 1),) + w.grid)


def emulate_blocks(emu_lib, w, steps, nb, edges=None, ordered=True, swap=False):
    """(f, g) of the whole domain after ``steps`` steps of the host emulation run as
    nb = (bx, by, bz) blocks with the library's per-axis halo exchange.  edges: per axis the
    block boundaries (default: as even as possible).  ordered=False packs every axis before
    any unpack (a negative control); swap=True moves each face with the buffer-free swap."""
    from lattice_boltzmann_cfd_gb300.slabs import split_ranges
    cfg, keep = make_config(w, "aa")
    N = w.cells
    fo = np.full((w.lattice, N), np.nan, np.float32)
    go = np.full((max(w.thermal, 1), N), np.nan, np.float32)
    rho = np.ascontiguousarray(w.rho0, np.float32)
    u = np.ascontiguousarray(w.u0, np.float32)
    T = np.ascontiguousarray(w.T_init, np.float32) if w.thermal else None
    if edges is None:
        edges = []
        for a in range(3):
            r = split_ranges(w.shape[a], nb[a])
            edges.append([x[0] for x in r] + [r[-1][1]])
    flat = np.array([e for a in range(3) for e in edges[a]], np.int32)
    nbs = np.array(nb, np.int32)
    vp = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = emu_lib.emu_run_blocks(ctypes.byref(cfg), vp(rho), vp(u), vp(T), int(steps), vp(nbs),
                                vp(flat), int(bool(ordered)), int(bool(swap)), vp(fo), vp(go))
    assert rc == 0, rc
    return fo.reshape((w.lattice,) + w.grid), go.reshape((max(w.thermal, 1),) + w.grid)


def slab_cases():
    """Problems whose outer axis is periodic (the slabs form a ring) or walled, with solid
    cells and thermal Dirichlet faces on both kinds of axis."""
    c3 = W.perturbed(W.cavity3d(shape=(9, 7, 13)), seed=31)
    sol = np.zeros(c3.grid, np.uint8)
    sol[3:6, 2:5, 3:6] = 1          # straddles the slab faces at z = 4 and z = 5
    rb = dataclasses.replace(       # heated from below: Dirichlet faces on the outer axis
        c3, name="D3Q19 MRT + D3Q7 Rayleigh-Benard 9x7x13 perturbed", solid=sol, gbeta=0.01,
        face_T=("adiabatic",) * 4 + ("dirichlet", "dirichlet"),
        T_wall=(0.0, 0.0, 0.0, 0.0, 0.4, -0.3))
    cs = W.perturbed(W.channel_sphere(shape=(10, 9, 12), center=(4, 4, 0), radius=3.0), seed=32)
    ring = dataclasses.replace(     # periodic z with the sphere across the wrap
        cs, name="D3Q19 MRT channel periodic-z 10x9x12 + sphere across the wrap",
        face_flow=("periodic", "periodic", "wall", "wall", "periodic", "periodic"),
        g_body=(1e-4, 0.0, 2e-5))
    c2 = dataclasses.replace(W.perturbed(W.cavity2d(shape=(10, 11, 1)), seed=33), gbeta=0.01)
    c2p = dataclasses.replace(
        c2, name=c2.name + " periodic-y",
        face_flow=("wall", "wall", "periodic", "periodic", "periodic", "periodic"))
    d27 = W.perturbed(W.channel_sphere(shape=(8, 7, 10), center=(3, 3, 0), radius=2.5,
                                       lattice=27), seed=38)
    d27 = dataclasses.replace(
        d27, name="D3Q27 CM channel periodic-z 8x7x10 + sphere across the wrap",
        face_flow=("periodic", "periodic", "wall", "wall", "periodic", "periodic"),
        g_body=(1e-4, 0.0, 2e-5))
    return [W.random_periodic(shape=(7, 6, 11), seed=34),
            W.random_periodic(shape=(7, 6, 11), seed=35, collision="bgk"),
            W.random_periodic(shape=(7, 6, 9), seed=39, lattice=27), d27,
            ring, rb, dataclasses.replace(c3, collision="bgk"), c2, c2p,
            W.random_periodic(shape=(9, 10, 1), seed=36, lattice=9)]


def outer_walls_case(shape=(12, 7, 11), seed=37):
    """Walls and Dirichlet faces only at the ends of the outer axis, periodic elsewhere, no
    solid: as slabs, the end ones run the masked kernels and the inner ones do not."""
    c = W.perturbed(W.cavity3d(shape=shape), seed=seed)
    return dataclasses.replace(
        c, name=f"D3Q19 MRT + D3Q7 walls on z only {shape[0]}x{shape[1]}x{shape[2]}",
        face_flow=("periodic",) * 4 + ("wall", "wall"), gbeta=0.01,
        face_T=("adiabatic",) * 4 + ("dirichlet", "dirichlet"),
        T_wall=(0.0, 0.0, 0.0, 0.0, 0.4, -0.3))


def faces_only_cases(large=False):
    """Walled problems without solid cells or immersed-boundary samples: their AA step
    kernels compute the link mask of every cell from the coordinates.  large: sizes that
    span several thread blocks along x with ragged tails (for the GPU)."""
    s3, s2, s27, sz = (((70, 40, 37), (300, 181, 1), (66, 20, 18), (64, 20, 24)) if large
                       else ((9, 7, 6), (10, 8, 1), (8, 6, 7), (7, 6, 9)))
    c3 = W.perturbed(W.cavity3d(shape=s3), seed=51)
    c2 = dataclasses.replace(W.perturbed(W.cavity2d(shape=s2), seed=52), gbeta=0.01)
    c2y = dataclasses.replace(
        c2, name=c2.name + ", walls and Dirichlet faces on y only",
        face_flow=("periodic", "periodic", "wall", "wall", "periodic", "periodic"),
        face_T=("adiabatic", "adiabatic", "dirichlet", "dirichlet", "adiabatic", "adiabatic"),
        T_wall=(0.0, 0.0, 0.3, -0.2, 0.0, 0.0))
    q27 = W.random_periodic(shape=s27, seed=53, lattice=27, nu=0.05)
    q27 = dataclasses.replace(q27, name=f"D3Q27 CM box {s27[0]}x{s27[1]}x{s27[2]}, walls",
                              face_flow=("wall",) * 6, g_body=(1e-4, -2e-5, 3e-5))
    return [c3, c2, c2y, q27, outer_walls_case(shape=sz, seed=54)]


def box_edge_cases():
    """Solid cells against the faces: a block across the periodic x faces (its widened box
    wraps, so the whole x axis is inside), a block on a wall face (the box is clipped), one
    solid cell in a corner of a periodic box, and a 2-D cavity with a solid strip along a
    Dirichlet wall."""
    ch = W.perturbed(W.channel_sphere(shape=(11, 9, 8), center=(5, 4, 4), radius=0.0), seed=61)
    sol = np.zeros(ch.grid, np.uint8)
    sol[3:5, 2:4, 0] = 1          # z, y, x = 0: across the periodic x faces
    sol[0, 5:7, 6:8] = 1          # on the z = 0 wall
    a = dataclasses.replace(ch, solid=sol, name="channel, solids on a periodic face and a wall")
    rp = W.random_periodic(shape=(7, 6, 5), seed=62)
    sol = np.zeros(rp.grid, np.uint8)
    sol[0, 0, 0] = 1
    b = dataclasses.replace(rp, solid=sol, name="periodic box, one solid corner cell")
    c2 = W.perturbed(W.cavity2d(shape=(12, 9, 1)), seed=63)
    sol = np.zeros(c2.grid, np.uint8)
    sol[0, 3:6, 0] = 1            # along the hot x = 0 wall
    c = dataclasses.replace(c2, solid=sol, gbeta=0.01, name="2-D cavity, solid strip on a wall")
    return [a, b, c]


def with_zero_solid_array(w):
    """The same problem with an all-zero solid array instead of none."""
    return dataclasses.replace(w, solid=np.zeros(w.grid, np.uint8),
                               name=w.name + " (zero solid array)")


def emulate_loaded_mask(emu_lib, w, steps):
    """emulate() with the link mask loaded for every cell in the AA steps, instead of
    computed from the coordinates outside the solid cells' box as the kernels do."""
    emu_lib.emu_set_loaded_mask(1)
    try:
        return emulate(emu_lib, w, steps)
    finally:
        emu_lib.emu_set_loaded_mask(0)


def degenerate_cases():
    """Grids of extent 1 or 2 along some axes (every neighbour is the cell itself or its one
    neighbour, through a wrap or a wall), on every lattice."""
    out = []
    for shape in ((1, 1, 1), (1, 2, 3), (3, 1, 2), (2, 3, 1)):
        out.append(W.random_periodic(shape=shape, seed=50 + sum(shape)))
        walled = W.perturbed(W.cavity3d(shape=shape), seed=60 + sum(shape))
        out.append(dataclasses.replace(walled, name=walled.name + f" {shape}", gbeta=0.02))
    for shape in ((1, 1, 1), (1, 5, 1), (4, 1, 1)):
        out.append(W.random_periodic(shape=shape, seed=70 + sum(shape), lattice=9))
        c2 = W.perturbed(W.cavity2d(shape=shape), seed=80 + sum(shape))
        out.append(dataclasses.replace(c2, name=c2.name + f" {shape}", gbeta=0.02))
    for shape in ((1, 1, 1), (2, 1, 3)):
        out.append(W.random_periodic(shape=shape, seed=90 + sum(shape), lattice=27))
        ch = W.perturbed(W.channel_sphere(shape=shape, center=(0, 0, 0), radius=0.0,
                                          lattice=27), seed=95 + sum(shape))
        out.append(dataclasses.replace(ch, name=ch.name + f" {shape}", solid=None,
                                       g_body=(1e-3, 0.0, 0.0)))
    return out


def small_cases():
    """Small problems covering every lattice, collision, boundary kind and forcing."""
    cases = [W.random_periodic(shape=(6, 5, 4), seed=1),
             W.random_periodic(shape=(6, 5, 4), seed=1, collision="bgk"),
             W.random_periodic(shape=(7, 5, 1), seed=2, lattice=9),
             W.taylor_green(n=8)]
    cs = W.perturbed(W.channel_sphere(shape=(12, 10, 9), center=(5, 4, 4), radius=2.5), seed=3)
    cases.append(dataclasses.replace(cs, g_body=(1e-4, 2e-5, -1e-5)))
    c3 = W.perturbed(W.cavity3d(shape=(9, 7, 6)), seed=4)
    sol = np.zeros(c3.grid, np.uint8)
    sol[2:4, 3:5, 4:6] = 1
    cases.append(dataclasses.replace(c3, solid=sol, gbeta=0.01))
    cases.append(dataclasses.replace(c3, collision="bgk", gbeta=0.02, up_axis=0))
    c2 = dataclasses.replace(W.perturbed(W.cavity2d(shape=(10, 8, 1)), seed=5), gbeta=0.01)
    cases.append(c2)
    ibs = W.channel_ib_sphere(shape=(14, 12, 11), center=(6.3, 5.7, 5.2), radius=2.6,
                              gx=1e-4, samples_per_area=2.0)
    cases.append(dataclasses.replace(W.perturbed(ibs, seed=6), name=ibs.name + " perturbed"))
    ib2 = W.perturbed(W.cavity2d(shape=(12, 10, 1)), seed=8)
    x2 = np.array([[3.3, 4.1, 0.0], [5.7, 2.2, 0.0], [7.1, 6.6, 0.0], [9.4, 5.0, 0.0]],
                  np.float32)
    cases.append(dataclasses.replace(ib2, name=ib2.name + " + IB", gbeta=0.01, ib_x=x2,
                                     ib_ub=np.full((4, 3), 0.01, np.float32),
                                     ib_w=np.array([1.0, 0.5, 0.8, 1.2], np.float32)))
    cases.append(dataclasses.replace(
        c2, face_flow=("periodic", "periodic", "wall", "wall", "periodic", "periodic"),
        face_T=("adiabatic", "adiabatic", "dirichlet", "dirichlet", "adiabatic", "adiabatic"),
        T_wall=(0.0, 0.0, 0.3, -0.2, 0.0, 0.0)))
    cases += d3q27_cases()
    return cases


def d3q27_cases():
    """D3Q27 central moments: periodic, periodic with a distinct rate per moment group, and a
    forced channel (walls in y, z) around a solid sphere."""
    rp = W.random_periodic(shape=(6, 5, 4), seed=11, lattice=27, nu=0.05)
    distinct = dataclasses.replace(
        W.random_periodic(shape=(5, 6, 7), seed=12, lattice=27, nu=0.08),
        name="D3Q27 CM periodic 5x6x7, distinct rates",
        rates={"bulk": 1.1, "r3": 1.3, "r4": 1.5, "r5": 1.7, "r6": 0.9},
        g_body=(2e-4, -1e-4, 5e-5))
    ch = W.perturbed(W.channel_sphere(shape=(12, 10, 9), center=(5, 4, 4), radius=2.5,
                                      lattice=27), seed=13)
    ch = dataclasses.replace(ch, g_body=(1e-4, 2e-5, -1e-5))
    ib = W.channel_ib_sphere(shape=(14, 12, 11), center=(6.3, 5.7, 5.2), radius=2.6,
                             gx=1e-4, samples_per_area=2.0, lattice=27)
    ib = dataclasses.replace(W.perturbed(ib, seed=14), name=ib.name + " perturbed")
    return [rp, distinct, ch, ib]


def split_steps(n):
    """Uneven chunks so that parity is carried across lbm_step calls (97 + 103 = 200)."""
    out = []
    while n > 0:
        c = min(n, 97 if not out else 103)
        out.append(c)
        n -= c
    return out


def gpu_states(w, checkpoints, window_fn=None, edit=None, streaming="aa"):
    """{steps: dict} of the CUDA path's results (numpy), stepping in uneven chunks."""
    import torch
    from lattice_boltzmann_cfd_gb300 import Simulation
    sim = Simulation(w, edit=edit, streaming=streaming)
    dev = sim.device
    T = torch.from_numpy(np.ascontiguousarray(w.T_init)).to(dev) if w.thermal else None
    sim.init_equilibrium(torch.from_numpy(np.ascontiguousarray(w.rho0)).to(dev),
                         torch.from_numpy(np.ascontiguousarray(w.u0)).to(dev), T)
    out, done = {}, 0
    for n in sorted(checkpoints):
        for c in split_steps(n - done):
            sim.step(c)
        done = n
        rho, u, Tt = sim.macroscopic()
        f, g = sim.populations()
        r = dict(rho=rho, u=u, T=Tt, f=f, g=g)
        if window_fn is None:
            r = {k: (None if v is None else v.cpu().numpy()) for k, v in r.items()}
        else:
            r = window_fn(r)
        r["diag"] = sim.diagnostics(allow_nonfinite=True)
        r["parity"] = sim.parity
        out[n] = r
    torch.cuda.synchronize()
    sim.close()
    return out


def compare_fields(w, got, ref, tol=TOL_FIELDS, pop_tol=None):
    """Max-abs differences over fluid cells; asserts within tolerance."""
    fluid = fluid_of(w)
    errs = {"rho": np.abs(got["rho"] - ref["rho"])[fluid].max(),
            "u": np.abs(got["u"] - ref["u"])[:, fluid].max(),
            "f": np.abs(got["f"] - ref["f"])[:, fluid].max()}
    if w.thermal:
        errs["T"] = np.abs(got["T"] - ref["T"])[fluid].max()
        errs["g"] = np.abs(got["g"] - ref["g"])[:, fluid].max()
    pop_tol = tol if pop_tol is None else pop_tol
    for k, e in errs.items():
        lim = pop_tol if k in ("f", "g") else tol
        assert e <= lim, f"{w.name}: {k} max-abs {e:.3e} > {lim:.1e}"
    return errs
