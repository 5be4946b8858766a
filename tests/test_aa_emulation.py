"""Host emulation of the CUDA path's steps (in-place AA, two-buffer PULL and SPLIT)
against the oracle (CPU).

The library's own per-cell functions run on the CPU with each step written into a
NaN-filled second buffer, so a slot read after another cell overwrote it, a slot written
twice or a slot left unwritten would show up as a stale or NaN value.  Matching the
two-buffer oracle at both parities therefore checks that every cell writes exactly the
slots it reads, that wall links redirect correctly and that the logical read-out is
parity-aware.  The link mask is compared bit for bit with a brute-force builder."""
import numpy as np
import pytest

from parity_util import (box_edge_cases, degenerate_cases, emulate, emulate_blocks,
                         emulate_loaded_mask, emulate_slabs, faces_only_cases, fluid_of, mask_brute_force,
                         oracle_states, outer_walls_case, slab_cases, small_cases)

CASES = small_cases()


@pytest.mark.parametrize("mode,narrow", [("aa", True), ("aa", False), ("pull", True),
                                         ("pull", False), ("split", True)],
                         ids=["aa-idx32", "aa-idx64", "pull-idx32", "pull-idx64", "split-idx32"])
@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_emulated_step_matches_oracle(oracle_mod, emu_lib, w, mode, narrow):
    if w.lattice == 27 and mode != "aa":
        pytest.skip("D3Q27 runs the AA layout only")
    ref = oracle_states(oracle_mod, w, [1, 2, 5, 6])
    fluid = fluid_of(w)
    for n, r in ref.items():
        f, g, _ = emulate(emu_lib, w, n, narrow, mode)
        assert not np.isnan(f[:, fluid]).any()
        assert np.abs(f - r["f"])[:, fluid].max() < 1e-6, n
        if w.thermal:
            assert np.abs(g - r["g"])[:, fluid].max() < 1e-6, n


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_link_mask_bit_exact(emu_lib, w):
    _, _, m = emulate(emu_lib, w, 0)
    if w.solid is None and all(k == "periodic" for k in w.face_flow[:2 * w.dim]):
        assert not m.any()
    else:
        assert np.array_equal(m, mask_brute_force(w))


@pytest.mark.parametrize("lattice,shape", [(19, (1, 1, 1)), (19, (2, 3, 1)), (19, (33, 7, 5)),
                                           (9, (1, 1, 1)), (9, (65, 3, 1)), (19, (4, 4, 4)),
                                           (27, (1, 1, 1)), (27, (3, 5, 2)), (27, (33, 7, 5))])
def test_neighbour_indices_stay_in_grid(emu_lib, lattice, shape):
    """The wrapped neighbour offsets of the AA odd step always name a cell of the grid
    (checked for every cell and direction, both signs)."""
    import ctypes
    emu_lib.emu_count_bad_indices.restype = ctypes.c_longlong
    assert emu_lib.emu_count_bad_indices(lattice, *shape) == 0


@pytest.mark.parametrize("d", [1, 2, 3, 7, 9, 31, 33, 63, 65, 70, 255, 257, 258, 300, 1000,
                               4095, 4097, 65535, 65537, 1 << 20, (1 << 20) + 1,
                               (1 << 30) + 3, (1 << 31) - 1, 1 << 31])
def test_division_by_multiply_and_shift(emu_lib, d):
    """The step kernels' division by an invariant divisor (multiply, shift) equals the
    quotient for the numerators 0 .. 70000, and around every sampled multiple of d up to
    2^31 - 1."""
    import ctypes
    emu_lib.emu_divisor_errors.restype = ctypes.c_longlong
    emu_lib.emu_divisor_errors.argtypes = [ctypes.c_uint, ctypes.c_uint, ctypes.c_uint,
                                           ctypes.c_longlong]
    assert emu_lib.emu_divisor_errors(d, 0, 70000, 200000) == 0
    assert emu_lib.emu_divisor_errors(d, (1 << 31) - 70000, (1 << 31) - 1, 10) == 0


@pytest.mark.parametrize("dim,shape,lo,hi", [
    (3, (258, 7, 5), 0, 5), (3, (258, 7, 5), 2, 4), (3, (33, 1, 3), 0, 3), (3, (1, 1, 1), 0, 1),
    (3, (70, 40, 37), 1, 36), (2, (300, 181, 1), 0, 181), (2, (300, 181, 1), 179, 181),
    (2, (65, 3, 1), 1, 2)])
def test_linear_step_launch_covers_each_cell_once(emu_lib, dim, shape, lo, hi):
    """The 1-D step launch used when rows are not a multiple of 32 cells: thread t of the
    planes [lo, hi) is cell lo * plane + t in storage order, and the thread after the last
    cell is outside."""
    import ctypes
    emu_lib.emu_linear_mapping_errors.restype = ctypes.c_longlong
    assert emu_lib.emu_linear_mapping_errors(dim, *shape, lo, hi) == 0


# ------------------------------------------------------------- slab decomposition ---

SLAB_CASES = slab_cases() + [outer_walls_case()]


def _slab_counts(w):
    n = w.shape[w.dim - 1]
    return sorted({1, 2, 3, n})    # n: one owned plane per slab


@pytest.mark.parametrize("w", SLAB_CASES, ids=[c.name for c in SLAB_CASES])
def test_slabs_match_single_domain_bitwise(oracle_mod, emu_lib, w):
    """The domain run as slabs along its outer axis, with a FILL exchange after every even
    step and a DRAIN after every odd one, holds bit for bit the single domain's state at
    both parities.  Every step writes into a NaN-filled buffer, so a ghost slot the odd step
    reads but FILL did not supply, or a boundary slot DRAIN did not return, would surface
    as NaN.  The single domain itself is checked against the oracle."""
    fluid = fluid_of(w)
    ref = oracle_states(oracle_mod, w, [5])[5]
    for n in (1, 2, 5, 6):
        f1, g1, _ = emulate(emu_lib, w, n)
        if n == 5:
            assert np.abs(f1 - ref["f"])[:, fluid].max() < 1e-6
        for k in _slab_counts(w):
            fs, gs = emulate_slabs(emu_lib, w, n, k)
            assert not np.isnan(fs).any(), (n, k)
            assert np.array_equal(fs, f1), (n, k)
            if w.thermal:
                assert not np.isnan(gs).any(), (n, k)
                assert np.array_equal(gs, g1), (n, k)


# ------------------------------------------------------------ block decomposition ---

def _block_layouts(w):
    """Splits along two and three axes, with one-plane blocks and ragged ends."""
    if w.dim == 2:
        return [(2, 2, 1), (3, 2, 1), (w.shape[0], 1, 1), (2, w.shape[1], 1)]
    return [(2, 2, 1), (1, 2, 2), (2, 1, 3), (2, 2, 2), (3, 3, 2)]


@pytest.mark.parametrize("w", SLAB_CASES, ids=[c.name for c in SLAB_CASES])
def test_blocks_match_single_domain_bitwise(emu_lib, w):
    """The domain run as blocks split along several axes, exchanging axis by axis (z, y, x)
    after every step, through buffers or with the buffer-free swap, holds bit for bit the
    single domain's state at both parities.  The
    links that cross a block's edge or corner go to the diagonal neighbour through the ghost
    rows of the axis exchanged before, so a missing hop would leave a NaN or a stale value
    at the cells along the edges."""
    for n in (1, 2, 5, 6):
        f1, g1, _ = emulate(emu_lib, w, n)
        for nb in _block_layouts(w):
            for swap in (False, True):
                fb, gb = emulate_blocks(emu_lib, w, n, nb, swap=swap)
                assert not np.isnan(fb).any(), (n, nb, swap)
                assert np.array_equal(fb, f1), (n, nb, swap)
                if w.thermal:
                    assert not np.isnan(gb).any(), (n, nb, swap)
                    assert np.array_equal(gb, g1), (n, nb, swap)


def test_blocks_along_the_slab_axis_equal_slabs(emu_lib):
    """Blocks split along the outer axis only are slabs: both runners agree bit for bit."""
    w = SLAB_CASES[0]
    for n in (3, 4):
        fs, _ = emulate_slabs(emu_lib, w, n, 3)
        fb, _ = emulate_blocks(emu_lib, w, n, (1, 1, 3))
        assert np.array_equal(fs, fb)


@pytest.mark.parametrize("w", [SLAB_CASES[0], SLAB_CASES[5], SLAB_CASES[7]],
                         ids=["periodic", "cavity3d-solid", "cavity2d"])
def test_blocks_catch_a_missing_diagonal_hop(emu_lib, w):
    """Negative control: packing every axis before any unpack drops the second hop of the
    diagonal links, and the state differs from the single domain, but only next to the
    block edges (the cells off them still agree)."""
    nb = (2, 2, 1) if w.dim == 2 else (1, 2, 2)
    f1, _, _ = emulate(emu_lib, w, 2)
    fb, _ = emulate_blocks(emu_lib, w, 2, nb, ordered=False)
    bad = ~(fb == f1).all(axis=0)          # per cell (z, y, x)
    assert bad.any()
    # the split axes' block boundaries, as (array axis, planes next to a boundary)
    from lattice_boltzmann_cfd_gb300.slabs import split_ranges
    near = np.zeros(w.grid, bool)
    for a in range(3):
        if nb[a] < 2:
            continue
        ax = 2 - a
        r = split_ranges(w.shape[a], nb[a])
        cuts = [x[0] for x in r] + [r[-1][1]]
        planes = {(c + d) % w.shape[a] for c in cuts for d in (-2, -1, 0, 1)}
        idx = [slice(None)] * near.ndim
        idx[ax] = sorted(planes)
        m = np.zeros(w.grid, bool)
        m[tuple(idx)] = True
        near |= m
    assert not (bad & ~near).any()


DEGENERATE = degenerate_cases()


@pytest.mark.parametrize("mode", ["aa", "pull", "split"])
@pytest.mark.parametrize("w", DEGENERATE, ids=[c.name for c in DEGENERATE])
def test_degenerate_grids(oracle_mod, emu_lib, w, mode):
    """Extents of 1 or 2: the wrapped or walled neighbour is the cell itself or its twin."""
    if w.lattice == 27 and mode != "aa":
        pytest.skip("D3Q27 runs the AA layout only")
    ref = oracle_states(oracle_mod, w, [1, 2, 5, 6])
    fluid = fluid_of(w)
    for n, r in ref.items():
        f, g, m = emulate(emu_lib, w, n, True, mode)
        assert np.abs(f - r["f"])[:, fluid].max() < 1e-6, n
        if w.thermal:
            assert np.abs(g - r["g"])[:, fluid].max() < 1e-6, n
    assert np.array_equal(emulate(emu_lib, w, 0)[2], mask_brute_force(w))


WALLED = faces_only_cases() + [c for c in small_cases() + slab_cases()
                               if c.solid is not None and getattr(c, "ib_x", None) is None]


@pytest.mark.parametrize("w", WALLED, ids=[c.name for c in WALLED])
def test_mask_from_coordinates_equals_loaded_mask(oracle_mod, emu_lib, w):
    """The AA step with the link mask computed from the coordinates outside the solid cells'
    box (as the kernels run it) and with the mask loaded for every cell are bit-identical at
    both parities, and match the oracle.  (The emulation also checks, at every cell off a
    ghost plane, that the computed mask equals the built one.)"""
    fluid = fluid_of(w)
    ref = oracle_states(oracle_mod, w, [5, 6])
    for n in (5, 6):
        f1, g1, m1 = emulate(emu_lib, w, n)
        f2, g2, m2 = emulate_loaded_mask(emu_lib, w, n)
        assert np.array_equal(m1, m2)
        assert np.array_equal(f1, f2), n
        assert np.array_equal(g1, g2), n
        assert np.abs(f1 - ref[n]["f"])[:, fluid].max() < 1e-6, n
        if w.thermal:
            assert np.abs(g1 - ref[n]["g"])[:, fluid].max() < 1e-6, n


BOX_EDGES = box_edge_cases()


@pytest.mark.parametrize("w", BOX_EDGES, ids=[c.name for c in BOX_EDGES])
def test_solid_box_at_the_faces(oracle_mod, emu_lib, w):
    """The box around solids that touch a periodic face or a wall: the computed masks equal
    the built ones (checked inside the emulation at every cell), the step equals the
    loaded-mask step bit for bit, and both match the oracle."""
    fluid = fluid_of(w)
    ref = oracle_states(oracle_mod, w, [3, 4])
    for n in (3, 4):
        f1, g1, _ = emulate(emu_lib, w, n)
        f2, g2, _ = emulate_loaded_mask(emu_lib, w, n)
        assert np.array_equal(f1, f2) and np.array_equal(g1, g2), n
        assert np.abs(f1 - ref[n]["f"])[:, fluid].max() < 1e-6, n
        if w.thermal:
            assert np.abs(g1 - ref[n]["g"])[:, fluid].max() < 1e-6, n


def _race_cases():
    """Tiny grids for the brute-force read/write-set check: every lattice and boundary
    kind, solids, slab ghost planes and a degenerate extent."""
    import dataclasses
    from lattice_boltzmann_cfd_gb300 import workloads as W
    rp = W.random_periodic(shape=(4, 4, 4), seed=71)
    bgk2 = W.random_periodic(shape=(3, 4, 1), seed=72, collision="bgk", lattice=9)
    c3 = W.perturbed(W.cavity3d(shape=(5, 4, 3)), seed=73)
    sol = np.zeros(c3.grid, np.uint8)
    sol[1, 2, 2] = 1
    c3 = dataclasses.replace(c3, solid=sol, gbeta=0.01, name=c3.name + " + solid cell")
    c2 = W.perturbed(W.cavity2d(shape=(5, 4, 1)), seed=74)
    sol = np.zeros(c2.grid, np.uint8)
    sol[0, 1, 3] = 1
    c2 = dataclasses.replace(c2, solid=sol, gbeta=0.01, name=c2.name + " + solid cell")
    q27 = W.perturbed(W.channel_sphere(shape=(4, 4, 4), center=(1, 2, 2), radius=0.0,
                                       lattice=27), seed=75)
    halo = dataclasses.replace(W.random_periodic(shape=(4, 3, 5), seed=76),
                               face_flow=("periodic",) * 4 + ("halo", "halo"),
                               name="D3Q19 slab 4x3x5 with ghost planes")
    thin = dataclasses.replace(W.perturbed(W.cavity3d(shape=(1, 2, 3)), seed=77), gbeta=0.02,
                               name="cavity 1x2x3")
    return [rp, bgk2, c3, c2, q27, halo, outer_walls_case(shape=(4, 3, 5), seed=78), thin]


RACE = _race_cases()


@pytest.mark.parametrize("odd", [0, 1], ids=["even", "odd"])
@pytest.mark.parametrize("w", RACE, ids=[c.name for c in RACE])
def test_aa_step_reads_and_writes_the_same_slots(emu_lib, w, odd):
    """Race-freedom of the in-place step, by brute force over every slot: each cell writes
    exactly the slots whose values it uses, and no slot is written by two cells."""
    import ctypes
    from lattice_boltzmann_cfd_gb300.solver import make_config
    cfg, keep = make_config(w, "aa")
    emu_lib.emu_race_violations.restype = ctypes.c_longlong
    assert emu_lib.emu_race_violations(ctypes.byref(cfg), odd) == 0


def _overlap_cases():
    """Slabs with HALO faces (both ends, or one end next to a wall) on every lattice, with
    walls, solids next to the slab faces and thermal Dirichlet faces."""
    import dataclasses
    from lattice_boltzmann_cfd_gb300 import workloads as W
    from lattice_boltzmann_cfd_gb300.slabs import slab_part
    rp = W.random_periodic(shape=(4, 3, 12), seed=81)
    c3 = W.perturbed(W.cavity3d(shape=(4, 3, 12)), seed=82)
    sol = np.zeros(c3.grid, np.uint8)
    sol[4, 1, 1] = 1     # next to the second slab's low boundary plane
    sol[7, 2, 2] = 1
    c3 = dataclasses.replace(c3, solid=sol, gbeta=0.01, name=c3.name + " + solids")
    rb = dataclasses.replace(c3, face_T=("adiabatic",) * 4 + ("dirichlet", "dirichlet"),
                             T_wall=(0.0, 0.0, 0.0, 0.0, 0.4, -0.3), name="Rayleigh-Benard")
    c2 = W.perturbed(W.cavity2d(shape=(5, 13, 1)), seed=83)
    q27 = W.random_periodic(shape=(3, 3, 12), seed=84, lattice=27)
    out = []
    for w in (rp, c3, rb, c2, q27):
        for r in range(2):
            local, sides, planes = slab_part(w, 2, r)
            out.append((f"{w.name} slab {r} of 2", local, sides))
    return out


OVERLAP = _overlap_cases()


@pytest.mark.parametrize("next_odd", [1, 0], ids=["FILL then odd", "DRAIN then even"])
@pytest.mark.parametrize("case", OVERLAP, ids=[c[0] for c in OVERLAP])
def test_exchange_overlaps_the_interior_without_races(emu_lib, case, next_odd):
    """The overlapped slab order runs a step's halo exchange beside the next step's launch
    over the interior planes.  By brute force over slots: no interior cell reads or writes a
    slot the pack reads or the unpack writes.  Widening the launch by the first owned plane
    next to a HALO face does produce such pairs, so the check is not vacuous."""
    import ctypes
    from lattice_boltzmann_cfd_gb300.slabs import plane_groups
    from lattice_boltzmann_cfd_gb300.solver import make_config
    name, local, (low, high) = case
    cfg, keep = make_config(local, "aa")
    n = local.shape[local.dim - 1]
    interior, boundary = plane_groups(n, low, high)
    assert len(interior) == 1
    (ilo, ihi), = interior
    emu_lib.emu_overlap_violations.restype = ctypes.c_longlong
    assert emu_lib.emu_overlap_violations(ctypes.byref(cfg), next_odd, ilo, ihi) == 0
    wider = (ilo - 1, ihi) if low else (ilo, ihi + 1)
    assert emu_lib.emu_overlap_violations(ctypes.byref(cfg), next_odd, *wider) > 0


def test_plane_groups_cover_each_plane_once():
    from lattice_boltzmann_cfd_gb300.slabs import plane_groups
    for n in range(1, 12):
        for low in (False, True):
            for high in (False, True):
                interior, boundary = plane_groups(n, low, high)
                covered = [k for lo, hi in interior + boundary for k in range(lo, hi)]
                assert sorted(covered) == list(range(n)), (n, low, high)
                for lo, hi in interior:
                    assert lo >= (2 if low else 0) and hi <= (n - 2 if high else n)



def _block_overlap_cases():
    """Blocks with HALO faces on two or three axes (ghost rows meeting at edges and corners),
    on every lattice, with walls, solids next to the block faces and Dirichlet faces."""
    import dataclasses
    from lattice_boltzmann_cfd_gb300 import workloads as W
    from lattice_boltzmann_cfd_gb300.blocks import block_part
    rp = W.random_periodic(shape=(10, 10, 10), seed=91)
    c3 = W.perturbed(W.cavity3d(shape=(10, 10, 10)), seed=92)
    sol = np.zeros(c3.grid, np.uint8)
    sol[4, 5, 4] = 1     # next to the blocks' faces at z = 5 and y = 5
    sol[6, 4, 6] = 1
    c3 = dataclasses.replace(c3, solid=sol, gbeta=0.01, name=c3.name + " + solids")
    c2 = W.perturbed(W.cavity2d(shape=(10, 11, 1)), seed=93)
    q27 = W.random_periodic(shape=(9, 9, 9), seed=94, lattice=27)
    out = []
    for w, nb, blocks in ((rp, (1, 2, 2), (0, 3)), (rp, (2, 2, 2), (0, 7)), (c3, (2, 2, 2), (0, 5)),
                          (c2, (2, 2, 1), (0, 3)), (q27, (2, 2, 2), (0, 6))):
        for b in blocks:
            local, sides, coords = block_part(w, nb, b)
            out.append((f"{w.name} block {b} of {nb}", local, sides))
    return out


BLOCK_OVERLAP = _block_overlap_cases()


@pytest.mark.parametrize("next_odd", [1, 0], ids=["FILL then odd", "DRAIN then even"])
@pytest.mark.parametrize("case", BLOCK_OVERLAP, ids=[c[0] for c in BLOCK_OVERLAP])
def test_block_exchange_overlaps_the_interior_without_races(emu_lib, case, next_odd):
    """The overlapped block order runs a step's exchange (every HALO face of every axis)
    beside the next step's launch over the interior box.  By brute force over slots: no
    interior cell reads or writes a slot a pack reads or an unpack writes.  Widening the box
    by one plane towards any HALO face produces such pairs."""
    import ctypes
    from lattice_boltzmann_cfd_gb300.blocks import block_groups
    from lattice_boltzmann_cfd_gb300.solver import make_config
    name, local, sides = case
    cfg, keep = make_config(local, "aa")
    (lo, hi), boundary = block_groups(local.shape, sides, local.dim)
    f = emu_lib.emu_box_overlap_violations
    f.restype = ctypes.c_longlong
    box = lambda v: (ctypes.c_int * 3)(*v)
    assert f(ctypes.byref(cfg), next_odd, box(lo), box(hi)) == 0
    for a in range(local.dim):
        for s in (0, 1):
            if not sides[a][s]:
                continue
            wlo, whi = list(lo), list(hi)
            if s == 0:
                wlo[a] -= 1
            else:
                whi[a] += 1
            assert f(ctypes.byref(cfg), next_odd, box(wlo), box(whi)) > 0, (a, s)


def test_block_groups_cover_each_cell_once():
    import itertools
    from lattice_boltzmann_cfd_gb300.blocks import block_groups
    for dim in (2, 3):
        for ext in ((7, 6, 5), (4, 9, 6), (3, 3, 3), (8, 5, 1)):
            ext = ext if dim == 3 else (ext[0], ext[1], 1)
            for flags in itertools.product((False, True), repeat=2 * dim):
                sides = [(flags[2 * a], flags[2 * a + 1]) if a < dim else (False, False)
                         for a in range(3)]
                interior, boundary = block_groups(ext, sides, dim)
                seen = np.zeros(ext[::-1], int)
                for lo, hi in ([interior] if interior else []) + boundary:
                    seen[lo[2]:hi[2], lo[1]:hi[1], lo[0]:hi[0]] += 1
                assert (seen == 1).all(), (ext, sides)
                if interior:
                    lo, hi = interior
                    for a in range(dim):
                        assert lo[a] >= (2 if sides[a][0] else 0)
                        assert hi[a] <= ext[a] - (2 if sides[a][1] else 0)
