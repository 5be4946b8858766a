"""Block partitioning (the domain cut along several axes) with the per-axis halo exchange,
on the GPU through the C ABI.

The blocks together must hold bit for bit the state of one domain run with the same kernels,
at both AA parities, and match the fp64 oracle run on the undivided domain.  A block whose
faces are all HALO or periodic and which holds no solid cell runs the unmasked kernels even
when the undivided domain (which has walls) runs the masked ones; where that mixes the two
kernel families the comparison with the undivided domain is within fp32 rounding instead
of bitwise (the oracle comparison is the same either way).
"""
import dataclasses
import datetime
import os
import socket

import numpy as np
import pytest

from lattice_boltzmann_cfd_gb300 import capi
from lattice_boltzmann_cfd_gb300 import workloads as W
from parity_util import TOL_FIELDS, compare_fields, oracle_states, outer_walls_case, slab_cases

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    capi.load()


def _dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _single(w, steps):
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    sim = Simulation(w)
    sim.init_equilibrium(_dev(w.rho0), _dev(w.u0), _dev(w.T_init))
    sim.step(steps)
    f, g = sim.populations()
    out = (f.cpu().numpy(), None if g is None else g.cpu().numpy(), sim.diagnostics())
    sim.close()
    return out


def _masked(w):
    return any(k == "wall" for k in w.face_flow[:2 * w.dim]) or (
        w.solid is not None and bool(w.solid.any()))


def _same_family(w, nb):
    """Every block runs the kernel family of the undivided domain."""
    from lattice_boltzmann_cfd_gb300.blocks import block_part
    want = _masked(w)
    return all(_masked(block_part(w, nb, b)[0]) == want for b in range(nb[0] * nb[1] * nb[2]))


def _blocks(w, nb, chunks, exchange="auto"):
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    dom = BlockDomain(w, nb, exchange=exchange)
    dom.init_equilibrium()
    for c in chunks:
        dom.step(c)
    f, g = dom.populations()
    rho, u, T = dom.macroscopic()
    got = {"rho": rho.cpu().numpy(), "u": u.cpu().numpy(),
           "T": None if T is None else T.cpu().numpy(), "f": f.cpu().numpy(),
           "g": None if g is None else g.cpu().numpy()}
    d = dom.diagnostics()
    dom.close()
    return got, d


def _large_cases():
    """Grids spanning several thread blocks along x with ragged tails."""
    rp = W.random_periodic(shape=(300, 20, 23), seed=81)
    cs = W.perturbed(W.channel_sphere(shape=(150, 24, 22), center=(40, 12, 11), radius=6,
                                      gx=1e-5), seed=82)
    cs = dataclasses.replace(cs, name=cs.name + " perturbed")
    c3 = W.perturbed(W.cavity3d(shape=(70, 40, 37)), seed=83)
    c2 = W.perturbed(W.cavity2d(shape=(300, 181, 1)), seed=84)
    return [rp, cs, c3, c2]


CASES = slab_cases() + [outer_walls_case()] + _large_cases()


def _layouts(w):
    if w.dim == 2:
        return [(2, 2, 1), (3, 2, 1), (2, 3, 1)]
    return [(2, 2, 1), (1, 2, 2), (2, 2, 2), (3, 2, 2)]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_blocks_equal_single_domain(oracle_mod, w):
    """Each block layout, exchanged with the buffer-free swap (and one layout through
    buffers), against the undivided domain (bitwise where the kernel families agree) and the
    fp64 oracle (1e-6 on the populations, 2e-5 on rho, u, T), at 7 and 8 steps; the summed
    diagnostics agree with the undivided domain's."""
    ref = oracle_states(oracle_mod, w, [7, 8])
    for steps in (7, 8):
        f1, g1, d1 = _single(w, steps)
        runs = [(nb, "swap") for nb in _layouts(w)] + [(_layouts(w)[-1], "buffers")]
        for nb, exchange in runs:
            got, ds = _blocks(w, nb, [3, steps - 3], exchange)
            compare_fields(w, got, ref[steps], tol=TOL_FIELDS, pop_tol=1e-6)
            if _same_family(w, nb):
                assert np.array_equal(got["f"], f1), (steps, nb)
                if w.thermal:
                    assert np.array_equal(got["g"], g1), (steps, nb)
            else:
                assert np.abs(got["f"] - f1).max() < 1e-6, (steps, nb)
                if w.thermal:
                    assert np.abs(got["g"] - g1).max() < 1e-6, (steps, nb)
            assert ds["fluid_cells"] == d1["fluid_cells"]
            assert ds["finite"]
            assert abs(ds["mass"] - d1["mass"]) <= 1e-9 * abs(d1["mass"])
            cells = d1["fluid_cells"]
            assert np.allclose(ds["momentum"], d1["momentum"], rtol=0, atol=1e-7 * cells)
            fscale = max(1e-30, float(np.abs(d1["force"]).max()))
            assert np.allclose(ds["force"], d1["force"], rtol=0, atol=1e-5 * fscale)
            if w.thermal:
                hscale = max(1e-30, float(np.abs(d1["heat"]).max()))
                assert np.allclose(ds["heat"], d1["heat"], rtol=0, atol=1e-6 * hscale)
                # the Nusselt numbers, recomputed from the parts' sums with the whole
                # domain's extents, against the library's own on the undivided domain
                assert np.allclose(ds["uT"], d1["uT"], rtol=0, atol=1e-7 * cells)
                for key in ("nu_hot", "nu_cold"):
                    assert abs(ds[key] - d1[key]) <= 1e-5 * max(1.0, abs(d1[key])), key
                assert abs(ds["nu_volume"] - d1["nu_volume"]) <= 1e-3


@pytest.mark.parametrize("w,nb", [
    (W.perturbed(W.cavity3d(shape=(70, 40, 37)), seed=83), (2, 2, 2)),
    (W.perturbed(W.cavity2d(shape=(300, 181, 1)), seed=84), (2, 2, 1))],
    ids=["cavity3d 70x40x37 2x2x2", "cavity2d 300x181 2x2"])
def test_blocks_200_and_201_steps_against_the_oracle(oracle_mod, w, nb):
    """Blocks over 200 and 201 steps against the oracle on the undivided domain (2e-5 on the
    fields and populations, heat sums 1e-4 relative)."""
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    ref = oracle_states(oracle_mod, w, [200, 201])
    dom = BlockDomain(w, nb)
    dom.init_equilibrium()
    done = 0
    for n in (200, 201):
        dom.step(n - done)
        done = n
        f, g = dom.populations()
        rho, u, T = dom.macroscopic()
        got = {"rho": rho.cpu().numpy(), "u": u.cpu().numpy(), "T": T.cpu().numpy(),
               "f": f.cpu().numpy(), "g": g.cpu().numpy()}
        compare_fields(w, got, ref[n])
        assert np.allclose(dom.diagnostics()["heat"], ref[n]["diag"]["heat"], rtol=1e-4,
                           atol=1e-3)
    dom.close()


OVERLAP_CASES = [CASES[i] for i in (0, 3, 5, 7, 8)] + _large_cases()


@pytest.mark.parametrize("w", OVERLAP_CASES, ids=[c.name for c in OVERLAP_CASES])
def test_overlapped_blocks_equal_plain_order(w):
    """The overlapped block order (interior box, boundary boxes, the exchange of every axis on
    a second stream beside the next step's interior) gives the plain order's state bit for
    bit, through the swap and through buffers."""
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    for steps in (7, 8):
        for nb, exchange in [(nb, "swap") for nb in _layouts(w)] + [(_layouts(w)[0], "buffers")]:
            got = {}
            for overlap in (False, True):
                dom = BlockDomain(w, nb, exchange=exchange, overlap=overlap)
                dom.init_equilibrium()
                for c in (3, steps - 3):
                    dom.step(c)
                f, g = dom.populations()
                got[overlap] = (f.cpu().numpy(), None if g is None else g.cpu().numpy())
                dom.close()
            assert np.array_equal(got[True][0], got[False][0]), (steps, nb, exchange)
            if w.thermal:
                assert np.array_equal(got[True][1], got[False][1]), (steps, nb, exchange)


def test_step_box_equals_step():
    """lbm_step_box over any partition of the grid into boxes, in any order, is lbm_step(1)
    at both parities; a box that overlaps one already stepped is refused."""
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    cases = [W.perturbed(W.cavity3d(shape=(70, 20, 13)), seed=95),
             W.perturbed(W.cavity2d(shape=(100, 23, 1)), seed=96),
             W.random_periodic(shape=(40, 12, 11), seed=97, lattice=27),
             W.random_periodic(shape=(66, 10, 9), seed=98)]      # rows of 66: linear launch
    rng = np.random.default_rng(11)
    for w in cases:
        ext = list(w.shape)
        ref, sim = Simulation(w), Simulation(w)
        for s_ in (ref, sim):
            s_.init_equilibrium(_dev(w.rho0), _dev(w.u0), _dev(w.T_init))
        for step in range(4):
            ref.step(1)
            # cut every axis at random points: the product of the pieces tiles the grid
            cuts = []
            for a in range(3):
                k = min(2, ext[a] - 1)
                c = sorted(rng.choice(np.arange(1, ext[a]), size=k, replace=False)) if k else []
                edges = [0] + [int(v) for v in c] + [ext[a]]
                cuts.append(list(zip(edges[:-1], edges[1:])))
            boxes = [((x[0], y[0], z[0]), (x[1], y[1], z[1]))
                     for x in cuts[0] for y in cuts[1] for z in cuts[2]]
            rng.shuffle(boxes)
            for i, (lo, hi) in enumerate(boxes):
                sim.step_box(lo, hi)
                if i == 0 and len(boxes) > 1:
                    with pytest.raises(capi.LbmError) as e:
                        sim.step_box(lo, hi)                         # already stepped
                    assert e.value.status == capi.LBM_ERR_ARG
                    with pytest.raises(capi.LbmError) as e:
                        sim.step(1)
                    assert e.value.status == capi.LBM_ERR_STATE
            assert sim.parity == (step + 1) % 2
            fa, ga = ref.populations()
            fb, gb = sim.populations()
            assert torch.equal(fa, fb), (w.name, step)
            if w.thermal:
                assert torch.equal(ga, gb), (w.name, step)
        for lo, hi in (((0, 0, 0), (ext[0] + 1, ext[1], ext[2])), ((1, 0, 0), (1, ext[1], ext[2])),
                       ((-1, 0, 0), (2, 2, 1))):
            with pytest.raises(capi.LbmError):
                sim.step_box(lo, hi)
        ref.close()
        sim.close()
    # the box launches take neither the two-buffer layouts nor immersed-boundary capacity
    wp = W.random_periodic(shape=(16, 8, 6), seed=99)
    for kw in ({"streaming": "pull"}, {"edit": lambda cfg: setattr(cfg, "ib_max_samples", 4)}):
        s_ = Simulation(wp, **kw)
        s_.init_equilibrium(_dev(wp.rho0), _dev(wp.u0))
        with pytest.raises(capi.LbmError) as e:
            s_.step_box((0, 0, 0), (16, 8, 6))
        assert e.value.status == capi.LBM_ERR_UNSUPPORTED
        s_.close()


def test_axis_halo_calls_are_checked():
    """Per-axis halo calls: the plane size of each axis, only HALO sides, axes in range,
    the same parity rules as the outer-axis calls."""
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    w = W.random_periodic(shape=(16, 8, 10), seed=86)
    w = dataclasses.replace(w, face_flow=("halo", "halo", "wall", "halo", "periodic",
                                          "periodic"))
    sim = Simulation(w)
    assert capi.lbm_halo_axis_bytes(sim.ctx, 0) == 4 * 5 * 8 * 10
    assert capi.lbm_halo_axis_bytes(sim.ctx, 1) == 4 * 5 * 16 * 10
    assert capi.lbm_halo_axis_bytes(sim.ctx, 2) == 4 * 5 * 16 * 8
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_axis_bytes(sim.ctx, 3)
    buf = torch.empty(5 * 16 * 10, device="cuda")
    sim.init_equilibrium(_dev(w.rho0), _dev(w.u0))
    sim.step(1)
    capi.lbm_halo_axis_pack(sim.ctx, 0, 1, capi.LBM_HALO_FILL, buf)
    capi.lbm_halo_axis_pack(sim.ctx, 1, 1, capi.LBM_HALO_FILL, buf)
    for axis, side in ((1, 0), (2, 0), (2, 1), (3, 0), (-1, 0)):
        with pytest.raises(capi.LbmError):
            capi.lbm_halo_axis_pack(sim.ctx, axis, side, capi.LBM_HALO_FILL, buf)
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_axis_unpack(sim.ctx, 0, 0, capi.LBM_HALO_DRAIN, buf)   # parity 1
    sim.step(1)
    capi.lbm_halo_axis_unpack(sim.ctx, 0, 0, capi.LBM_HALO_DRAIN, buf)
    torch.cuda.synchronize()
    sim.close()


def test_swap_calls_are_checked():
    """lbm_halo_axis_swap: both faces HALO, the same step, lattices and face extents."""
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    base = W.random_periodic(shape=(16, 8, 10), seed=90)
    w = dataclasses.replace(base, face_flow=("periodic",) * 4 + ("halo", "halo"))
    a, b = Simulation(w), Simulation(w)
    wz = dataclasses.replace(w, shape=(16, 8, 7), rho0=w.rho0[:7], u0=w.u0[:, :7])
    c = Simulation(wz)                                   # another z extent: still one face
    wy = dataclasses.replace(w, shape=(16, 9, 10), rho0=np.ones((10, 9, 16), np.float32),
                             u0=np.zeros((3, 10, 9, 16), np.float32))
    d = Simulation(wy)                                   # another y extent: not the same face
    for sim, ww in ((a, w), (b, w), (c, wz), (d, wy)):
        sim.init_equilibrium(_dev(ww.rho0), _dev(ww.u0))
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_axis_swap(a.ctx, b.ctx, 2, capi.LBM_HALO_FILL)     # parity 0
    for sim in (a, b, c, d):
        sim.step(1)
    capi.lbm_halo_axis_swap(a.ctx, b.ctx, 2, capi.LBM_HALO_FILL)
    capi.lbm_halo_axis_swap(a.ctx, c.ctx, 2, capi.LBM_HALO_FILL)
    capi.lbm_halo_axis_swap(a.ctx, a.ctx, 2, capi.LBM_HALO_FILL)         # a ring of one
    for args in ((a.ctx, d.ctx, 2, capi.LBM_HALO_FILL),                  # faces differ
                 (a.ctx, b.ctx, 0, capi.LBM_HALO_FILL),                  # x is periodic
                 (a.ctx, b.ctx, 3, capi.LBM_HALO_FILL),
                 (a.ctx, b.ctx, 2, capi.LBM_HALO_DRAIN),                 # parity 1
                 (a.ctx, b.ctx, 2, 7)):
        with pytest.raises(capi.LbmError):
            capi.lbm_halo_axis_swap(*args)
    b.step(1)
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_axis_swap(a.ctx, b.ctx, 2, capi.LBM_HALO_FILL)     # not the same step
    a.step(1)
    capi.lbm_halo_axis_swap(a.ctx, b.ctx, 2, capi.LBM_HALO_DRAIN)
    torch.cuda.synchronize()
    for sim in (a, b, c, d):
        sim.close()


def test_batched_swaps_equal_one_swap_per_face(monkeypatch):
    """lbm_halo_axis_swap_many (every face of an axis in one launch) gives bit for bit the
    state of one lbm_halo_axis_swap per face, in 3-D (faces on two and three axes, a
    periodic ring of two blocks) and 2-D."""
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain

    def one_by_one(lo, hi, axis, phase):
        for a, b in zip(lo, hi):
            capi.lbm_halo_axis_swap(a, b, axis, phase)

    for w, nb in ((W.perturbed(W.cavity3d(shape=(40, 22, 18)), seed=101), (2, 2, 2)),
                  (W.random_periodic(shape=(30, 20, 16), seed=102), (1, 2, 4)),
                  (W.perturbed(W.cavity2d(shape=(70, 41, 1)), seed=103), (3, 2, 1))):
        got = []
        for batched in (True, False):
            with monkeypatch.context() as m:
                if not batched:
                    m.setattr(capi, "lbm_halo_axis_swap_many", one_by_one)
                dom = BlockDomain(w, nb)
                dom.init_equilibrium()
                dom.step(7)
                f, g = dom.populations()
                got.append((f.cpu().numpy(), None if g is None else g.cpu().numpy()))
                dom.close()
        assert np.array_equal(got[0][0], got[1][0]), w.name
        if w.thermal:
            assert np.array_equal(got[0][1], got[1][1]), w.name


def test_batched_swap_calls_are_checked():
    """lbm_halo_axis_swap_many: 1 to 32 pairs, each face once, the checks of a single swap
    on every pair."""
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    w = W.random_periodic(shape=(16, 12, 10), seed=104)
    dom = BlockDomain(w, (1, 2, 2))
    dom.init_equilibrium()
    dom.step(1)                                     # parity 1: FILL is due
    ctx = [b.ctx for b in dom.blocks]
    pairs = dom.pairs(2)
    lo, hi = [ctx[a] for a, _ in pairs], [ctx[b] for _, b in pairs]
    capi.lbm_halo_axis_swap_many(lo, hi, 2, capi.LBM_HALO_FILL)
    for args, text in ((([lo[0], lo[0]], [hi[0], hi[1]]), "two pairs"),   # a face twice
                       (([], []), "n must lie"),                           # no pair
                       ((lo * 17, hi * 17), "n must lie")):                # 34 pairs
        with pytest.raises(capi.LbmError, match=text):
            capi.lbm_halo_axis_swap_many(args[0], args[1], 2, capi.LBM_HALO_FILL)
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_axis_swap_many(lo, hi, 2, capi.LBM_HALO_DRAIN)   # parity 1
    with pytest.raises(capi.LbmError):
        capi.lbm_halo_axis_swap_many(lo, hi, 0, capi.LBM_HALO_FILL)    # x is not split
    torch.cuda.synchronize()
    dom.close()


# ------------------------------------------------------------- one block per rank ---

STEPS = (7, 8)


def _case(name):
    if name == "periodic 2x2":
        return W.random_periodic(shape=(40, 12, 20), seed=87), (2, 1, 2)
    if name == "cavity3d 2x2":
        return W.perturbed(W.cavity3d(shape=(36, 20, 22)), seed=88), (1, 2, 2)
    return W.perturbed(W.cavity2d(shape=(70, 30, 1)), seed=89), (2, 2, 1)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, name, overlap, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from lattice_boltzmann_cfd_gb300.blocks import DistBlockDomain
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=120))
    w, nb = _case(name)
    d = DistBlockDomain(w, nb, rank, world, device="cuda:0", transport="host", overlap=overlap)
    d.init_equilibrium()
    res, done = {}, 0
    for n in STEPS:
        d.step(n - done)
        done = n
        f, g = d.populations()
        res[n] = (f.cpu().numpy(), None if g is None else g.cpu().numpy())
    res["diag"] = d.global_diagnostics()      # a collective: every rank calls it
    out[rank] = res
    d.close()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("overlap", [False, True], ids=["plain", "overlap"])
@pytest.mark.parametrize("name", ["periodic 2x2", "cavity3d 2x2", "cavity2d 2x2"])
def test_four_ranks_share_the_gpu(oracle_mod, name, overlap):
    """Four gloo ranks, one block each, on the one GPU of the test box, in the plain and the
    overlapped order: the halo kernels write and read page-locked host buffers and the
    waiting is on the host, in the gloo messages.  The gathered owned cells equal the undivided domain bit for bit and match
    the fp64 oracle."""
    import torch.multiprocessing as mp
    from lattice_boltzmann_cfd_gb300.blocks import block_part, owned_slices
    w, nb = _case(name)
    world = nb[0] * nb[1] * nb[2]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), name, overlap, out), nprocs=world, join=True)
    ref = oracle_states(oracle_mod, w, list(STEPS))
    for n in STEPS:
        f1, g1, _ = _single(w, n)
        f = np.full_like(f1, np.nan)
        g = None if g1 is None else np.full_like(g1, np.nan)
        for r in range(world):
            _, sides, coords = block_part(w, nb, r)
            own = owned_slices(sides, coords)
            sel = np.ix_(*(np.array(coords[a])[own[2 - a]] for a in (2, 1, 0)))
            f[(slice(None),) + sel] = out[r][n][0]
            if g is not None:
                g[(slice(None),) + sel] = out[r][n][1]
        assert np.array_equal(f, f1), n
        if w.thermal:
            assert np.array_equal(g, g1), n
        assert np.abs(f - ref[n]["f"]).max() <= 1e-6
        if w.thermal:
            assert np.abs(g - ref[n]["g"]).max() <= 1e-6
    # the all-reduced diagnostics after the last step, against the undivided domain's
    d1 = _single(w, STEPS[-1])[2]
    for r in range(world):
        dg = out[r]["diag"]
        assert dg["fluid_cells"] == d1["fluid_cells"] and dg["finite"]
        assert abs(dg["mass"] - d1["mass"]) <= 1e-9 * abs(d1["mass"])
        assert np.allclose(dg["momentum"], d1["momentum"], rtol=0, atol=1e-7 * d1["fluid_cells"])
        if w.thermal:
            for key in ("nu_hot", "nu_cold"):
                assert abs(dg[key] - d1[key]) <= 1e-5 * max(1.0, abs(d1[key])), key
            assert abs(dg["nu_volume"] - d1["nu_volume"]) <= 1e-3


def test_checkpoint_resume_across_decompositions():
    """Whole-domain populations taken from one decomposition after 100 or 101 steps resume in
    another (slabs -> blocks, blocks -> slabs, blocks -> one domain and back): the remaining
    steps give the state of 201 straight steps within fp32 rounding (the read-out adds the
    rest weights back in fp32)."""
    from lattice_boltzmann_cfd_gb300.slabs import SlabDomain
    from lattice_boltzmann_cfd_gb300.blocks import BlockDomain
    from lattice_boltzmann_cfd_gb300.solver import Simulation
    w = W.perturbed(W.cavity3d(shape=(40, 20, 18)), seed=91)
    f_ref, g_ref, _ = _single(w, 201)

    def run(dom, n):
        dom.init_equilibrium()
        dom.step(n)
        return dom.populations()

    def single():
        s = Simulation(w)
        s.init_equilibrium(_dev(w.rho0), _dev(w.u0), _dev(w.T_init))
        return s

    makers = {"slabs": lambda: SlabDomain(w, 3), "blocks": lambda: BlockDomain(w, (1, 2, 2)),
              "blocks x": lambda: BlockDomain(w, (2, 1, 2))}
    for k in (100, 101):
        for src, dst in (("slabs", "blocks"), ("blocks", "slabs"), ("blocks x", "single"),
                         ("single", "blocks x")):
            if src == "single":
                a = single()
                a.step(k)
                f, g = a.populations()
            else:
                a = makers[src]()
                f, g = run(a, k)
            b = single() if dst == "single" else makers[dst]()
            b.set_populations(f, g)
            b.step(201 - k)
            fb, gb = b.populations()
            assert np.abs(fb.cpu().numpy() - f_ref).max() < 1e-6, (k, src, dst)
            assert np.abs(gb.cpu().numpy() - g_ref).max() < 1e-6, (k, src, dst)
            a.close()
            b.close()
