"""The candidate block edges of the immersed-boundary sample ordering search ("GPU
Optimization for High-Quality Kinetic Fluid Simulation", Sec. 4, Eq. 11): l runs over
{2, ..., L_m}, L_m the smallest edge of the samples' bounding box in cells (capped)."""
import dataclasses

import numpy as np

from lattice_boltzmann_cfd_gb300 import workloads as W
from lattice_boltzmann_cfd_gb300.tuning import default_candidates


def _with_samples(w, x):
    x = np.asarray(x, np.float32)
    return dataclasses.replace(w, ib_x=x, ib_ub=np.zeros_like(x),
                               ib_w=np.ones(len(x), np.float32))


def test_sphere_candidates_span_its_diameter():
    w = W.channel_ib_sphere(shape=(64, 48, 48), center=(20.3, 23.7, 24.2), radius=8)
    c = default_candidates(w)
    # the samples lie on the sphere: the bounding box edge is just under the diameter 16
    assert c[0] == 2 and c == list(range(2, c[-1] + 1))
    assert 15 <= c[-1] <= 17


def test_smallest_edge_of_the_box_decides():
    w = W.channel_ib_sphere(shape=(64, 48, 48), center=(20.3, 23.7, 24.2), radius=8)
    box = [[0, 0, 0], [30.5, 9.2, 20.0], [1, 2, 3]]          # extents 30.5, 9.2, 20
    # an extent of 9.2 spans floor(9.2) + 1 = 10 cells
    assert default_candidates(_with_samples(w, box)) == list(range(2, 11))
    assert default_candidates(_with_samples(w, box), cap=5) == [2, 3, 4, 5]


def test_flat_or_single_sample_sets_keep_the_smallest_edge():
    w = W.channel_ib_sphere(shape=(64, 48, 48), center=(20.3, 23.7, 24.2), radius=8)
    flat = [[0, 0, 5], [10, 10, 5], [3, 7, 5]]                 # no extent along z
    assert default_candidates(_with_samples(w, flat)) == [2]
    assert default_candidates(_with_samples(w, [[4, 4, 4]])) == [2]

