"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU. Each test names what it pins:
  * hand-derived worked examples (tests/golden/*.json);
  * the pages' pulse numbering Z -> Y -> X and the dependency chain;
  * brute-force halo membership: every periodic image within the cutoff of a
    domain's upper faces appears exactly once in its halo, nothing else does,
    and each halo value is bit-exactly x or fl(x + L) as the image demands;
  * the expected halo volume (closed form) within Poisson spread;
  * momentum conservation and per-atom force sums in fp64 within an fp32
    rounding bound;
  * special and invalid cases.
"""
import math

import numpy as np
import pytest

from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import Oracle, OracleError
from tests import pins


@pytest.mark.parametrize("name", ["two_slab_x.json", "corner_relay_xy.json"])
def test_golden_worked_example(name):
    pins.check_golden(name)


def test_pulse_numbering_and_dependency_chain():
    pins.check_pulse_dependencies()


@pytest.mark.parametrize("name", ["C1", "C2", "C3"])
def test_brute_force_exactly_once(name):
    o, pos = pins.built(W.WORKLOADS[name])
    pins.check_brute_force(o, pos)


@pytest.mark.parametrize("box,dims,cutoff,n", [
    ((3.0, 3.0, 3.0), (3, 3, 3), 0.6, 2700),      # 27 domains, 1 pulse per dim
    ((5.0, 5.0, 3.0), (5, 5, 1), 1.5, 3000),      # 2 pulses in X and in Y
    ((6.0, 4.0, 5.0), (4, 1, 5), 1.3, 3000),      # X 1 pulse (w=1.5), Z 2 pulses (w=1)
    ((4.0, 4.0, 4.0), (2, 2, 2), 2.0, 1500),      # cutoff equal to the slab width
    ((4.0, 4.5, 4.0), (1, 3, 1), 2.9, 1500),      # np = 2 = n - 1 (largest allowed)
    ((2.0, 2.0, 2.0), (2, 2, 2), 0.5, 0),         # no atoms: every pulse empty
    ((2.0, 2.0, 2.0), (2, 2, 2), 0.5, 7),         # ragged, mostly empty pulses
])
def test_brute_force_shapes(box, dims, cutoff, n):
    w = W.custom("t", n, box, dims, cutoff, seed=11 + n)
    o, pos = pins.built(w)
    pins.check_brute_force(o, pos)


def boundary_points():
    below = float(np.nextafter(np.float32(4.0), np.float32(0)))
    vals = [0.0, 1.0, 2.0, 3.0, below, float(np.nextafter(np.float32(1.0), np.float32(0))),
            float(np.nextafter(np.float32(3.0), np.float32(0))), 0.5, 2.5]
    return np.array([[a, b, c] for a in vals for b in vals[:5] for c in vals[:4]], np.float32)


def test_brute_force_boundary_atoms():
    """Atoms exactly on slab faces, at 0, at the largest fp32 below L and at
    distance exactly r_c from a face (the strict test keeps them out)."""
    pts = boundary_points()
    o = Oracle((4.0, 4.0, 4.0), (2, 2, 2), 1.0)
    o.build(pts)
    pins.check_brute_force(o, pts)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
def test_halo_volume_closed_form(name):
    w = W.WORKLOADS[name]
    o, _ = pins.built(w)
    vol = np.prod(w.box)
    density = w.n_atoms / vol
    ext = np.prod([(b / n) + (w.cutoff if n > 1 else 0.0) for b, n in zip(w.box, w.dims)])
    own = np.prod([b / n for b, n in zip(w.box, w.dims)])
    expected_total = (ext - own) * density * o.n_domains
    got = int(o.halo.sum())
    sigma = math.sqrt(expected_total)
    assert abs(got - expected_total) < 5 * sigma + 1, (got, expected_total)


@pytest.mark.parametrize("name", ["C1", "C2", "C3"])
def test_force_momentum_and_per_atom(name):
    w = W.WORKLOADS[name]
    o, _ = pins.built(w)
    pins.check_forces(o, w)


def test_coordinate_replay_reproduces_build():
    o, _ = pins.built(W.WORKLOADS["C2"])
    pins.check_replay(o)


def test_single_domain_is_identity():
    w = W.custom("one", 500, (3.0, 3.0, 3.0), (1, 1, 1), 1.0, seed=3)
    o, pos = pins.built(w)
    assert o.n_pulses == 0 and o.total_slots == 500 and o.total_entries == 0
    assert np.array_equal(o.coords(), pos)
    f = W.forces(w, 500)
    g = f.copy()
    o.exchange_forces(g)
    assert np.array_equal(f, g)


def test_two_domains_symmetric():
    """2x1x1 with one pulse: each domain is both neighbours of the other; the
    halo of domain 0 comes from domain 1 unshifted, that of domain 1 from
    domain 0 shifted by +L."""
    o, pos = pins.built(W.WORKLOADS["C1"])
    origin, shift = pins.origins(o)
    assert o.n_pulses == 1
    assert int(o.table[0, 0, 2]) == 1 and int(o.table[0, 1, 2]) == 0
    assert int(o.table[0, 0, 4]) == 1 and int(o.table[0, 1, 4]) == 0
    h0 = slice(int(o.dom_offset[0] + o.home[0]), int(o.dom_offset[0] + o.home[0] + o.halo[0]))
    h1 = slice(int(o.dom_offset[1] + o.home[1]), int(o.dom_offset[1] + o.home[1] + o.halo[1]))
    assert np.all(shift[h0] == 0) and np.all(shift[h1][:, 0] == 1)


@pytest.mark.parametrize("box,dims,cutoff,err", [
    ((3.0, 3.0, 3.0), (2, 1, 1), 0.0, -1),
    ((3.0, 3.0, 3.0), (2, 1, 1), -1.0, -1),
    ((3.0, 3.0, 3.0), (0, 1, 1), 1.0, -1),
    ((3.0, 0.0, 3.0), (2, 1, 1), 1.0, -1),
    ((3.0, 3.0, 3.0), (2, 1, 1), 1.6, -2),         # np = 2 = n
    ((12.0, 6.0, 6.0), (16, 1, 1), 12.0, -2),
])
def test_invalid_setup(box, dims, cutoff, err):
    with pytest.raises(OracleError) as ei:
        Oracle(box, dims, cutoff)
    assert ei.value.code == err


@pytest.mark.parametrize("bad", [-0.25, 3.0, 3.5, float("nan")])
def test_atom_outside_box(bad):
    o = Oracle((3.0, 3.0, 3.0), (2, 1, 1), 1.0)
    pos = np.array([[1.0, 1.0, 1.0], [bad, 1.0, 1.0]], np.float32)
    with pytest.raises(OracleError) as ei:
        o.build(pos)
    assert ei.value.code == -3
