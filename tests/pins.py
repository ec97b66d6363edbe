"""Reusable pin checks of an oracle build (raise AssertionError on failure).

They are used on the committed oracle (tests/test_oracle.py) and on mutated
copies of it (tests/test_oracle_mutations.py), which must each fail one.
"""
import json
import os

import numpy as np

from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import Oracle
from tests import bruteforce as BF
from tests.helpers import fp64_image_sums, home_slots, trace_origins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # unit roundoff of fp32 round-to-nearest


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def origins(o):
    return trace_origins(o.n_domains, o.dom_offset, o.home, o.home_ids, o.table, o.maps, o.pulse_dim)


def built(w, lib_path=None):
    o = Oracle(w.box, w.dims, w.cutoff, lib_path=lib_path)
    pos = W.positions(w)
    o.build(pos)
    return o, pos


def check_golden(name, lib_path=None):
    g = golden(name)
    o = Oracle(g["box"], g["dims"], g["cutoff"], lib_path=lib_path)
    o.build(np.array(g["positions"], np.float32))
    assert [[int(d), int(k)] for d, k in zip(o.pulse_dim, o.pulse_k)] == g["pulses"]
    assert o.dom_offset.tolist() == g["dom_offset"]
    assert o.home.tolist() == g["home"]
    assert o.halo.tolist() == g["halo"]
    assert o.home_ids.tolist() == g["home_ids"]
    for p, rows in enumerate(g["table"]):
        for r, row in enumerate(rows):
            t = o.table[p, r]
            assert [int(t[1]), int(t[2]), int(t[3]), int(t[4]), int(t[5])] == row, (p, r)
            assert o.map_of(p, r).tolist() == g["maps"][p][r], (p, r)
    assert np.array_equal(o.coords(), np.array(g["coords"], np.float32))
    # forces (s+1, 10(s+1), -(s+1)) reduced in reverse pulse order
    s = np.arange(o.total_slots, dtype=np.float32) + 1
    f = np.stack([s, 10 * s, -s], axis=1).astype(np.float32)
    o.exchange_forces(f)
    fx = np.array(g["forces_x_after"], np.float32)
    assert np.array_equal(f[:, 0], fx)
    assert np.array_equal(f[:, 1], 10 * fx)
    assert np.array_equal(f[:, 2], -fx)


def check_pulse_dependencies(lib_path=None):
    g = golden("pulse_dependencies.json")
    w = W.WORKLOADS["C2"]
    o = Oracle(g["box"], g["dims"], g["cutoff"], lib_path=lib_path)
    assert [[int(d), int(k)] for d, k in zip(o.pulse_dim, o.pulse_k)] == g["pulses"]
    # The dependent tail of pulse p (local index >= home count) must come from
    # the receive ranges of exactly the earlier pulses the pages list.
    o.build(W.positions(w))
    for p, waits in enumerate(g["coord_waits"]):
        seen = set()
        for r in range(o.n_domains):
            m = o.map_of(p, r)
            split = int(o.table[p, r, 5])
            assert np.all(m[:split] < o.home[r]) and np.all(m[split:] >= o.home[r])
            for j in m[split:]:
                for q in range(p):
                    rows = [t for t in o.table[q] if int(t[2]) == r]
                    assert len(rows) == 1
                    lo_, n_ = int(rows[0][3]), int(rows[0][1])
                    if lo_ <= j < lo_ + n_:
                        seen.add(q)
        assert sorted(seen) == waits, (p, sorted(seen), waits)


def check_brute_force(o, pos):
    origin, shift = origins(o)
    assert np.all(origin >= 0)
    coords = o.coords()
    cells = [(r % o.dims[0], (r // o.dims[0]) % o.dims[1], r // (o.dims[0] * o.dims[1]))
             for r in range(o.n_domains)]
    total_halo = 0
    for r in range(o.n_domains):
        lo_, h, n_halo = int(o.dom_offset[r]), int(o.home[r]), int(o.halo[r])
        got_ids = origin[lo_ + h: lo_ + h + n_halo]
        # exactly once: no atom appears twice in one halo
        assert len(np.unique(got_ids)) == len(got_ids), f"duplicate image in halo of {r}"
        ids, vals = BF.halo_of_domain(pos, o.box, o.dims, o.cutoff, cells[r])
        assert sorted(got_ids.tolist()) == sorted(ids.tolist()), f"halo set of domain {r}"
        order = np.argsort(got_ids, kind="stable")
        exp = vals[np.argsort(ids, kind="stable")]
        got = coords[lo_ + h: lo_ + h + n_halo][order]
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32)), f"halo values of {r}"
        # home slots hold the inputs unchanged
        assert np.array_equal(coords[lo_: lo_ + h], pos[origin[lo_: lo_ + h]])
        total_halo += n_halo
    return total_halo


def check_forces(o, w):
    f_pre = W.forces(w, o.total_slots)
    f = f_pre.copy()
    o.exchange_forces(f)
    origin, _ = origins(o)
    s64, a64, cnt = fp64_image_sums(origin, f_pre, o.n_atoms)
    hs = home_slots(o.n_domains, o.dom_offset, o.home)
    ids = origin[hs]
    got = f[hs].astype(np.float64)
    # per atom: the fp32 sum of m+1 terms is within m*u*sum|terms| (first order)
    bound = (cnt[ids] - 1)[:, None] * U * a64[ids] * 1.0001 + 1e-30
    assert np.all(np.abs(got - s64[ids]) <= bound)
    # momentum: total over all slots before == total over home slots after
    p_before = f_pre.astype(np.float64).sum(axis=0)
    p_after = got.sum(axis=0)
    mom_bound = ((cnt - 1)[:, None] * U * a64).sum(axis=0) * 1.0001 + 1e-12
    assert np.all(np.abs(p_before - p_after) <= mom_bound)
    assert int(cnt.sum()) == o.total_slots


def check_replay(o):
    """The per-step coordinate exchange, run on an array whose halo slots
    were poisoned, reproduces the build's halo bit for bit."""
    x = o.coords().copy()
    hs = home_slots(o.n_domains, o.dom_offset, o.home)
    mask = np.ones(o.total_slots, bool)
    mask[hs] = False
    x[mask] = np.nan
    o.exchange_coords(x)
    assert np.array_equal(x.view(np.uint32), o.coords().view(np.uint32))
