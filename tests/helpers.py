"""Shared test helpers: trace which input atom fills every slot of a layout,
and fp64 reference sums for the force checks."""
from __future__ import annotations

import numpy as np


def layout_lengths(n_domains, home, table):
    """Slots per domain (home plus every receive range) read off a pulse table
    whose rows are (map_off, size, recv, recv_off, shift, ...)."""
    length = np.array(home, np.int64).copy()
    for p in range(table.shape[0]):
        for r in range(n_domains):
            q = int(table[p, r, 2])
            length[q] = max(length[q], int(table[p, r, 3] + table[p, r, 1]))
    return length


def trace_origins(n_domains, dom_offset, home, home_ids, table, maps, pulse_dim):
    """origin[slot] = input atom index held by that slot (home or halo) and
    shift[slot, d] = number of +L_d shifts applied on the way, replaying each
    pulse's gather packed[i] = data[map[i]] with ids instead of coordinates."""
    length = layout_lengths(n_domains, home, table)
    total = int(dom_offset[-1] + length[-1]) if n_domains else 0
    origin = np.full(total, -1, np.int64)
    shift = np.zeros((total, 3), np.int8)
    k = 0
    for r in range(n_domains):
        h = int(home[r])
        origin[dom_offset[r]: dom_offset[r] + h] = home_ids[k: k + h]
        k += h
    for p in range(table.shape[0]):
        d = int(pulse_dim[p])
        for r in range(n_domains):
            off, size, q, roff, sh = (int(v) for v in table[p, r, :5])
            m = maps[off: off + size].astype(np.int64)
            src = dom_offset[r] + m
            dst = dom_offset[q] + roff + np.arange(size)
            origin[dst] = origin[src]
            shift[dst] = shift[src]
            if sh:
                shift[dst, d] += 1
    return origin, shift


def fp64_image_sums(origin, f_pre, n_atoms):
    """fp64 sum of the pre-reduction forces over all images of each atom, the
    matching sum of absolute values (for error bounds) and the image counts."""
    f64 = f_pre.astype(np.float64)
    s = np.zeros((n_atoms, 3))
    a = np.zeros((n_atoms, 3))
    cnt = np.zeros(n_atoms, np.int64)
    np.add.at(s, origin, f64)
    np.add.at(a, origin, np.abs(f64))
    np.add.at(cnt, origin, 1)
    return s, a, cnt


def home_slots(n_domains, dom_offset, home):
    return np.concatenate([np.arange(dom_offset[r], dom_offset[r] + home[r]) for r in range(n_domains)]
                          ) if n_domains else np.zeros(0, np.int64)
