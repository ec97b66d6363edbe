"""Brute-force halo membership, independent of the staged-forwarding algorithm.

For every target domain R and every atom a this decides directly, image by
image, whether the periodic image of a lies in R's halo, instead of relaying
atoms pulse by pulse. Per dimension d with n_d > 1 the image a + s_d*L_d
(s_d in {0, 1}, because the halo extends above a domain) is k_d cells above R.
It belongs to R's halo iff 0 <= k_d <= np_d in every such dimension, not all
k_d are zero, and at each of the k_d hops the sender's cutoff test passes in
that sender's own frame (unshifted until the hop from cell 0 has added L_d).

This is the "every atom within r_c of a domain's boundary, under periodic
images, appears exactly once in its halo" statement written out with the same
geometric readings as the exchange (send down, fp32 strict cutoff test on
x - lo of the sender, fp32 shift). It is used only to pin the oracle.
"""
from __future__ import annotations

import math

import numpy as np


def geometry(box, dims, cutoff):
    box = [float(b) for b in box]
    dims = [int(n) for n in dims]
    np_d = []
    lo = []
    for d in range(3):
        if dims[d] > 1:
            np_d.append(int(math.ceil(cutoff / (box[d] / dims[d]))))
        else:
            np_d.append(0)
        lo.append(np.array([np.float32(c * box[d] / dims[d]) for c in range(dims[d])], np.float32))
    return np_d, lo


def home_cells(pos, box, dims):
    x = pos.astype(np.float64)
    cells = np.empty(pos.shape, np.int64)
    for d in range(3):
        c = np.floor(x[:, d] * dims[d] / box[d]).astype(np.int64)
        cells[:, d] = np.minimum(c, dims[d] - 1)
    return cells


def halo_of_domain(pos, box, dims, cutoff, cell_r):
    """Return (ids, values[fp32, n x 3]) of the images in the halo of the
    domain whose cell is ``cell_r``; ids are input atom indices."""
    pos = np.asarray(pos, np.float32)
    n = pos.shape[0]
    np_d, lo = geometry(box, dims, cutoff)
    cells = home_cells(pos, box, dims)
    rcf = np.float32(cutoff)
    ok = np.ones(n, bool)
    any_hop = np.zeros(n, bool)
    vals = pos.copy()
    for d in range(3):
        nd = dims[d]
        if nd == 1:
            continue
        c = cells[:, d]
        cr = cell_r[d]
        s = (c < cr).astype(np.int64)            # image above R needs the +L copy
        k = c + s * nd - cr
        in_range = k <= np_d[d]
        x = pos[:, d]
        xs = (x + np.float32(box[d])).astype(np.float32)
        hops_ok = np.ones(n, bool)
        for j in range(max(np_d[d], 0)):
            active = in_range & (k > j)
            v = cr + k - j                           # virtual cell of the j-th sender
            wrapped = v >= nd
            actual = np.where(wrapped, v - nd, v)
            actual = np.clip(actual, 0, nd - 1)
            val = np.where(wrapped, x, np.where(s == 1, xs, x)).astype(np.float32)
            rel = (val - lo[d][actual]).astype(np.float32)
            hops_ok &= ~active | (rel < rcf)
        ok &= in_range & hops_ok
        any_hop |= k > 0
        vals[:, d] = np.where(s == 1, xs, x)
    sel = ok & any_hop
    return np.nonzero(sel)[0], vals[sel]
