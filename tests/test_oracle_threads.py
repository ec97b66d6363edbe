"""The oracle's threaded exchanges (each pulse's senders spread over OpenMP
threads, pulse order kept) against its plain loops, bit for bit.

Within one pulse a sender writes only its receiver's receive range of that
pulse and reads only its own home and earlier ranges (forces: adds into its
own earlier slots, reads its receiver's range of the pulse), so the senders of
a pulse are independent and any thread count gives identical results. The
threaded form is what the CPU baseline times on all host cores.
"""
import numpy as np
import pytest

from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import Oracle


def _same_bits(a, b):
    return np.array_equal(a.view(np.int32), b.view(np.int32))


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_threaded_exchange_matches_plain(name, threads):
    w = W.WORKLOADS[name]
    o = Oracle(w.box, w.dims, w.cutoff)
    o.build(W.positions(w))
    x = o.coords()
    x_par = x.copy()
    f = W.forces(w, o.total_slots)
    f_par = f.copy()
    for _ in range(2):   # the second step forwards the first step's halos again
        o.exchange_coords(x)
        o.exchange_coords_par(x_par, threads)
        o.exchange_forces(f)
        o.exchange_forces_par(f_par, threads)
    assert _same_bits(x, x_par)
    assert _same_bits(f, f_par)


def test_max_threads_is_positive():
    w = W.WORKLOADS["C1"]
    o = Oracle(w.box, w.dims, w.cutoff)
    assert o.max_threads() >= 1
