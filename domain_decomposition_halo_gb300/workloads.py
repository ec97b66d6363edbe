"""Seeded synthetic workloads for the staged halo exchange.

This module only draws random inputs. It holds none of the exchange's
arithmetic (no cell assignment, no cutoff test, no shift), so that both the
CUDA path and the CPU oracle can take their inputs from it without sharing
any of the method.

The workloads stand in for the water-ethanol systems (45,000 to 23M atoms,
~100 atoms/nm^3) that "A Practical Guide to GPU-Initiated Communication for
Molecular Dynamics at Scale" benchmarks in its section "A leap in scaling
performance"; those systems are not available here.

Recipe (all generators are numpy PCG64, ``numpy.random.default_rng``):

* positions: fp64 uniform draws cast to fp32. A value whose fp32 rounding is
  not below the box length is replaced by the largest fp32 below it, so every
  position lies in [0, L).
* ``order="random"``: atoms uniform over the whole box, in draw order.
* ``order="grouped"``: the box is cut into the decomposition's uniform slabs
  (c*L/n .. (c+1)*L/n per dimension); each slab box gets ``n_atoms / n_dom``
  atoms drawn uniformly inside it, slab boxes in x-fastest order. Atoms are
  therefore grouped by domain and in random order within each domain.
* forces: one fp32 float3 per slot of the exchange layout (home and halo,
  every domain, in layout order) from ``default_rng(seed + 1000)``: uniform
  in [-1, 1] or standard normal.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Tuple

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    n_atoms: int
    box: Tuple[float, float, float]
    dims: Tuple[int, int, int]
    cutoff: float
    forces: str          # "uniform" (U[-1,1]) or "normal" (N(0,1))
    order: str           # "random" or "grouped"
    seed: int

    def describe(self) -> str:
        b = "x".join(f"{v:g}" for v in self.box)
        d = "x".join(str(v) for v in self.dims)
        return (f"{self.n_atoms} atoms, box {b} nm, {d} domains, cutoff {self.cutoff:g} nm, "
                f"{self.order} order, forces {self.forces}, seed {self.seed}")


# The five configurations: a 2-domain slab case, a 2x2x2 case with relayed
# edge/corner halos, a 16-slab case whose slabs are thinner than the cutoff
# (two pulses with forwarding), and two large bandwidth cases with scattered
# in-domain order.
WORKLOADS = {
    "C1": Workload("C1", 3000, (3.1, 3.1, 3.1), (2, 1, 1), 1.2, "uniform", "random", 1),
    "C2": Workload("C2", 24000, (6.2, 6.2, 6.2), (2, 2, 2), 1.0, "uniform", "random", 2),
    "C3": Workload("C3", 43200, (12.0, 6.0, 6.0), (16, 1, 1), 1.0, "normal", "random", 3),
    "C4": Workload("C4", 1_000_000, (21.5, 21.5, 21.5), (4, 4, 4), 1.2, "normal", "grouped", 4),
    "C5": Workload("C5", 12_000_000, (49.3, 49.3, 49.3), (8, 8, 4), 1.0, "normal", "grouped", 5),
}


def _below(box_len: float) -> np.float32:
    """Largest fp32 value strictly below ``box_len`` (compared in fp64)."""
    v = np.float32(box_len)
    while float(v) >= box_len:
        v = np.nextafter(v, np.float32(0.0))
    return v


def _clip_to_box(col32: np.ndarray, box_len: float) -> None:
    bad = col32.astype(np.float64) >= box_len
    if bad.any():
        col32[bad] = _below(box_len)


def positions(w: Workload) -> np.ndarray:
    """fp32 array [n_atoms, 3] of positions in [0, L) per the recipe above."""
    rng = np.random.default_rng(w.seed)
    n = w.n_atoms
    out = np.empty((n, 3), dtype=np.float32)
    if w.order == "random":
        for d in range(3):
            out[:, d] = rng.uniform(0.0, w.box[d], size=n).astype(np.float32)
    elif w.order == "grouped":
        nx, ny, nz = w.dims
        n_dom = nx * ny * nz
        if n % n_dom:
            raise ValueError("grouped order needs n_atoms divisible by the domain count")
        per = n // n_dom
        k = 0
        for cz in range(nz):
            for cy in range(ny):
                for cx in range(nx):
                    cell = (cx, cy, cz)
                    for d in range(3):
                        lo = cell[d] * w.box[d] / w.dims[d]
                        hi = (cell[d] + 1) * w.box[d] / w.dims[d]
                        out[k:k + per, d] = rng.uniform(lo, hi, size=per).astype(np.float32)
                    k += per
    else:
        raise ValueError(f"unknown order {w.order!r}")
    for d in range(3):
        _clip_to_box(out[:, d], w.box[d])
    return out


def forces(w: Workload, n_slots: int) -> np.ndarray:
    """fp32 array [n_slots, 3]: one force per layout slot (home and halo)."""
    rng = np.random.default_rng(w.seed + 1000)
    if w.forces == "uniform":
        f = rng.uniform(-1.0, 1.0, size=(n_slots, 3))
    elif w.forces == "normal":
        f = rng.standard_normal(size=(n_slots, 3))
    else:
        raise ValueError(f"unknown force law {w.forces!r}")
    return f.astype(np.float32)


def custom(name: str, n_atoms: int, box, dims, cutoff: float, seed: int,
           forces_law: str = "uniform", order: str = "random") -> Workload:
    """A workload outside the fixed table (edge cases, small sweeps)."""
    return Workload(name, int(n_atoms), tuple(float(b) for b in box), tuple(int(d) for d in dims),
                    float(cutoff), forces_law, order, int(seed))
