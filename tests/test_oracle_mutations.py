"""Mutation check of the oracle's pins.

Each case copies the committed oracle source, plants one plausible mistake
(a wrong sign, index, bound, order or a dropped term), compiles the copy with
gcc and runs the pins on it. Every mutant must fail at least one pin; the
unmodified copy must pass them all. Nothing here touches a GPU.
"""
import json
import os
import shutil
import subprocess
import sys

import numpy as np
import pytest

from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import compile_oracle, Oracle
from tests import pins
from tests.test_oracle import boundary_points

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "hx_oracle.c")

MUTANTS = {
    "forces_forward_order": ("for (int p = o->n_pulses - 1; p >= 0; --p)", "for (int p = 0; p < o->n_pulses; ++p)"),
    "no_periodic_shift_at_build": ("if (shift) v[d] = v[d] + o->boxf[d];", ";"),
    "shift_in_last_cell": ("const int shift = (c[d] == 0);", "const int shift = (c[d] == o->dims[d] - 1);"),
    "cutoff_not_strict": ("if (rel < o->rcf)", "if (rel <= o->rcf)"),
    "forward_all_local_atoms": ("if (k == 0) { cb = 0; ce = snap[r]; }", "if (1) { cb = 0; ce = snap[r]; }"),
    "send_to_upper_neighbour": ("c[d] = (c[d] - 1 + o->dims[d]) % o->dims[d];", "c[d] = (c[d] + 1) % o->dims[d];"),
    "pulse_order_xyz": ("for (int d = 2; d >= 0; --d) {", "for (int d = 0; d < 3; ++d) {"),
    "force_overwrite_not_accumulate": ("dst[3 * (int64_t)m[i] + 0] += src[3 * i + 0];", "dst[3 * (int64_t)m[i] + 0] = src[3 * i + 0];"),
    "force_dropped_z": ("dst[3 * (int64_t)m[i] + 2] += src[3 * i + 2];", ";"),
    "lo_face_off_by_one": ("o->lo[d][c] = (float)((double)c * box[d] / dims[d]);", "o->lo[d][c] = (float)((double)(c + 1) * box[d] / dims[d]);"),
    "replay_without_shift": ("if (o->t_shift[t]) {", "if (0) {"),
    "replay_wrong_receiver_offset": ("float* dst = x + 3 * (o->dom_offset[o->t_recv[t]] + o->t_off[t]);", "float* dst = x + 3 * (o->dom_offset[o->t_recv[t]] + o->t_off[t] + 1);"),
    "forces_read_sender_slots": ("const float* src = f + 3 * (o->dom_offset[o->t_recv[t]] + o->t_off[t]);", "const float* src = f + 3 * (o->dom_offset[r] + o->t_off[t]);"),
    "home_cell_rounding": ("int cd = (int)floor(x * (double)o->dims[d] / o->box[d]);", "int cd = (int)floor(x * (double)o->dims[d] / o->box[d] + 0.5);"),
    "split_counts_dependents": ("if (m[i] < o->home[r]) split = (int32_t)(i + 1);", "if (m[i] >= o->home[r]) split = (int32_t)(i + 1);"),
}


def _run_pins(lib):
    """Return the list of pins that failed on the oracle built at ``lib``."""
    failed = []
    checks = [
        ("golden_two_slab", lambda: pins.check_golden("two_slab_x.json", lib)),
        ("golden_corner", lambda: pins.check_golden("corner_relay_xy.json", lib)),
        ("pulse_dependencies", lambda: pins.check_pulse_dependencies(lib)),
    ]
    for name in ("C2", "C3"):
        w = W.WORKLOADS[name]
        checks.append((f"brute_{name}", lambda w=w: pins.check_brute_force(*pins.built(w, lib))))
        checks.append((f"forces_{name}", lambda w=w: pins.check_forces(pins.built(w, lib)[0], w)))
    checks.append(("replay_C2", lambda: pins.check_replay(pins.built(W.WORKLOADS["C2"], lib)[0])))

    def boundary():
        pts = boundary_points()
        o = Oracle((4.0, 4.0, 4.0), (2, 2, 2), 1.0, lib_path=lib)
        o.build(pts)
        pins.check_brute_force(o, pts)
    checks.append(("boundary", boundary))
    for name, fn in checks:
        try:
            fn()
        except Exception:  # noqa: BLE001 - any failure of a pin counts
            failed.append(name)
    return failed


def _run_pins_isolated(lib):
    """Run the pins in a child process: a mutant may corrupt memory, and a
    crash of the child also counts as a caught mutant."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-m", "tests.test_oracle_mutations", lib],
                          cwd=root, capture_output=True, text=True, timeout=600)
    if proc.returncode != 0:
        return ["crashed"]
    return json.loads(proc.stdout.strip().splitlines()[-1])


def _mutant_lib(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} must be unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    return compile_oracle(str(path), str(tmp_path / f"lib{name}.so"))


def test_unmodified_copy_passes(tmp_path):
    shutil.copy(SRC, tmp_path / "same.c")
    lib = compile_oracle(str(tmp_path / "same.c"), str(tmp_path / "libsame.so"))
    assert _run_pins_isolated(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _mutant_lib(tmp_path, name, old, new)
    failed = _run_pins_isolated(lib)
    assert failed, f"mutant {name} passed every pin"


if __name__ == "__main__":
    print(json.dumps(_run_pins(sys.argv[1])))
