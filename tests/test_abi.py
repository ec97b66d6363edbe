"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function include/hx.h declares; the host-side plan agrees with
the oracle; argument errors come back as codes."""
import ctypes
import os
import re

import numpy as np
import pytest

from domain_decomposition_halo_gb300 import hx as HX
from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import Oracle, OracleError

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hx.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(hx_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("hx_init", "hx_build_maps", "hx_exchange_coords", "hx_exchange_forces", "hx_destroy"):
        assert must in names
    assert sorted(HX.SIGNATURES) == names


def test_library_exports_every_declared_symbol():
    lib = HX.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name
    # device code for sm_103a is inside the shared object
    blob = open(HX.library_path(), "rb").read()
    assert b"sm_103a" in blob or b"sm_103" in blob


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5"])
def test_plan_matches_oracle(name):
    w = W.WORKLOADS[name]
    pd, pk = HX.query_plan(w.box, w.dims, w.cutoff)
    o = Oracle(w.box, w.dims, w.cutoff)
    assert pd.tolist() == o.pulse_dim.tolist()
    assert pk.tolist() == o.pulse_k.tolist()


@pytest.mark.parametrize("box,dims,cutoff,err", [
    ((3.0, 3.0, 3.0), (2, 1, 1), 0.0, HX.HX_ERR_ARG),
    ((3.0, 3.0, 3.0), (2, 1, 1), float("nan"), HX.HX_ERR_ARG),
    ((3.0, 3.0, 3.0), (0, 1, 1), 1.0, HX.HX_ERR_ARG),
    ((3.0, -1.0, 3.0), (2, 1, 1), 1.0, HX.HX_ERR_ARG),
    ((3.0, 3.0, 3.0), (2, 1, 1), 1.6, HX.HX_ERR_PULSES),
    ((12.0, 6.0, 6.0), (16, 1, 1), 12.0, HX.HX_ERR_PULSES),
    ((64.0, 64.0, 64.0), (17, 17, 17), 1.0, HX.HX_ERR_ARG),   # more domains than supported
])
def test_plan_errors(box, dims, cutoff, err):
    with pytest.raises(HX.HXError) as ei:
        HX.query_plan(box, dims, cutoff)
    assert ei.value.code == err
    if err == HX.HX_ERR_PULSES:
        with pytest.raises(OracleError):
            Oracle(box, dims, cutoff)


def test_init_validates_before_touching_a_device():
    lib = HX.load_library()
    h = ctypes.c_void_p()
    b = np.array([3.0, 3.0, 3.0])
    d = np.array([2, 1, 1], np.int32)
    assert lib.hx_init(ctypes.byref(h), b.ctypes.data, d.ctypes.data, -1.0, 0, 0, 0) == HX.HX_ERR_ARG
    assert lib.hx_init(None, b.ctypes.data, d.ctypes.data, 1.0, 0, 0, 0) == HX.HX_ERR_ARG
    assert lib.hx_init(ctypes.byref(h), b.ctypes.data, d.ctypes.data, 1.0, 0, 0x10, 0) == HX.HX_ERR_ARG   # no such flag
    assert lib.hx_exchange_coords(None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_status(None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_exchange_coords_host(None, None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_exchange_forces_host(None, None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_exchange_coords_host_packed(None, None, None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_exchange_forces_host_packed(None, None, None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_debug_sweep_waits(None, 1) == HX.HX_ERR_ARG
    assert lib.hx_status_async(None, None, None) == HX.HX_ERR_ARG
    assert lib.hx_get_resolved_counts(None, None, None, None) == HX.HX_ERR_ARG
    lib.hx_destroy(None)
    assert lib.hx_error_string(HX.HX_ERR_TIMEOUT)


def test_many_pulses_plan():
    # 2 pulses in each of three dims: Z0 Z1 Y0 Y1 X0 X1
    pd, pk = HX.query_plan((5.0, 5.0, 5.0), (5, 5, 5), 1.5)
    assert pd.tolist() == [2, 2, 1, 1, 0, 0] and pk.tolist() == [0, 1, 0, 1, 0, 1]


C_PROGRAM = r"""
#include <stdio.h>
#include "hx.h"
int main(void) {
  double box[3] = {5.0, 5.0, 5.0};
  int dims[3] = {5, 5, 5};
  int np = 0;
  int32_t pd[HX_MAX_PULSES], pk[HX_MAX_PULSES];
  hx_handle h = NULL;
  int rc = hx_query_plan(box, dims, 1.5, &np, pd, pk);
  printf("%d %d", rc, np);
  for (int i = 0; i < np; ++i) printf(" %d:%d", pd[i], pk[i]);
  printf(" | %d", hx_init(&h, box, dims, -1.0, 0, 0, 0));
  printf(" %d", hx_exchange_coords(NULL, NULL, NULL));
  printf(" %d\n", hx_status_async(NULL, NULL, NULL));
  hx_destroy(NULL);
  return 0;
}
"""


def test_boundary_is_plain_c(tmp_path):
    """include/hx.h compiles as C99 (no C++ or torch types) and a C program
    links libhx.so and calls it: the plan of three dimensions with two pulses
    each, and argument errors returned as codes."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib = HX.load_library()
    libdir = os.path.dirname(HX.library_path())
    src = tmp_path / "boundary.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "boundary"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", libdir, "-lhx", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    done = subprocess.run(cmd, capture_output=True, text=True)
    assert done.returncode == 0, done.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out[:2] == ["0", "6"]
    assert out[2:8] == ["2:0", "2:1", "1:0", "1:1", "0:0", "0:1"]
    assert out[8] == "|" and out[9:] == [str(HX.HX_ERR_ARG)] * 3
    assert lib is not None
