"""ctypes front end of the CPU oracle (``hx_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` import this module. The product package never does.

``build()`` compiles the C file with gcc (``-O2 -ffp-contract=off``) into
``oracle/_build/libhx_oracle.so``; ``Oracle`` wraps one decomposition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hx_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libhx_oracle.so")

ERRORS = {0: "ok", -1: "argument", -2: "pulses", -3: "range", -8: "memory"}

_libs = {}


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 -ffp-contract=off of one oracle source into a shared object,
    with OpenMP when the compiler has it (the threaded exchanges), else
    without (they then run on one thread)."""
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    done = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True)
    if done.returncode != 0:
        subprocess.run(base, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_oracle(_SRC, _LIB)
    return _LIB


def _load(path: Optional[str] = None) -> ctypes.CDLL:
    path = path or build()
    if path not in _libs:
        lib = ctypes.CDLL(path)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.oracle_create.restype = P
        lib.oracle_create.argtypes = [P, P, ctypes.c_double, P]
        lib.oracle_destroy.argtypes = [P]
        lib.oracle_build.restype = ctypes.c_int
        lib.oracle_build.argtypes = [P, P, I64]
        for name in ("oracle_num_pulses", "oracle_num_domains"):
            getattr(lib, name).restype = ctypes.c_int
            getattr(lib, name).argtypes = [P]
        for name in ("oracle_total_slots", "oracle_total_entries"):
            getattr(lib, name).restype = I64
            getattr(lib, name).argtypes = [P]
        lib.oracle_pulse_list.argtypes = [P, P, P]
        lib.oracle_lo_table.argtypes = [P, ctypes.c_int, P]
        lib.oracle_get_layout.argtypes = [P, P, P, P]
        lib.oracle_get_home_ids.argtypes = [P, P]
        lib.oracle_get_maps.argtypes = [P, P, P]
        lib.oracle_get_coords.argtypes = [P, P]
        lib.oracle_exchange_coords.argtypes = [P, P]
        lib.oracle_exchange_forces.argtypes = [P, P]
        lib.oracle_exchange_coords_par.argtypes = [P, P, ctypes.c_int]
        lib.oracle_exchange_forces_par.argtypes = [P, P, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        _ = I32
        _libs[path] = lib
    return _libs[path]


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle error {code} ({ERRORS.get(code, '?')})")
        self.code = code


class Oracle:
    """One decomposition: set-up, build (layout + maps + halo), exchanges."""

    TABLE_FIELDS = ("map_off", "size", "recv", "recv_off", "shift", "split")

    def __init__(self, box, dims, cutoff: float, lib_path: Optional[str] = None):
        self._lib = _load(lib_path)
        b = np.ascontiguousarray(box, dtype=np.float64)
        d = np.ascontiguousarray(dims, dtype=np.int32)
        err = ctypes.c_int(0)
        h = self._lib.oracle_create(_ptr(b), _ptr(d), float(cutoff), ctypes.byref(err))
        if not h:
            raise OracleError(err.value)
        self._h = h
        self.box = tuple(float(v) for v in box)
        self.dims = tuple(int(v) for v in dims)
        self.cutoff = float(cutoff)
        self.n_domains = self._lib.oracle_num_domains(h)
        self.n_pulses = self._lib.oracle_num_pulses(h)
        pd = np.zeros(max(self.n_pulses, 1), np.int32)
        pk = np.zeros(max(self.n_pulses, 1), np.int32)
        self._lib.oracle_pulse_list(h, _ptr(pd), _ptr(pk))
        self.pulse_dim = pd[: self.n_pulses].copy()
        self.pulse_k = pk[: self.n_pulses].copy()
        self.built = False

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.oracle_destroy(h)
            self._h = None

    def lo_table(self, d: int) -> np.ndarray:
        out = np.zeros(self.dims[d], np.float32)
        self._lib.oracle_lo_table(self._h, d, _ptr(out))
        return out

    def build(self, pos: np.ndarray) -> None:
        pos = np.ascontiguousarray(pos, dtype=np.float32).reshape(-1, 3)
        rc = self._lib.oracle_build(self._h, _ptr(pos), pos.shape[0])
        if rc != 0:
            raise OracleError(rc)
        self.n_atoms = pos.shape[0]
        self.total_slots = int(self._lib.oracle_total_slots(self._h))
        self.total_entries = int(self._lib.oracle_total_entries(self._h))
        nd = self.n_domains
        self.dom_offset = np.zeros(nd, np.int64)
        self.home = np.zeros(nd, np.int32)
        self.halo = np.zeros(nd, np.int32)
        self._lib.oracle_get_layout(self._h, _ptr(self.dom_offset), _ptr(self.home), _ptr(self.halo))
        self.home_ids = np.zeros(max(self.n_atoms, 1), np.int32)
        self._lib.oracle_get_home_ids(self._h, _ptr(self.home_ids))
        self.home_ids = self.home_ids[: self.n_atoms]
        self.maps = np.zeros(max(self.total_entries, 1), np.int32)
        table = np.zeros((max(self.n_pulses * nd, 1), 6), np.int64)
        self._lib.oracle_get_maps(self._h, _ptr(self.maps), _ptr(table))
        self.maps = self.maps[: self.total_entries]
        # table[p, r] = (map_off, size, recv, recv_off, shift, split)
        self.table = table[: self.n_pulses * nd].reshape(self.n_pulses, nd, 6)
        self.built = True

    def coords(self) -> np.ndarray:
        out = np.zeros((max(self.total_slots, 1), 3), np.float32)
        self._lib.oracle_get_coords(self._h, _ptr(out))
        return out[: self.total_slots]

    def map_of(self, p: int, r: int) -> np.ndarray:
        off, size = int(self.table[p, r, 0]), int(self.table[p, r, 1])
        return self.maps[off: off + size]

    def exchange_coords(self, x: np.ndarray) -> None:
        """In place on a C-contiguous fp32 [total_slots, 3] array."""
        assert x.dtype == np.float32 and x.flags.c_contiguous and x.shape == (self.total_slots, 3)
        self._lib.oracle_exchange_coords(self._h, _ptr(x))

    def exchange_forces(self, f: np.ndarray) -> None:
        """In place on a C-contiguous fp32 [total_slots, 3] array."""
        assert f.dtype == np.float32 and f.flags.c_contiguous and f.shape == (self.total_slots, 3)
        self._lib.oracle_exchange_forces(self._h, _ptr(f))

    def exchange_coords_par(self, x: np.ndarray, threads: int) -> None:
        """``exchange_coords`` with each pulse's senders on ``threads`` threads."""
        assert x.dtype == np.float32 and x.flags.c_contiguous and x.shape == (self.total_slots, 3)
        self._lib.oracle_exchange_coords_par(self._h, _ptr(x), int(threads))

    def exchange_forces_par(self, f: np.ndarray, threads: int) -> None:
        """``exchange_forces`` with each pulse's senders on ``threads`` threads."""
        assert f.dtype == np.float32 and f.flags.c_contiguous and f.shape == (self.total_slots, 3)
        self._lib.oracle_exchange_forces_par(self._h, _ptr(f), int(threads))

    def max_threads(self) -> int:
        """OpenMP's default thread count, or 1 if the oracle was built without OpenMP."""
        return int(self._lib.oracle_max_threads())
