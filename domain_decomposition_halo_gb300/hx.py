"""Python binding of libhx (ctypes): argument marshalling only.

Every step of the halo exchange runs in libhx's CUDA kernels; this module only
passes device pointers, sizes and streams through the C ABI declared in
``include/hx.h``. There is no fallback: if the library cannot be loaded the
import of a handle raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from . import build as _build

HX_OK = 0
HX_ERR_ARG = -1
HX_ERR_PULSES = -2
HX_ERR_RANGE = -3
HX_ERR_CAPACITY = -4
HX_ERR_CUDA = -5
HX_ERR_TIMEOUT = -6
HX_ERR_STATE = -7
HX_ERR_NOMEM = -8

HX_FLAG_UNORDERED_FORCES = 0x1
HX_FLAG_NO_GRAPH = 0x2
HX_FLAG_FINE_WAITS = 0x8
HX_FLAG_SWEEP_FORCES = 0x40
HX_FLAG_RESOLVED = 0x100
HX_FLAG_BULK_STORE = 0x200
HX_FLAG_PDL = 0x400

HX_MAX_PULSES = 32

# Every function declared in include/hx.h with its ctypes signature.
_P, _I, _U, _D, _I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_double, ctypes.c_int64
SIGNATURES = {
    "hx_query_plan": (_I, [_P, _P, _D, _P, _P, _P]),
    "hx_init": (_I, [_P, _P, _P, _D, _I, _U, _U]),
    "hx_build_maps": (_I, [_P, _P, _I64, _P, _I64, _P, _P]),
    "hx_get_counts": (_I, [_P, _P, _P, _P, _P]),
    "hx_get_resolved_counts": (_I, [_P, _P, _P, _P]),
    "hx_get_layout": (_I, [_P, _P, _P, _P]),
    "hx_get_home_ids": (_I, [_P, _P, _P]),
    "hx_get_maps": (_I, [_P, _P, _I64, _P]),
    "hx_exchange_coords": (_I, [_P, _P, _P]),
    "hx_exchange_forces": (_I, [_P, _P, _P]),
    "hx_exchange_coords_host": (_I, [_P, _P, _P, _P]),
    "hx_exchange_forces_host": (_I, [_P, _P, _P, _P]),
    "hx_exchange_coords_host_packed": (_I, [_P, _P, _P, _P, _P]),
    "hx_exchange_forces_host_packed": (_I, [_P, _P, _P, _P, _P]),
    "hx_exchange_coords_unfused": (_I, [_P, _P, _P]),
    "hx_exchange_forces_unfused": (_I, [_P, _P, _P]),
    "hx_exchange_coords_static": (_I, [_P, _P, _P]),
    "hx_noop": (_I, [_P, _P]),
    "hx_status": (_I, [_P, _P, _P]),
    "hx_status_async": (_I, [_P, _P, _P]),
    "hx_clear_status": (_I, [_P, _P]),
    "hx_debug_drop_signal": (_I, [_P, _I, _I, _I]),
    "hx_debug_sweep_waits": (_I, [_P, _I]),
    "hx_error_string": (ctypes.c_char_p, [_I]),
    "hx_destroy": (None, [_P]),
}

_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libhx.so (building it in-tree first if asked); raise if impossible."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path) or not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError(f"libhx.so is missing at {path}; build it with domain_decomposition_halo_gb300.build")
        path = _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class HXError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        msg = load_library().hx_error_string(code).decode()
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")
        self.code = code


def _check(code: int, what: str) -> None:
    if code != HX_OK:
        raise HXError(code, what)


def query_plan(box, dims, cutoff: float) -> Tuple[np.ndarray, np.ndarray]:
    """Global pulse list (dims, index within dim) without a GPU."""
    lib = load_library()
    b = np.ascontiguousarray(box, np.float64)
    d = np.ascontiguousarray(dims, np.int32)
    n = ctypes.c_int(0)
    pd = np.zeros(HX_MAX_PULSES, np.int32)
    pk = np.zeros(HX_MAX_PULSES, np.int32)
    _check(lib.hx_query_plan(b.ctypes.data, d.ctypes.data, float(cutoff), ctypes.byref(n), pd.ctypes.data,
                             pk.ctypes.data), "hx_query_plan")
    return pd[: n.value].copy(), pk[: n.value].copy()


def _stream_ptr(stream, device: int = 0) -> Optional[int]:
    if stream is None:
        return _current_raw_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _current_raw_stream(device: int) -> int:
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(device)
    return torch.cuda.current_stream(device).cuda_stream


class HaloExchange:
    """One decomposition on one GPU: build maps once, exchange every step."""

    def __init__(self, box, dims, cutoff: float, device: int = 0, flags: int = 0, timeout_us: int = 0):
        self._lib = load_library()
        b = np.ascontiguousarray(box, np.float64)
        d = np.ascontiguousarray(dims, np.int32)
        h = ctypes.c_void_p()
        _check(self._lib.hx_init(ctypes.byref(h), b.ctypes.data, d.ctypes.data, float(cutoff), int(device),
                                 int(flags), int(timeout_us)), "hx_init")
        self._h = h
        self._hv = h.value
        self._fn = {name: getattr(self._lib, name) for name in SIGNATURES}
        self._validated = {}   # argument name -> (id, data_ptr, numel) of the last tensor that passed the checks
        self.device = int(device)
        self.box = tuple(float(v) for v in box)
        self.dims = tuple(int(v) for v in dims)
        self.cutoff = float(cutoff)
        self.flags = int(flags)
        self.n_atoms = 0
        self.total_slots = 0

    # ------------------------------------------------------------ lifetime
    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.hx_destroy(self._h)
        self._h = None
        self._hv = None
        self._validated = {}

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ------------------------------------------------------------ build
    def _check_tensor(self, t, numel: int, what: str, dtype=None):
        import torch
        dtype = dtype or torch.float32
        if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
            raise ValueError(f"{what} must be a contiguous {dtype} CUDA tensor")
        if t.device.index != self.device:
            raise ValueError(f"{what} is on cuda:{t.device.index}, the handle on cuda:{self.device}")
        if t.numel() < numel:
            raise ValueError(f"{what} holds {t.numel()} elements, {numel} needed")

    def build_maps(self, pos, coords=None, stream=None) -> int:
        """Build from positions (CUDA fp32 [n, 3]); fill ``coords`` (CUDA fp32
        [slots, 3]) when given. Returns the number of slots of the layout."""
        n = pos.numel() // 3
        self._check_tensor(pos, 3 * n, "pos")
        needed = ctypes.c_int64(0)
        cap = coords.numel() // 3 if coords is not None else 0
        if coords is not None:
            self._check_tensor(coords, 0, "coords")
        rc = self._lib.hx_build_maps(self._h, pos.data_ptr() if n else None, n,
                                     coords.data_ptr() if coords is not None else None, cap,
                                     ctypes.byref(needed), _stream_ptr(stream, self.device))
        if rc not in (HX_OK, HX_ERR_CAPACITY) or (rc == HX_ERR_CAPACITY and coords is not None):
            _check(rc, "hx_build_maps")
        self.n_atoms = n
        self.total_slots = int(needed.value)
        return self.total_slots

    def counts(self) -> Tuple[int, int, int, int]:
        nd, npl = ctypes.c_int(0), ctypes.c_int(0)
        ts, te = ctypes.c_int64(0), ctypes.c_int64(0)
        _check(self._lib.hx_get_counts(self._h, ctypes.byref(nd), ctypes.byref(npl), ctypes.byref(ts),
                                       ctypes.byref(te)), "hx_get_counts")
        return nd.value, npl.value, ts.value, te.value

    def resolved_counts(self) -> Tuple[int, int, int]:
        """Resolved mode's force trees: (pairs, quads, general)."""
        a, b, c = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        _check(self._lib.hx_get_resolved_counts(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
               "hx_get_resolved_counts")
        return a.value, b.value, c.value

    def layout(self):
        nd = self.counts()[0]
        off = np.zeros(nd, np.int64)
        home = np.zeros(nd, np.int32)
        halo = np.zeros(nd, np.int32)
        _check(self._lib.hx_get_layout(self._h, off.ctypes.data, home.ctypes.data, halo.ctypes.data),
               "hx_get_layout")
        return off, home, halo

    def home_ids(self, out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty(max(self.n_atoms, 1), dtype=torch.int32, device=f"cuda:{self.device}")[: self.n_atoms]
        if self.n_atoms:
            self._check_tensor(out, self.n_atoms, "home_ids", torch.int32)
        _check(self._lib.hx_get_home_ids(self._h, out.data_ptr() if self.n_atoms else None, _stream_ptr(stream, self.device)),
               "hx_get_home_ids")
        return out

    def maps(self):
        nd, npl, _, te = self.counts()
        m = np.zeros(max(te, 1), np.int32)
        table = np.zeros((max(npl * nd, 1), 6), np.int64)
        _check(self._lib.hx_get_maps(self._h, m.ctypes.data, max(te, 1), table.ctypes.data), "hx_get_maps")
        return m[:te], table[: npl * nd].reshape(npl, nd, 6)

    # ------------------------------------------------------------ per step
    def _step_ptr(self, t, what: str) -> int:
        """Data pointer of a per-step buffer. The full checks run once per
        tensor object and storage; later calls with the same tensor only
        compare its pointer and size."""
        ptr = t.data_ptr()
        key = (id(t), ptr, t.numel(), self.total_slots)
        if self._validated.get(what) != key:
            self._check_tensor(t, 3 * self.total_slots, what)
            self._validated[what] = key
        return ptr

    def exchange_coords(self, coords, stream=None) -> None:
        rc = self._fn["hx_exchange_coords"](self._hv, self._step_ptr(coords, "coords"),
                                            _stream_ptr(stream, self.device))
        if rc:
            _check(rc, "hx_exchange_coords")

    def exchange_forces(self, forces, stream=None) -> None:
        rc = self._fn["hx_exchange_forces"](self._hv, self._step_ptr(forces, "forces"),
                                            _stream_ptr(stream, self.device))
        if rc:
            _check(rc, "hx_exchange_forces")

    def _check_host(self, t, what: str) -> None:
        if t.is_cuda or t.dtype.itemsize != 4 or not t.is_floating_point() or not t.is_contiguous():
            raise ValueError(f"{what} must be a contiguous float32 host tensor (page-locked)")
        if t.numel() < 3 * self.total_slots:
            raise ValueError(f"{what} holds {t.numel()} elements, {3 * self.total_slots} needed")

    def exchange_coords_host(self, coords_host, coords_dev, stream=None) -> None:
        """Home coordinates from ``coords_host`` (page-locked CPU fp32 [slots, 3])
        into ``coords_dev``, the coordinate exchange there, and every halo
        slot back into ``coords_host``; queued on ``stream``."""
        self._check_host(coords_host, "coords_host")
        self._check_tensor(coords_dev, 3 * self.total_slots, "coords_dev")
        _check(self._lib.hx_exchange_coords_host(self._h, coords_host.data_ptr(), coords_dev.data_ptr(),
                                                 _stream_ptr(stream, self.device)), "hx_exchange_coords_host")

    def exchange_forces_host(self, forces_host, forces_dev, stream=None) -> None:
        """Every slot's force from ``forces_host`` into ``forces_dev``, the force
        exchange there, and every home force back into ``forces_host``."""
        self._check_host(forces_host, "forces_host")
        self._check_tensor(forces_dev, 3 * self.total_slots, "forces_dev")
        _check(self._lib.hx_exchange_forces_host(self._h, forces_host.data_ptr(), forces_dev.data_ptr(),
                                                 _stream_ptr(stream, self.device)), "hx_exchange_forces_host")

    def _check_host_packed(self, t, n_slots: int, what: str) -> None:
        if t.is_cuda or t.dtype.itemsize != 4 or not t.is_floating_point() or not t.is_contiguous():
            raise ValueError(f"{what} must be a contiguous float32 host tensor (page-locked for asynchronous copies)")
        if t.numel() < 3 * n_slots:
            raise ValueError(f"{what} holds {t.numel()} elements, {3 * n_slots} needed")

    def exchange_coords_host_packed(self, home_host, halo_host, coords_dev, stream=None) -> None:
        """Packed home coordinates from ``home_host`` (CPU fp32 [n_atoms, 3], layout
        order) into ``coords_dev``'s home slots, the coordinate exchange there,
        and every halo slot packed into ``halo_host`` (CPU fp32 [halo slots, 3]);
        queued on ``stream``."""
        n_home = self.n_atoms
        self._check_host_packed(home_host, n_home, "home_host")
        self._check_host_packed(halo_host, self.total_slots - n_home, "halo_host")
        self._check_tensor(coords_dev, 3 * self.total_slots, "coords_dev")
        _check(self._lib.hx_exchange_coords_host_packed(self._h, home_host.data_ptr(), halo_host.data_ptr(),
                                                        coords_dev.data_ptr(), _stream_ptr(stream, self.device)),
               "hx_exchange_coords_host_packed")

    def exchange_forces_host_packed(self, forces_host, home_forces_host, forces_dev, stream=None) -> None:
        """Every slot's force from ``forces_host`` (CPU fp32 [slots, 3]) into
        ``forces_dev``, the force exchange there, and the home forces packed
        into ``home_forces_host`` (CPU fp32 [n_atoms, 3], layout order)."""
        self._check_host_packed(forces_host, self.total_slots, "forces_host")
        self._check_host_packed(home_forces_host, self.n_atoms, "home_forces_host")
        self._check_tensor(forces_dev, 3 * self.total_slots, "forces_dev")
        _check(self._lib.hx_exchange_forces_host_packed(self._h, forces_host.data_ptr(), home_forces_host.data_ptr(),
                                                        forces_dev.data_ptr(), _stream_ptr(stream, self.device)),
               "hx_exchange_forces_host_packed")

    def exchange_coords_unfused(self, coords, stream=None) -> None:
        self._check_tensor(coords, 3 * self.total_slots, "coords")
        _check(self._lib.hx_exchange_coords_unfused(self._h, coords.data_ptr(), _stream_ptr(stream, self.device)),
               "hx_exchange_coords_unfused")

    def exchange_forces_unfused(self, forces, stream=None) -> None:
        self._check_tensor(forces, 3 * self.total_slots, "forces")
        _check(self._lib.hx_exchange_forces_unfused(self._h, forces.data_ptr(), _stream_ptr(stream, self.device)),
               "hx_exchange_forces_unfused")

    def exchange_coords_static(self, coords, stream=None) -> None:
        """hx_exchange_coords without any device allocation: for callers that
        must not allocate while they run (see include/hx.h)."""
        self._check_tensor(coords, 3 * self.total_slots, "coords")
        _check(self._lib.hx_exchange_coords_static(self._h, coords.data_ptr(), _stream_ptr(stream, self.device)),
               "hx_exchange_coords_static")

    def noop(self, stream=None) -> None:
        rc = self._fn["hx_noop"](self._hv, _stream_ptr(stream, self.device))
        if rc:
            _check(rc, "hx_noop")

    # ------------------------------------------------------------ status
    def status(self, stream=None) -> Tuple[int, int]:
        detail = ctypes.c_int(-1)
        rc = self._lib.hx_status(self._h, _stream_ptr(stream, self.device), ctypes.byref(detail))
        return rc, detail.value

    def status_async(self, out, stream=None) -> None:
        """Queue the sticky status and detail into ``out`` (a CPU int32 tensor of
        2 elements, page-locked for an asynchronous copy) without synchronising;
        ``out`` holds them once ``stream`` has passed this call."""
        import torch
        if out.is_cuda or out.dtype != torch.int32 or out.numel() < 2 or not out.is_contiguous():
            raise ValueError("out must be a contiguous int32 host tensor of 2 elements")
        _check(self._lib.hx_status_async(self._h, out.data_ptr(), _stream_ptr(stream, self.device)), "hx_status_async")

    def clear_status(self, stream=None) -> None:
        _check(self._lib.hx_clear_status(self._h, _stream_ptr(stream, self.device)), "hx_clear_status")

    def debug_drop_signal(self, direction: int, domain: int, pulse: int = 0) -> None:
        _check(self._lib.hx_debug_drop_signal(self._h, int(direction), int(domain), int(pulse)),
               "hx_debug_drop_signal")

    def debug_sweep_waits(self, mode: int) -> None:
        """Force sweep waits: 0 automatic, 1 segment by segment, 2 whole unit."""
        _check(self._lib.hx_debug_sweep_waits(self._h, int(mode)), "hx_debug_sweep_waits")
