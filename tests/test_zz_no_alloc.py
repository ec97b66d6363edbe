"""hx_exchange_coords_static: the coordinate exchange for callers that must
not allocate device memory while they run (an engine that reserves the whole
GPU for its own arena, or code that may only use memory it has accounted
for). Its scratch is a fixed file-scope device array instead of handle
memory. Checked through the C-ABI against hx_exchange_coords, bit for bit
(the tolerance of every coordinate test), on two calls in a row; also that
the calls leave the device's free memory unchanged, that a time-out of the
static call reaches hx_status, and that a work list beyond the array's size
is refused before anything is launched.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from domain_decomposition_halo_gb300 import hx as HX  # noqa: E402
from domain_decomposition_halo_gb300 import workloads as W  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["C2", "C5"])
@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_RESOLVED, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE])
def test_static_scratch_matches_regular_exchange(name, flags):
    w = W.WORKLOADS[name]
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff, flags=flags)
    pos = torch.from_numpy(W.positions(w)).cuda()
    n = hx.build_maps(pos)
    base = torch.empty((n, 3), device="cuda")
    hx.build_maps(pos, base)
    off, home, _ = hx.layout()
    is_home = torch.zeros(n, dtype=torch.bool, device="cuda")
    for r in range(len(off)):
        is_home[int(off[r]): int(off[r] + home[r])] = True
    lib = HX.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        x = base.clone()
        x[is_home] = x[is_home] * (1.0 - 1e-4 * (call + 1))   # different homes each call
        x[~is_home] = float("nan")                             # halos must all be rewritten
        ref = x.clone()
        hx.exchange_coords(ref)
        got = x.clone()
        rc = lib.hx_exchange_coords_static(hx._h, got.data_ptr(), stream)
        assert rc == HX.HX_OK, HX.load_library().hx_error_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(ref.view(torch.int32), got.view(torch.int32)), f"call {call}"
    assert hx.status()[0] == HX.HX_OK
    hx.close()


def test_static_scratch_rejects_unbuilt_handle():
    w = W.WORKLOADS["C1"]
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff)
    x = torch.zeros((4, 3), device="cuda")
    rc = HX.load_library().hx_exchange_coords_static(hx._h, x.data_ptr(), None)
    assert rc == HX.HX_ERR_STATE
    assert HX.load_library().hx_exchange_coords_static(None, x.data_ptr(), None) == HX.HX_ERR_ARG


def _static(hx, x, stream=None):
    lib = HX.load_library()
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return lib.hx_exchange_coords_static(hx._h, x.data_ptr(), s)


@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_RESOLVED])
def test_static_call_allocates_no_device_memory(flags):
    """The set-up (symbol address, kernel module) happens in hx_build_maps,
    so from the first static call on the device's free memory stays put."""
    w = W.WORKLOADS["C2"]
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff, flags=flags)
    pos = torch.from_numpy(W.positions(w)).cuda()
    n = hx.build_maps(pos)
    x = torch.empty((n, 3), device="cuda")
    hx.build_maps(pos, x)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _static(hx, x) == HX.HX_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert hx.status()[0] == HX.HX_OK
    hx.close()


@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE])
def test_static_call_timeout_reaches_status(flags):
    """Failure detection on the static path: a (domain, pulse) that never
    signals (host-side fault injection) makes its waiters give up after the
    bounded wait; hx_status of the calling handle reports it, hx_clear_status
    clears it, and the next static call matches the regular exchange."""
    w = W.WORKLOADS["C2"]
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff, flags=flags, timeout_us=20000)
    pos = torch.from_numpy(W.positions(w)).cuda()
    n = hx.build_maps(pos)
    base = torch.empty((n, 3), device="cuda")
    hx.build_maps(pos, base)
    hx.debug_drop_signal(0, 3, 0)
    x = base.clone()
    assert _static(hx, x) == HX.HX_OK
    rc, detail = hx.status()
    assert rc == HX.HX_ERR_TIMEOUT
    assert detail // 65536 == 0
    hx.debug_drop_signal(0, -1)
    hx.clear_status()
    assert hx.status()[0] == HX.HX_OK
    ref = base.clone()
    hx.exchange_coords(ref)
    got = base.clone()
    assert _static(hx, got) == HX.HX_OK
    torch.cuda.synchronize()
    assert hx.status()[0] == HX.HX_OK
    assert torch.equal(ref.view(torch.int32), got.view(torch.int32))
    hx.close()


def test_static_call_refuses_a_work_list_beyond_its_array():
    """64 x 64 slabs with 16 pulses in each of X and Y: 32 * 4096 signalled
    items, and with every item's chunks more than HX_STATIC_MAX_FLAGS flags.
    The static call returns HX_ERR_CAPACITY and launches nothing; the regular
    exchange runs."""
    box, dims, cutoff = (64.0, 64.0, 1.0), (64, 64, 1), 15.5
    rng = np.random.default_rng(11)
    pos = (rng.random((4 * 4096, 3)) * np.array(box)).astype(np.float32)
    hx = HX.HaloExchange(box, dims, cutoff)
    pos_t = torch.from_numpy(pos).cuda()
    n = hx.build_maps(pos_t)
    x = torch.empty((n, 3), device="cuda")
    hx.build_maps(pos_t, x)
    before = x.clone()
    assert _static(hx, x) == HX.HX_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int32), x.view(torch.int32))
    hx.exchange_coords(x)
    torch.cuda.synchronize()
    assert hx.status()[0] == HX.HX_OK
    hx.close()
