"""hx_exchange_coords_static: the coordinate exchange for callers that must
not allocate device memory while they run (an engine that reserves the whole
GPU for its own arena, or code that may only use memory it has accounted
for). Its scratch is a fixed file-scope device array instead of handle
memory. Checked through the C-ABI against hx_exchange_coords, bit for bit
(the tolerance of every coordinate test), on two calls in a row.

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
@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_TILES, HX.HX_FLAG_SWEEP,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES, HX.HX_FLAG_CLUSTER,
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
