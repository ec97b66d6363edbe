"""The fused exchange beside a concurrently running local kernel (the pages'
section "SM occupancy and kernel scheduling": the local non-bonded work fills
the SMs while the halo exchange runs).

A low-priority stream runs memory-bound elementwise kernels (thousands of
short blocks each) while one coordinate and one force exchange run on a
high-priority stream. The persistent exchange grid then becomes resident
only as the other kernel's blocks retire, so its warps may wait for
producers that are not yet resident; every device wait is bounded by a
short limit (20 ms), so a stall shows up as HX_ERR_TIMEOUT instead of a
hang. Each step must leave the device status OK and match the CPU oracle
bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from domain_decomposition_halo_gb300 import hx as HX  # noqa: E402
from domain_decomposition_halo_gb300 import workloads as W  # noqa: E402

from .test_gpu_parity import Case, _bits  # noqa: E402

pytestmark = pytest.mark.gpu

MODES = [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE,
         HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES,
         HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_PDL,
         HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL, HX.HX_FLAG_RESOLVED]


@pytest.mark.parametrize("name", ["C2", "C4"])
@pytest.mark.parametrize("flags", MODES)
def test_exchange_beside_a_concurrent_kernel(name, flags):
    c = Case(W.WORKLOADS[name], flags=flags, timeout_us=20000)
    o = c.o
    hm = c.home_mask()
    x0 = o.coords().copy()
    x0[~hm] = np.nan                      # every halo slot must be rewritten
    x_ref = x0.copy()
    o.exchange_coords(x_ref)
    f0 = W.forces(c.w, o.total_slots)
    f_ref = f0.copy()
    o.exchange_forces(f_ref)
    lo = torch.cuda.Stream(priority=0)
    hi = torch.cuda.Stream(priority=-5)
    filler = torch.ones(64 * 2 ** 20, device="cuda")   # 256 MB per elementwise launch
    xt = torch.from_numpy(x0).cuda()
    ft = torch.from_numpy(f0).cuda()
    x0t, f0t = xt.clone(), ft.clone()
    for rep in range(6):
        xt.copy_(x0t)
        ft.copy_(f0t)
        torch.cuda.synchronize()
        with torch.cuda.stream(lo):
            for _ in range(8):
                filler.mul_(1.0000001)
        c.hx.exchange_coords(xt, stream=hi)
        c.hx.exchange_forces(ft, stream=hi)
        torch.cuda.synchronize()
        rc, detail = c.hx.status(stream=hi)
        assert rc == HX.HX_OK, f"rep {rep}: status {rc}, detail {detail}"
        assert np.array_equal(_bits(xt.cpu().numpy()), _bits(x_ref)), f"rep {rep}: coordinates"
        assert np.array_equal(_bits(ft.cpu().numpy()), _bits(f_ref)), f"rep {rep}: forces"
    c.hx.close()
