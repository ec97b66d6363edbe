"""GPU parity of libhx against the CPU oracle, through the C ABI.

Maps, layout, home order and coordinates must match bit for bit; forces bit
for bit in ordered mode and within 1e-6 of the sum of absolute values of the
reduced terms (the scale of each sum) in unordered mode.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from domain_decomposition_halo_gb300 import hx as HX
from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import Oracle

pytestmark = pytest.mark.gpu

ALL_MODES = [0, HX.HX_FLAG_NO_GRAPH, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_NO_GRAPH,
             HX.HX_FLAG_SWEEP_FORCES, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES,
             HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_NO_GRAPH, HX.HX_FLAG_RESOLVED,
             HX.HX_FLAG_RESOLVED | HX.HX_FLAG_NO_GRAPH, HX.HX_FLAG_BULK_STORE,
             HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE, HX.HX_FLAG_RESOLVED | HX.HX_FLAG_PDL,
             HX.HX_FLAG_PDL, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_PDL,
             HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_PDL,
             HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_NO_GRAPH,
             HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL]


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


class Case:
    """A workload built on both sides."""

    def __init__(self, w, flags=0, timeout_us=0, pos=None):
        self.w = w
        self.pos = W.positions(w) if pos is None else pos
        self.o = Oracle(w.box, w.dims, w.cutoff)
        self.o.build(self.pos)
        self.hx = HX.HaloExchange(w.box, w.dims, w.cutoff, flags=flags, timeout_us=timeout_us)
        self.pos_t = torch.from_numpy(self.pos).cuda()
        self.slots = self.hx.build_maps(self.pos_t)
        self.coords = torch.full((max(self.slots, 1), 3), float("nan"), device="cuda")[: self.slots]
        self.hx.build_maps(self.pos_t, self.coords)
        torch.cuda.synchronize()

    def home_mask(self):
        m = np.zeros(self.o.total_slots, bool)
        for r in range(self.o.n_domains):
            m[self.o.dom_offset[r]: self.o.dom_offset[r] + self.o.home[r]] = True
        return m


def check_build(c: Case):
    o = c.o
    assert c.slots == o.total_slots
    off, home, halo = c.hx.layout()
    assert np.array_equal(off, o.dom_offset)
    assert np.array_equal(home, o.home)
    assert np.array_equal(halo, o.halo)
    ids = c.hx.home_ids().cpu().numpy()
    assert np.array_equal(ids, o.home_ids)
    maps, table = c.hx.maps()
    assert np.array_equal(maps, o.maps)
    assert np.array_equal(table, o.table)
    assert np.array_equal(_bits(c.coords.cpu().numpy()), _bits(o.coords()))


def check_coord_steps(c: Case, steps=3, unfused=False):
    o = c.o
    rng = np.random.default_rng(123)
    hm = c.home_mask()
    x = o.coords().copy()
    for s in range(steps):
        # move home atoms a little (stays inside the box: exchanged values are
        # compared, not re-partitioned), poison every halo slot
        if s > 0 and hm.any():
            x[hm] = (x[hm] * np.float32(0.999) + np.float32(1e-3) * rng.random((hm.sum(), 3), np.float32)).astype(np.float32)
        x[~hm] = np.nan
        xt = torch.from_numpy(x).cuda()
        if unfused:
            c.hx.exchange_coords_unfused(xt)
        else:
            c.hx.exchange_coords(xt)
        o.exchange_coords(x)
        assert np.array_equal(_bits(xt.cpu().numpy()), _bits(x)), f"coordinate step {s}"
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)


def check_force_steps(c: Case, steps=2, ordered=True, unfused=False):
    o = c.o
    for s in range(steps):
        f = W.forces(c.w, o.total_slots)
        if s:
            f = (f * np.float32(1.0 + s)).astype(np.float32)
        ft = torch.from_numpy(f).cuda()
        if unfused:
            c.hx.exchange_forces_unfused(ft)
        else:
            c.hx.exchange_forces(ft)
        ref = f.copy()
        o.exchange_forces(ref)
        got = ft.cpu().numpy()
        if ordered:
            assert np.array_equal(_bits(got), _bits(ref)), f"force step {s}"
        else:
            scale = np.abs(f).copy()
            o.exchange_forces(scale)
            assert np.all(np.abs(got.astype(np.float64) - ref) <= 1e-6 * scale + 1e-30), f"force step {s}"
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
@pytest.mark.parametrize("flags", ALL_MODES)
def test_parity_configs(name, flags):
    c = Case(W.WORKLOADS[name], flags=flags)
    check_build(c)
    check_coord_steps(c)
    check_force_steps(c)


@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_RESOLVED,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES])
def test_parity_c5_full_size(flags):
    """12M atoms, 256 domains: the bench's configuration and launch path."""
    c = Case(W.WORKLOADS["C5"], flags=flags)
    check_build(c)
    check_coord_steps(c, steps=2)
    check_force_steps(c, steps=1)


@pytest.mark.parametrize("name", ["C2", "C3", "C4"])
@pytest.mark.parametrize("extra", [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE])
def test_unordered_forces(name, extra):
    c = Case(W.WORKLOADS[name], flags=HX.HX_FLAG_UNORDERED_FORCES | extra)
    check_force_steps(c, steps=2, ordered=False)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
def test_unfused_baseline(name):
    c = Case(W.WORKLOADS[name])
    check_coord_steps(c, steps=2, unfused=True)
    check_force_steps(c, steps=1, unfused=True)


@pytest.mark.parametrize("box,dims,cutoff,n", [
    ((3.0, 3.0, 3.0), (1, 1, 1), 1.0, 500),       # no pulses: identity
    ((2.0, 2.0, 2.0), (2, 2, 2), 0.5, 0),         # no atoms: every pulse empty, still signalled
    ((2.0, 2.0, 2.0), (2, 2, 2), 0.5, 7),         # ragged, mostly empty pulses
    ((5.0, 5.0, 3.0), (5, 5, 1), 1.5, 30000),     # 2 pulses in X and Y, forwarding chains
    ((5.0, 5.0, 5.0), (5, 5, 5), 1.5, 40000),     # 6 pulses
    ((6.0, 4.0, 5.0), (4, 1, 5), 1.3, 30000),     # mixed pulse counts
    ((4.0, 4.5, 4.0), (1, 3, 1), 2.9, 20000),     # np = n - 1
    ((3.0, 3.0, 3.0), (3, 3, 3), 0.6, 2700),      # 27 domains
    ((40.0, 3.0, 3.0), (40, 1, 1), 1.0, 36000),   # many small domains along one dim
])
@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_RESOLVED, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE])
def test_parity_shapes(box, dims, cutoff, n, flags):
    w = W.custom("shape", n, box, dims, cutoff, seed=7 + n)
    pulse_dims, _ = HX.query_plan(box, dims, cutoff)
    copies_bound = int(np.prod([1 + int(np.sum(pulse_dims == d)) for d in range(3)]))
    if flags & HX.HX_FLAG_RESOLVED and copies_bound > 8:
        # a home atom may have more than 7 copies: the resolved tables refuse
        # the plan at build time if one does (and are exact if none does)
        try:
            c = Case(w, flags=flags)
        except HX.HXError as e:
            assert e.code == HX.HX_ERR_PULSES
            return
    else:
        c = Case(w, flags=flags)
    check_build(c)
    check_coord_steps(c)
    check_force_steps(c)


def _copies_per_atom(o):
    """Copies of each home atom, replaying the oracle's maps: a received
    slot's origin is the origin of the slot it was sent from."""
    origin = np.full(o.total_slots, -1, np.int64)
    for r in range(o.n_domains):
        origin[o.dom_offset[r]: o.dom_offset[r] + o.home[r]] = np.arange(o.dom_offset[r], o.dom_offset[r] + o.home[r])
    for p in range(o.n_pulses):
        for r in range(o.n_domains):
            m = o.map_of(p, r)
            q, off = int(o.table[p, r, 2]), int(o.table[p, r, 3])
            dst = o.dom_offset[q] + off
            origin[dst: dst + len(m)] = origin[o.dom_offset[r] + m]
    halo = np.concatenate([origin[o.dom_offset[r] + o.home[r]: o.dom_offset[r] + o.home[r] + o.halo[r]]
                           for r in range(o.n_domains)])
    assert np.all(halo >= 0)
    return np.bincount(halo, minlength=o.total_slots)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
def test_resolved_tree_classes(name):
    """Resolved mode's force trees: one per home atom with copies; an atom
    with one copy is a pair; corner trees of four nodes may be quads; the
    general class holds the rest. Parity of every class is in
    test_parity_configs."""
    c = Case(W.WORKLOADS[name], flags=HX.HX_FLAG_RESOLVED)
    pairs, quads, general = c.hx.resolved_counts()
    copies = _copies_per_atom(c.o)
    assert pairs == int(np.sum(copies == 1))
    assert pairs + quads + general == int(np.sum(copies > 0))
    assert quads <= int(np.sum(copies == 3))
    if name in ("C2", "C4"):   # 1 pulse per dimension: corners are quads, 3-dimension corners general
        assert quads == int(np.sum(copies == 3)) and quads > 0 and general == int(np.sum(copies == 7)) > 0
    if name == "C3":           # 2 pulses along x: relayed copies make three-node chains
        assert quads == 0 and general == int(np.sum(copies == 2)) > 0
    if name == "C1":
        assert quads == 0 and general == 0
    if name == "C1":   # a handle in another mode has no trees
        assert Case(W.WORKLOADS[name], flags=HX.HX_FLAG_FINE_WAITS).hx.resolved_counts() == (0, 0, 0)


@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES])
def test_misaligned_buffers(flags):
    """Caller buffers that start 4, 8 or 12 bytes past a 16-byte boundary (the
    bulk-store pack and the slot sweep move 16-byte-aligned middles in bulk
    and the edges with plain loads and stores)."""
    w = W.WORKLOADS["C2"]
    c = Case(w, flags=flags)
    for shift in (1, 2, 3):
        x = c.o.coords().copy()
        hm = c.home_mask()
        x[~hm] = np.nan
        big = torch.zeros(x.size + 8, device="cuda")
        xt = big[shift: shift + x.size].view(-1, 3)
        xt.copy_(torch.from_numpy(x))
        c.hx.exchange_coords(xt)
        c.o.exchange_coords(x)
        assert np.array_equal(_bits(xt.cpu().numpy()), _bits(x))
        f = W.forces(w, c.o.total_slots)
        fbig = torch.zeros(f.size + 8, device="cuda")
        ft = fbig[shift: shift + f.size].view(-1, 3)
        ft.copy_(torch.from_numpy(f))
        c.hx.exchange_forces(ft)
        ref = f.copy()
        c.o.exchange_forces(ref)
        assert np.array_equal(_bits(ft.cpu().numpy()), _bits(ref))
    assert c.hx.status()[0] == 0


def test_boundary_atoms():
    below = float(np.nextafter(np.float32(4.0), np.float32(0)))
    vals = [0.0, 1.0, 2.0, 3.0, below, float(np.nextafter(np.float32(1.0), np.float32(0))),
            float(np.nextafter(np.float32(3.0), np.float32(0))), 0.5, 2.5, -0.0]
    pts = np.array([[a, b, c] for a in vals for b in vals[:6] for c in vals[:4]], np.float32)
    w = W.custom("edge", len(pts), (4.0, 4.0, 4.0), (2, 2, 2), 1.0, seed=0)
    c = Case(w, pos=pts)
    check_build(c)
    check_coord_steps(c)


def test_many_steps_reuse_signals():
    """Epoch-valued signals are never reset between launches: 200 steps."""
    for flags in (0, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES, HX.HX_FLAG_RESOLVED,
                  HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE, HX.HX_FLAG_RESOLVED | HX.HX_FLAG_PDL,
                  HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL):
        c = Case(W.WORKLOADS["C2"], flags=flags)
        x = c.o.coords().copy()
        xt = torch.from_numpy(x).cuda()
        f0 = W.forces(c.w, c.o.total_slots)
        for _ in range(200):
            c.hx.exchange_coords(xt)
            ft = torch.from_numpy(f0).cuda()
            c.hx.exchange_forces(ft)
        ref = f0.copy()
        c.o.exchange_forces(ref)
        assert np.array_equal(_bits(ft.cpu().numpy()), _bits(ref))
        assert np.array_equal(_bits(xt.cpu().numpy()), _bits(x))
        assert c.hx.status()[0] == 0


def test_side_stream():
    c = Case(W.WORKLOADS["C2"])
    s = torch.cuda.Stream()
    x = c.o.coords().copy()
    hm = c.home_mask()
    x[~hm] = np.nan
    with torch.cuda.stream(s):
        xt = torch.from_numpy(x).cuda(non_blocking=False)
        c.hx.exchange_coords(xt, stream=s)
    s.synchronize()
    c.o.exchange_coords(x)
    assert np.array_equal(_bits(xt.cpu().numpy()), _bits(x))


def test_rebuild_replaces_maps():
    c = Case(W.WORKLOADS["C1"])
    w2 = W.WORKLOADS["C2"]
    hx = HX.HaloExchange(w2.box, w2.dims, w2.cutoff)
    pos = torch.from_numpy(W.positions(w2)).cuda()
    n1 = hx.build_maps(pos)
    coords = torch.empty((n1, 3), device="cuda")
    hx.build_maps(pos, coords)
    pos2 = W.positions(W.custom("again", 20000, w2.box, w2.dims, w2.cutoff, seed=99))
    o2 = Oracle(w2.box, w2.dims, w2.cutoff)
    o2.build(pos2)
    n2 = hx.build_maps(torch.from_numpy(pos2).cuda())
    coords2 = torch.empty((n2, 3), device="cuda")
    hx.build_maps(torch.from_numpy(pos2).cuda(), coords2)
    assert np.array_equal(_bits(coords2.cpu().numpy()), _bits(o2.coords()))
    del c


def test_errors():
    w = W.WORKLOADS["C1"]
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff)
    x = torch.zeros((10, 3), device="cuda")
    with pytest.raises(HX.HXError) as ei:
        hx._check_tensor = lambda *a, **k: None       # reach the C ABI's own state check
        hx.exchange_coords(x)
    assert ei.value.code == HX.HX_ERR_STATE
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff)
    bad = torch.from_numpy(np.array([[1.0, 1.0, 1.0], [3.2, 1.0, 1.0]], np.float32)).cuda()
    with pytest.raises(HX.HXError) as ei:
        hx.build_maps(bad)
    assert ei.value.code == HX.HX_ERR_RANGE
    nan = torch.from_numpy(np.array([[float("nan"), 1.0, 1.0]], np.float32)).cuda()
    with pytest.raises(HX.HXError) as ei:
        hx.build_maps(nan)
    assert ei.value.code == HX.HX_ERR_RANGE
    pos = torch.from_numpy(W.positions(w)).cuda()
    n = hx.build_maps(pos)
    small = torch.empty((n - 1, 3), device="cuda")
    with pytest.raises(HX.HXError) as ei:
        hx.build_maps(pos, small)
    assert ei.value.code == HX.HX_ERR_CAPACITY
    # resolved coordinates with swept forces is not a mode; 0x4, 0x10, 0x20 and
    # 0x80 are retired or unassigned bits
    for bad in (HX.HX_FLAG_RESOLVED | HX.HX_FLAG_SWEEP_FORCES, 0x4, 0x10, 0x20, 0x80):
        with pytest.raises(HX.HXError) as ei:
            HX.HaloExchange(w.box, w.dims, w.cutoff, flags=bad)
        assert ei.value.code == HX.HX_ERR_ARG
    with pytest.raises(HX.HXError):
        HX.HaloExchange(w.box, w.dims, w.cutoff, device=torch.cuda.device_count())


@pytest.mark.parametrize("direction", [0, 1])
@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_BULK_STORE, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES |
                                   HX.HX_FLAG_PDL])
def test_dropped_signal_times_out_and_recovers(direction, flags):
    """Failure detection without a device fault: a (domain, pulse) that never
    signals makes its waiters give up after the bounded wait; the kernel
    finishes, hx_status reports HX_ERR_TIMEOUT and the item, and after
    hx_clear_status the exchange is correct again."""
    c = Case(W.WORKLOADS["C2"], flags=flags, timeout_us=20000)
    nd = c.o.n_domains
    pulse = 0 if direction == 0 else c.o.n_pulses - 1
    c.hx.debug_drop_signal(direction, 3, pulse)
    x = c.o.coords().copy()
    xt = torch.from_numpy(x).cuda()
    f = W.forces(c.w, c.o.total_slots)
    ft = torch.from_numpy(f).cuda()
    if direction == 0:
        c.hx.exchange_coords(xt)
    else:
        c.hx.exchange_forces(ft)
    rc, detail = c.hx.status()
    assert rc == HX.HX_ERR_TIMEOUT
    # the first wait to give up is on the dropped item, or on an item of the
    # same direction that was itself held up by it (waits time out together)
    assert detail // 65536 == direction
    item = detail % 65536
    p_item = item // nd
    if direction == 1 and flags & HX.HX_FLAG_SWEEP_FORCES:
        # a unit is labelled by its first map's (pulse, domain); a cascade can
        # report any unit downstream of the dropped one
        assert 0 <= item < c.o.n_pulses * nd
    else:
        assert item == pulse * nd + 3 or (p_item > pulse if direction == 0 else p_item < pulse)
    c.hx.debug_drop_signal(direction, -1)
    c.hx.clear_status()
    assert c.hx.status()[0] == 0
    check_coord_steps(c, steps=2)
    check_force_steps(c, steps=1)


@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL])
def test_status_async_reports_without_synchronising(flags):
    """hx_status_async queues the sticky status on the stream: OK after a clean
    exchange, HX_ERR_TIMEOUT with the same detail as hx_status after a dropped
    signal, and OK again once cleared."""
    c = Case(W.WORKLOADS["C2"], flags=flags, timeout_us=20000)
    out = torch.full((2,), 7, dtype=torch.int32).pin_memory()
    xt = torch.from_numpy(c.o.coords().copy()).cuda()
    c.hx.exchange_coords(xt)
    c.hx.status_async(out)
    torch.cuda.synchronize()
    assert out.tolist() == [HX.HX_OK, -1]
    c.hx.debug_drop_signal(0, 3, 0)
    c.hx.exchange_coords(xt)
    c.hx.status_async(out)
    torch.cuda.synchronize()
    rc, detail = c.hx.status()
    assert rc == HX.HX_ERR_TIMEOUT and out.tolist() == [rc, detail]
    c.hx.debug_drop_signal(0, -1)
    c.hx.clear_status()
    c.hx.exchange_coords(xt)
    c.hx.status_async(out)
    torch.cuda.synchronize()
    assert out.tolist() == [HX.HX_OK, -1]
    with pytest.raises(ValueError):
        c.hx.status_async(torch.empty(2, dtype=torch.int32, device="cuda"))


@pytest.mark.parametrize("name", ["C4", "C5"])
@pytest.mark.parametrize("flags", [HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_RESOLVED | HX.HX_FLAG_PDL,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_PDL,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_PDL, HX.HX_FLAG_PDL,
                                   HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES |
                                   HX.HX_FLAG_PDL])
def test_back_to_back_steps(name, flags):
    """Forty coordinate + force exchanges queued back to back on one stream
    (no synchronisation between them, so consecutive launches may overlap
    their start-up) give the oracle's result of the same forty steps, bit
    for bit: coordinates are idempotent, forces accumulate every step."""
    c = Case(W.WORKLOADS[name], flags=flags)
    x = c.o.coords().copy()
    f = W.forces(c.w, c.o.total_slots)
    xt = torch.from_numpy(x).cuda()
    ft = torch.from_numpy(f).cuda()
    for _ in range(40):
        c.hx.exchange_coords(xt)
        c.hx.exchange_forces(ft)
    torch.cuda.synchronize()
    assert c.hx.status()[0] == 0
    for _ in range(40):
        c.o.exchange_coords(x)
        c.o.exchange_forces(f)
    assert np.array_equal(_bits(xt.cpu().numpy()), _bits(x))
    assert np.array_equal(_bits(ft.cpu().numpy()), _bits(f))


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
@pytest.mark.parametrize("flags", [HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES,
                                   HX.HX_FLAG_RESOLVED, 0])
def test_host_buffer_exchanges(name, flags):
    """hx_exchange_coords_host / hx_exchange_forces_host: home coordinates in,
    halo coordinates out; every force in, home forces out; bit-exact."""
    w = W.WORKLOADS[name]
    c = Case(w, flags=flags)
    o = c.o
    hm = c.home_mask()
    x0 = o.coords()
    ref = x0.copy()
    o.exchange_coords(ref)
    host = torch.from_numpy(x0.copy()).pin_memory()
    host.numpy()[~hm] = np.nan   # halo slots come only from the exchange
    dev = torch.full((c.slots, 3), float("nan"), device="cuda")
    for _ in range(2):           # a second call on the same buffers gives the same result
        c.hx.exchange_coords_host(host, dev)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(host.numpy()), _bits(ref))
    f0 = W.forces(w, c.slots)
    fref = f0.copy()
    o.exchange_forces(fref)
    fh = torch.from_numpy(f0.copy()).pin_memory()
    fd = torch.full((c.slots, 3), float("nan"), device="cuda")
    c.hx.exchange_forces_host(fh, fd)
    torch.cuda.synchronize()
    got = fh.numpy()
    assert np.array_equal(_bits(got[hm]), _bits(fref[hm]))     # home forces: the reduced sums
    assert np.array_equal(_bits(got[~hm]), _bits(f0[~hm]))     # halo forces: left as given
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4"])
@pytest.mark.parametrize("flags", [HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL,
                                   HX.HX_FLAG_RESOLVED | HX.HX_FLAG_PDL, 0])
def test_host_packed_exchanges(name, flags):
    """hx_exchange_coords_host_packed / hx_exchange_forces_host_packed: packed
    home coordinates in, packed halo coordinates out (layout order); every
    slot's force in, packed home forces out; bit-exact, twice on the same
    buffers, inputs left as given."""
    w = W.WORKLOADS[name]
    c = Case(w, flags=flags)
    o = c.o
    hm = c.home_mask()
    x0 = o.coords()
    ref = x0.copy()
    o.exchange_coords(ref)
    home = torch.from_numpy(x0[hm].copy()).pin_memory()
    halo = torch.full((int((~hm).sum()), 3), float("nan")).pin_memory()
    dev = torch.full((c.slots, 3), float("nan"), device="cuda")
    for _ in range(2):
        c.hx.exchange_coords_host_packed(home, halo, dev)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(halo.numpy()), _bits(ref[~hm]))
        assert np.array_equal(_bits(dev.cpu().numpy()), _bits(ref))
        assert np.array_equal(_bits(home.numpy()), _bits(x0[hm]))
    f0 = W.forces(w, c.slots)
    fref = f0.copy()
    o.exchange_forces(fref)
    fh = torch.from_numpy(f0.copy()).pin_memory()
    hf = torch.full((int(hm.sum()), 3), float("nan")).pin_memory()
    fd = torch.full((c.slots, 3), float("nan"), device="cuda")
    for _ in range(2):
        c.hx.exchange_forces_host_packed(fh, hf, fd)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(hf.numpy()), _bits(fref[hm]))   # home forces: the reduced sums
        assert np.array_equal(_bits(fh.numpy()), _bits(f0))         # the input is left as given
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)


def test_host_packed_full_size():
    """The packed host-buffer calls on the 12M-atom workload in the bench's
    modes: packed halo coordinates and home forces bit-exact against the
    oracle."""
    w = W.WORKLOADS["C5"]
    c = Case(w, flags=HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL)
    o = c.o
    hm = c.home_mask()
    x0 = o.coords()
    ref = x0.copy()
    o.exchange_coords(ref)
    home = torch.from_numpy(x0[hm].copy()).pin_memory()
    halo = torch.empty((int((~hm).sum()), 3)).pin_memory()
    dev = torch.empty((c.slots, 3), device="cuda")
    c.hx.exchange_coords_host_packed(home, halo, dev)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(halo.numpy()), _bits(ref[~hm]))
    f0 = W.forces(w, c.slots)
    fref = f0.copy()
    o.exchange_forces(fref)
    hf = torch.empty((int(hm.sum()), 3)).pin_memory()
    c.hx.exchange_forces_host_packed(torch.from_numpy(f0).pin_memory(), hf, dev)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(hf.numpy()), _bits(fref[hm]))
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)


def test_host_packed_misaligned_pageable_and_rebuild():
    """Packed buffers 4 bytes off a 16-byte boundary and in pageable memory
    (synchronous copies) give the same bits; a rebuild with more atoms grows
    the packing buffer; undersized buffers are refused before any copy."""
    w = W.WORKLOADS["C2"]
    pos = W.positions(w)
    c = Case(w, flags=HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES, pos=pos[: len(pos) // 2].copy())
    for step, p in enumerate((pos[: len(pos) // 2].copy(), pos)):
        if step:
            c = Case(w, flags=HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_SWEEP_FORCES, pos=p)
        o = c.o
        hm = c.home_mask()
        ref = o.coords().copy()
        o.exchange_coords(ref)
        nh, nl = int(hm.sum()), int((~hm).sum())
        store = torch.empty(3 * nh + 1, dtype=torch.float32).pin_memory()
        home = store[1:].view(nh, 3)                       # 4 bytes past a 16-byte boundary
        home.copy_(torch.from_numpy(o.coords()[hm]))
        halo = torch.from_numpy(np.full((nl, 3), np.nan, np.float32))   # pageable
        dev = torch.empty((c.slots, 3), device="cuda")
        c.hx.exchange_coords_host_packed(home, halo, dev)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(halo.numpy()), _bits(ref[~hm]))
        with pytest.raises(ValueError):
            c.hx.exchange_coords_host_packed(home[:-1], halo, dev)
        with pytest.raises(ValueError):
            c.hx.exchange_forces_host_packed(torch.empty((c.slots - 1, 3)), torch.empty((nh, 3)), dev)
    # the same handle rebuilt with more atoms: the packing buffer grows with it
    hx = HX.HaloExchange(w.box, w.dims, w.cutoff, flags=HX.HX_FLAG_FINE_WAITS)
    for p in (pos[: len(pos) // 3], pos):
        o = Oracle(w.box, w.dims, w.cutoff)
        o.build(p)
        pt = torch.from_numpy(p.copy()).cuda()
        n = hx.build_maps(pt)
        dev = torch.empty((n, 3), device="cuda")
        hx.build_maps(pt, dev)
        hm = np.zeros(n, bool)
        for r in range(o.n_domains):
            hm[o.dom_offset[r]: o.dom_offset[r] + o.home[r]] = True
        ref = o.coords().copy()
        o.exchange_coords(ref)
        halo = torch.empty((int((~hm).sum()), 3)).pin_memory()
        hx.exchange_coords_host_packed(torch.from_numpy(o.coords()[hm].copy()).pin_memory(), halo, dev)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(halo.numpy()), _bits(ref[~hm]))
    hx.close()


SWEEP = HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES


@pytest.mark.parametrize("name", ["C2", "C3", "C4"] + [f"rand{k}" for k in (9, 20, 25, 31)])
@pytest.mark.parametrize("pdl", [0, HX.HX_FLAG_PDL])
def test_sweep_wait_modes(name, pdl):
    """The force sweep with its waits forced segment by segment and forced per
    whole unit, on shapes with one and two pulses per dimension: ordered forces
    bit-exact against the oracle in both, over several steps."""
    w = _random_shape(int(name[4:])) if name.startswith("rand") else W.WORKLOADS[name]
    try:
        c = Case(w, flags=SWEEP | pdl)
    except HX.HXError as e:   # the sweep serves at most 8 pulses
        assert e.code == HX.HX_ERR_PULSES
        pytest.skip("more pulses than the force sweep serves")
    f0 = W.forces(w, c.slots)
    ref = f0.copy()
    c.o.exchange_forces(ref)
    for mode in (1, 2, 0):
        c.hx.debug_sweep_waits(mode)
        for _ in range(3):
            ft = torch.from_numpy(f0.copy()).cuda()
            c.hx.exchange_forces(ft)
            torch.cuda.synchronize()
            assert np.array_equal(_bits(ft.cpu().numpy()), _bits(ref)), (name, mode)
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)
    with pytest.raises(HX.HXError):
        c.hx.debug_sweep_waits(3)


def test_sweep_segment_waits_full_size():
    """The 12M-atom workload takes whole-unit waits by default: its forces with
    segment waits forced are the same bits."""
    w = W.WORKLOADS["C5"]
    c = Case(w, flags=SWEEP | HX.HX_FLAG_PDL)
    f0 = W.forces(w, c.slots)
    ref = f0.copy()
    c.o.exchange_forces(ref)
    c.hx.debug_sweep_waits(1)
    for _ in range(2):
        ft = torch.from_numpy(f0.copy()).cuda()
        c.hx.exchange_forces(ft)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(ft.cpu().numpy()), _bits(ref))
    rc, det = c.hx.status()
    assert rc == 0, (rc, det)


def test_host_buffer_rules():
    w = W.WORKLOADS["C2"]
    c = Case(w, flags=HX.HX_FLAG_FINE_WAITS)
    dev = torch.empty((c.slots, 3), device="cuda")
    with pytest.raises(ValueError):
        c.hx.exchange_coords_host(torch.empty((c.slots - 1, 3)).pin_memory(), dev)   # too small
    with pytest.raises(ValueError):
        c.hx.exchange_coords_host(dev, dev)                                            # not a host tensor
    # pageable memory: refused unless this system maps it for the device
    pageable = torch.from_numpy(c.o.coords().copy())
    try:
        c.hx.exchange_coords_host(pageable, dev)
        torch.cuda.synchronize()
        ref = c.o.coords().copy()
        c.o.exchange_coords(ref)
        assert np.array_equal(_bits(pageable.numpy()), _bits(ref))
    except HX.HXError as e:
        assert e.code == HX.HX_ERR_ARG


def test_host_buffer_misaligned():
    """A host buffer one float off the device buffer's 16-byte phase: the
    range copies take their word-by-word path; results stay bit-exact."""
    w = W.WORKLOADS["C2"]
    c = Case(w, flags=HX.HX_FLAG_FINE_WAITS)
    o = c.o
    hm = c.home_mask()
    ref = o.coords().copy()
    o.exchange_coords(ref)
    store = torch.empty(3 * c.slots + 1, dtype=torch.float32).pin_memory()
    host = store[1:].view(c.slots, 3)               # 4 bytes past a 16-byte boundary
    assert host.data_ptr() % 16 == 4
    host.copy_(torch.from_numpy(o.coords()))
    host.numpy()[~hm] = np.nan
    dev = torch.full((c.slots, 3), float("nan"), device="cuda")
    c.hx.exchange_coords_host(host, dev)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(host.numpy()), _bits(ref))
    f0 = W.forces(w, c.slots)
    fref = f0.copy()
    o.exchange_forces(fref)
    fstore = torch.empty(3 * c.slots + 1, dtype=torch.float32).pin_memory()
    fh = fstore[1:].view(c.slots, 3)
    fh.copy_(torch.from_numpy(f0))
    c.hx.exchange_forces_host(fh, torch.empty_like(dev))
    torch.cuda.synchronize()
    assert np.array_equal(_bits(fh.numpy()[hm]), _bits(fref[hm]))


def _random_shape(seed):
    """A seeded random decomposition: 1-4 slabs per dimension, slab widths
    0.4-3 nm, a cutoff below (n_d - 1) slab widths wherever n_d > 1, and
    0-20000 atoms."""
    rng = np.random.default_rng(1000 + seed)
    dims = [int(v) for v in rng.integers(1, 5, 3)]
    width = [float(v) for v in rng.uniform(0.4, 3.0, 3)]
    box = tuple(round(dims[d] * width[d], 3) for d in range(3))
    cutoff = float(rng.uniform(0.3, 1.5))
    limits = [box[d] / dims[d] * (dims[d] - 1) for d in range(3) if dims[d] > 1]
    if limits:
        cutoff = min(cutoff, 0.95 * min(limits))
    n = int(rng.integers(0, 20000))
    return W.custom(f"random{seed}", n, box, tuple(dims), cutoff, seed=2000 + seed,
                    forces_law="normal" if seed % 2 else "uniform")


@pytest.mark.parametrize("seed", range(32))
@pytest.mark.parametrize("flags", ALL_MODES + [HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES])
def test_random_shapes(seed, flags):
    w = _random_shape(seed)
    pulse_dims, _ = HX.query_plan(w.box, w.dims, w.cutoff)
    copies_bound = int(np.prod([1 + int(np.sum(pulse_dims == d)) for d in range(3)]))
    try:
        c = Case(w, flags=flags)
    except HX.HXError as e:   # resolved tables hold at most 7 copies per atom
        assert flags & HX.HX_FLAG_RESOLVED and copies_bound > 8 and e.code == HX.HX_ERR_PULSES
        return
    check_build(c)
    check_coord_steps(c)
    check_force_steps(c)
