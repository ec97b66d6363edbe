"""Host-side logic of bench.py that needs no GPU."""
import numpy as np

import bench
from domain_decomposition_halo_gb300 import workloads as W


def test_reference_sample_keeps_per_domain_geometry():
    w = W.WORKLOADS["C5"]
    for k in range(1, 6):
        s = bench.sample_workload(w, k)
        per_dom_box = [b / n for b, n in zip(s.box, s.dims)]
        assert np.allclose(per_dom_box, [b / n for b, n in zip(w.box, w.dims)])
        n_dom = s.dims[0] * s.dims[1] * s.dims[2]
        assert s.n_atoms // n_dom == w.n_atoms // (w.dims[0] * w.dims[1] * w.dims[2])
        assert n_dom == (w.dims[0] * w.dims[1] * w.dims[2]) >> k
        assert s.cutoff == w.cutoff and s.order == w.order and s.forces == w.forces
        assert all(n >= 2 for n in s.dims)


def test_flag_names():
    from domain_decomposition_halo_gb300 import hx as HX
    assert bench.hx_flags("fine") == HX.HX_FLAG_FINE_WAITS
    assert bench.hx_flags("pages") == 0
    assert bench.hx_flags("fine,nograph,unordered") == (HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_NO_GRAPH |
                                                        HX.HX_FLAG_UNORDERED_FORCES)


def test_traffic_needs_matching_digest(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "domain_decomposition_halo_gb300" / "csrc").mkdir(parents=True)
    for name in sorted({n for files in bench.KERNEL_SOURCES.values() for n in files}):
        (tmp_path / "domain_decomposition_halo_gb300" / "csrc" / name).write_text("x")
    (tmp_path / "profiles").mkdir()
    digest = bench.kernel_source_digest("sweep")
    (tmp_path / "profiles" / "k_C5.md").write_text(f"traffic_bytes_per_launch: 123\nkernel_source_digest: {digest}\n")
    assert bench.profiled_traffic("k", "C5", "sweep") == 123.0
    (tmp_path / "profiles" / "k_C5.md").write_text("traffic_bytes_per_launch: 123\nkernel_source_digest: 0000\n")
    assert bench.profiled_traffic("k", "C5", "sweep") is None


def test_kernel_impl_names_the_launched_kernels():
    default = bench.hx_flags("fine,bulkstore,sweepf")
    assert bench.kernel_impl(default, 0).startswith("k_coords_bulk<chunk flags>")
    assert bench.kernel_impl(default, 1).startswith("k_sweep<1>")
    assert bench.kernel_impl(0, 1).startswith("k_forces_fused<last arrival, ordered>")
    assert bench.kernel_impl(bench.hx_flags("resolved"), 1).startswith("k_resolved_forces")


def test_launch_label_follows_the_flags():
    assert bench.launch_label(bench.hx_flags("fine,bulkstore,sweepf,pdl")).startswith("one direct launch with programmatic")
    assert bench.launch_label(bench.hx_flags("fine,nograph")) == "one direct launch per direction per step"
    assert bench.launch_label(0) == "one CUDA-graph launch per direction per step"


def test_step_distribution_nearest_rank_p90():
    d = bench.step_distribution([10.0 - k for k in range(10)])   # 1..10, unsorted
    assert d == {"median": 5.5, "p90": 9.0, "min": 1.0, "max": 10.0, "n": 10}
    d = bench.step_distribution(list(range(1, 21)))
    assert d["p90"] == 18 and d["median"] == 10.5
    assert bench.step_distribution([3.0])["p90"] == 3.0


def test_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d = tmp_path / "domain_decomposition_halo_gb300" / "csrc"
    d.mkdir(parents=True)
    names = sorted({n for files in bench.KERNEL_SOURCES.values() for n in files})
    for name in names:
        (d / name).write_text('int f(int a) { return a + 1; }  // add\nconst char* s = "a // b";\n')
    first = bench.kernel_source_digest("chunks")
    (d / "hx_kernels.cu").write_text(
        '/* a block\n comment */ int f(int a) {\n  return a + 1;   // another\n}\nconst char* s = "a // b";\n')
    assert bench.kernel_source_digest("chunks") == first
    (d / "hx_kernels.cu").write_text('int f(int a) { return a + 2; }\nconst char* s = "a // b";\n')
    assert bench.kernel_source_digest("chunks") != first
    (d / "hx_kernels.cu").write_text('int f(int a) { return a + 1; }\nconst char* s = "a // c";\n')
    assert bench.kernel_source_digest("chunks") != first   # text inside a string is code


def test_digest_is_per_kernel_family(tmp_path, monkeypatch):
    """A change to the chunk kernels leaves the sweep's profile valid, and a
    change to the shared header voids both."""
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d = tmp_path / "domain_decomposition_halo_gb300" / "csrc"
    d.mkdir(parents=True)
    for name in sorted({n for files in bench.KERNEL_SOURCES.values() for n in files}):
        (d / name).write_text(f"int {name.split('.')[0]}_v = 1;\n")
    chunks, sweep = bench.kernel_source_digest("chunks"), bench.kernel_source_digest("sweep")
    (d / "hx_kernels.cu").write_text("int hx_kernels_v = 2;\n")
    assert bench.kernel_source_digest("sweep") == sweep
    assert bench.kernel_source_digest("chunks") != chunks
    (d / "hx_internal.h").write_text("int hx_internal_v = 2;\n")
    assert bench.kernel_source_digest("sweep") != sweep


def test_kernel_family_follows_the_flags():
    f = bench.hx_flags("fine,bulkstore,sweepf,pdl")
    assert bench.kernel_family(f, 0) == "chunks" and bench.kernel_family(f, 1) == "sweep"
    assert bench.kernel_family(bench.hx_flags("resolved"), 1) == "resolved"
    assert bench.kernel_family(bench.hx_flags("fine"), 1) == "chunks"

def test_launch_mean_leaves_out_host_stalls():
    # one interval that holds a host stall (the queue ran dry) must not move the kernel's duration
    ts = [80.0] * 999 + [33000.0]
    mean, dropped = bench.launch_mean(ts)
    assert dropped == 1 and mean == 80.0
    mean, dropped = bench.launch_mean([1.0, 2.0, 3.0])
    assert dropped == 0 and mean == 2.0
