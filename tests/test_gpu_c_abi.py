"""The C ABI from a plain C program on the GPU: cudaMalloc'd buffers, the map
build, one coordinate and one force exchange, no Python in the data path. The
results are compared with the oracle bit for bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from domain_decomposition_halo_gb300 import hx as HX
from domain_decomposition_halo_gb300 import workloads as W
from oracle.oracle import Oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <cuda_runtime.h>
#include "hx.h"

static float* read_floats(const char* path, long n) {
  float* p = (float*)malloc(sizeof(float) * (size_t)n);
  FILE* f = fopen(path, "rb");
  if (!p || !f || fread(p, sizeof(float), (size_t)n, f) != (size_t)n) exit(3);
  fclose(f);
  return p;
}

static void write_floats(const char* path, const float* p, long n) {
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(p, sizeof(float), (size_t)n, f) != (size_t)n) exit(4);
  fclose(f);
}

#define CHECK(x) do { int rc_ = (x); if (rc_ != HX_OK) { fprintf(stderr, "%s: %d\n", #x, rc_); return 1; } } while (0)

int main(int argc, char** argv) {
  /* argv: dir n_atoms box cutoff nx ny nz flags */
  if (argc != 9) return 2;
  const char* dir = argv[1];
  const long n = atol(argv[2]);
  double box[3] = {atof(argv[3]), atof(argv[3]), atof(argv[3])};
  const double cutoff = atof(argv[4]);
  int dims[3] = {atoi(argv[5]), atoi(argv[6]), atoi(argv[7])};
  const unsigned flags = (unsigned)atoi(argv[8]);
  char path[1024];
  snprintf(path, sizeof(path), "%s/pos.f32", dir);
  float* pos = read_floats(path, 3 * n);
  float *d_pos = NULL, *d_x = NULL, *d_f = NULL;
  if (cudaMalloc((void**)&d_pos, sizeof(float) * 3 * (size_t)n) != cudaSuccess) return 5;
  cudaMemcpy(d_pos, pos, sizeof(float) * 3 * (size_t)n, cudaMemcpyHostToDevice);
  hx_handle h = NULL;
  CHECK(hx_init(&h, box, dims, cutoff, 0, flags, 0));
  int64_t slots = 0;
  CHECK(hx_build_maps(h, d_pos, n, NULL, 0, &slots, NULL));
  if (cudaMalloc((void**)&d_x, sizeof(float) * 3 * (size_t)slots) != cudaSuccess) return 5;
  if (cudaMalloc((void**)&d_f, sizeof(float) * 3 * (size_t)slots) != cudaSuccess) return 5;
  CHECK(hx_build_maps(h, d_pos, n, d_x, slots, &slots, NULL));
  CHECK(hx_exchange_coords(h, d_x, NULL));
  snprintf(path, sizeof(path), "%s/forces.f32", dir);
  float* f = read_floats(path, 3 * slots);
  cudaMemcpy(d_f, f, sizeof(float) * 3 * (size_t)slots, cudaMemcpyHostToDevice);
  CHECK(hx_exchange_forces(h, d_f, NULL));
  int detail = 0;
  CHECK(hx_status(h, NULL, &detail));
  float* x = (float*)malloc(sizeof(float) * 3 * (size_t)slots);
  if (!x) return 6;
  cudaMemcpy(x, d_x, sizeof(float) * 3 * (size_t)slots, cudaMemcpyDeviceToHost);
  cudaMemcpy(f, d_f, sizeof(float) * 3 * (size_t)slots, cudaMemcpyDeviceToHost);
  snprintf(path, sizeof(path), "%s/coords_out.f32", dir);
  write_floats(path, x, 3 * slots);
  snprintf(path, sizeof(path), "%s/forces_out.f32", dir);
  write_floats(path, f, 3 * slots);
  printf("%lld\n", (long long)slots);
  hx_destroy(h);
  cudaFree(d_pos);
  cudaFree(d_x);
  cudaFree(d_f);
  free(pos);
  free(x);
  free(f);
  return 0;
}
"""


@pytest.mark.parametrize("flags", [0, HX.HX_FLAG_FINE_WAITS | HX.HX_FLAG_BULK_STORE | HX.HX_FLAG_SWEEP_FORCES | HX.HX_FLAG_PDL])
def test_c_program_exchanges_match_oracle(tmp_path, flags):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    HX.load_library()
    libdir = os.path.dirname(HX.library_path())
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "exchange.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "exchange"
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           str(src), "-L", libdir, "-lhx", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", str(exe)]
    done = subprocess.run(cmd, capture_output=True, text=True)
    assert done.returncode == 0, done.stderr
    w = W.WORKLOADS["C2"]          # a cube, so one box length serves all three dimensions
    pos = W.positions(w)
    o = Oracle(w.box, w.dims, w.cutoff)
    o.build(pos)
    f0 = W.forces(w, o.total_slots)
    pos.astype(np.float32).tofile(tmp_path / "pos.f32")
    f0.astype(np.float32).tofile(tmp_path / "forces.f32")
    args = [str(exe), str(tmp_path), str(len(pos)), repr(w.box[0]), repr(w.cutoff),
            str(w.dims[0]), str(w.dims[1]), str(w.dims[2]), str(flags)]
    run = subprocess.run(args, capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert int(run.stdout.split()[0]) == o.total_slots
    x = np.fromfile(tmp_path / "coords_out.f32", dtype=np.float32).reshape(-1, 3)
    f = np.fromfile(tmp_path / "forces_out.f32", dtype=np.float32).reshape(-1, 3)
    ref_f = f0.copy()
    o.exchange_forces(ref_f)
    assert np.array_equal(x.view(np.uint32), o.coords().view(np.uint32))
    assert np.array_equal(f.view(np.uint32), ref_f.view(np.uint32))
