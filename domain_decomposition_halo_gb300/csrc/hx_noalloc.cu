// hx_exchange_coords_static: the fused coordinate exchange without any
// device allocation of its own.
//
// Some callers must not allocate device memory while they run: an MD engine
// or framework that reserves all of the GPU's memory for its own arena, or
// code that may only use memory it has accounted for. The regular exchange
// keeps its signal flags and control block in memory the handle allocated,
// and instantiates a CUDA graph (which allocates) on its first call with each
// buffer. This entry point keeps that scratch in one fixed file-scope device
// array instead, launches the kernel directly, and never calls cudaMalloc,
// cudaFree or anything that allocates. The handle itself (hx_init,
// hx_build_maps) still allocates, once, before the steps.
#include <mutex>

#include "hx.h"
#include "hx_internal.h"

namespace hx {
namespace {

constexpr size_t kStaticFlags = HX_STATIC_MAX_FLAGS;
constexpr int kMaxDevices = 64;

struct StaticScratch {
  Ctrl ctrl;
  unsigned long long flags[kStaticFlags];
  unsigned int arrivals[kStaticFlags];
};

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) StaticScratch g_scratch;

std::mutex g_mutex;
StaticScratch* g_address[kMaxDevices] = {};

// Device address of g_scratch on `device` (which must be current); looked up
// once per device. In host code the symbol itself is only a stand-in.
StaticScratch* scratch_on(int device, int* rc) {
  *rc = HX_OK;
  if (device < 0 || device >= kMaxDevices) {
    *rc = HX_ERR_ARG;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_address[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      *rc = HX_ERR_CUDA;
      return nullptr;
    }
    g_address[device] = static_cast<StaticScratch*>(p);
  }
  return g_address[device];
}

}  // namespace
}  // namespace hx

extern "C" int hx_exchange_coords_static(hx_handle h, float* coords, void* stream) {
  if (!h) return HX_ERR_ARG;
  const int device = hx::handle_device(h);
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return HX_ERR_CUDA;
  if (cur != device && cudaSetDevice(device) != cudaSuccess) return HX_ERR_CUDA;
  int rc = HX_OK;
  hx::StaticScratch* sc = hx::scratch_on(device, &rc);
  if (!sc) return rc;
  return hx::launch_coords_with_scratch(h, coords, static_cast<cudaStream_t>(stream), &sc->ctrl, sc->flags,
                                         sc->arrivals, hx::kStaticFlags);
}
