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
// hx_build_maps) still allocates, once, before the steps: hx_build_maps also
// looks up the array's device address and loads the kernel the static call
// will launch (with lazy module loading, the first touch of a module loads
// its code and static data, which allocates), so a static call only reads
// what the handle holds.
#include <atomic>

#include "hx.h"
#include "hx_internal.h"
#include "hx_runtime.h"

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

// Per device, the handle whose static call last used the array (its control
// block then holds that call's status). Host bookkeeping only.
std::atomic<const hx_ctx*> g_last_user[kMaxDevices];

}  // namespace

// At build time, with the handle's device current: the array's device address
// (in host code its symbol is only a stand-in) and the static call's kernel
// loaded. Looked up per handle, so a handle made in a new context (after a
// device reset) never sees a stale address.
int static_prepare(hx_ctx* h) {
  h->static_scratch = nullptr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return HX_ERR_CUDA;
  }
  const void* fn = static_kernel(h);
  if (fn) {
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, fn) != cudaSuccess) {
      cudaGetLastError();
      return HX_ERR_CUDA;
    }
  }
  h->static_scratch = p;
  return HX_OK;
}

// hx_status / hx_clear_status: the static path's status, when this handle made
// the device's last static call.
int static_status(const hx_ctx* h, int* status, int* detail) {
  *status = 0;
  *detail = -1;
  if (h->device < 0 || h->device >= kMaxDevices || !h->static_scratch) return HX_OK;
  if (g_last_user[h->device].load() != h) return HX_OK;
  Ctrl c;
  if (cudaMemcpy(&c, &static_cast<StaticScratch*>(h->static_scratch)->ctrl, sizeof(c), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return HX_ERR_CUDA;
  *status = c.status;
  *detail = c.detail;
  return HX_OK;
}

int static_clear(const hx_ctx* h, cudaStream_t s) {
  if (h->device < 0 || h->device >= kMaxDevices || !h->static_scratch) return HX_OK;
  if (g_last_user[h->device].load() != h) return HX_OK;
  Ctrl* c = &static_cast<StaticScratch*>(h->static_scratch)->ctrl;
  if (cudaMemsetAsync(&c->status, 0, 2 * sizeof(int), s) != cudaSuccess) return HX_ERR_CUDA;
  return HX_OK;
}

void static_forget(const hx_ctx* h) {
  if (h->device < 0 || h->device >= kMaxDevices) return;
  const hx_ctx* expected = h;
  g_last_user[h->device].compare_exchange_strong(expected, nullptr);
}

}  // namespace hx

extern "C" int hx_exchange_coords_static(hx_handle h, float* coords, void* stream) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (!h->static_scratch) return HX_ERR_CUDA;   // the build could not prepare the static path
  if (h->device < 0 || h->device >= hx::kMaxDevices) return HX_ERR_ARG;
  hx_rt::DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  hx::StaticScratch* sc = static_cast<hx::StaticScratch*>(h->static_scratch);
  const int rc = hx::launch_coords_with_scratch(h, coords, static_cast<cudaStream_t>(stream), &sc->ctrl, sc->flags,
                                                sc->arrivals, hx::kStaticFlags);
  if (rc == HX_OK) hx::g_last_user[h->device].store(h);
  return rc;
}
