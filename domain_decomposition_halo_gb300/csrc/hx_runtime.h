// Host-side internals of libhx shared by the runtime and C-ABI (hx_api.cu)
// and the work-table builders (hx_tables.cu): the handle, the decomposition
// plan and the device allocation helpers.
#pragma once

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "hx.h"
#include "hx_host.h"
#include "hx_internal.h"

namespace hx_rt {

using namespace hx;

constexpr int kGraphCache = 16;

struct GraphEntry {
  int kind;        // 0 coords, 1 forces, 2 noop
  void* ptr;
  cudaGraphExec_t exec;
};

// Makes `device` current for the life of the guard and gives the caller's
// current device back at the end, so that an entry point leaves the calling
// thread's device as it found it. ok() is false when the switch failed.
class DeviceGuard {
 public:
  explicit DeviceGuard(int device) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      ok_ = false;
      return;
    }
    if (prev_ != device) {
      ok_ = cudaSetDevice(device) == cudaSuccess;
      switched_ = ok_;
    }
  }
  ~DeviceGuard() {
    if (switched_) cudaSetDevice(prev_);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = true;
  bool switched_ = false;
};

template <class T>
cudaError_t dev_alloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), sizeof(T) * count);
}

template <class T>
void dev_free(T*& p) {
  if (p) cudaFree(p);
  p = nullptr;
}

struct Plan {
  double box[3];
  int dims[3];
  double cutoff;
  float boxf[3];
  float rcf;
  int np[3];
  int n_pulses;
  int pulse_dim[HX_MAX_PULSES];
  int pulse_k[HX_MAX_PULSES];
  int ndom;
  std::vector<float> lo[3];
};

}  // namespace hx_rt

#define HX_CUDA(call)                       \
  do {                                      \
    cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return HX_ERR_CUDA; \
  } while (0)

using namespace hx;
using namespace hx_rt;

struct hx_ctx {
  Plan pl;
  int device = 0;
  unsigned flags = 0;
  unsigned long long timeout_ns = 0;
  int sm_count = 0;

  bool built = false;
  int64_t n_atoms = 0;
  int64_t total_slots = 0;
  int64_t total_entries = 0;
  std::vector<int64_t> dom_offset;
  std::vector<int32_t> home, halo;
  // per (pulse p, sender r), index p * ndom + r
  std::vector<int64_t> t_map_off;
  std::vector<int32_t> t_size, t_recv, t_off, t_shift, t_split;

  int32_t* d_maps = nullptr;
  int32_t* d_home_ids = nullptr;
  ChunkSlot* d_chunks[2] = {nullptr, nullptr};   // fused coordinate / force chunk lists (self-contained records)
  Wait* d_waits[2] = {nullptr, nullptr};
  Chunk* d_uchunks = nullptr;                // unfused per-pulse chunk list
  unsigned long long* d_flags = nullptr;     // [2][n_items]
  unsigned int* d_blk = nullptr;             // [2][n_items]
  Ctrl* d_ctrl = nullptr;                    // [2]
  int* d_status = nullptr;                   // [2]: hx_status_async's status and detail, on the device
  int n_chunks[2] = {0, 0};
  int grid[2] = {0, 0};
  size_t n_flags = 1;                        // flags (and election counters) per direction
  int family[2] = {0, 0};                    // kernel family of each direction's fused path (Family)
  Unit* d_units[2] = {nullptr, nullptr};
  UnitSeg* d_segs[2] = {nullptr, nullptr};
  Wait* d_twaits[2] = {nullptr, nullptr};
  int n_units[2] = {0, 0};
  std::vector<int> u_begin;                  // per pulse, first unfused chunk (P + 1 entries)
  std::vector<GraphEntry> graphs;
  ResSeg* d_res_segs = nullptr;              // resolved mode: halo segments
  uint32_t* d_res_om = nullptr;              // ... origin and shift mask per halo slot
  int4* d_res_recs = nullptr;                // ... force trees: pairs and quads, general ones apart
  TreeRec* d_res_trees = nullptr;
  int64_t n_res_halo = 0, n_res_segs = 0, n_res_pairs = 0, n_res_quads = 0, n_res_trees = 0;
  CopyChunk* d_home_chunks = nullptr;        // host-buffer calls: every domain's home range
  CopyChunk* d_halo_chunks = nullptr;        // ... and halo range, in pieces of one block each
  int n_home_chunks = 0, n_halo_chunks = 0;
  int sweep_waits = 0;                      // force sweep: 0 by units per warp, 1 segment waits, 2 whole-unit waits
  float* d_pack = nullptr;                  // packed host-buffer calls: the home or halo ranges end to end
  int64_t pack_slots = 0;                   // its size in slots (allocated by the first packed call)
  void* static_scratch = nullptr;            // hx_exchange_coords_static: device address of its scratch array
};

namespace hx_rt {

// hx_api.cu
void cell_of(const Plan& pl, int r, int c[3]);
int neighbour(const Plan& pl, int r, int d, int step);
const void* kernel_for(hx_ctx* h, int kind);
size_t fused_smem(const hx_ctx* h, int dir);   // dynamic shared memory of a direction's fused kernel
int reset_signals(hx_ctx* h, cudaStream_t s);
int64_t resolved_blocks(int64_t n, int per);
int resolved_per_thread(const hx_ctx* h, int64_t n, int most);

// hx_tables.cu: every work table of a built handle, from the maps
int build_tables(hx_ctx* h, cudaStream_t s);

}  // namespace hx_rt
