// Internal tables shared by the host runtime and the kernels of libhx.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace hx {

constexpr int kThreads = 256;          // threads per block of every exchange kernel
constexpr int kUnroll = 4;             // entries in flight per thread
constexpr int kPass = kThreads * kUnroll;  // entries per block pass (1024)

// One (sender, pulse) unit: pulse p of sender r sends S entries to its lower
// neighbour q along dim(p). Index t = p * n_domains + r.
struct Item {
  int64_t src_base;   // first slot of the sender's array (dom_offset[r])
  int64_t dst_base;   // first slot of the receive range in q (dom_offset[q] + off)
  int64_t map_off;    // first entry of this map in the maps array
  int32_t size;       // S
  int32_t split;      // entries [0, split) read home slots (independent)
  int32_t dim;        // 0, 1, 2
  int32_t do_shift;   // 1 when the sender sits in cell 0 along dim
  float shift;        // (float)L_dim
  int32_t coord_chunks;  // chunks of the coordinate exchange for this item
  int32_t force_chunks;  // chunks of the force exchange for this item
  int32_t pad;
};

// A contiguous range of map entries of one item, claimed by one block.
struct Chunk {
  int32_t item;
  int32_t begin;
  int32_t end;
  int32_t wait_off;   // waits in the direction's wait list before the body
  int32_t wait_cnt;
  int32_t halo_src;   // 1 when the entries read slots written during the launch
};

// Wait for item `item` of the same direction to have signalled this epoch;
// `chunks` = how many chunk signals complete it (counter mode).
struct Wait {
  int32_t item;
  int32_t chunks;
};

// Per-direction control block (device memory, zeroed at build time).
struct Ctrl {
  unsigned int ticket;        // next chunk to hand out (minus gridDim.x)
  unsigned int exit_count;    // blocks that finished this launch (wraps)
  unsigned long long epoch;   // launches completed
  int status;                 // 0 or an HX_ERR_* code (sticky)
  int detail;                 // item of the first wait that gave up
  int drop_item;              // debug: item whose signals are dropped, or -1
  int pad;
};

struct DirParams {
  const Item* items;
  const Chunk* chunks;
  const Wait* waits;
  const int32_t* maps;
  unsigned long long* flags;  // per item: epoch flag or arrival counter
  unsigned int* blk_count;    // per item: last-block election counters
  Ctrl* ctrl;
  int n_chunks;
  int direction;              // 0 coordinates, 1 forces
  unsigned long long timeout_ns;
};

// Unfused baseline: one launch per pulse over that pulse's chunk range.
struct PulseParams {
  const Item* items;
  const Chunk* chunks;
  const int32_t* maps;
  int chunk_begin;
};

// ---- launch wrappers (hx_kernels.cu) ----
enum SignalMode { kLastBlock = 0, kCounter = 1 };

const void* coords_kernel(int signal_mode);
const void* forces_kernel(int signal_mode, bool ordered);
const void* noop_kernel();
int max_blocks_per_sm(const void* fn);

cudaError_t launch_pack_pulse(float* x, const PulseParams& p, int n_chunks, cudaStream_t s);
cudaError_t launch_unpack_pulse(float* f, const PulseParams& p, int n_chunks, cudaStream_t s);

// ---- map builder (hx_build.cu) ----
struct BuildTile {          // candidates [local_begin, local_begin + n) of one sender
  int32_t sender;
  int32_t local_begin;
  int32_t n;
  int32_t buf;              // 0 = home coordinates, 1 + p = receive buffer of pulse p
  int64_t elem_begin;       // index of the first candidate in that buffer
  float lo;                 // lower face of the sender along the pulse's dim
  float shift;              // (float)L_dim
  int32_t do_shift;
  int32_t pad;
};

constexpr int kPartTile = 2048;   // atoms per partition tile
constexpr int kSelTile = 2048;    // candidates per selection tile

cudaError_t launch_cells(const float* pos, int64_t n, const int* dims, const double* box,
                         int ndom, int32_t* dom_id, int32_t* hist, int ntiles, int* err,
                         cudaStream_t s);
cudaError_t launch_scatter_home(const float* pos, int64_t n, int ndom, const int32_t* dom_id,
                                const int32_t* hist_scanned, int ntiles, int32_t* home_ids,
                                float* home_xyz, int32_t* home_dom, cudaStream_t s);
cudaError_t scan_exclusive(const int32_t* in, int32_t* out, int64_t n, cudaStream_t s);
cudaError_t launch_select_count(const BuildTile* tiles, int ntiles, const float* const* bufs,
                                int dim, float rc, int32_t* tile_count, cudaStream_t s);
cudaError_t launch_select_write(const BuildTile* tiles, int ntiles, const float* const* bufs,
                                int dim, float rc, const int32_t* tile_off, int32_t* map_out,
                                float* recv_out, cudaStream_t s);
cudaError_t launch_place_home(const float* home_xyz, const int32_t* home_dom,
                              const int64_t* home_start, const int64_t* dom_offset, int64_t n,
                              float* coords, cudaStream_t s);

}  // namespace hx
