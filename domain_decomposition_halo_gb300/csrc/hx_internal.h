// Internal tables shared by the host runtime and the kernels of libhx.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "hx.h"

struct hx_ctx;

namespace hx {

#ifndef HX_ROUNDS
#define HX_ROUNDS 8
#endif
#ifndef HX_MIN_BLOCKS
#define HX_MIN_BLOCKS 3
#endif
#ifndef HX_POLL_NAP_MIN_NS
#define HX_POLL_NAP_MIN_NS 32
#endif
#ifndef HX_POLL_NAP_MAX_NS
#define HX_POLL_NAP_MAX_NS 256
#endif

constexpr int kThreads = 256;                 // threads per block of the exchange kernels
constexpr int kWarps = kThreads / 32;         // independent warps per block
constexpr int kRounds = HX_ROUNDS;            // 32-entry rounds per warp chunk
constexpr int kChunk = 32 * kRounds;          // map entries per warp chunk
constexpr int kMinBlocks = HX_MIN_BLOCKS;     // resident blocks per SM the register budget allows

// One warp's unit of work: up to kChunk consecutive entries of one
// (sender, pulse) map. Everything the warp needs is in this 64-byte record,
// so a chunk costs one descriptor load.
enum ChunkFlags : int32_t {
  kHaloSrc = 1,      // entries read slots written earlier in the same launch
  kSignal = 2,       // some later chunk waits for this chunk (or for its item)
  kShift = 4,        // add `shift` to component `dim` (coordinates only)
};

struct alignas(16) Chunk {
  int64_t src;        // first slot of the sender's array (gather source / force targets)
  int64_t dst;        // receiver-side slot of this chunk's first entry
  int64_t map;        // index of this chunk's first entry in the maps array
  int32_t n;          // entries (0..kChunk; 0 only for a pure signal)
  int32_t item;       // pulse * n_domains + sender
  int32_t item_chunks;  // chunks that make up the item (signal arithmetic)
  int32_t wait_off;   // this chunk's waits in the direction's wait list
  int32_t wait_cnt;
  int32_t flags;      // ChunkFlags
  int32_t dim;        // component the shift applies to
  float shift;        // (float)L_dim
};
static_assert(sizeof(Chunk) == 64, "chunk descriptor must stay one 64-byte record");

// Wait for `item` of the same direction to have been signalled by all of its
// `chunks` in the current launch (per-chunk flags: `item` is the chunk's
// position in the list and `chunks` is 1).
struct Wait {
  int32_t item;
  int32_t chunks;
};

// A chunk of the fused lists as one self-contained record: its descriptor,
// its map run and its first waits, so that a warp fetches everything it
// needs for a chunk with one set of 16-byte copies and no dependent load
// (waits past kWaitSlots stay in the direction's wait list).
constexpr int kWaitSlots = 32;
struct alignas(16) ChunkSlot {
  Chunk rec;
  int32_t map[kChunk];
  Wait waits[kWaitSlots];
};
static_assert(sizeof(ChunkSlot) % 16 == 0, "chunk slots are copied in 16-byte pieces");

// Per-direction control block (device memory; zeroed at build and by
// hx_clear_status, never reset between launches).
struct Ctrl {
  unsigned long long epoch;   // launches of this direction completed since the last
                              // reset: a launch reads it at its start (its own epoch is
                              // that + 1) and its last block to finish stores its epoch
  int status;                 // 0 or an HX_ERR_* code (sticky)
  int detail;                 // item of the first wait that gave up
  int drop_item;              // debug: item whose signals are dropped, or -1
  unsigned exits;             // blocks of the running launch that have finished
  int pad[2];
};
static_assert(sizeof(Ctrl) == 32, "control block must stay 32 bytes");

struct DirParams {
  const ChunkSlot* chunks;
  const Wait* waits;
  const int32_t* maps;
  unsigned long long* flags;  // epoch flags: per item (last-arrival signals) or per chunk (fine waits)
  unsigned int* arrivals;     // per item: last-arrival election counters
  Ctrl* ctrl;
  unsigned long long n_chunks;
  int direction;              // 0 coordinates, 1 forces
  int late_dependents;        // 1: under programmatic launch, the next kernel is scheduled only
                              // as this grid's blocks exit (not as they start)
  unsigned long long timeout_ns;
};

// Unfused baseline: one launch per pulse over that pulse's chunks.
struct PulseParams {
  const Chunk* chunks;
  const int32_t* maps;
  int chunk_begin;
  int n_chunks;
};

// kLastArrival: per-item epoch flag stored by the item's last chunk (the
// pages' last-block election); kChunkFlag: one epoch flag per chunk, for
// chunk-granular waits.
enum SignalMode { kLastArrival = 0, kChunkFlag = 2 };

// ---- exchange kernels (hx_kernels.cu) ----
const void* coords_kernel(int signal_mode, bool bulk_store);   // bulk_store: gather to shared memory, bulk copy out
const void* forces_kernel(int signal_mode, bool ordered);
size_t chunk_smem_bytes(int dir, bool bulk_store);              // dynamic shared memory of a fused chunk kernel's block
const void* noop_kernel();
int max_blocks_per_sm(const void* fn, size_t smem);            // sets the kernel's dynamic shared memory limit first
cudaError_t launch_pack_pulse(float* x, const PulseParams& p, cudaStream_t s);

// ---- resolved kernels (hx_resolved.cu): the forwarding unrolled at build time ----
constexpr int kTreeNodes = 8;             // a home atom and at most 7 copies
struct alignas(16) TreeRec {
  int32_t node[kTreeNodes];               // global slots; node[0] is the home atom
  uint8_t ev[kTreeNodes];                 // adds in order: target (low 4 bits) += source (high 4 bits)
  int32_t n_nodes;                        // nodes used; n_nodes - 1 adds
  int32_t pad;
};
static_assert(sizeof(TreeRec) == 48, "tree record must stay 48 bytes");
// Coordinates: one block per segment of consecutive halo slots of one domain
// (up to kResSeg; the build sizes segments for the decomposition). Per halo
// slot one word: the origin home slot in the low 29 bits, the shift mask
// (bit d: add box[d] to component d) in the top 3.
constexpr int kResThreads = 256;
constexpr int kResSlotsPerThread = 4;     // at most; the build picks 1..4 gathers in flight per thread
constexpr int kResSeg = kResThreads * kResSlotsPerThread;   // largest segment
constexpr int kResOriginBits = 29;
struct ResSeg {
  int32_t k;                              // first halo index of the segment
  int32_t slot;                           // its global slot
  int32_t n;                              // halo slots in the segment, 1..kResSeg
  int32_t pad;
};
static_assert(sizeof(ResSeg) == 16, "segment record must stay 16 bytes");
// Forces: one 16-byte record per tree, in home-slot order of its root:
//   pair (root, copy, -1, -1):  root += copy
//   quad (a, b, c, d):          a += c; b += d; a += b   (c, d received in
//                                one later pulse than b: a corner atom's two
//                                copies and the copy of its first copy)
// Other trees (general) keep a TreeRec and run in blocks of their own before
// the record blocks, one tree a thread, their adds replayed from the record.
constexpr int kResTreesPerThread = 2;      // at most; the build picks 1..2
struct ResolvedParams {
  const ResSeg* segs;
  const uint32_t* origin_mask;            // per halo slot
  const int4* recs;                       // pairs and quads
  const TreeRec* trees;                   // general trees
  int64_t n_segs;
  int64_t n_recs, n_trees;
  int32_t trees_per_thread;
  int32_t rec_blocks;                     // blocks of the records, after the general blocks
  float box[3];
  int pad;
};
const void* resolved_kernel(int kind);    // 0 coordinates, 1 forces (ordered)
cudaError_t launch_unpack_pulse(float* f, const PulseParams& p, cudaStream_t s);

// ---- unit records of the slot-sweep kernels (hx_sweep.cu) ----
//
// A unit is up to kSweepSlots consecutive slots of one domain's array, inside
// one range (home, or the slots received in one pulse), with one segment per
// (sender, pulse) map that has entries inside it. Coordinates: a unit is a
// source - its warp stages it in shared memory once and serves the gathers of
// every pulse that selects from it. Forces: a unit is a target - its warp
// stages it, adds every pulse's contributions in reverse pulse order in
// shared memory, and writes it back.
constexpr int kInlineSegs = 4;       // segments carried inside the unit record
constexpr int kInlineWaits = 2;      // waits carried inside the unit record

struct alignas(16) UnitSeg {   // entries [map, map + n) of one (sender, pulse) map that fall in the unit
  int64_t map;        // first entry in the maps array
  int64_t other;      // receiver-side slot of that entry (coordinates: destination, forces: source)
  int32_t n;
  int32_t dim;
  float shift;
  int32_t do_shift;
  int32_t map_off;    // stage byte offset of the region the map run is copied to
  int32_t src_off;    // stage byte offset of the region the received-force run is copied to
  int32_t dep;        // forces: how many of the unit's waits (listed segment by segment) are
                      // for the units of the same launch that write this segment's received run
  int32_t pad;
};
static_assert(sizeof(UnitSeg) == 48, "segment record must stay 48 bytes");

struct alignas(16) Unit {  // one 256-byte record, read by 16 threads in one round trip
  int64_t base;       // caller-array slot of the unit's first slot
  int32_t n;          // slots in the unit
  int32_t local_a;    // local index of the first slot within its domain
  int32_t seg_cnt;
  int32_t extra_off;  // segments past kInlineSegs in the direction's overflow list
  int32_t wait_off;   // producer units to wait for (positions in the list)
  int32_t wait_cnt;
  int32_t flags;      // kSignal: other units of the launch wait for this one
  int32_t item;       // pulse * n_domains + domain of its first segment (status, fault injection)
  int32_t entries;    // entries of all segments
  Wait wait_inline[kInlineWaits];   // the first waits (also in the wait list), read with the record
  int32_t pad;
  UnitSeg seg[kInlineSegs];
};
static_assert(sizeof(Unit) == 256, "unit record must stay 256 bytes");

struct UnitParams {
  const Unit* units;
  const UnitSeg* extra;       // segments past kInlineSegs
  const Wait* waits;
  const int32_t* maps;
  unsigned long long* flags;  // per unit: epoch flag
  Ctrl* ctrl;
  unsigned long long n_units;
  int direction;
  int seg_waits;              // 1: dependent segments wait for their own producers (see k_sweep)
  unsigned long long timeout_ns;
};

// Kernel family of one direction's fused exchange.
enum Family : int { kFamChunks = 0, kFamSweep = 2, kFamResolved = 4 };

// ---- slot-sweep kernels (hx_sweep.cu): one warp per unit, same unit records ----
#ifndef HX_SWEEP_SLOTS
#define HX_SWEEP_SLOTS 256
#endif
#ifndef HX_SWEEP_ENTRIES
#define HX_SWEEP_ENTRIES 256
#endif
constexpr int kSweepSlots = HX_SWEEP_SLOTS;       // slots of one unit: a warp's staged tile
constexpr int kSweepEntries = HX_SWEEP_ENTRIES;   // map entries of one unit at most
#ifndef HX_SWEEP_BATCH
#define HX_SWEEP_BATCH 1
#endif
constexpr int kSweepBatch = HX_SWEEP_BATCH;       // consecutive units a warp takes in one claim
#ifndef HX_SEG_WAIT_UNITS_PER_WARP
#define HX_SEG_WAIT_UNITS_PER_WARP 4
#endif
constexpr int kSegWaitUnitsPerWarp = HX_SEG_WAIT_UNITS_PER_WARP;   // segment-by-segment waits up to this
                                                                    // many units a warp
constexpr int kSweepSegs = 8;                     // segments (pulses) of one unit at most
static_assert(1 + 2 * kSweepSegs <= 32, "a sweep unit stages one run per lane");
// Stage layout of one warp: slots, then map runs, then (forces) received
// runs; every run has a 16-byte-aligned region 16 bytes longer than itself.
constexpr int kSweepSlotBytes = kSweepSlots * 12 + 16;
constexpr int kSweepMapBytes = kSweepEntries * 4 + 32 * kSweepSegs;
constexpr int kSweepSrcBytes = kSweepEntries * 12 + 32 * kSweepSegs;
constexpr int sweep_stage_bytes(int kind) {
  return kSweepSlotBytes + kSweepMapBytes + (kind == 1 ? kSweepSrcBytes : 0);
}
const void* sweep_kernel(int kind);              // 0 coordinates, 1 forces
size_t sweep_smem_bytes(int kind);               // dynamic shared memory of a block
int sweep_blocks_per_sm(int kind);

// ---- launch with caller-independent scratch (hx_api.cu, for hx_noalloc.cu) ----
// Runs the handle's fused coordinate exchange with its signal flags, election
// counters and control block at the given device addresses instead of the
// handle's own; clears them first on `s`. No allocation. HX_ERR_CAPACITY when
// the handle's work list needs more than `max_flags` flags.
int launch_coords_with_scratch(hx_ctx* h, float* coords, cudaStream_t s, Ctrl* ctrl, unsigned long long* flags,
                               unsigned int* arrivals, size_t max_flags);
const void* static_kernel(const hx_ctx* h);   // the kernel launch_coords_with_scratch launches (NULL: none)
// hx_noalloc.cu: the static path's set-up at build time, its status for
// hx_status / hx_clear_status, and its bookkeeping at hx_destroy.
int static_prepare(hx_ctx* h);
int static_status(const hx_ctx* h, int* status, int* detail);
int static_clear(const hx_ctx* h, cudaStream_t s);
void static_forget(const hx_ctx* h);

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

cudaError_t launch_cells(const float* pos, int64_t n, const int* dims, const float* faces,
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
