// Exchange kernels of libhx (sm_103a).
//
// Coordinates: one persistent launch for every pulse ("Enabling parallelism
// across pulses through kernel fusion"; fusedPulsesPackAndSendKernel). The
// work is cut into warp chunks of up to 256 entries of one (sender, pulse)
// map, listed in a topological order (a chunk only waits for items listed
// before it) chosen for L2 locality. Warp w of the persistent grid takes the
// list positions w, w + W, w + 2W, ... in order, so a waiting chunk only
// waits for chunks that running warps own and reach first. Warps never
// synchronise with each other inside a block: like the pages' per-warp TMA
// variant ("NVLink path: TMA-based direct stores"), each warp gathers,
// stores and signals on its own.
//
// A chunk gathers x[src + map[i]], applies the periodic shift, and stores
// straight into the receiver's slots (the NVLink-path "pack directly into
// the peer's coordinate array": here the same HBM). A chunk of forwarded
// entries has its map entries at hand, then its lanes wait with acquire
// loads at gpu scope until the items that filled those slots have signalled
// (packHaloCoords). After its stores a chunk signals its item, when anybody
// waits for it: either the pages' hierarchical scheme (signalPeerOnLastBlock:
// a counting atomic with release semantics elects the last chunk, which
// stores the epoch flag with release) or, with chunk-granular waits, one
// epoch flag per chunk.
//
// Forces: the same skeleton in reverse pulse order ("Force halo exchange:
// Reversing the dependency chain"): a chunk of (sender r, pulse p) adds the
// received halo-slot forces of its receiver into r's targets through the map
// (unpackRecvBufKernel<accumulate=true>) once every item that writes those
// targets or those slots in a later pulse has signalled.
//
// Every wait is bounded by %globaltimer; a wait that runs out records
// HX_ERR_TIMEOUT in the control block and the warp carries on, so a kernel
// always finishes.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

constexpr int kErrTimeout = -6;
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned kPollNapMinNs = HX_POLL_NAP_MIN_NS;   // back-off between flag polls: first nap
constexpr unsigned kPollNapMaxNs = HX_POLL_NAP_MAX_NS;   // ... doubling up to this

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Counting increment (wraps to 0 after `mod`) with acquire-release at gpu
// scope: each chunk's stores are released before its increment, and the
// electing (last) chunk acquires all of them before it publishes the flag.
__device__ __forceinline__ unsigned atom_inc_acq_rel(unsigned* p, unsigned mod) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(mod) : "memory");
  return old;
}

// Programmatic dependent launch (HX_FLAG_PDL): let the stream's next kernel
// be scheduled now, and wait for the previous kernel to complete before
// reading or claiming anything. Both are no-ops in a launch without the
// programmatic-serialization attribute.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A scattered slot (12 bytes at a 4-byte-aligned address): read as three
// 4-byte words (an 8-byte + 4-byte split of the read was measured slower for
// the gathers), written as an 8-byte and a 4-byte store, one L2 write request
// fewer than three words.
template <bool RO>
__device__ __forceinline__ void load_slot(const float* p, float& a, float& b, float& c) {
  a = RO ? __ldg(p) : p[0];
  b = RO ? __ldg(p + 1) : p[1];
  c = RO ? __ldg(p + 2) : p[2];
}

__device__ __forceinline__ void store_slot(float* p, float a, float b, float c) {
  const bool lo8 = (reinterpret_cast<uintptr_t>(p) & 7u) == 0u;
  *reinterpret_cast<float2*>(lo8 ? p : p + 1) = lo8 ? make_float2(a, b) : make_float2(b, c);
  *(lo8 ? p + 2 : p) = lo8 ? c : a;
}

__device__ __forceinline__ Chunk load_chunk(const Chunk* p) {
  const int4* q = reinterpret_cast<const int4*>(p);
  union {
    int4 v[4];
    Chunk c;
  } u;
  u.v[0] = __ldg(q);
  u.v[1] = __ldg(q + 1);
  u.v[2] = __ldg(q + 2);
  u.v[3] = __ldg(q + 3);
  return u.c;
}

// Whole warp: wait until every producer in the chunk's wait list has
// signalled at this epoch. The lanes take the list in strides of 32 (the
// first kWaitSlots entries from the copy in shared memory), so a chunk with
// several producers pays about one flag round trip, not one per producer.
// Each lane polls with acquire loads at gpu scope and a short back-off
// between polls; the closing __syncwarp orders every lane's acquire before
// the warp's loads. A wait that gives up (timeout, or another wait already
// failed) records the status and lets the chunk proceed without the
// guarantee.
template <int MODE>
__device__ void wait_chunk(const DirParams& P, const Chunk& ch, const Wait* waits, unsigned long long epoch) {
  const int lane = threadIdx.x & 31;
  for (int w = lane; w < ch.wait_cnt; w += 32) {
    const Wait wt = w < kWaitSlots ? waits[w] : P.waits[ch.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    unsigned long long t0 = 0;
    unsigned iter = 0, nap = 0;
    // epoch flags (per item or per chunk) are compared for equality, as the
    // pages' signal wait does
    while (ld_acquire_u64(flag) != epoch) {
      if ((iter++ & 15u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) break;
        if (now - t0 > P.timeout_ns) {
          if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0) {
            // report the (sender, pulse) item, also when the wait was on one chunk of it
            const int item = (MODE == kChunkFlag) ? P.chunks[wt.item].rec.item : wt.item;
            atomicExch(&P.ctrl->detail, P.direction * 65536 + item);
          }
          break;
        }
      }
      nap = nap ? min(2u * nap, kPollNapMaxNs) : kPollNapMinNs;
      __nanosleep(nap);
    }
  }
  __syncwarp();
}

// Lane 0 only, after the warp's stores (ordered by the preceding __syncwarp).
template <int MODE>
__device__ __forceinline__ void signal_chunk(const DirParams& P, const Chunk& ch, unsigned long long c,
                                             unsigned long long epoch, int drop_item) {
  const bool drop = ch.item == drop_item;
  if (MODE == kChunkFlag) {
    if (!drop) st_release_u64(P.flags + c, epoch);
  } else {
    const unsigned last = static_cast<unsigned>(ch.item_chunks - 1);
    const unsigned old = atom_inc_acq_rel(P.arrivals + ch.item, last);
    if (old == last && !drop) st_release_u64(P.flags + ch.item, epoch);
  }
}

__device__ __forceinline__ void load_map(const int32_t* __restrict__ map, int n, int (&j)[kRounds]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int e = u * 32 + lane;
    j[u] = (e < n) ? __ldg(map + e) : -1;
  }
}

// Store the warp's round of 32 consecutive entries as 96 contiguous floats
// with three coalesced 128-byte stores (transposed through shared memory).
__device__ __forceinline__ void store_round(float* __restrict__ dst, int n_round, const float (&v)[3],
                                            float* stage) {
  const int lane = threadIdx.x & 31;
  if (lane < n_round) {
    stage[3 * lane + 0] = v[0];
    stage[3 * lane + 1] = v[1];
    stage[3 * lane + 2] = v[2];
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int idx = k * 32 + lane;
    if (idx < 3 * n_round) dst[idx] = stage[idx];
  }
  __syncwarp();
}

// Where a chunk's map entries come from: registers loaded up front (the
// unfused kernels) or the chunk's record in shared memory, read as each
// round is issued (the fused loop: no registers held for the map).
struct RegMap {
  const int (&j)[kRounds];
  __device__ __forceinline__ int operator()(int u) const { return j[u]; }
};
struct SmemMap {
  const int32_t* m;
  int n;
  __device__ __forceinline__ int operator()(int u) const {
    const int e = u * 32 + static_cast<int>(threadIdx.x & 31);
    return e < n ? m[e] : -1;
  }
};

// Coordinates of one chunk: gather (+shift) and store into the receiver.
// Home slots are never written by the coordinate kernel, so independent
// chunks read them through the read-only path.
template <class Map>
__device__ __forceinline__ void gather_chunk(const float* __restrict__ x, const Chunk& ch, const Map& j,
                                             float (&v)[kRounds][3]) {
  const float* src = x + 3 * ch.src;
  const bool halo = (ch.flags & kHaloSrc) != 0;
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int ju = j(u);
    if (ju >= 0) {
      const float* s = src + 3 * static_cast<int64_t>(ju);
      if (halo) load_slot<false>(s, v[u][0], v[u][1], v[u][2]);
      else load_slot<true>(s, v[u][0], v[u][1], v[u][2]);
    }
  }
}

template <class Map>
__device__ __forceinline__ void coords_chunk(float* __restrict__ x, const Chunk& ch, const Map& j, float* stage) {
  float v[kRounds][3];
  gather_chunk(x, ch, j, v);
  if (ch.flags & kShift) {   // no add otherwise: unshifted values keep every bit (-0.0 included)
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      if (ch.dim == 0) v[u][0] = __fadd_rn(v[u][0], ch.shift);
      else if (ch.dim == 1) v[u][1] = __fadd_rn(v[u][1], ch.shift);
      else v[u][2] = __fadd_rn(v[u][2], ch.shift);
    }
  }
  float* dst = x + 3 * ch.dst;
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int n_round = ch.n - u * 32;
    if (n_round <= 0) break;
    store_round(dst + 96 * u, n_round < 32 ? n_round : 32, v[u], stage);
  }
}

// Forces of one chunk: targets[map[i]] += received[i], x then y then z
// (the unfused kernels; the fused loop stages the received run).
template <bool ORDERED>
__device__ __forceinline__ void forces_chunk(float* __restrict__ f, const Chunk& ch, const int (&j)[kRounds]) {
  const int lane = threadIdx.x & 31;
  float* tgt = f + 3 * ch.src;
  const float* rcv = f + 3 * ch.dst;
  constexpr int kHalf = kRounds / 2;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float g[kHalf][3];
    float t[kHalf][3];
#pragma unroll
    for (int u = 0; u < kHalf; ++u) {
      const int e = (h * kHalf + u) * 32 + lane;
      if (e < ch.n) {
        const float* s = rcv + 3 * static_cast<int64_t>(e);
        g[u][0] = s[0];
        g[u][1] = s[1];
        g[u][2] = s[2];
      }
    }
    if (ORDERED) {
#pragma unroll
      for (int u = 0; u < kHalf; ++u) {
        const int jj = j[h * kHalf + u];
        if (jj >= 0) {
          const float* p = tgt + 3 * static_cast<int64_t>(jj);
          t[u][0] = p[0];
          t[u][1] = p[1];
          t[u][2] = p[2];
        }
      }
#pragma unroll
      for (int u = 0; u < kHalf; ++u) {
        const int jj = j[h * kHalf + u];
        if (jj >= 0)
          store_slot(tgt + 3 * static_cast<int64_t>(jj), __fadd_rn(t[u][0], g[u][0]), __fadd_rn(t[u][1], g[u][1]),
                     __fadd_rn(t[u][2], g[u][2]));
      }
    } else {
#pragma unroll
      for (int u = 0; u < kHalf; ++u) {
        const int jj = j[h * kHalf + u];
        if (jj >= 0) {
          float* p = tgt + 3 * static_cast<int64_t>(jj);
          atomicAdd(p, g[u][0]);
          atomicAdd(p + 1, g[u][1]);
          atomicAdd(p + 2, g[u][2]);
        }
      }
    }
  }
}

// Bulk-store pack (the pages' TMA variant, "Optimizing for efficient
// transfers across NVIDIA NVLink-connected GPUs": gather into shared memory,
// then one bulk copy to the peer). The warp gathers its chunk into its
// shared-memory stage, laid out at the destination's address mod 16; lane 0
// stores the 16-byte-aligned middle with one cp.async.bulk shared -> global,
// and the lanes store the words around it. The store completes
// asynchronously: the stage is reused only after the copy has read it, and a
// signal follows only once the copy is complete and ordered before the
// release (bulk_store_done).
constexpr int kBulkStageBytes = kChunk * 12 + 16;
#ifndef HX_BULK_MIN_ENTRIES
#define HX_BULK_MIN_ENTRIES 96
#endif
// Chunks of fewer entries take the plain-store path even in the bulk-store
// kernel: for a small chunk the bulk copy's completion round trip before the
// release costs more than the lanes' own stores (one GB300, back to back with
// programmatic launch: 32-entry chunks 14.9 us per step with plain stores and
// 15.6 with bulk stores on 8 domains; 256-entry chunks 27.9 with bulk stores
// and 28.7 with plain ones on 64 domains).
constexpr int kBulkMinEntries = HX_BULK_MIN_ENTRIES;
constexpr int kPipe = 2;         // chunks in a warp's pipeline: in use, next one in flight

// A warp's shared memory in the fused chunk kernels: the chunk pipeline and
// the stage (coordinates: a 32-entry transposed round, or the whole chunk for
// the bulk store; forces: the chunk's received run).
template <int KIND>
struct alignas(16) ChunkWarpSmem {
  ChunkSlot slot[kPipe];
  alignas(16) unsigned char stage[KIND == 0 ? 96 * 4 : kBulkStageBytes];
};

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

template <class Map>
__device__ __forceinline__ void coords_chunk_bulk(float* __restrict__ x, const Chunk& ch, const Map& j,
                                                  unsigned char* stage) {
  const int lane = threadIdx.x & 31;
  float v[kRounds][3];
  gather_chunk(x, ch, j, v);
  if (ch.flags & kShift) {   // no add otherwise: unshifted values keep every bit (-0.0 included)
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      if (ch.dim == 0) v[u][0] = __fadd_rn(v[u][0], ch.shift);
      else if (ch.dim == 1) v[u][1] = __fadd_rn(v[u][1], ch.shift);
      else v[u][2] = __fadd_rn(v[u][2], ch.shift);
    }
  }
  float* dst = x + 3 * ch.dst;
  const unsigned long long gd = reinterpret_cast<unsigned long long>(dst);
  float* sv = reinterpret_cast<float*>(stage + (gd & 15ull));
  // the previous chunk's bulk store has read the stage
  if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int e = u * 32 + lane;
    if (e < ch.n) {
      sv[3 * e + 0] = v[u][0];
      sv[3 * e + 1] = v[u][1];
      sv[3 * e + 2] = v[u][2];
    }
  }
  __syncwarp();
  const unsigned bytes = 12u * static_cast<unsigned>(ch.n);
  const unsigned long long a0 = (gd + 15ull) & ~15ull, a1 = (gd + bytes) & ~15ull;
  if (a1 > a0) {
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the lanes' stage writes, to the copy
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\tcp.async.bulk.commit_group;" ::"l"(
                       a0),
                   "r"(smem_u32(stage + (gd & 15ull) + (a0 - gd))), "r"(static_cast<unsigned>(a1 - a0))
                   : "memory");
    }
    const int head = static_cast<int>((a0 - gd) / 4), tail = static_cast<int>((gd + bytes - a1) / 4);
    if (lane < head) dst[lane] = sv[lane];
    else if (lane >= 4 && lane < 4 + tail) {
      const int k = static_cast<int>((a1 - gd) / 4) + (lane - 4);
      dst[k] = sv[k];
    }
  } else {
    for (int k = lane; k < 3 * ch.n; k += 32) dst[k] = sv[k];
  }
}

// Lane 0, before a release that covers a bulk-stored chunk: the copy has
// completed and is ordered before later generic accesses.
__device__ __forceinline__ void bulk_store_done() {
  asm volatile("cp.async.bulk.wait_group 0;\n\tfence.proxy.async.global;" ::: "memory");
}

// Chunk pipeline of one warp in shared memory. While the warp works on its
// chunk k, the whole record of chunk k+1 (descriptor, map run, first waits)
// is copied in with cp.async: a warp's claims are static (below), so it
// knows its next chunk ahead, and a chunk starts with everything at hand.
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// All but the `n` most recently committed groups of this thread have landed.
template <int n>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory"); }

// Whole warp: one chunk record, in 16-byte pieces (committed as one group).
__device__ __forceinline__ void fetch_chunk(ChunkSlot& s, const ChunkSlot* src) {
  const int lane = threadIdx.x & 31;
  constexpr int kPieces = static_cast<int>(sizeof(ChunkSlot) / 16);
  const int4* g = reinterpret_cast<const int4*>(src);
  int4* d = reinterpret_cast<int4*>(&s);
#pragma unroll
  for (int k = lane; k < kPieces; k += 32) cp_async_16(d + k, g + k);
  cp_async_commit();
}

// Forces of one chunk: targets[map[i]] += received[i], x then y then z. The
// received run (contiguous slots) is copied into the warp's stage with
// cp.async (16-byte pieces for its aligned middle, words for the ragged ends;
// the stage keeps the run's address mod 16) while the targets are loaded
// into registers, so a chunk costs one round trip before its adds. The
// stage's copy is committed as the newest group; the caller has committed
// its other copies before.
template <bool ORDERED, class Map>
__device__ __forceinline__ void forces_chunk_staged(float* __restrict__ f, const Chunk& ch, const Map& j,
                                                    unsigned char* stage) {
  const int lane = threadIdx.x & 31;
  const unsigned long long g = reinterpret_cast<unsigned long long>(f + 3 * ch.dst);
  const unsigned bytes = 12u * static_cast<unsigned>(ch.n);
  unsigned char* base = stage + (g & 15ull);   // base[k] holds the byte at g + k
  const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
  if (a1 > a0) {
    const int pieces = static_cast<int>((a1 - a0) / 16);
    for (int k = lane; k < pieces; k += 32)
      cp_async_16(base + (a0 - g) + 16 * k, reinterpret_cast<const void*>(a0 + 16ull * k));
    const int head = static_cast<int>((a0 - g) / 4), tail = static_cast<int>((g + bytes - a1) / 4);
    if (lane < head) cp_async_4(base + 4 * lane, reinterpret_cast<const void*>(g + 4ull * lane));
    else if (lane >= 4 && lane < 4 + tail)
      cp_async_4(base + (a1 - g) + 4 * (lane - 4), reinterpret_cast<const void*>(a1 + 4ull * (lane - 4)));
  } else {
    for (int k = lane; k < static_cast<int>(bytes / 4); k += 32)
      cp_async_4(base + 4 * k, reinterpret_cast<const void*>(g + 4ull * k));
  }
  cp_async_commit();
  float* tgt = f + 3 * ch.src;
  float t[kRounds][3];
  if (ORDERED) {
#pragma unroll
    for (int u = 0; u < kRounds; ++u) {
      const int ju = j(u);
      if (ju >= 0) load_slot<false>(tgt + 3 * static_cast<int64_t>(ju), t[u][0], t[u][1], t[u][2]);
    }
  }
  cp_async_wait<0>();   // this lane's copies of the run (and anything committed before)
  __syncwarp();         // ... and every other lane's
  const float* rcv = reinterpret_cast<const float*>(base);
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    const int jj = j(u);
    if (jj >= 0) {
      const int e = u * 32 + lane;
      float* p = tgt + 3 * static_cast<int64_t>(jj);
      if (ORDERED) {
        store_slot(p, __fadd_rn(t[u][0], rcv[3 * e + 0]), __fadd_rn(t[u][1], rcv[3 * e + 1]),
                   __fadd_rn(t[u][2], rcv[3 * e + 2]));
      } else {
        atomicAdd(p, rcv[3 * e + 0]);
        atomicAdd(p + 1, rcv[3 * e + 1]);
        atomicAdd(p + 2, rcv[3 * e + 2]);
      }
    }
  }
  __syncwarp();   // the stage is read before the next chunk's copy into it
}

// Persistent warp loop shared by both directions. KIND 0 = coordinates,
// 1 = forces ordered, 2 = forces unordered, 3 = coordinates by bulk stores.
//
// Claims are static: warp w of the launch takes list positions w, w + W,
// w + 2W, ... (W warps), in that order. The list is in a topological order
// of the waits and every warp is resident, so the smallest unfinished
// position always belongs to a warp that has finished all its earlier
// positions and whose producers all sit at smaller positions: the launch
// always progresses. No atomic ticket is drawn (thousands of warps drawing
// from one counter at launch serialise for microseconds). The launch's epoch
// is read from the control block at the start; the launch's last block to
// finish stores it there for the next launch.
template <int MODE, int KIND>
__device__ __forceinline__ void run_warps(float* __restrict__ buf, const DirParams& P, ChunkWarpSmem<KIND>& S) {
  const int lane = threadIdx.x & 31;
  const unsigned long long W = static_cast<unsigned long long>(gridDim.x) * kWarps;
  const unsigned long long N = P.n_chunks;
  unsigned long long c = static_cast<unsigned long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (!P.late_dependents) allow_dependents();
  wait_prerequisites();   // before the first flag, table or buffer access
  const unsigned long long epoch = ld_relaxed_u64(&P.ctrl->epoch) + 1ull;
  if (c < N) {
    const int drop_item = ld_relaxed_s32(&P.ctrl->drop_item);
    fetch_chunk(S.slot[0], P.chunks + c);
    cp_async_wait<0>();
    __syncwarp();
    int b = 0;
    while (true) {
      const ChunkSlot& cur = S.slot[b];
      const Chunk ch = cur.rec;
      const SmemMap j{cur.map, ch.n};
      const unsigned long long c1 = c + W;
      if (c1 < N) fetch_chunk(S.slot[b ^ 1], P.chunks + c1);
      if (ch.wait_cnt > 0) wait_chunk<MODE>(P, ch, cur.waits, epoch);
      if (KIND == 0) coords_chunk(buf, ch, j, reinterpret_cast<float*>(S.stage));
      else if (KIND == 3) {
        if (ch.n >= kBulkMinEntries) {
          coords_chunk_bulk(buf, ch, j, S.stage);
        } else {   // small chunk: plain stores, once the previous bulk store has read the stage
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();
          coords_chunk(buf, ch, j, reinterpret_cast<float*>(S.stage));
        }
      }
      else forces_chunk_staged<KIND == 1>(buf, ch, j, S.stage);
      if (ch.flags & kSignal) {
        __syncwarp();
        if (lane == 0) {
          if (KIND == 3) bulk_store_done();
          signal_chunk<MODE>(P, ch, c, epoch, drop_item);
        }
      }
      if (c1 >= N) break;
      c = c1;
      b ^= 1;
      cp_async_wait<0>();   // the next chunk's record
      __syncwarp();
    }
    if (KIND == 3 && lane == 0) bulk_store_done();   // nothing in flight when the warp exits
  }
  // The launch's last block to finish publishes its epoch for the next launch
  // of this direction (which reads it after this grid has completed).
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned done = atomicAdd(&P.ctrl->exits, 1u);
    if (done == gridDim.x - 1) {
      P.ctrl->exits = 0u;
      st_relaxed_u64(&P.ctrl->epoch, epoch);
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_coords_fused(float* __restrict__ x, DirParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  run_warps<MODE, 0>(x, P, reinterpret_cast<ChunkWarpSmem<0>*>(smem_raw)[threadIdx.x >> 5]);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_coords_bulk(float* __restrict__ x, DirParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  run_warps<MODE, 3>(x, P, reinterpret_cast<ChunkWarpSmem<3>*>(smem_raw)[threadIdx.x >> 5]);
}

template <int MODE, bool ORDERED>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_forces_fused(float* __restrict__ f, DirParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int K = ORDERED ? 1 : 2;
  run_warps<MODE, K>(f, P, reinterpret_cast<ChunkWarpSmem<K>*>(smem_raw)[threadIdx.x >> 5]);
}

// Unfused baseline: one warp per chunk of one pulse, stream order between pulses.
__global__ void __launch_bounds__(kThreads) k_pack_pulse(float* __restrict__ x, PulseParams P) {
  __shared__ float s_stage[kWarps][96];
  const int c = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (c >= P.n_chunks) return;
  Chunk ch = load_chunk(P.chunks + P.chunk_begin + c);
  ch.flags |= kHaloSrc;   // earlier pulses' slots were written by earlier launches: any load path works
  int j[kRounds];
  load_map(P.maps + ch.map, ch.n, j);
  coords_chunk(x, ch, RegMap{j}, s_stage[threadIdx.x >> 5]);
}

__global__ void __launch_bounds__(kThreads) k_unpack_pulse(float* __restrict__ f, PulseParams P) {
  const int c = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (c >= P.n_chunks) return;
  const Chunk ch = load_chunk(P.chunks + P.chunk_begin + c);
  int j[kRounds];
  load_map(P.maps + ch.map, ch.n, j);
  forces_chunk<true>(f, ch, j);
}

__global__ void k_noop() {}

}  // namespace

const void* coords_kernel(int signal_mode, bool bulk_store) {
  if (bulk_store)
    return signal_mode == kChunkFlag ? reinterpret_cast<const void*>(&k_coords_bulk<kChunkFlag>)
                                     : reinterpret_cast<const void*>(&k_coords_bulk<kLastArrival>);
  return signal_mode == kChunkFlag ? reinterpret_cast<const void*>(&k_coords_fused<kChunkFlag>)
                                   : reinterpret_cast<const void*>(&k_coords_fused<kLastArrival>);
}

const void* forces_kernel(int signal_mode, bool ordered) {
  if (signal_mode == kChunkFlag)
    return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kChunkFlag, true>)
                   : reinterpret_cast<const void*>(&k_forces_fused<kChunkFlag, false>);
  return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kLastArrival, true>)
                 : reinterpret_cast<const void*>(&k_forces_fused<kLastArrival, false>);
}

const void* noop_kernel() { return reinterpret_cast<const void*>(&k_noop); }

size_t chunk_smem_bytes(int dir, bool bulk_store) {
  if (dir == 1) return kWarps * sizeof(ChunkWarpSmem<1>);
  return kWarps * (bulk_store ? sizeof(ChunkWarpSmem<3>) : sizeof(ChunkWarpSmem<0>));
}

int max_blocks_per_sm(const void* fn, size_t smem) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_pack_pulse(float* x, const PulseParams& p, cudaStream_t s) {
  if (p.n_chunks <= 0) return cudaSuccess;
  k_pack_pulse<<<(p.n_chunks + kWarps - 1) / kWarps, kThreads, 0, s>>>(x, p);
  return cudaGetLastError();
}

cudaError_t launch_unpack_pulse(float* f, const PulseParams& p, cudaStream_t s) {
  if (p.n_chunks <= 0) return cudaSuccess;
  k_unpack_pulse<<<(p.n_chunks + kWarps - 1) / kWarps, kThreads, 0, s>>>(f, p);
  return cudaGetLastError();
}

}  // namespace hx
