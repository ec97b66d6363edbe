// Exchange kernels of libhx (sm_103a).
//
// Coordinates: one persistent launch for every pulse ("Enabling parallelism
// across pulses through kernel fusion"; fusedPulsesPackAndSendKernel). The
// work is cut into warp chunks of up to 256 entries of one (sender, pulse)
// map, listed in a topological order (a chunk only waits for items listed
// before it) chosen for L2 locality. A warp takes its first chunk by its
// global warp index and every further one by an atomic ticket, so a waiting
// chunk can only wait for chunks that running warps already own. Warps never
// synchronise with each other inside a block: like the pages' per-warp TMA
// variant ("NVLink path: TMA-based direct stores"), each warp gathers,
// stores and signals on its own.
//
// A chunk gathers x[src + map[i]], applies the periodic shift, and stores
// straight into the receiver's slots (the NVLink-path "pack directly into
// the peer's coordinate array": here the same HBM). A chunk of forwarded
// entries loads its map entries, then lane 0 waits with acquire loads at gpu
// scope until the items that filled those slots have signalled
// (packHaloCoords). After its stores a chunk signals its item, when anybody
// waits for it: either the pages' hierarchical scheme (signalPeerOnLastBlock:
// a counting atomic with release semantics elects the last chunk, which
// stores the epoch flag with release) or one release-add per chunk to an
// arrival counter.
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

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
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

// Lane 0 only. Returns false when a wait gave up (timeout, or another wait
// already failed), in which case the chunk proceeds without the guarantee.
template <int MODE>
__device__ bool wait_chunk(const DirParams& P, const Chunk& ch, unsigned long long epoch) {
  for (int w = 0; w < ch.wait_cnt; ++w) {
    const Wait wt = P.waits[ch.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    const unsigned long long target =
        (MODE == kCounter) ? epoch * static_cast<unsigned long long>(wt.chunks) : epoch;
    unsigned long long t0 = 0;
    unsigned iter = 0;
    // epoch flags (per item or per chunk) are compared for equality, as the
    // pages' signal wait does; arrival counters only grow
    while ((MODE == kCounter) ? (ld_acquire_u64(flag) < target) : (ld_acquire_u64(flag) != target)) {
      if ((iter++ & 31u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) return false;
        if (now - t0 > P.timeout_ns) {
          if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0) {
            // report the (sender, pulse) item, also when the wait was on one chunk of it
            const int item = (MODE == kChunkFlag) ? P.chunks[wt.item].item : wt.item;
            atomicExch(&P.ctrl->detail, P.direction * 65536 + item);
          }
          return false;
        }
      }
    }
  }
  return true;
}

// Lane 0 only, after the warp's stores (ordered by the preceding __syncwarp).
template <int MODE>
__device__ __forceinline__ void signal_chunk(const DirParams& P, const Chunk& ch, unsigned long long c,
                                             unsigned long long epoch, int drop_item) {
  const bool drop = ch.item == drop_item;
  if (MODE == kChunkFlag) {
    if (!drop) st_release_u64(P.flags + c, epoch);
  } else if (MODE == kCounter) {
    if (!drop) red_release_add_u64(P.flags + ch.item, 1ull);
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

// Coordinates of one chunk: gather (+shift) and store into the receiver.
// Home slots are never written by the coordinate kernel, so independent
// chunks read them through the read-only path.
__device__ __forceinline__ void coords_chunk(float* __restrict__ x, const Chunk& ch, const int (&j)[kRounds],
                                             float* stage) {
  const float* src = x + 3 * ch.src;
  float v[kRounds][3];
  const bool halo = (ch.flags & kHaloSrc) != 0;
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    if (j[u] >= 0) {
      const float* s = src + 3 * static_cast<int64_t>(j[u]);
      if (halo) {
        v[u][0] = s[0];
        v[u][1] = s[1];
        v[u][2] = s[2];
      } else {
        v[u][0] = __ldg(s);
        v[u][1] = __ldg(s + 1);
        v[u][2] = __ldg(s + 2);
      }
    }
  }
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

// Forces of one chunk: targets[map[i]] += received[i], x then y then z.
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
        if (jj >= 0) {
          float* p = tgt + 3 * static_cast<int64_t>(jj);
          p[0] = __fadd_rn(t[u][0], g[u][0]);
          p[1] = __fadd_rn(t[u][1], g[u][1]);
          p[2] = __fadd_rn(t[u][2], g[u][2]);
        }
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

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void coords_chunk_bulk(float* __restrict__ x, const Chunk& ch, const int (&j)[kRounds],
                                                  unsigned char* stage) {
  const int lane = threadIdx.x & 31;
  const float* src = x + 3 * ch.src;
  float v[kRounds][3];
  const bool halo = (ch.flags & kHaloSrc) != 0;
#pragma unroll
  for (int u = 0; u < kRounds; ++u) {
    if (j[u] >= 0) {
      const float* s = src + 3 * static_cast<int64_t>(j[u]);
      if (halo) {
        v[u][0] = s[0];
        v[u][1] = s[1];
        v[u][2] = s[2];
      } else {
        v[u][0] = __ldg(s);
        v[u][1] = __ldg(s + 1);
        v[u][2] = __ldg(s + 2);
      }
    }
  }
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
    if (j[u] >= 0) {
      const int e = u * 32 + lane;
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

// Persistent warp loop shared by both directions. KIND 0 = coordinates,
// 1 = forces ordered, 2 = forces unordered, 3 = coordinates by bulk stores.
template <int MODE, int KIND>
__device__ __forceinline__ void run_warps(float* __restrict__ buf, const DirParams& P, float* stage) {
  const int lane = threadIdx.x & 31;
  const unsigned long long W = static_cast<unsigned long long>(gridDim.x) * kWarps;
  const unsigned long long N = P.n_chunks;
  unsigned long long c = static_cast<unsigned long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  allow_dependents();
  wait_prerequisites();   // before the first ticket, flag or buffer access
  if (c >= N) return;
  const int drop_item = *reinterpret_cast<const volatile int*>(&P.ctrl->drop_item);
  unsigned long long base = ~0ull;   // first ticket of this launch: (epoch - 1) * N
  unsigned long long epoch = 0;
  while (c < N) {
    unsigned long long t = 0;
    if (lane == 0) t = atomicAdd(&P.ctrl->ticket, 1ull);
    const Chunk ch = load_chunk(P.chunks + c);
    int j[kRounds];
    load_map(P.maps + ch.map, ch.n, j);
    t = __shfl_sync(kFull, t, 0);
    if (base == ~0ull) {   // every ticket of one launch lies in [base, base + N)
      base = t - t % N;
      epoch = base / N + 1ull;
    }
    if (ch.wait_cnt > 0) {
      if (lane == 0) wait_chunk<MODE>(P, ch, epoch);
      __syncwarp();
    }
    if (KIND == 0) coords_chunk(buf, ch, j, stage);
    else if (KIND == 3) coords_chunk_bulk(buf, ch, j, reinterpret_cast<unsigned char*>(stage));
    else forces_chunk<KIND == 1>(buf, ch, j);
    if (ch.flags & kSignal) {
      __syncwarp();
      if (lane == 0) {
        if (KIND == 3) bulk_store_done();
        signal_chunk<MODE>(P, ch, c, epoch, drop_item);
      }
    }
    c = (t - base) + W;
  }
  if (KIND == 3 && lane == 0) bulk_store_done();   // nothing in flight when the warp exits
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_coords_fused(float* __restrict__ x, DirParams P) {
  __shared__ float s_stage[kWarps][96];
  run_warps<MODE, 0>(x, P, s_stage[threadIdx.x >> 5]);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_coords_bulk(float* __restrict__ x, DirParams P) {
  __shared__ __align__(16) float s_stage[kWarps][kBulkStageBytes / 4];
  run_warps<MODE, 3>(x, P, s_stage[threadIdx.x >> 5]);
}

template <int MODE, bool ORDERED>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_forces_fused(float* __restrict__ f, DirParams P) {
  run_warps<MODE, ORDERED ? 1 : 2>(f, P, nullptr);
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
  coords_chunk(x, ch, j, s_stage[threadIdx.x >> 5]);
}

__global__ void __launch_bounds__(kThreads) k_unpack_pulse(float* __restrict__ f, PulseParams P) {
  const int c = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (c >= P.n_chunks) return;
  const Chunk ch = load_chunk(P.chunks + P.chunk_begin + c);
  int j[kRounds];
  load_map(P.maps + ch.map, ch.n, j);
  forces_chunk<true>(f, ch, j);
}

// Cluster path: the whole exchange in one thread-block cluster. Pulse after
// pulse (forces last pulse first), the cluster's warps take the pulse's
// chunks; a cluster barrier with release/acquire semantics separates the
// pulses, so a pulse reads every slot that earlier pulses stored (forwarding)
// or added into (forces). No flags, tickets or spin waits: the pages' "each
// waits for all preceding pulse signals", with the cluster barrier as the
// signal. Meant for decompositions small enough that the dependency chain
// and the launch, not bandwidth, set the step time.
__device__ __forceinline__ void cluster_sync_release_acquire() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int KIND>
__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kClusterThreads, 1)
    k_cluster(float* __restrict__ buf, ClusterParams P) {
  constexpr int kCtaWarps = kClusterThreads / 32;
  __shared__ float s_stage[kCtaWarps][96];
  const int warp = threadIdx.x >> 5;
  const int gw = blockIdx.x * kCtaWarps + warp;   // the grid is the one cluster
  const int W = kClusterCtas * kCtaWarps;
  for (int k = 0; k < P.n_pulses; ++k) {
    const int p = KIND == 0 ? k : P.n_pulses - 1 - k;
    for (int c = P.begin[p] + gw; c < P.begin[p + 1]; c += W) {
      const Chunk ch = load_chunk(P.chunks + c);   // flags carry kHaloSrc: halo sources by plain loads
      int j[kRounds];
      load_map(P.maps + ch.map, ch.n, j);
      if (KIND == 0) coords_chunk(buf, ch, j, s_stage[warp]);
      else forces_chunk<true>(buf, ch, j);
    }
    if (k + 1 < P.n_pulses) cluster_sync_release_acquire();
  }
}

__global__ void k_noop() {}

}  // namespace

const void* coords_kernel(int signal_mode, bool bulk_store) {
  if (bulk_store) {
    if (signal_mode == kChunkFlag) return reinterpret_cast<const void*>(&k_coords_bulk<kChunkFlag>);
    return signal_mode == kCounter ? reinterpret_cast<const void*>(&k_coords_bulk<kCounter>)
                                   : reinterpret_cast<const void*>(&k_coords_bulk<kLastArrival>);
  }
  if (signal_mode == kChunkFlag) return reinterpret_cast<const void*>(&k_coords_fused<kChunkFlag>);
  return signal_mode == kCounter ? reinterpret_cast<const void*>(&k_coords_fused<kCounter>)
                                 : reinterpret_cast<const void*>(&k_coords_fused<kLastArrival>);
}

const void* forces_kernel(int signal_mode, bool ordered) {
  if (signal_mode == kChunkFlag)
    return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kChunkFlag, true>)
                   : reinterpret_cast<const void*>(&k_forces_fused<kChunkFlag, false>);
  if (signal_mode == kCounter)
    return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kCounter, true>)
                   : reinterpret_cast<const void*>(&k_forces_fused<kCounter, false>);
  return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kLastArrival, true>)
                 : reinterpret_cast<const void*>(&k_forces_fused<kLastArrival, false>);
}

const void* noop_kernel() { return reinterpret_cast<const void*>(&k_noop); }

const void* cluster_kernel(int kind) {
  return kind == 0 ? reinterpret_cast<const void*>(&k_cluster<0>) : reinterpret_cast<const void*>(&k_cluster<1>);
}

int max_blocks_per_sm(const void* fn) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, 0) != cudaSuccess) return 0;
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
