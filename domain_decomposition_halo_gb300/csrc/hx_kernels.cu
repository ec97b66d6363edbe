// Exchange kernels of libhx (sm_103a).
//
// Coordinates: one persistent launch for every pulse ("Enabling parallelism
// across pulses through kernel fusion"; fusedPulsesPackAndSendKernel). Work is
// cut into chunks of map entries, handed out in a topological order (all
// independent chunks first, then the dependent tails pulse by pulse), first
// by block index and then by an atomic ticket, so a chunk only ever waits for
// chunks handed out before it. A chunk gathers x[src + map[i]], applies the
// periodic shift and stores straight into the receiver's slots (the
// NVLink-path "pack directly into the peer's coordinate array", here the
// same HBM). A dependent chunk first loads its map entries, then thread 0
// waits with acquire loads at gpu scope for the signals of earlier pulses
// into its sender (packHaloCoords' wait on every preceding pulse), then the
// block gathers. When the block has stored its chunk it signals: either the
// pages' hierarchical scheme (signalPeerOnLastBlock: a counting atomic with
// release at gpu scope elects the last block, which stores the epoch flag
// with release) or one release-add per chunk to an arrival counter.
//
// Forces: the same skeleton in reverse pulse order ("Force halo exchange:
// Reversing the dependency chain"): a chunk of (sender r, pulse p) adds the
// received halo-slot forces of its receiver into r's targets through the map
// (unpackRecvBufKernel<accumulate=true>) once every later pulse that writes
// those targets or those slots has signalled.
//
// Every wait is bounded by %globaltimer; a wait that runs out records
// HX_ERR_TIMEOUT in the control block and the block carries on, so a kernel
// always finishes.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

constexpr int kErrTimeout = -6;

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
// scope: every block's stores are released before its increment, and the
// electing block acquires all of them before it publishes the flag.
__device__ __forceinline__ unsigned atom_inc_acq_rel(unsigned* p, unsigned mod) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(mod) : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long load_epoch(const Ctrl* c) {
  return *reinterpret_cast<const volatile unsigned long long*>(&c->epoch);
}

// Thread 0 only. Returns false when a wait gave up (timeout or an earlier
// error), in which case the caller proceeds without the guarantee.
template <int MODE>
__device__ bool wait_chunk(const DirParams& P, const Chunk& ch, unsigned long long epoch) {
  for (int w = 0; w < ch.wait_cnt; ++w) {
    const Wait wt = P.waits[ch.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    const unsigned long long target =
        (MODE == kCounter) ? epoch * static_cast<unsigned long long>(wt.chunks) : epoch;
    unsigned long long t0 = 0;
    unsigned iter = 0;
    // last-block flags hold an epoch (compare for equality, as the pages'
    // signal wait does); counters only grow
    while ((MODE == kCounter) ? (ld_acquire_u64(flag) < target) : (ld_acquire_u64(flag) != target)) {
      if ((iter++ & 31u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) return false;
        if (now - t0 > P.timeout_ns) {
          if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0)
            atomicExch(&P.ctrl->detail, P.direction * 65536 + wt.item);
          return false;
        }
      }
    }
  }
  return true;
}

template <int MODE>
__device__ void signal_item(const DirParams& P, int item, int chunks, unsigned long long epoch) {
  const bool drop = (item == *reinterpret_cast<const volatile int*>(&P.ctrl->drop_item));
  if (MODE == kCounter) {
    if (!drop) red_release_add_u64(P.flags + item, 1ull);
  } else {
    const unsigned last = static_cast<unsigned>(chunks - 1);
    const unsigned old = atom_inc_acq_rel(P.blk_count + item, last);
    if (old == last && !drop) st_release_u64(P.flags + item, epoch);
  }
}

// Last block out resets the ticket and publishes the epoch for the next launch.
__device__ void block_exit(const DirParams& P, unsigned long long epoch) {
  if (threadIdx.x == 0) {
    const unsigned last = gridDim.x - 1;
    const unsigned old = atom_inc_acq_rel(&P.ctrl->exit_count, last);
    if (old == last) {
      P.ctrl->ticket = 0u;
      *reinterpret_cast<volatile unsigned long long*>(&P.ctrl->epoch) = epoch;
    }
  }
}

__device__ __forceinline__ void load_map(const int32_t* __restrict__ map, int base, int end,
                                         int (&j)[kUnroll]) {
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int i = base + u * kThreads + static_cast<int>(threadIdx.x);
    j[u] = (i < end) ? __ldg(map + i) : -1;
  }
}

// Gather float3 x[src + j] (+shift along dim) for the thread's entries.
// Home slots are read-only during the coordinate kernel, so independent
// entries may use the read-only path; halo slots written by other blocks of
// this launch are read at L2 (.cg).
__device__ __forceinline__ void gather(const float* __restrict__ src, const int (&j)[kUnroll],
                                       bool halo_src, float (&v)[kUnroll][3]) {
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    if (j[u] >= 0) {
      const float* s = src + 3 * static_cast<int64_t>(j[u]);
      if (halo_src) {
        v[u][0] = __ldcg(s);
        v[u][1] = __ldcg(s + 1);
        v[u][2] = __ldcg(s + 2);
      } else {
        v[u][0] = __ldg(s);
        v[u][1] = __ldg(s + 1);
        v[u][2] = __ldg(s + 2);
      }
    }
  }
}

__device__ __forceinline__ void apply_shift(const Item& it, float (&v)[kUnroll][3]) {
  if (!it.do_shift) return;  // no add at all: keeps -0.0 and every bit of unshifted values
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    if (it.dim == 0) v[u][0] = __fadd_rn(v[u][0], it.shift);
    else if (it.dim == 1) v[u][1] = __fadd_rn(v[u][1], it.shift);
    else v[u][2] = __fadd_rn(v[u][2], it.shift);
  }
}

// Store the warp's 32 consecutive entries [wb, wb + 32) as 96 contiguous
// floats with three coalesced 128-byte stores (transposed through shared).
__device__ __forceinline__ void store_warp(float* __restrict__ dst, int wb, int end,
                                           const float (&v)[3], float* stage) {
  const int lane = threadIdx.x & 31;
  const int n = min(32, end - wb);
  if (n <= 0) return;
  if (lane < n) {
    stage[3 * lane + 0] = v[0];
    stage[3 * lane + 1] = v[1];
    stage[3 * lane + 2] = v[2];
  }
  __syncwarp();
  float* d = dst + 3 * static_cast<int64_t>(wb);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int idx = k * 32 + lane;
    if (idx < 3 * n) d[idx] = stage[idx];
  }
  __syncwarp();
}

// Load the warp's 32 consecutive received forces [wb, wb + 32) coalesced.
__device__ __forceinline__ void load_warp(const float* __restrict__ srcv, int wb, int end,
                                          float (&g)[3], float* stage) {
  const int lane = threadIdx.x & 31;
  const int n = min(32, end - wb);
  if (n <= 0) return;
  const float* s = srcv + 3 * static_cast<int64_t>(wb);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int idx = k * 32 + lane;
    if (idx < 3 * n) stage[idx] = __ldcg(s + idx);
  }
  __syncwarp();
  if (lane < n) {
    g[0] = stage[3 * lane + 0];
    g[1] = stage[3 * lane + 1];
    g[2] = stage[3 * lane + 2];
  }
  __syncwarp();
}

// Body of one coordinate chunk; `j` already holds the first pass's map entries.
__device__ __forceinline__ void coords_body(float* __restrict__ x, const Item& it, const Chunk& ch,
                                            const int32_t* __restrict__ map, bool halo_src,
                                            int (&j)[kUnroll], float* stage) {
  const float* src = x + 3 * it.src_base;
  float* dst = x + 3 * it.dst_base;
  const int warp = threadIdx.x >> 5;
  for (int base = ch.begin; base < ch.end; base += kPass) {
    float v[kUnroll][3];
    gather(src, j, halo_src, v);
    apply_shift(it, v);
    if (base + kPass < ch.end) load_map(map, base + kPass, ch.end, j);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) store_warp(dst, base + u * kThreads + warp * 32, ch.end, v[u], stage);
  }
}

// Body of one force chunk; `j` already holds the first pass's map entries.
template <bool ORDERED>
__device__ __forceinline__ void forces_body(float* __restrict__ f, const Item& it, const Chunk& ch,
                                            const int32_t* __restrict__ map, int (&j)[kUnroll],
                                            float* stage) {
  float* tgt = f + 3 * it.src_base;
  const float* rcv = f + 3 * it.dst_base;
  const int warp = threadIdx.x >> 5;
  for (int base = ch.begin; base < ch.end; base += kPass) {
    float g[kUnroll][3];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) load_warp(rcv, base + u * kThreads + warp * 32, ch.end, g[u], stage);
    int jj[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) jj[u] = j[u];
    if (base + kPass < ch.end) load_map(map, base + kPass, ch.end, j);
    if (ORDERED) {
      float t[kUnroll][3];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (jj[u] >= 0) {
          const float* p = tgt + 3 * static_cast<int64_t>(jj[u]);
          t[u][0] = __ldcg(p);
          t[u][1] = __ldcg(p + 1);
          t[u][2] = __ldcg(p + 2);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (jj[u] >= 0) {
          float* p = tgt + 3 * static_cast<int64_t>(jj[u]);
          p[0] = __fadd_rn(t[u][0], g[u][0]);
          p[1] = __fadd_rn(t[u][1], g[u][1]);
          p[2] = __fadd_rn(t[u][2], g[u][2]);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (jj[u] >= 0) {
          float* p = tgt + 3 * static_cast<int64_t>(jj[u]);
          atomicAdd(p, g[u][0]);
          atomicAdd(p + 1, g[u][1]);
          atomicAdd(p + 2, g[u][2]);
        }
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) k_coords_fused(float* __restrict__ x, DirParams P) {
  __shared__ float s_stage[kThreads / 32][96];
  __shared__ int s_next;
  const unsigned long long epoch = load_epoch(P.ctrl) + 1ull;
  float* stage = s_stage[threadIdx.x >> 5];
  int c = blockIdx.x;
  while (c < P.n_chunks) {
    unsigned ticket = 0;
    if (threadIdx.x == 0) ticket = atomicAdd(&P.ctrl->ticket, 1u);
    const Chunk ch = P.chunks[c];
    const Item it = P.items[ch.item];
    const int32_t* map = P.maps + it.map_off;
    int j[kUnroll];
    load_map(map, ch.begin, ch.end, j);
    if (ch.wait_cnt > 0) {
      if (threadIdx.x == 0) wait_chunk<MODE>(P, ch, epoch);
      __syncthreads();
    }
    coords_body(x, it, ch, map, ch.halo_src != 0, j, stage);
    __syncthreads();
    if (threadIdx.x == 0) {
      signal_item<MODE>(P, ch.item, it.coord_chunks, epoch);
      s_next = static_cast<int>(ticket + gridDim.x);
    }
    __syncthreads();
    c = s_next;
  }
  block_exit(P, epoch);
}

template <int MODE, bool ORDERED>
__global__ void __launch_bounds__(kThreads) k_forces_fused(float* __restrict__ f, DirParams P) {
  __shared__ float s_stage[kThreads / 32][96];
  __shared__ int s_next;
  const unsigned long long epoch = load_epoch(P.ctrl) + 1ull;
  float* stage = s_stage[threadIdx.x >> 5];
  int c = blockIdx.x;
  while (c < P.n_chunks) {
    unsigned ticket = 0;
    if (threadIdx.x == 0) ticket = atomicAdd(&P.ctrl->ticket, 1u);
    const Chunk ch = P.chunks[c];
    const Item it = P.items[ch.item];
    const int32_t* map = P.maps + it.map_off;
    int j[kUnroll];
    load_map(map, ch.begin, ch.end, j);
    if (ch.wait_cnt > 0) {
      if (threadIdx.x == 0) wait_chunk<MODE>(P, ch, epoch);
      __syncthreads();
    }
    forces_body<ORDERED>(f, it, ch, map, j, stage);
    __syncthreads();
    if (threadIdx.x == 0) {
      signal_item<MODE>(P, ch.item, it.force_chunks, epoch);
      s_next = static_cast<int>(ticket + gridDim.x);
    }
    __syncthreads();
    c = s_next;
  }
  block_exit(P, epoch);
}

// Unfused baseline: one block per chunk of one pulse, stream order between pulses.
__global__ void __launch_bounds__(kThreads) k_pack_pulse(float* __restrict__ x, PulseParams P) {
  __shared__ float s_stage[kThreads / 32][96];
  const Chunk ch = P.chunks[P.chunk_begin + blockIdx.x];
  const Item it = P.items[ch.item];
  const int32_t* map = P.maps + it.map_off;
  int j[kUnroll];
  load_map(map, ch.begin, ch.end, j);
  coords_body(x, it, ch, map, true, j, s_stage[threadIdx.x >> 5]);
}

__global__ void __launch_bounds__(kThreads) k_unpack_pulse(float* __restrict__ f, PulseParams P) {
  __shared__ float s_stage[kThreads / 32][96];
  const Chunk ch = P.chunks[P.chunk_begin + blockIdx.x];
  const Item it = P.items[ch.item];
  const int32_t* map = P.maps + it.map_off;
  int j[kUnroll];
  load_map(map, ch.begin, ch.end, j);
  forces_body<true>(f, it, ch, map, j, s_stage[threadIdx.x >> 5]);
}

__global__ void k_noop() {}

}  // namespace

const void* coords_kernel(int signal_mode) {
  return signal_mode == kCounter ? reinterpret_cast<const void*>(&k_coords_fused<kCounter>)
                                 : reinterpret_cast<const void*>(&k_coords_fused<kLastBlock>);
}

const void* forces_kernel(int signal_mode, bool ordered) {
  if (signal_mode == kCounter)
    return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kCounter, true>)
                   : reinterpret_cast<const void*>(&k_forces_fused<kCounter, false>);
  return ordered ? reinterpret_cast<const void*>(&k_forces_fused<kLastBlock, true>)
                 : reinterpret_cast<const void*>(&k_forces_fused<kLastBlock, false>);
}

const void* noop_kernel() { return reinterpret_cast<const void*>(&k_noop); }

int max_blocks_per_sm(const void* fn) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, 0) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_pack_pulse(float* x, const PulseParams& p, int n_chunks, cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  k_pack_pulse<<<n_chunks, kThreads, 0, s>>>(x, p);
  return cudaGetLastError();
}

cudaError_t launch_unpack_pulse(float* f, const PulseParams& p, int n_chunks, cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  k_unpack_pulse<<<n_chunks, kThreads, 0, s>>>(f, p);
  return cudaGetLastError();
}

}  // namespace hx
