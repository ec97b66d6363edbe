// Tile-staged exchange kernels of libhx (sm_103a).
//
// Same operation as the chunk kernels of hx_kernels.cu: the gather
// packed[i] = x[map[i]] of packSendBufKernel and the accumulation
// forces[map[i]] += packed[i] of unpackRecvBufKernel<accumulate>, fused over
// all pulses with per-unit release/acquire signals ("Enabling parallelism
// across pulses through kernel fusion"). The unit of work is a tile of up to
// kTile consecutive slots of one domain's array with up to kTileEntries map
// entries falling in it:
//   - coordinates: the tile is a source. Its slots and the runs of every map
//     that selects from it are copied into shared memory by TMA bulk copies;
//     each map run's gathers are served from shared memory and stored as
//     coalesced runs straight into the receiver's slots;
//   - forces: the tile is a target. Its slots, the map runs and the received
//     force runs are copied in; the runs are added last pulse first, so each
//     slot is the fp32 sum in reverse pulse order ("Force halo exchange:
//     Reversing the dependency chain"), and the tile is written back.
// Two stages per block: while one unit is processed, the copies of the
// block's next unit are in flight, and its 256-byte record is already in
// shared memory. With random in-domain order nearly every 64-byte granule of
// a domain's slots holds a selected atom, so copying whole tiles moves about
// the DRAM bytes that scattered 12-byte accesses would, as sequential
// streams, and every per-entry access stays in shared memory.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

constexpr int kErrTimeout = -6;

template <int KIND>
struct StageLayout {
  static constexpr int kTileBytes = kTile * 12 + 16;
  static constexpr int kMapBytes = kTileEntries * 4 + 32 * kTileSegs;
  static constexpr int kSrcBytes = KIND == 1 ? kTileEntries * 12 + 32 * kTileSegs : 0;
  static constexpr int kBytes = kTileBytes + kMapBytes + kSrcBytes;
};

template <int KIND>
struct alignas(16) TileSmem {
  alignas(16) unsigned char stage[2][StageLayout<KIND>::kBytes];
  TileUnit desc[2];                               // records of the current and the next unit
  TileSeg extra[2][kTileSegs - kInlineSegs];      // their segments past the inline ones
  float out[kWarps][96];                          // per-warp transpose for coalesced runs (coordinates)
  unsigned long long mbar[2];                     // bulk-copy completion, one per stage
  unsigned long long next_unit;
  unsigned long long launch;                      // launches completed before this one
  int prefetched[2];
};

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

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned smem_addr(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Global -> shared bulk copy (TMA); both addresses and the size are
// multiples of 16 bytes.
__device__ __forceinline__ void bulk_load(void* dst, unsigned long long src, unsigned bytes, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void record_timeout(const TileParams& P, int item) {
  if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0) atomicExch(&P.ctrl->detail, P.direction * 65536 + item);
}

// Threads 0..15: copy unit c's record into `d`, then (when it has more than
// kInlineSegs segments) its overflow segments into `extra`. Ends with a
// block barrier.
template <int KIND>
__device__ void load_desc(const TileParams& P, unsigned long long c, TileUnit* d, TileSeg* extra) {
  if (threadIdx.x < 16)
    reinterpret_cast<int4*>(d)[threadIdx.x] = __ldg(reinterpret_cast<const int4*>(P.units + c) + threadIdx.x);
  __syncthreads();
  const int more = d->seg_cnt - kInlineSegs;
  if (more > 0) {
    for (int w = threadIdx.x; w < 3 * more; w += kThreads)
      reinterpret_cast<int4*>(extra)[w] = __ldg(reinterpret_cast<const int4*>(P.extra + d->extra_off) + w);
    __syncthreads();
  }
}

__device__ __forceinline__ const TileSeg& seg_of(const TileUnit& d, const TileSeg* extra, int s) {
  return s < kInlineSegs ? d.seg[s] : extra[s - kInlineSegs];
}

// Thread 0: are (block = wait until) all producer tiles of u at this epoch?
__device__ bool producers_done(const TileParams& P, const TileUnit& u, unsigned long long epoch, bool block) {
  for (int w = 0; w < u.wait_cnt; ++w) {
    const Wait wt = P.waits[u.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    if (ld_acquire_u64(flag) == epoch) continue;
    if (!block) return false;
    unsigned long long t0 = 0;
    unsigned iter = 0;
    while (ld_acquire_u64(flag) != epoch) {
      if ((iter++ & 31u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) return true;
        if (now - t0 > P.timeout_ns) {
          record_timeout(P, __ldg(&P.units[wt.item].item));
          return true;
        }
      }
    }
  }
  return true;
}

// Run k of a unit: 0 = its slots, then per segment its map run and (forces)
// its received-force run.
template <int KIND>
__device__ __forceinline__ void run_of(const float* __restrict__ x, const TileParams& P, const TileUnit& d,
                                       const TileSeg* extra, int k, unsigned long long& g, unsigned& bytes,
                                       unsigned& region) {
  if (k == 0) {
    g = reinterpret_cast<unsigned long long>(x + 3 * d.base);
    bytes = 12u * static_cast<unsigned>(d.n);
    region = 0;
    return;
  }
  const int per = KIND == 1 ? 2 : 1;
  const TileSeg& sg = seg_of(d, extra, (k - 1) / per);
  if ((k - 1) % per == 0) {
    g = reinterpret_cast<unsigned long long>(P.maps + sg.map);
    bytes = 4u * static_cast<unsigned>(sg.n);
    region = static_cast<unsigned>(sg.map_off);
  } else {
    g = reinterpret_cast<unsigned long long>(x + 3 * sg.other);
    bytes = 12u * static_cast<unsigned>(sg.n);
    region = static_cast<unsigned>(sg.src_off);
  }
}

// All threads: start the copies of a unit into stage buffer `st`. Every run
// lands at (its global address mod 16) inside its 16-byte-aligned region;
// thread 0 bulk-copies the aligned middles (one mbarrier phase), and the
// head and tail words (under 16 bytes each) go by plain loads.
template <int KIND>
__device__ void issue_stage(const float* __restrict__ x, const TileParams& P, const TileUnit& d,
                            const TileSeg* extra, unsigned char* st, unsigned long long* bar) {
  const int n_runs = 1 + (KIND == 1 ? 2 : 1) * d.seg_cnt;
  if (threadIdx.x == 0) {
    unsigned total = 0;
    for (int k = 0; k < n_runs; ++k) {
      unsigned long long g;
      unsigned bytes, region;
      run_of<KIND>(x, P, d, extra, k, g, bytes, region);
      const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
      if (a1 > a0) total += static_cast<unsigned>(a1 - a0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier generic use of the stage
    mbar_arrive_expect_tx(bar, total);
    for (int k = 0; k < n_runs; ++k) {
      unsigned long long g;
      unsigned bytes, region;
      run_of<KIND>(x, P, d, extra, k, g, bytes, region);
      const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
      if (a1 > a0) bulk_load(st + region + (g & 15ull) + (a0 - g), a0, static_cast<unsigned>(a1 - a0), bar);
    }
  }
  for (int k = threadIdx.x >> 3; k < n_runs; k += kThreads / 8) {
    unsigned long long g;
    unsigned bytes, region;
    run_of<KIND>(x, P, d, extra, k, g, bytes, region);
    const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
    const int w = threadIdx.x & 7;
    if (a1 > a0) {
      const unsigned head = static_cast<unsigned>(a0 - g) / 4, tail = static_cast<unsigned>(g + bytes - a1) / 4;
      unsigned long long word;
      if (w < 4) {
        if (static_cast<unsigned>(w) >= head) continue;
        word = g + 4ull * w;
      } else {
        if (static_cast<unsigned>(w - 4) >= tail) continue;
        word = a1 + 4ull * (w - 4);
      }
      *reinterpret_cast<float*>(st + region + (g & 15ull) + (word - g)) = *reinterpret_cast<const float*>(word);
    } else {   // a run of under 32 bytes: every word by plain loads
      for (unsigned o = 4u * w; o < bytes; o += 32u)
        *reinterpret_cast<float*>(st + region + (g & 15ull) + o) = *reinterpret_cast<const float*>(g + o);
    }
  }
}

// Coordinates: out[i] = tile[map[i] - local_a] (+shift), per segment, as
// coalesced 96-float runs per warp round of 32 entries.
__device__ void coords_unit(float* __restrict__ x, const TileParams& P, const TileUnit& d, const TileSeg* extra,
                            const unsigned char* st, float (*out)[96]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* tile = reinterpret_cast<const float*>(st + (reinterpret_cast<unsigned long long>(x + 3 * d.base) & 15ull));
  float* stage = out[warp];
  for (int s = 0; s < d.seg_cnt; ++s) {
    const TileSeg& sg = seg_of(d, extra, s);
    const int32_t* map = reinterpret_cast<const int32_t*>(
        st + sg.map_off + (reinterpret_cast<unsigned long long>(P.maps + sg.map) & 15ull));
    float* dst = x + 3 * sg.other;
    const int rounds = (sg.n + 31) / 32;
    for (int r = warp; r < rounds; r += kWarps) {
      const int e = r * 32 + lane;
      const int n_round = min(32, sg.n - r * 32);
      if (e < sg.n) {
        const int j = map[e] - d.local_a;
        float v0 = tile[3 * j], v1 = tile[3 * j + 1], v2 = tile[3 * j + 2];
        if (sg.do_shift) {
          if (sg.dim == 0) v0 = __fadd_rn(v0, sg.shift);
          else if (sg.dim == 1) v1 = __fadd_rn(v1, sg.shift);
          else v2 = __fadd_rn(v2, sg.shift);
        }
        stage[3 * lane] = v0;
        stage[3 * lane + 1] = v1;
        stage[3 * lane + 2] = v2;
      }
      __syncwarp();
      float* dd = dst + 96 * static_cast<int64_t>(r);
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int idx = q * 32 + lane;
        if (idx < 3 * n_round) dd[idx] = stage[idx];
      }
      __syncwarp();
    }
  }
}

// Forces: segments come last pulse first; within one segment every target
// is distinct, and a barrier between segments keeps each slot's sum in
// reverse pulse order. Then the tile goes back.
__device__ void forces_unit(float* __restrict__ f, const TileUnit& d, const TileSeg* extra, unsigned char* st,
                            const TileParams& P) {
  float* tile = reinterpret_cast<float*>(st + (reinterpret_cast<unsigned long long>(f + 3 * d.base) & 15ull));
  for (int s = 0; s < d.seg_cnt; ++s) {
    const TileSeg& sg = seg_of(d, extra, s);
    const int32_t* map = reinterpret_cast<const int32_t*>(
        st + sg.map_off + (reinterpret_cast<unsigned long long>(P.maps + sg.map) & 15ull));
    const float* src = reinterpret_cast<const float*>(
        st + sg.src_off + (reinterpret_cast<unsigned long long>(f + 3 * sg.other) & 15ull));
    for (int e = threadIdx.x; e < sg.n; e += kThreads) {
      float* t = tile + 3 * (map[e] - d.local_a);
      t[0] = __fadd_rn(t[0], src[3 * e]);
      t[1] = __fadd_rn(t[1], src[3 * e + 1]);
      t[2] = __fadd_rn(t[2], src[3 * e + 2]);
    }
    __syncthreads();
  }
  float* out = f + 3 * d.base;
  for (int k = threadIdx.x; k < 3 * d.n; k += kThreads) out[k] = tile[k];
}

template <int KIND>
__global__ void __launch_bounds__(kThreads) k_tiles(float* __restrict__ x, TileParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<KIND>& S = *reinterpret_cast<TileSmem<KIND>*>(smem_raw);
  const unsigned long long N = P.n_units;
  unsigned long long c = blockIdx.x;
  if (c >= N) return;
  const unsigned long long G = gridDim.x;
  if (threadIdx.x == 0) {
    mbar_init(&S.mbar[0], 1);
    mbar_init(&S.mbar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the ticket of this block's first unit numbers the launch and names the next unit
    const unsigned long long t = atomicAdd(&P.ctrl->ticket, 1ull);
    S.launch = t / N;
    S.next_unit = (t % N) + G;
    S.prefetched[0] = S.prefetched[1] = 0;
  }
  load_desc<KIND>(P, c, &S.desc[0], S.extra[0]);   // its barrier publishes the fields above
  const unsigned long long epoch = S.launch + 1ull;
  const unsigned long long base = S.launch * N;
  const int drop_item = *reinterpret_cast<const volatile int*>(&P.ctrl->drop_item);
  unsigned parity[2] = {0u, 0u};
  unsigned long long nxt = S.next_unit;
  int cur = 0;
  while (c < N) {
    const TileUnit& d = S.desc[cur];
    unsigned long long t_next = 0;
    if (threadIdx.x == 0 && nxt < N) t_next = atomicAdd(&P.ctrl->ticket, 1ull);   // the ticket of `nxt`
    // the current unit: when it was not prefetched, wait for its producers and copy it now
    if (!S.prefetched[cur]) {
      if (threadIdx.x == 0) {
        producers_done(P, d, epoch, true);
        if (d.wait_cnt > 0) asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncthreads();
      issue_stage<KIND>(x, P, d, S.extra[cur], S.stage[cur], &S.mbar[cur]);
    }
    // the next unit's record, then its copies when nothing it reads is still being written
    if (nxt < N) {
      load_desc<KIND>(P, nxt, &S.desc[cur ^ 1], S.extra[cur ^ 1]);
      if (threadIdx.x == 0) {
        const bool ready = producers_done(P, S.desc[cur ^ 1], epoch, false);
        if (ready && S.desc[cur ^ 1].wait_cnt > 0) asm volatile("fence.proxy.async.global;" ::: "memory");
        S.prefetched[cur ^ 1] = ready ? 1 : 0;
      }
      __syncthreads();
      if (S.prefetched[cur ^ 1]) issue_stage<KIND>(x, P, S.desc[cur ^ 1], S.extra[cur ^ 1], S.stage[cur ^ 1], &S.mbar[cur ^ 1]);
    }
    {
      unsigned long long t0 = 0;
      unsigned iter = 0;
      while (!mbar_try_wait(&S.mbar[cur], parity[cur])) {
        if ((++iter & 63u) == 0u) {   // a bulk copy always completes; bound the wait all the same
          const unsigned long long now = global_timer_ns();
          if (t0 == 0) t0 = now;
          if (now - t0 > P.timeout_ns) {
            if (threadIdx.x == 0) record_timeout(P, d.item);
            break;
          }
        }
      }
      parity[cur] ^= 1u;
    }
    __syncthreads();   // plain-loaded edges of the runs are visible too
    if (KIND == 0) coords_unit(x, P, d, S.extra[cur], S.stage[cur], S.out);
    else forces_unit(x, d, S.extra[cur], S.stage[cur], P);
    __syncthreads();
    if (threadIdx.x == 0) {
      if ((d.flags & kSignal) && d.item != drop_item) st_release_u64(P.flags + c, epoch);
      S.prefetched[cur] = 0;
      S.next_unit = (nxt < N) ? (t_next - base) + G : N;
    }
    __syncthreads();
    c = nxt;
    nxt = S.next_unit;
    cur ^= 1;
  }
}

}  // namespace

const void* tiles_kernel(int kind) {
  return kind == 0 ? reinterpret_cast<const void*>(&k_tiles<0>) : reinterpret_cast<const void*>(&k_tiles<1>);
}

size_t tiles_smem_bytes(int kind) { return kind == 0 ? sizeof(TileSmem<0>) : sizeof(TileSmem<1>); }

int tiles_blocks_per_sm(int kind) {
  const void* fn = tiles_kernel(kind);
  const size_t smem = tiles_smem_bytes(kind);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

}  // namespace hx
