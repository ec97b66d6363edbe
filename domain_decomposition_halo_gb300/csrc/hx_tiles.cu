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
// Each block is a producer/consumer pipeline. One producer warp draws
// tickets, loads unit records, waits for their producers and issues the bulk
// copies into a ring of 3 (forces) or 4 (coordinates) stages guarded by
// full/empty mbarriers. Eight consumer warps process the staged units and
// send the signals. With random in-domain order nearly every 64-byte granule
// of a domain's slots holds a selected atom, so copying whole tiles moves
// about the DRAM bytes that scattered 12-byte accesses would, as sequential
// streams, and every per-entry access stays in shared memory. The one
// producer per block serialises the control path of every unit; the slot
// sweep (hx_sweep.cu) gives each warp its own units instead.
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
struct Stages {
  static constexpr int kCount = KIND == 1 ? 3 : 4;   // ring depth: as many as 2-3 blocks per SM allow
};

template <int KIND>
struct alignas(16) TileSmem {
  alignas(16) unsigned char stage[Stages<KIND>::kCount][StageLayout<KIND>::kBytes];
  TileUnit desc[Stages<KIND>::kCount];                      // record of the unit in each stage
  TileSeg extra[Stages<KIND>::kCount][kTileSegs - kInlineSegs];
  float out[kTileConsumerWarps][96];                        // per-warp transpose (coordinates)
  unsigned long long full[Stages<KIND>::kCount];            // copies of a stage landed (producer -> consumers)
  unsigned long long empty[Stages<KIND>::kCount];           // consumers done with a stage (consumers -> producer)
  long long unit_of[Stages<KIND>::kCount];                  // unit in each stage, -1 = no more units
  unsigned long long epoch;
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

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bounded wait for the phase of `bar` with the given parity; false on time-out.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity, unsigned long long limit_ns);

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

__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity, unsigned long long limit_ns) {
  unsigned long long t0 = 0;
  unsigned iter = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++iter & 63u) == 0u) {
      const unsigned long long now = global_timer_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > limit_ns) return false;
    }
  }
  return true;
}

// Named barrier of the consumer warps only (the producer warp runs ahead).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kTileConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ void record_timeout(const TileParams& P, int item) {
  if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0) atomicExch(&P.ctrl->detail, P.direction * 65536 + item);
}

// Producer warp: copy unit c's record into `d`, and its segments past the
// inline ones into `extra`.
__device__ void load_desc(const TileParams& P, unsigned long long c, TileUnit* d, TileSeg* extra) {
  const int lane = threadIdx.x & 31;
  if (lane < 16)
    reinterpret_cast<int4*>(d)[lane] = __ldg(reinterpret_cast<const int4*>(P.units + c) + lane);
  __syncwarp();
  const int more = d->seg_cnt - kInlineSegs;
  for (int w = lane; w < 3 * more; w += 32)
    reinterpret_cast<int4*>(extra)[w] = __ldg(reinterpret_cast<const int4*>(P.extra + d->extra_off) + w);
  __syncwarp();
}

__device__ __forceinline__ const TileSeg& seg_of(const TileUnit& d, const TileSeg* extra, int s) {
  return s < kInlineSegs ? d.seg[s] : extra[s - kInlineSegs];
}

// Producer warp: wait until every tile that u reads has been signalled at
// this epoch. Lanes take the wait list in strides of 32 and the warp joins at
// the end, so one unit's flags are polled in parallel rather than one after
// another. A wait that runs out records a timeout and gives up.
__device__ void producers_wait(const TileParams& P, const TileUnit& u, unsigned long long epoch) {
  const int lane = threadIdx.x & 31;
  for (int w = lane; w < u.wait_cnt; w += 32) {
    const Wait wt = P.waits[u.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    unsigned long long t0 = 0;
    unsigned iter = 0;
    while (ld_acquire_u64(flag) != epoch) {
      if ((iter++ & 31u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) break;
        if (now - t0 > P.timeout_ns) {
          record_timeout(P, __ldg(&P.units[wt.item].item));
          break;
        }
      }
    }
  }
  __syncwarp();   // orders every lane's acquire before lane 0 issues the copies
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

// Producer warp: start the copies of a unit into stage buffer `st`. Every
// run lands at (its global address mod 16) inside its 16-byte-aligned
// region; the head and tail words (under 16 bytes each) go by plain loads of
// the warp's lanes, then lane 0 arrives on `full` expecting the bytes of the
// aligned middles and issues them as bulk copies.
template <int KIND>
__device__ void issue_stage(const float* __restrict__ x, const TileParams& P, const TileUnit& d,
                            const TileSeg* extra, unsigned char* st, unsigned long long* full) {
  const int lane = threadIdx.x & 31;
  const int n_runs = 1 + (KIND == 1 ? 2 : 1) * d.seg_cnt;
  for (int k = lane >> 3; k < n_runs; k += 4) {
    unsigned long long g;
    unsigned bytes, region;
    run_of<KIND>(x, P, d, extra, k, g, bytes, region);
    const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
    const int w = lane & 7;
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
  __syncwarp();
  if (lane == 0) {
    unsigned total = 0;
    for (int k = 0; k < n_runs; ++k) {
      unsigned long long g;
      unsigned bytes, region;
      run_of<KIND>(x, P, d, extra, k, g, bytes, region);
      const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
      if (a1 > a0) total += static_cast<unsigned>(a1 - a0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier generic use of the stage
    mbar_arrive_expect_tx(full, total);
    for (int k = 0; k < n_runs; ++k) {
      unsigned long long g;
      unsigned bytes, region;
      run_of<KIND>(x, P, d, extra, k, g, bytes, region);
      const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
      if (a1 > a0) bulk_load(st + region + (g & 15ull) + (a0 - g), a0, static_cast<unsigned>(a1 - a0), full);
    }
  }
  __syncwarp();
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
    for (int r = warp; r < rounds; r += kTileConsumerWarps) {
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
    for (int e = threadIdx.x; e < sg.n; e += kTileConsumerWarps * 32) {
      float* t = tile + 3 * (map[e] - d.local_a);
      t[0] = __fadd_rn(t[0], src[3 * e]);
      t[1] = __fadd_rn(t[1], src[3 * e + 1]);
      t[2] = __fadd_rn(t[2], src[3 * e + 2]);
    }
    consumers_sync();
  }
  float* out = f + 3 * d.base;
  for (int k = threadIdx.x; k < 3 * d.n; k += kTileConsumerWarps * 32) out[k] = tile[k];
}

template <int KIND>
__global__ void __launch_bounds__(kTileThreads) k_tiles(float* __restrict__ x, TileParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<KIND>& S = *reinterpret_cast<TileSmem<KIND>*>(smem_raw);
  constexpr int kS = Stages<KIND>::kCount;
  const unsigned long long N = P.n_units;
  if (blockIdx.x >= N) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kS; ++k) {
      mbar_init(&S.full[k], 1);
      mbar_init(&S.empty[k], kTileConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kTileConsumerWarps) {
    // ---------------- producer: records, waits, copies, tickets ----------------
    unsigned long long c = blockIdx.x, base = 0, epoch = 0, t = 0;
    if (lane == 0) {
      t = atomicAdd(&P.ctrl->ticket, 1ull);   // the ticket of the first unit numbers the launch
      base = t - t % N;
      epoch = base / N + 1ull;
      S.epoch = epoch;
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    base = __shfl_sync(0xffffffffu, base, 0);
    epoch = __shfl_sync(0xffffffffu, epoch, 0);
    unsigned long long nxt = (t - base) + gridDim.x;
    unsigned empty_parity[kS];
    for (int k = 0; k < kS; ++k) empty_parity[k] = 1u;   // a fresh stage counts as emptied
    int slot = 0;
    while (c < N) {
      if (!mbar_wait(&S.empty[slot], empty_parity[slot], P.timeout_ns)) {
        if (lane == 0) record_timeout(P, -1);
      }
      empty_parity[slot] ^= 1u;
      unsigned long long tn = 0;
      if (lane == 0 && nxt < N) tn = atomicAdd(&P.ctrl->ticket, 1ull);   // the ticket of `nxt`
      load_desc(P, c, &S.desc[slot], S.extra[slot]);
      producers_wait(P, S.desc[slot], epoch);
      if (lane == 0) {
        if (S.desc[slot].wait_cnt > 0) asm volatile("fence.proxy.async.global;" ::: "memory");
        S.unit_of[slot] = static_cast<long long>(c);
      }
      __syncwarp();
      issue_stage<KIND>(x, P, S.desc[slot], S.extra[slot], S.stage[slot], &S.full[slot]);
      tn = __shfl_sync(0xffffffffu, tn, 0);
      c = nxt;
      nxt = (c < N) ? (tn - base) + gridDim.x : N;
      slot = slot + 1 == kS ? 0 : slot + 1;
    }
    // no more units: hand the consumers an end marker
    if (!mbar_wait(&S.empty[slot], empty_parity[slot], P.timeout_ns)) {
      if (lane == 0) record_timeout(P, -1);
    }
    if (lane == 0) {
      S.unit_of[slot] = -1;
      mbar_arrive(&S.full[slot]);
    }
    return;
  }

  // ---------------- consumers: shared-memory work, stores, signals ----------------
  const int drop_item = *reinterpret_cast<const volatile int*>(&P.ctrl->drop_item);
  unsigned full_parity[kS];
  for (int k = 0; k < kS; ++k) full_parity[k] = 0u;
  int slot = 0;
  while (true) {
    if (!mbar_wait(&S.full[slot], full_parity[slot], P.timeout_ns)) {
      if (threadIdx.x == 0) record_timeout(P, -1);
    }
    full_parity[slot] ^= 1u;
    const long long c = S.unit_of[slot];
    if (c < 0) break;
    const TileUnit& d = S.desc[slot];
    if (KIND == 0) coords_unit(x, P, d, S.extra[slot], S.stage[slot], S.out);
    else forces_unit(x, d, S.extra[slot], S.stage[slot], P);
    consumers_sync();   // every store of this unit is issued
    if (threadIdx.x == 0 && (d.flags & kSignal) && d.item != drop_item)
      st_release_u64(P.flags + c, S.epoch);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
    slot = slot + 1 == kS ? 0 : slot + 1;
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
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kTileThreads, smem) != cudaSuccess) return 0;
  return n;
}

}  // namespace hx
