// Tile-staged exchange kernels of libhx (sm_103a).
//
// Same operation as the chunk kernels of hx_kernels.cu: the gather
// packed[i] = x[map[i]] of packSendBufKernel and the accumulation
// forces[map[i]] += packed[i] of unpackRecvBufKernel<accumulate>, fused over
// all pulses with per-unit release/acquire signals ("Enabling parallelism
// across pulses through kernel fusion"). The unit of work is a tile of
// consecutive slots instead of a run of map entries:
//   - coordinates: a block copies a source tile into shared memory (a TMA
//     bulk copy for home slots, plain coalesced loads for halo slots that
//     other blocks wrote in this launch, after waiting for them) and serves
//     the gathers of every pulse that selects from it, storing each pulse's
//     output run straight into the receiver's slots;
//   - forces: a block copies a target tile into shared memory, adds the
//     received halo forces of every pulse that targets it - last pulse first,
//     so each slot is the fp32 sum in reverse pulse order ("Force halo
//     exchange: Reversing the dependency chain") - and writes it back.
// With random in-domain order nearly every 64-byte granule of a domain's
// slots holds a selected atom, so reading whole tiles moves about the same
// DRAM bytes as scattered 12-byte accesses, as sequential streams, and all
// per-entry traffic stays in shared memory.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

constexpr int kErrTimeout = -6;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kTileBytes = kTile * 12;

struct alignas(16) TileSmem {
  alignas(16) unsigned char buf[kTileBytes + 16];   // tile image, shifted by (address mod 16)
  float stage[kWarps][96];                          // per-warp transpose for coalesced runs
  unsigned long long mbar;                          // completion of the bulk copy
  unsigned long long next;                          // next unit of this block
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
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
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

// Bulk copy global -> shared (TMA), completing on `bar`. Both addresses and
// the size are multiples of 16 bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void record_timeout(const TileParams& P, int item) {
  if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0) atomicExch(&P.ctrl->detail, P.direction * 65536 + item);
}

// Thread 0: wait until every producer tile of this unit has stored this
// launch's epoch (acquire, gpu scope). Bounded by the handle's timeout.
__device__ void wait_unit(const TileParams& P, const TileUnit& u, unsigned long long epoch) {
  for (int w = 0; w < u.wait_cnt; ++w) {
    const Wait wt = P.waits[u.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    unsigned long long t0 = 0;
    unsigned iter = 0;
    while (ld_acquire_u64(flag) != epoch) {
      if ((iter++ & 31u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) return;
        if (now - t0 > P.timeout_ns) {
          record_timeout(P, P.units[wt.item].item);
          return;
        }
      }
    }
  }
}

// Copy the unit's slots [base, base + n) into S.buf. Returns the shared
// address of the tile's first float. `parity` tracks the mbarrier phase.
__device__ float* load_tile(float* __restrict__ x, const TileParams& P, const TileUnit& u, TileSmem& S,
                            unsigned& parity) {
  const int tid = threadIdx.x;
  const unsigned long long g0 = reinterpret_cast<unsigned long long>(x + 3 * u.base);
  const unsigned long long g1 = g0 + 12ull * static_cast<unsigned long long>(u.n);
  float* tile = reinterpret_cast<float*>(S.buf + (g0 & 15ull));
  const unsigned long long a0 = (g0 + 15ull) & ~15ull;
  const unsigned long long a1 = g1 & ~15ull;
  const bool bulk = !(u.flags & kHaloSrc) && a1 > a0;
  if (!bulk) {
    const float* src = x + 3 * u.base;
    for (int k = tid; k < 3 * u.n; k += blockDim.x) tile[k] = src[k];
    __syncthreads();
    return tile;
  }
  if (tid == 0) {
    const unsigned bytes = static_cast<unsigned>(a1 - a0);
    mbar_expect_tx(&S.mbar, bytes);
    bulk_load(reinterpret_cast<unsigned char*>(tile) + (a0 - g0), reinterpret_cast<const void*>(a0), bytes,
              &S.mbar);
  }
  // the unaligned head and tail (under 16 bytes each) by plain loads
  const int head = static_cast<int>((a0 - g0) / 4), tail_from = static_cast<int>((a1 - g0) / 4);
  if (tid < head) tile[tid] = x[3 * u.base + tid];
  if (tid >= 32 && tid - 32 + tail_from < 3 * u.n && tid - 32 < 4)
    tile[tid - 32 + tail_from] = x[3 * u.base + tid - 32 + tail_from];
  unsigned long long t0 = 0;
  unsigned iter = 0;
  while (!mbar_try_wait(&S.mbar, parity)) {
    if ((++iter & 63u) == 0u) {   // a bulk copy always completes; bound the wait all the same
      const unsigned long long now = global_timer_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > P.timeout_ns) {
        if (tid == 0) record_timeout(P, u.item);
        break;
      }
    }
  }
  parity ^= 1u;
  __syncthreads();
  return tile;
}

// Coordinates: for every segment, out[i] = tile[map[i] - local_a] (+shift),
// stored as coalesced 96-float runs per warp round of 32 entries.
__device__ void coords_unit(float* __restrict__ x, const TileParams& P, const TileUnit& u, const float* tile,
                            TileSmem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* stage = S.stage[warp];
  for (int sidx = 0; sidx < u.seg_cnt; ++sidx) {
    const TileSeg sg = P.segs[u.seg_off + sidx];
    const int32_t* map = P.maps + sg.map;
    float* dst = x + 3 * sg.other;
    const int rounds = (sg.n + 31) / 32;
    for (int r0 = warp; r0 < rounds; r0 += 4 * kWarps) {
      int j[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = (r0 + k * kWarps) * 32 + lane;
        j[k] = (e < sg.n) ? __ldg(map + e) - u.local_a : -1;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = r0 + k * kWarps;
        if (r >= rounds) break;
        const int n_round = min(32, sg.n - r * 32);
        if (j[k] >= 0) {
          float v0 = tile[3 * j[k]], v1 = tile[3 * j[k] + 1], v2 = tile[3 * j[k] + 2];
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
        float* d = dst + 96 * static_cast<int64_t>(r);
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int idx = q * 32 + lane;
          if (idx < 3 * n_round) d[idx] = stage[idx];
        }
        __syncwarp();
      }
    }
  }
}

// Forces: segments come last pulse first; within one segment every target is
// distinct, so the adds of one pulse are independent, and a barrier between
// segments keeps the reverse pulse order of each slot's sum.
__device__ void forces_unit(float* __restrict__ f, const TileParams& P, const TileUnit& u, float* tile,
                            TileSmem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* stage = S.stage[warp];
  for (int sidx = 0; sidx < u.seg_cnt; ++sidx) {
    const TileSeg sg = P.segs[u.seg_off + sidx];
    const int32_t* map = P.maps + sg.map;
    const float* src = f + 3 * sg.other;
    const int rounds = (sg.n + 31) / 32;
    for (int r0 = warp; r0 < rounds; r0 += 4 * kWarps) {
      int j[4];
      float g[4][3];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = (r0 + k * kWarps) * 32 + lane;
        j[k] = (e < sg.n) ? __ldg(map + e) - u.local_a : -1;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = r0 + k * kWarps;
        if (r >= rounds) break;
        const int n_round = min(32, sg.n - r * 32);
        const float* s = src + 96 * static_cast<int64_t>(r);
#pragma unroll
        for (int q = 0; q < 3; ++q) {
          const int idx = q * 32 + lane;
          if (idx < 3 * n_round) stage[idx] = s[idx];
        }
        __syncwarp();
        g[k][0] = stage[3 * lane];
        g[k][1] = stage[3 * lane + 1];
        g[k][2] = stage[3 * lane + 2];
        __syncwarp();
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (j[k] >= 0) {
          float* t = tile + 3 * j[k];
          t[0] = __fadd_rn(t[0], g[k][0]);
          t[1] = __fadd_rn(t[1], g[k][1]);
          t[2] = __fadd_rn(t[2], g[k][2]);
        }
      }
    }
    __syncthreads();
  }
  float* out = f + 3 * u.base;
  for (int k = threadIdx.x; k < 3 * u.n; k += blockDim.x) out[k] = tile[k];
}

template <int KIND>
__global__ void __launch_bounds__(kThreads) k_tiles(float* __restrict__ x, TileParams P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem& S = *reinterpret_cast<TileSmem*>(smem_raw);
  const unsigned long long N = P.n_units;
  unsigned long long c = blockIdx.x;
  if (c >= N) return;
  if (threadIdx.x == 0) mbar_init(&S.mbar, 1);
  __syncthreads();
  const int drop_item = *reinterpret_cast<const volatile int*>(&P.ctrl->drop_item);
  unsigned parity = 0;
  unsigned long long base = ~0ull, epoch = 0;   // thread 0 only
  while (c < N) {
    unsigned long long t = 0;
    if (threadIdx.x == 0) t = atomicAdd(&P.ctrl->ticket, 1ull);
    const TileUnit u = P.units[c];
    if (threadIdx.x == 0 && base == ~0ull) {   // every ticket of one launch lies in [base, base + N)
      base = t - t % N;
      epoch = base / N + 1ull;
    }
    if (u.wait_cnt > 0) {
      if (threadIdx.x == 0) wait_unit(P, u, epoch);
      __syncthreads();
    }
    float* tile = load_tile(x, P, u, S, parity);
    if (KIND == 0) coords_unit(x, P, u, tile, S);
    else forces_unit(x, P, u, tile, S);
    __syncthreads();
    if (threadIdx.x == 0) {
      if ((u.flags & kSignal) && u.item != drop_item) st_release_u64(P.flags + c, epoch);
      S.next = (t - base) + gridDim.x;
    }
    __syncthreads();
    c = S.next;
  }
}

}  // namespace

const void* tiles_kernel(int kind) {
  return kind == 0 ? reinterpret_cast<const void*>(&k_tiles<0>) : reinterpret_cast<const void*>(&k_tiles<1>);
}

size_t tiles_smem_bytes() { return sizeof(TileSmem); }

int tiles_blocks_per_sm(int kind) {
  const void* fn = tiles_kernel(kind);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, tiles_smem_bytes()) != cudaSuccess) return 0;
  return n;
}

}  // namespace hx
