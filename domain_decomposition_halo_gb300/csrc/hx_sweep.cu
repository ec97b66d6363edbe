// Slot-sweep force exchange kernel of libhx (sm_103a).
//
// Same operation as the force chunk kernel of hx_kernels.cu: the
// accumulation forces[map[i]] += packed[i] of unpackRecvBufKernel<accumulate>,
// last pulse first ("Force halo exchange: Reversing the dependency chain").
//
// The two differ only in the unit of work. A chunk is a run of one pulse's
// map. A sweep unit is a run of up to kSweepSlots consecutive target slots
// of one sender's array, with every pulse's map entries that fall in it. Its
// slots, its map runs and the received force runs are staged in shared
// memory; the runs are added last pulse first and the slots are written
// back. (A coordinate form, with the unit as a gather source, was measured
// slower than the chunk kernels everywhere and is not built.)
//
// Why this pays on one GPU: with random in-domain order nearly every
// 64-byte granule of a sender's slots holds some pulse's target. The chunk
// kernel therefore reads and writes the whole home region once per pulse, in
// scattered 12-byte accesses. A sweep touches it once in total, as
// sequential streams, and every per-entry access stays in shared memory.
// Each contiguous run is one TMA bulk copy (cp.async.bulk) issued by one lane
// and completing on the warp's mbarrier, so moving a unit's bytes costs a
// handful of instructions instead of one per 128 bytes per lane.
//
// Dependencies and signals are per unit, as in the chunk kernels' fine mode
// ("Enabling parallelism across pulses through kernel fusion"): a unit waits
// for the receivers' units that still add into the slots it reads. Each warp
// is independent. Its claims are static batches of
// units in a topological order (warp w of W takes batches w, w + W, ...), so
// it never waits on a unit that no running warp owns.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

constexpr int kErrTimeout = -6;
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned kPollNapMinNs = HX_POLL_NAP_MIN_NS;   // back-off between flag polls: first nap
constexpr unsigned kPollNapMaxNs = HX_POLL_NAP_MAX_NS;   // ... doubling up to this

// A warp's stage buffer: the unit's slots, its map runs and (forces) its
// received runs, each in its own 16-byte-aligned region at the run's global
// address mod 16. The region offsets are in the unit's segment records.
template <int KIND>
struct alignas(16) WarpSmem {
  alignas(16) unsigned char stage[sweep_stage_bytes(KIND)];
  Unit desc[2];              // the current unit's record and the next one's
  unsigned long long bar;        // completion of the unit's bulk copies
  unsigned long long bar_late;   // completion of a late segment's received run
};

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

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
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

// Bounded wait for the phase of `bar` with the given parity; false on time-out.
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

// Global -> shared bulk copy (TMA); both addresses and the size are
// multiples of 16 bytes.
__device__ __forceinline__ void bulk_load(void* dst, unsigned long long src, unsigned bytes, unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void record_timeout(const UnitParams& P, int item) {
  if (atomicCAS(&P.ctrl->status, 0, kErrTimeout) == 0) atomicExch(&P.ctrl->detail, P.direction * 65536 + item);
}

__device__ __forceinline__ UnitSeg seg_at(const UnitParams& P, const Unit& d, int s) {
  return s < kInlineSegs ? d.seg[s] : P.extra[d.extra_off + s - kInlineSegs];
}

// Whole warp: wait until the units of d's waits [first, first + cnt) have
// been signalled at this epoch (the first waits come with the unit's record, the rest from the
// direction's wait list). Lanes take the wait list in strides of 32 and poll with
// acquire loads at gpu scope and a short back-off; the closing __syncwarp
// orders every lane's acquire before the warp's loads. A wait that runs out
// records a timeout and gives up.
__device__ void wait_units(const UnitParams& P, const Unit& d, unsigned long long epoch, int first, int cnt) {
  const int lane = threadIdx.x & 31;
  for (int w = first + lane; w < first + cnt; w += 32) {
    const Wait wt = w < kInlineWaits ? d.wait_inline[w] : P.waits[d.wait_off + w];
    const unsigned long long* flag = P.flags + wt.item;
    unsigned long long t0 = 0;
    unsigned iter = 0, nap = 0;
    while (ld_acquire_u64(flag) != epoch) {
      if ((iter++ & 15u) == 0u) {
        const unsigned long long now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (ld_relaxed_s32(&P.ctrl->status) != 0) break;
        if (now - t0 > P.timeout_ns) {
          record_timeout(P, __ldg(&P.units[wt.item].item));
          break;
        }
      }
      nap = nap ? min(2u * nap, kPollNapMaxNs) : kPollNapMinNs;
      __nanosleep(nap);
    }
  }
  __syncwarp();
}

// Whole warp, no blocking: one acquire poll of each of d's first 32 waits;
// returns a bit per dependent segment whose producers have all signalled at
// this epoch (a segment with a wait past the first 32 counts as not ready).
__device__ unsigned poll_segments(const UnitParams& P, const Unit& d, unsigned long long epoch) {
  const int lane = threadIdx.x & 31;
  bool pending = false;
  if (lane < d.wait_cnt) {
    const Wait wt = lane < kInlineWaits ? d.wait_inline[lane] : P.waits[d.wait_off + lane];
    pending = ld_acquire_u64(P.flags + wt.item) != epoch;
  }
  const unsigned pend = __ballot_sync(kFull, pending);
  unsigned ready = 0u;
  int wpos = 0;
  for (int s = 0; s < d.seg_cnt; ++s) {
    const int n = seg_at(P, d, s).dep;
    if (n > 0 && wpos + n <= 32) {
      const unsigned bits = (n == 32 ? kFull : ((1u << n) - 1u)) << wpos;
      if ((pend & bits) == 0u) ready |= 1u << s;
    }
    wpos += n;
  }
  return ready;
}

// Run k of a unit: 0 = its slots, then per segment its map run and (forces)
// its received-force run: global address, bytes, stage region offset.
// `dep`: the run is a received run that units of the same launch write.
template <int KIND>
__device__ __forceinline__ void run_of(const float* x, const UnitParams& P, const Unit& d, int k,
                                       unsigned long long& g, unsigned& bytes, unsigned& region, bool& dep) {
  dep = false;
  if (k == 0) {
    g = reinterpret_cast<unsigned long long>(x + 3 * d.base);
    bytes = 12u * static_cast<unsigned>(d.n);
    region = 0;
    return;
  }
  const int per = KIND == 1 ? 2 : 1;
  const UnitSeg sg = seg_at(P, d, (k - 1) / per);
  if ((k - 1) % per == 0) {
    g = reinterpret_cast<unsigned long long>(P.maps + sg.map);
    bytes = 4u * static_cast<unsigned>(sg.n);
    region = static_cast<unsigned>(sg.map_off);
  } else {
    g = reinterpret_cast<unsigned long long>(x + 3 * sg.other);
    bytes = 12u * static_cast<unsigned>(sg.n);
    region = static_cast<unsigned>(sg.src_off);
    dep = sg.dep != 0;
  }
}

// Whole warp: stage every run of the unit, one run per lane (a unit has at
// most 1 + 2 * kSweepSegs <= 32 runs). Each run lands at (its global address
// mod 16) inside its region. Lane 0 announces the bytes of all the runs'
// 16-byte-aligned middles on the warp's mbarrier; then every lane issues its
// run's middle as one bulk copy and copies the head and tail words (under 16
// bytes each) with plain loads. Runs of under 32 bytes go entirely by plain
// loads. The caller waits on the mbarrier and then on the warp (__syncwarp).
//
// `ready` has a bit per segment: the received run of a dependent segment
// (one that units of this launch write) is staged only when its bit is set,
// i.e. its producers have been seen signalled; the other runs always are.
// The mbarrier's arrival announces the bytes of the runs staged.
template <int KIND>
__device__ void stage_unit(const float* x, const UnitParams& P, const Unit& d, unsigned char* st,
                           unsigned long long* bar, unsigned ready = kFull) {
  const int lane = threadIdx.x & 31;
  const int n_runs = 1 + (KIND == 1 ? 2 : 1) * d.seg_cnt;
  unsigned long long g = 0, a0 = 0, a1 = 0;
  unsigned bytes = 0, region = 0, middle = 0;
  bool dep = false;
  if (lane < n_runs) {
    run_of<KIND>(x, P, d, lane, g, bytes, region, dep);
    a0 = (g + 15ull) & ~15ull;
    a1 = (g + bytes) & ~15ull;
    if (a1 > a0) middle = static_cast<unsigned>(a1 - a0);
  }
  const bool mine = !dep || ((ready >> ((lane - 1) / 2)) & 1u) != 0u;
  const unsigned total = __reduce_add_sync(kFull, mine ? middle : 0u);
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the stage's earlier generic use
    mbar_arrive_expect_tx(bar, total);
  }
  __syncwarp();
  if (lane < n_runs && mine) {
    unsigned char* dst = st + region + (g & 15ull);
    // Plain words: up to 3 before and 3 after an aligned middle, or a whole
    // run of under 32 bytes (at most 7 words). All loads are issued before
    // any store so that they are in flight together.
    if (middle > 0) bulk_load(dst + (a0 - g), a0, middle, bar);
    const unsigned nh = middle > 0 ? static_cast<unsigned>(a0 - g) / 4 : bytes / 4;
    const unsigned nt = middle > 0 ? static_cast<unsigned>(g + bytes - a1) / 4 : 0u;
    const unsigned tail0 = static_cast<unsigned>(a1 - g);
    float v[8];
#pragma unroll
    for (unsigned k = 0; k < 8; ++k) {
      const unsigned off = k < nh ? 4u * k : tail0 + 4u * (k - nh);
      if (k < nh + nt) v[k] = __ldcg(reinterpret_cast<const float*>(g + off));
    }
#pragma unroll
    for (unsigned k = 0; k < 8; ++k) {
      const unsigned off = k < nh ? 4u * k : tail0 + 4u * (k - nh);
      if (k < nh + nt) *reinterpret_cast<float*>(dst + off) = v[k];
    }
  }
}

// Warm L2 with the unit's runs (aligned middles; one run per lane). Lines
// whose producers have not signalled yet may be fetched early: L2 is where
// later stores land, so the unit's own bulk copies still read the final data.
template <int KIND>
__device__ void prefetch_unit(const float* x, const UnitParams& P, const Unit& d) {
  const int lane = threadIdx.x & 31;
  const int n_runs = 1 + (KIND == 1 ? 2 : 1) * d.seg_cnt;
  if (lane < n_runs) {
    unsigned long long g;
    unsigned bytes, region;
    bool dep;
    run_of<KIND>(x, P, d, lane, g, bytes, region, dep);
    const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
    if (a1 > a0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a0), "r"(static_cast<unsigned>(a1 - a0))
                   : "memory");
  }
}

// 16-byte global -> shared copy that completes asynchronously;
// cp_async_wait_all waits for all of this thread's copies.
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Lane 0: this warp's bulk stores have read the stage / have completed and
// are ordered before later generic accesses (before a release).
__device__ __forceinline__ void bulk_stores_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_stores_done() {
  asm volatile("cp.async.bulk.wait_group 0;\n\tfence.proxy.async.global;" ::: "memory");
}

// Write-back of a unit's staged slots: one bulk store for the 16-byte-aligned
// middle (the stage keeps the global address mod 16), plain stores for the
// words around it.
__device__ __forceinline__ void write_back(float* __restrict__ f, const Unit& d, float* tile) {
  const int lane = threadIdx.x & 31;
  const unsigned long long gt = reinterpret_cast<unsigned long long>(f + 3 * d.base);
  const unsigned bytes = 12u * static_cast<unsigned>(d.n);
  const unsigned long long a0 = (gt + 15ull) & ~15ull, a1 = (gt + bytes) & ~15ull;
  if (a1 > a0) {
    const unsigned head = static_cast<unsigned>(a0 - gt) / 4, tail = static_cast<unsigned>(gt + bytes - a1) / 4;
    if (lane == 0) {   // the aligned middle in one bulk store (its completion: bulk_stores_done)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the adds, to the copy
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\tcp.async.bulk.commit_group;" ::"l"(
                       a0),
                   "r"(smem_addr(tile + head)), "r"(static_cast<unsigned>(a1 - a0))
                   : "memory");
    }
    if (lane < static_cast<int>(head)) f[3 * d.base + lane] = tile[lane];
    else if (lane >= 4 && lane < 4 + static_cast<int>(tail)) {
      const int k = static_cast<int>((a1 - gt) / 4) + (lane - 4);
      f[3 * d.base + k] = tile[k];
    }
  } else {
    for (int k = lane; k < 3 * d.n; k += 32) f[3 * d.base + k] = tile[k];
  }
}

// Forces of one staged unit: each segment's received run added into the
// slots, segments in list order (last pulse first), a warp barrier between
// segments since one slot can be a target in several pulses; entries of one
// segment have distinct targets. Then the slots are written back.
//
// A dependent segment (one whose received run other units of this launch
// write) whose bit in `ready` is clear was not staged: it waits here for
// exactly its producers (its share of the unit's waits, which are listed
// segment by segment), then stages its run with one bulk copy completing on
// the warp's second mbarrier, so the unit adds its earlier segments while the
// producers of its later ones are still working.
__device__ __forceinline__ void forces_unit(float* __restrict__ f, const UnitParams& P, const Unit& d,
                                            WarpSmem<1>& S, unsigned long long epoch, unsigned ready,
                                            unsigned& parity_late) {
  const int lane = threadIdx.x & 31;
  const unsigned long long gt = reinterpret_cast<unsigned long long>(f + 3 * d.base);
  float* tile = reinterpret_cast<float*>(S.stage + (gt & 15ull));
  int wpos = 0;
  for (int s = 0; s < d.seg_cnt; ++s) {
    const UnitSeg sg = seg_at(P, d, s);
    const int32_t* smap = reinterpret_cast<const int32_t*>(
        S.stage + sg.map_off + (reinterpret_cast<unsigned long long>(P.maps + sg.map) & 15ull));
    const bool late = sg.dep > 0 && ((ready >> s) & 1u) == 0u;   // its run was not staged
    wpos += sg.dep;
    if (late) {
      wait_units(P, d, epoch, wpos - sg.dep, sg.dep);
      // the run into its stage region: one bulk copy of its aligned middle on
      // the late barrier, the words around it by lane 0's plain loads
      if (lane == 0) {
        const unsigned long long g = reinterpret_cast<unsigned long long>(f + 3 * sg.other);
        const unsigned bytes = 12u * static_cast<unsigned>(sg.n);
        const unsigned long long a0 = (g + 15ull) & ~15ull, a1 = (g + bytes) & ~15ull;
        const unsigned middle = a1 > a0 ? static_cast<unsigned>(a1 - a0) : 0u;
        unsigned char* dst = S.stage + sg.src_off + (g & 15ull);
        asm volatile("fence.proxy.async.global;" ::: "memory");       // the producers' stores, to the copy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stage's earlier generic use
        mbar_arrive_expect_tx(&S.bar_late, middle);
        if (middle > 0) bulk_load(dst + (a0 - g), a0, middle, &S.bar_late);
        const unsigned nh = middle > 0 ? static_cast<unsigned>(a0 - g) / 4 : bytes / 4;
        const unsigned nt = middle > 0 ? static_cast<unsigned>(g + bytes - a1) / 4 : 0u;
        for (unsigned k = 0; k < nh + nt; ++k) {
          const unsigned off = k < nh ? 4u * k : static_cast<unsigned>(a1 - g) + 4u * (k - nh);
          *reinterpret_cast<float*>(dst + off) = __ldcg(reinterpret_cast<const float*>(g + off));
        }
      }
      if (!mbar_wait(&S.bar_late, parity_late, P.timeout_ns)) {
        if (lane == 0) record_timeout(P, d.item);
      }
      parity_late ^= 1u;
      __syncwarp();   // lane 0's words are in place
    }
    {
      const float* src = reinterpret_cast<const float*>(
          S.stage + sg.src_off + (reinterpret_cast<unsigned long long>(f + 3 * sg.other) & 15ull));
      for (int i = lane; i < sg.n; i += 32) {
        float* t = tile + 3 * (smap[i] - d.local_a);
        t[0] = __fadd_rn(t[0], src[3 * i + 0]);
        t[1] = __fadd_rn(t[1], src[3 * i + 1]);
        t[2] = __fadd_rn(t[2], src[3 * i + 2]);
      }
    }
    __syncwarp();   // the next (earlier) pulse adds after this one
  }
  write_back(f, d, tile);
}


// KIND 1 = forces (ordered), the one direction the sweep serves.
template <int KIND>
__global__ void __launch_bounds__(kThreads, 3) k_sweep(float* __restrict__ buf, UnitParams P) {
  static_assert(KIND == 1, "the slot sweep serves the force exchange");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31;
  WarpSmem<KIND>& S = reinterpret_cast<WarpSmem<KIND>*>(smem_raw)[threadIdx.x >> 5];
  const unsigned long long W = static_cast<unsigned long long>(gridDim.x) * kWarps;
  const unsigned long long N = P.n_units;
  const unsigned long long NB = (N + kSweepBatch - 1) / kSweepBatch;   // batches of units per launch
  const unsigned long long b0 = static_cast<unsigned long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  // Under programmatic dependent launch the next kernel of the stream may be
  // scheduled once every block of this grid has started (so this grid is
  // wholly resident first, as the static claims need), and this grid waits
  // for the previous kernel to complete before it touches any table, flag
  // or force. Both instructions are no-ops in a plain stream-ordered launch.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The launch's epoch; its last block to finish stores it for the next
  // launch of this direction (which reads it after this grid has completed).
  const unsigned long long epoch = ld_relaxed_u64(&P.ctrl->epoch) + 1ull;
  if (b0 < NB) {
    unsigned long long c = b0 * kSweepBatch;
    const int drop_item = *reinterpret_cast<const volatile int*>(&P.ctrl->drop_item);
    if (lane == 0) {
      mbar_init(&S.bar, 1);
      mbar_init(&S.bar_late, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    unsigned parity = 0, parity_late = 0;
    // Units are claimed in batches of kSweepBatch consecutive units, and the
    // claims are static: warp w of the W warps takes batches w, w + W,
    // w + 2W, ... in order, so a warp works through its claims in list order
    // and the topological order keeps the launch deadlock-free (the smallest
    // unfinished unit's warp has finished its earlier units, and its
    // producers sit at smaller positions). The next unit's record is copied
    // in while the current unit is staged and processed.
    if (lane < 16)
      cp_async_16(reinterpret_cast<int4*>(&S.desc[0]) + lane, reinterpret_cast<const int4*>(P.units + c) + lane);
    cp_async_wait_all();
    __syncwarp();
    int b = 0;
    bool next_ready = false;   // the next unit's waits were seen satisfied ahead of time
    while (true) {
      const bool same_batch = (c + 1) % kSweepBatch != 0;
      const unsigned long long cn = same_batch ? c + 1 : (c / kSweepBatch + W) * kSweepBatch;   // this warp's next unit
      if (cn < N && lane < 16)
        cp_async_16(reinterpret_cast<int4*>(&S.desc[b ^ 1]) + lane, reinterpret_cast<const int4*>(P.units + cn) + lane);
      const Unit& d = S.desc[b];
      // The unit's waits. With segment waits (short lists, where the pulse
      // chain bounds the launch), one poll decides which dependent runs are
      // staged now; the others are read after their own segment's wait.
      // Otherwise the warp waits for all its producers before staging.
      unsigned ready = kFull;
      if (d.wait_cnt > 0) {
        if (!next_ready) {
          if (P.seg_waits) ready = poll_segments(P, d, epoch);
          else wait_units(P, d, epoch, 0, d.wait_cnt);
        }
        // bulk copies (async proxy) then read what other warps stored (generic proxy) before their signals
        if (lane == 0 && ready) asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
      }
      if (KIND == 1) {   // the previous unit's write-back has read the stage
        if (lane == 0) bulk_stores_read();
        __syncwarp();
      }
      stage_unit<KIND>(buf, P, d, S.stage, &S.bar, ready);
      if (cn < N) {   // the next record, then its runs into L2 while this unit's copies land
        cp_async_wait_all();
        __syncwarp();
        prefetch_unit<KIND>(buf, P, S.desc[b ^ 1]);
      }
      if (!mbar_wait(&S.bar, parity, P.timeout_ns)) {
        if (lane == 0) record_timeout(P, d.item);
      }
      parity ^= 1u;
      __syncwarp();   // the lanes' edge words are in place
      forces_unit(buf, P, d, S, epoch, ready, parity_late);
      // One acquire poll of the next unit's waits (when they all come with
      // its record), issued before this unit's signal so that the two round
      // trips overlap; if it finds them set, the next unit skips its wait.
      unsigned long long pv = epoch;
      bool poll_next = false;
      if (cn < N) {
        const Unit& dn = S.desc[b ^ 1];
        poll_next = dn.wait_cnt > 0 && dn.wait_cnt <= kInlineWaits;
        if (poll_next && lane < dn.wait_cnt) pv = ld_acquire_u64(P.flags + dn.wait_inline[lane].item);
      }
      if (d.flags & kSignal) {
        __syncwarp();   // every lane's stores precede lane 0's release
        if (lane == 0) {
          if (KIND == 1) bulk_stores_done();
          if (d.item != drop_item) st_release_u64(P.flags + c, epoch);
        }
      }
      next_ready = __all_sync(kFull, pv == epoch) && poll_next;   // every lane's acquire precedes the next staging
      if (cn >= N) break;
      cp_async_wait_all();   // the next record
      __syncwarp();          // ... for every lane; the stage is rewritten for the next unit
      c = cn;
      b ^= 1;
    }
    if (KIND == 1 && lane == 0) bulk_stores_done();   // nothing in flight when the warp exits
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned done = atomicAdd(&P.ctrl->exits, 1u);
    if (done == gridDim.x - 1) {
      P.ctrl->exits = 0u;
      st_relaxed_u64(&P.ctrl->epoch, epoch);
    }
  }
}

}  // namespace

const void* sweep_kernel(int) { return reinterpret_cast<const void*>(&k_sweep<1>); }

size_t sweep_smem_bytes(int) { return kWarps * sizeof(WarpSmem<1>); }

int sweep_blocks_per_sm(int kind) {
  const void* fn = sweep_kernel(kind);
  const size_t smem = sweep_smem_bytes(kind);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

}  // namespace hx
