// Resolved exchange kernels of libhx (sm_103a): the staged forwarding
// unrolled at build time, for decompositions where the dependency chain,
// not bandwidth, sets the step time.
//
// Coordinates. A halo slot received in pulse p holds what its sender held in
// the sent slot, plus the periodic shift of that pulse ("Dependency-aware
// packing": forwarded atoms are re-sent from the received slots). Following
// the senders back ends at one home atom, the slot's origin. Along the way
// each dimension adds its box length at most once (a forwarding path moves
// np_d < n_d cells, so it wraps at most once per dimension), and no add
// touches another component. So the slot's final value is the origin's
// value with fl(x_d + L_d) in each shifted component d: bit for bit the
// staged result, computed by one independent gather per slot.
//
// Forces. Reversed, every copy adds its value into the slot it was sent
// from ("Force halo exchange: Reversing the dependency chain"), so a home
// atom and all its copies form a tree whose edges are those adds. The
// staged order (pulses last to first) restricted to one tree is that tree's
// adds sorted by descending pulse, and adds of one pulse never chain (a slot
// received in pulse p is sent only in later pulses). Replaying a tree's adds
// in that order in registers gives every slot of the tree the staged fp32
// sums exactly. A thread loads a tree's record, its node values, adds, and
// stores the nodes that received adds. Most trees are an atom with one copy
// (one add) or a corner atom with two copies and the copy of its first copy
// (three adds in a fixed order); those two shapes get a 16-byte record and
// straight-line code, the rest a general record in blocks of their own,
// scheduled first because their threads take longest.
//
// Tables are numbered in slot order (halo slots, tree roots), so neighbouring
// threads touch neighbouring slots.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

// Programmatic dependent launch: let the next kernel of the stream be
// scheduled now (it waits in griddepcontrol.wait for this one), and wait for
// the previous kernel before reading what it wrote. Both are no-ops in a
// launch without the programmatic-serialization attribute.
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Up to kResSlotsPerThread halo slots per thread (as many as the segment
// holds), strided by the block so that every load and store instruction of
// a warp covers consecutive slots: slot = origin (+ shifts).
__global__ void __launch_bounds__(kResThreads) k_resolved_coords(float* __restrict__ x, ResolvedParams P) {
  allow_dependents();
  const ResSeg sg = P.segs[blockIdx.x];   // build-time tables, read before the wait
  uint32_t om[kResSlotsPerThread];
#pragma unroll
  for (int u = 0; u < kResSlotsPerThread; ++u) {
    const int j = u * kResThreads + static_cast<int>(threadIdx.x);
    om[u] = j < sg.n ? __ldg(P.origin_mask + sg.k + j) : 0u;
  }
  wait_prerequisites();
  float v[kResSlotsPerThread][3];
#pragma unroll
  for (int u = 0; u < kResSlotsPerThread; ++u) {   // every gather issued before any is used
    const int j = u * kResThreads + static_cast<int>(threadIdx.x);
    if (j < sg.n) {
      const float* s = x + 3 * static_cast<int64_t>(om[u] & ((1u << kResOriginBits) - 1u));
      v[u][0] = s[0];
      v[u][1] = s[1];
      v[u][2] = s[2];
    }
  }
#pragma unroll
  for (int u = 0; u < kResSlotsPerThread; ++u) {
    const int j = u * kResThreads + static_cast<int>(threadIdx.x);
    if (j < sg.n) {
      const unsigned mask = om[u] >> kResOriginBits;
      if (mask & 1u) v[u][0] = __fadd_rn(v[u][0], P.box[0]);   // no add otherwise: unshifted values keep every bit
      if (mask & 2u) v[u][1] = __fadd_rn(v[u][1], P.box[1]);
      if (mask & 4u) v[u][2] = __fadd_rn(v[u][2], P.box[2]);
      float* d = x + 3 * (static_cast<int64_t>(sg.slot) + j);
      d[0] = v[u][0];
      d[1] = v[u][1];
      d[2] = v[u][2];
    }
  }
}

__device__ __forceinline__ void load3(const float* f, int slot, float (&v)[3]) {
  const float* p = f + 3 * static_cast<int64_t>(slot);
  v[0] = p[0];
  v[1] = p[1];
  v[2] = p[2];
}
// A scattered slot written as an 8-byte and a 4-byte store (one L2 write
// request fewer than three words).
__device__ __forceinline__ void store3(float* f, int slot, const float (&v)[3]) {
  float* p = f + 3 * static_cast<int64_t>(slot);
  const bool lo8 = (reinterpret_cast<uintptr_t>(p) & 7u) == 0u;
  *reinterpret_cast<float2*>(lo8 ? p : p + 1) = lo8 ? make_float2(v[0], v[1]) : make_float2(v[1], v[2]);
  *(lo8 ? p + 2 : p) = lo8 ? v[2] : v[0];
}
__device__ __forceinline__ void add3(float (&a)[3], const float (&b)[3]) {
  a[0] = __fadd_rn(a[0], b[0]);
  a[1] = __fadd_rn(a[1], b[1]);
  a[2] = __fadd_rn(a[2], b[2]);
}

// A general tree: replay its adds in descending pulse order.
__device__ __forceinline__ void general_tree(float* __restrict__ f, const TreeRec& r) {
  float v[kTreeNodes][3];
#pragma unroll
  for (int j = 0; j < kTreeNodes; ++j)
    if (j < r.n_nodes) load3(f, r.node[j], v[j]);
  unsigned target = 0;   // nodes that receive an add
#pragma unroll
  for (int e = 0; e < kTreeNodes - 1; ++e) {
    if (e < r.n_nodes - 1) {
      const int tg = r.ev[e] & 15, sc = r.ev[e] >> 4;
      // registers are indexed through unrolled selects so that v stays in registers
#pragma unroll
      for (int a = 0; a < kTreeNodes; ++a) {
        if (a != tg) continue;
#pragma unroll
        for (int b = 0; b < kTreeNodes; ++b) {
          if (b != sc) continue;
          add3(v[a], v[b]);
        }
      }
      target |= 1u << tg;
    }
  }
#pragma unroll
  for (int j = 0; j < kTreeNodes; ++j)
    if (j < r.n_nodes && (target >> j & 1u)) store3(f, r.node[j], v[j]);
}

// General blocks (first in the grid): one general tree per thread. Record
// blocks: one or two pairs or quads per thread (strided by the block; all
// index loads, then all value loads issued before any add); pairs and quads
// share a warp.
__global__ void __launch_bounds__(kResThreads) k_resolved_forces(float* __restrict__ f, ResolvedParams P) {
  constexpr int U = kResTreesPerThread;
  allow_dependents();
  const int gen_blocks = static_cast<int>(gridDim.x) - P.rec_blocks;   // first: their threads take longest
  if (static_cast<int>(blockIdx.x) < gen_blocks) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kResThreads + threadIdx.x;
    if (t >= P.n_trees) return;
    const TreeRec r = P.trees[t];   // build-time table, read before the wait
    wait_prerequisites();
    general_tree(f, r);
    return;
  }
  const int per = P.trees_per_thread;
  const int64_t base = static_cast<int64_t>(static_cast<int>(blockIdx.x) - gen_blocks) * (kResThreads * per) + threadIdx.x;
  int4 rc[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {   // build-time table, read before the wait
    const int64_t t = base + u * kResThreads;
    rc[u] = u < per && t < P.n_recs ? __ldg(P.recs + t) : make_int4(-1, -1, -1, -1);
  }
  wait_prerequisites();
  float a[U][3], b[U][3], c[U][3], d[U][3];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (rc[u].x >= 0) {
      load3(f, rc[u].x, a[u]);
      load3(f, rc[u].y, b[u]);
      if (rc[u].z >= 0) {
        load3(f, rc[u].z, c[u]);
        load3(f, rc[u].w, d[u]);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (rc[u].x >= 0) {
      if (rc[u].z >= 0) {   // quad: the later pulse first, then the first copy into the atom
        add3(a[u], c[u]);
        add3(b[u], d[u]);
        add3(a[u], b[u]);
        store3(f, rc[u].y, b[u]);
      } else {              // pair: root += copy
        add3(a[u], b[u]);
      }
      store3(f, rc[u].x, a[u]);
    }
  }
}

}  // namespace

const void* resolved_kernel(int kind) {
  return kind == 0 ? reinterpret_cast<const void*>(&k_resolved_coords)
                   : reinterpret_cast<const void*>(&k_resolved_forces);
}

}  // namespace hx
