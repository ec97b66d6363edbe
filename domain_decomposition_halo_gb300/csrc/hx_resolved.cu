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
// sums exactly. One thread per tree: load the record, load the node values,
// add, store the nodes that received adds.
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

// One thread per halo slot: slot = origin (+ shifts).
__global__ void __launch_bounds__(256) k_resolved_coords(float* __restrict__ x, ResolvedParams P) {
  allow_dependents();
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= P.n_halo) return;
  const int2 so = __ldg(P.halo + k);   // (slot, origin): build-time tables, read before the wait
  const unsigned mask = __ldg(P.shift_mask + k);
  wait_prerequisites();
  float v0 = x[3 * static_cast<int64_t>(so.y) + 0];
  float v1 = x[3 * static_cast<int64_t>(so.y) + 1];
  float v2 = x[3 * static_cast<int64_t>(so.y) + 2];
  if (mask & 1u) v0 = __fadd_rn(v0, P.box[0]);   // no add otherwise: unshifted values keep every bit
  if (mask & 2u) v1 = __fadd_rn(v1, P.box[1]);
  if (mask & 4u) v2 = __fadd_rn(v2, P.box[2]);
  float* d = x + 3 * static_cast<int64_t>(so.x);
  d[0] = v0;
  d[1] = v1;
  d[2] = v2;
}

// One thread per tree: replay its adds in descending pulse order.
__global__ void __launch_bounds__(256) k_resolved_forces(float* __restrict__ f, ResolvedParams P) {
  allow_dependents();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= P.n_trees) return;
  const TreeRec r = P.trees[t];   // build-time table, read before the wait
  wait_prerequisites();
  float v[kTreeNodes][3];
#pragma unroll
  for (int j = 0; j < kTreeNodes; ++j) {
    if (j < r.n_nodes) {
      const float* p = f + 3 * static_cast<int64_t>(r.node[j]);
      v[j][0] = p[0];
      v[j][1] = p[1];
      v[j][2] = p[2];
    }
  }
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
          v[a][0] = __fadd_rn(v[a][0], v[b][0]);
          v[a][1] = __fadd_rn(v[a][1], v[b][1]);
          v[a][2] = __fadd_rn(v[a][2], v[b][2]);
        }
      }
      target |= 1u << tg;
    }
  }
#pragma unroll
  for (int j = 0; j < kTreeNodes; ++j) {
    if (j < r.n_nodes && (target >> j & 1u)) {
      float* p = f + 3 * static_cast<int64_t>(r.node[j]);
      p[0] = v[j][0];
      p[1] = v[j][1];
      p[2] = v[j][2];
    }
  }
}

}  // namespace

const void* resolved_kernel(int kind) {
  return kind == 0 ? reinterpret_cast<const void*>(&k_resolved_coords)
                   : reinterpret_cast<const void*>(&k_resolved_forces);
}

}  // namespace hx
