// GPU halo-map builder of libhx (sm_103a).
//
// The pages take the index maps as given (packSendBufKernel's `map`, the
// fused kernel's `indexMap`); these kernels make them:
//   1. home cells and a stable partition of the input into per-domain home
//      ranges (input order kept inside a domain);
//   2. per pulse in the global Z -> Y -> X order, the sender-frame cutoff
//      test on every candidate and a stable compaction of the selected local
//      indices into the pulse's maps (ascending local index, so the entries
//      that read forwarded halo atoms form the tail, as the dependency split
//      of "Enabling parallelism across pulses through kernel fusion" needs),
//      together with the shifted coordinates the receiver gets, which later
//      pulses read as their forwarded candidates.
// All selection decisions are one fp32 subtraction and a strict compare; the
// home cell is the fp64 floor of x * n / L, found by fp32 compares against
// face tables the host derives from that expression, so both are
// bit-reproducible.
#include <cstdint>

#include "hx_internal.h"

namespace hx {
namespace {

constexpr int kScanBlock = 2048;   // elements per scan block (256 threads x 8)
constexpr unsigned kFull = 0xffffffffu;

// Home cells by comparison against per-dimension face tables: faces[off[d]]
// is the smallest fp32 value whose fp64 widening reaches L_d (positions at or
// above it are out of range), faces[off[d] + c] (c = 1 .. n_d-1) the smallest
// fp32 x with min(n_d-1, floor((double)x * n_d / L_d)) >= c. That cell
// function is monotone in x, so counting the faces at or below x gives
// exactly the cell the fp64 expression gives, with fp32 compares only.
struct FaceTables {
  int dims[3];
  int off[3];
  int total;
};

__global__ void __launch_bounds__(256) k_cells(const float* __restrict__ pos, int64_t n, FaceTables g,
                                               const float* __restrict__ faces, int ndom,
                                               int32_t* __restrict__ dom_id, int32_t* __restrict__ hist,
                                               int ntiles, int* err) {
  extern __shared__ int s_mem[];
  int* s_hist = s_mem;
  float* s_face = reinterpret_cast<float*>(s_mem + ndom);
  for (int d = threadIdx.x; d < ndom; d += blockDim.x) s_hist[d] = 0;
  for (int k = threadIdx.x; k < g.total; k += blockDim.x) s_face[k] = faces[k];
  __syncthreads();
  const int64_t tile_start = static_cast<int64_t>(blockIdx.x) * kPartTile;
  for (int k = 0; k < kPartTile / 256; ++k) {
    const int64_t i = tile_start + k * 256 + threadIdx.x;
    if (i >= n) break;
    int c[3];
    bool ok = true;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
      const float x = pos[3 * i + d];
      const float* f = s_face + g.off[d];
      ok = ok && (x >= 0.0f && x < f[0]);   // NaN fails both
      int lo = 0, hi = g.dims[d] - 1;       // cell = number of faces f[1..n-1] at or below x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (f[mid] <= x) lo = mid;
        else hi = mid - 1;
      }
      c[d] = lo;
    }
    if (!ok) atomicOr(err, 1);
    const int r = c[0] + g.dims[0] * (c[1] + g.dims[1] * c[2]);
    dom_id[i] = r;
    atomicAdd(&s_hist[r], 1);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < ndom; d += blockDim.x)
    hist[static_cast<int64_t>(d) * ntiles + blockIdx.x] = s_hist[d];
}

// Stable scatter of one partition tile. Warp w owns the contiguous run
// [tile_start + 256 w, +256) and walks it 32 atoms at a time in input order;
// equal domains inside a step are ranked by lane with __match_any_sync.
__global__ void __launch_bounds__(256) k_scatter_home(const float* __restrict__ pos, int64_t n, int ndom,
                                                      const int32_t* __restrict__ dom_id,
                                                      const int32_t* __restrict__ hist_scanned, int ntiles,
                                                      int32_t* __restrict__ home_ids,
                                                      float* __restrict__ home_xyz,
                                                      int32_t* __restrict__ home_dom) {
  extern __shared__ int s_run[];   // [8][ndom]: per-warp counts, then running ranks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < 8 * ndom; e += blockDim.x) s_run[e] = 0;
  __syncthreads();
  const int64_t run_start = static_cast<int64_t>(blockIdx.x) * kPartTile + warp * 256;
  int* mine = s_run + warp * ndom;
  for (int step = 0; step < 8; ++step) {
    const int64_t i = run_start + step * 32 + lane;
    const bool valid = i < n;
    const int d = valid ? dom_id[i] : -1;
    const unsigned m = __match_any_sync(kFull, d);
    if (valid && lane == __ffs(m) - 1) mine[d] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  for (int d = threadIdx.x; d < ndom; d += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 8; ++w) {
      const int t = s_run[w * ndom + d];
      s_run[w * ndom + d] = run;
      run += t;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int step = 0; step < 8; ++step) {
    const int64_t i = run_start + step * 32 + lane;
    const bool valid = i < n;
    const int d = valid ? dom_id[i] : -1;
    const unsigned m = __match_any_sync(kFull, d);
    int rank = 0;
    if (valid) rank = mine[d] + __popc(m & lt);
    __syncwarp();
    if (valid && lane == __ffs(m) - 1) mine[d] += __popc(m);
    __syncwarp();
    if (valid) {
      const int64_t at = static_cast<int64_t>(hist_scanned[static_cast<int64_t>(d) * ntiles + blockIdx.x]) + rank;
      home_ids[at] = static_cast<int32_t>(i);
      home_dom[at] = d;
      home_xyz[3 * at + 0] = pos[3 * i + 0];
      home_xyz[3 * at + 1] = pos[3 * i + 1];
      home_xyz[3 * at + 2] = pos[3 * i + 2];
    }
  }
}

// Exclusive scan, level 1: each block scans kScanBlock elements and writes
// its total.
__global__ void __launch_bounds__(256) k_scan_block(const int32_t* __restrict__ in, int32_t* __restrict__ out,
                                                    int64_t n, int32_t* __restrict__ block_sums) {
  __shared__ int s_warp[8];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanBlock + threadIdx.x * 8;
  int v[8];
  int sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[k] = (base + k < n) ? in[base + k] : 0;
    sum += v[k];
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int warp_off = 0;
  for (int w = 0; w < warp; ++w) warp_off += s_warp[w];
  int run = warp_off + incl - sum;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (base + k < n) out[base + k] = run;
    run += v[k];
  }
  if (threadIdx.x == 255) block_sums[blockIdx.x] = warp_off + incl;
}

__global__ void k_scan_add(int32_t* __restrict__ out, int64_t n, const int32_t* __restrict__ block_off) {
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanBlock;
  const int add = block_off[blockIdx.x];
  for (int k = threadIdx.x; k < kScanBlock; k += blockDim.x)
    if (base + k < n) out[base + k] += add;
}

__device__ __forceinline__ float candidate(const float* const* bufs, const BuildTile& t, int e, int dim) {
  return bufs[t.buf][3 * (t.elem_begin + e) + dim];
}

__global__ void __launch_bounds__(256) k_select_count(const BuildTile* __restrict__ tiles,
                                                      const float* const* __restrict__ bufs, int dim,
                                                      float rc, int32_t* __restrict__ tile_count) {
  const BuildTile t = tiles[blockIdx.x];
  int total = 0;
  for (int k = 0; k < kSelTile / 256; ++k) {
    const int e = k * 256 + threadIdx.x;
    bool sel = false;
    if (e < t.n) sel = __fsub_rn(candidate(bufs, t, e, dim), t.lo) < rc;
    total += __syncthreads_count(sel);
  }
  if (threadIdx.x == 0) tile_count[blockIdx.x] = total;
}

// Stable compaction: candidates are visited in local order (round k covers
// [256 k, 256 k + 256), warp by warp, lane by lane), so the rank of a selected
// candidate is the number of selected candidates before it.
__global__ void __launch_bounds__(256) k_select_write(const BuildTile* __restrict__ tiles,
                                                      const float* const* __restrict__ bufs, int dim,
                                                      float rc, const int32_t* __restrict__ tile_off,
                                                      int32_t* __restrict__ map_out,
                                                      float* __restrict__ recv_out) {
  __shared__ int s_cnt[8];
  const BuildTile t = tiles[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  int running = tile_off[blockIdx.x];
  for (int k = 0; k < kSelTile / 256; ++k) {
    if (k * 256 >= t.n) break;   // uniform across the block
    const int e = k * 256 + threadIdx.x;
    bool sel = false;
    float v[3] = {0.f, 0.f, 0.f};
    if (e < t.n) {
      const float* s = bufs[t.buf] + 3 * (t.elem_begin + e);
      v[0] = s[0];
      v[1] = s[1];
      v[2] = s[2];
      sel = __fsub_rn(v[dim], t.lo) < rc;
    }
    const unsigned b = __ballot_sync(kFull, sel);
    if (lane == 0) s_cnt[warp] = __popc(b);
    __syncthreads();
    int before = running;
    int round_total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      if (w < warp) before += s_cnt[w];
      round_total += s_cnt[w];
    }
    if (sel) {
      const int at = before + __popc(b & lt);
      map_out[at] = t.local_begin + e;
      if (t.do_shift) v[dim] = __fadd_rn(v[dim], t.shift);
      recv_out[3 * static_cast<int64_t>(at) + 0] = v[0];
      recv_out[3 * static_cast<int64_t>(at) + 1] = v[1];
      recv_out[3 * static_cast<int64_t>(at) + 2] = v[2];
    }
    running += round_total;
    __syncthreads();
  }
}

__global__ void k_place_home(const float* __restrict__ home_xyz, const int32_t* __restrict__ home_dom,
                             const int64_t* __restrict__ home_start, const int64_t* __restrict__ dom_offset,
                             int64_t n, float* __restrict__ coords) {
  for (int64_t k = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = home_dom[k];
    const int64_t slot = dom_offset[r] + (k - home_start[r]);
    coords[3 * slot + 0] = home_xyz[3 * k + 0];
    coords[3 * slot + 1] = home_xyz[3 * k + 1];
    coords[3 * slot + 2] = home_xyz[3 * k + 2];
  }
}

}  // namespace

cudaError_t launch_cells(const float* pos, int64_t n, const int* dims, const float* faces, int ndom,
                         int32_t* dom_id, int32_t* hist, int ntiles, int* err, cudaStream_t s) {
  if (ntiles <= 0) return cudaSuccess;
  FaceTables g;
  int total = 0;
  for (int d = 0; d < 3; ++d) {
    g.dims[d] = dims[d];
    g.off[d] = total;
    total += dims[d];
  }
  g.total = total;
  const size_t smem = sizeof(int) * static_cast<size_t>(ndom) + sizeof(float) * static_cast<size_t>(total);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_cells, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_cells<<<ntiles, 256, smem, s>>>(pos, n, g, faces, ndom, dom_id, hist, ntiles, err);
  return cudaGetLastError();
}

cudaError_t launch_scatter_home(const float* pos, int64_t n, int ndom, const int32_t* dom_id,
                                const int32_t* hist_scanned, int ntiles, int32_t* home_ids, float* home_xyz,
                                int32_t* home_dom, cudaStream_t s) {
  if (ntiles <= 0) return cudaSuccess;
  const size_t smem = sizeof(int) * 8 * static_cast<size_t>(ndom);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_scatter_home, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_scatter_home<<<ntiles, 256, smem, s>>>(pos, n, ndom, dom_id, hist_scanned, ntiles, home_ids, home_xyz,
                                            home_dom);
  return cudaGetLastError();
}

cudaError_t scan_exclusive(const int32_t* in, int32_t* out, int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t nb = (n + kScanBlock - 1) / kScanBlock;
  int32_t* sums = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&sums), sizeof(int32_t) * 2 * nb, s);
  if (e != cudaSuccess) return e;
  int32_t* sums_scanned = sums + nb;
  k_scan_block<<<static_cast<unsigned>(nb), 256, 0, s>>>(in, out, n, sums);
  e = cudaGetLastError();
  if (e == cudaSuccess && nb > 1) {
    e = scan_exclusive(sums, sums_scanned, nb, s);
    if (e == cudaSuccess) {
      k_scan_add<<<static_cast<unsigned>(nb), 256, 0, s>>>(out, n, sums_scanned);
      e = cudaGetLastError();
    }
  }
  cudaError_t f = cudaFreeAsync(sums, s);
  return e != cudaSuccess ? e : f;
}

cudaError_t launch_select_count(const BuildTile* tiles, int ntiles, const float* const* bufs, int dim,
                                float rc, int32_t* tile_count, cudaStream_t s) {
  if (ntiles <= 0) return cudaSuccess;
  k_select_count<<<ntiles, 256, 0, s>>>(tiles, bufs, dim, rc, tile_count);
  return cudaGetLastError();
}

cudaError_t launch_select_write(const BuildTile* tiles, int ntiles, const float* const* bufs, int dim,
                                float rc, const int32_t* tile_off, int32_t* map_out, float* recv_out,
                                cudaStream_t s) {
  if (ntiles <= 0) return cudaSuccess;
  k_select_write<<<ntiles, 256, 0, s>>>(tiles, bufs, dim, rc, tile_off, map_out, recv_out);
  return cudaGetLastError();
}

cudaError_t launch_place_home(const float* home_xyz, const int32_t* home_dom, const int64_t* home_start,
                              const int64_t* dom_offset, int64_t n, float* coords, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  k_place_home<<<static_cast<unsigned>(blocks), 256, 0, s>>>(home_xyz, home_dom, home_start, dom_offset, n,
                                                              coords);
  return cudaGetLastError();
}

}  // namespace hx
