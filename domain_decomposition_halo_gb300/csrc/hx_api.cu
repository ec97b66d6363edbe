// Host runtime and C-ABI of libhx: decomposition plan, map-build driver,
// work tables of the fused kernels, CUDA-graph launch cache, status.
//
// The plan follows "A Practical Guide to GPU-Initiated Communication for
// Molecular Dynamics at Scale": pulses numbered globally Z -> Y -> X
// (section "Dependency-aware packing"); a dependent tail that waits for every
// earlier pulse into its sender; forces in reverse pulse order (section
// "Force halo exchange: Reversing the dependency chain").
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "hx.h"
#include "hx_host.h"
#include "hx_internal.h"

using namespace hx;

namespace {

constexpr int kGraphCache = 16;

struct GraphEntry {
  int kind;        // 0 coords, 1 forces, 2 noop
  void* ptr;
  cudaGraphExec_t exec;
};

template <class T>
cudaError_t dev_alloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), sizeof(T) * count);
}

template <class T>
void dev_free(T*& p) {
  if (p) cudaFree(p);
  p = nullptr;
}

struct Plan {
  double box[3];
  int dims[3];
  double cutoff;
  float boxf[3];
  float rcf;
  int np[3];
  int n_pulses;
  int pulse_dim[HX_MAX_PULSES];
  int pulse_k[HX_MAX_PULSES];
  int ndom;
  std::vector<float> lo[3];
};

int make_plan(const double box[3], const int dims[3], double cutoff, Plan* pl) {
  if (!box || !dims || !(cutoff > 0.0) || !std::isfinite(cutoff)) return HX_ERR_ARG;
  int64_t ndom = 1;
  for (int d = 0; d < 3; ++d) {
    if (dims[d] < 1 || !(box[d] > 0.0) || !std::isfinite(box[d])) return HX_ERR_ARG;
    ndom *= dims[d];
  }
  if (ndom > HX_MAX_DOMAINS) return HX_ERR_ARG;
  pl->cutoff = cutoff;
  pl->rcf = static_cast<float>(cutoff);
  pl->ndom = static_cast<int>(ndom);
  for (int d = 0; d < 3; ++d) {
    pl->box[d] = box[d];
    pl->dims[d] = dims[d];
    pl->boxf[d] = static_cast<float>(box[d]);
    if (dims[d] > 1) {
      const double w = box[d] / dims[d];
      const double np = std::ceil(cutoff / w);
      if (np >= dims[d]) return HX_ERR_PULSES;
      pl->np[d] = static_cast<int>(np);
    } else {
      pl->np[d] = 0;
    }
    pl->lo[d].resize(dims[d]);
    for (int c = 0; c < dims[d]; ++c) pl->lo[d][c] = static_cast<float>(static_cast<double>(c) * box[d] / dims[d]);
  }
  int p = 0;
  for (int d = 2; d >= 0; --d) {
    for (int k = 0; k < pl->np[d]; ++k) {
      if (p >= HX_MAX_PULSES) return HX_ERR_PULSES;
      pl->pulse_dim[p] = d;
      pl->pulse_k[p] = k;
      ++p;
    }
  }
  pl->n_pulses = p;
  return HX_OK;
}

// The home cell min(n-1, floor((double)x * n / L)) of an fp32 position.
int home_cell(float x, int n, double L) {
  const int c = static_cast<int>(std::floor(static_cast<double>(x) * static_cast<double>(n) / L));
  return c > n - 1 ? n - 1 : c;
}

float float_of_bits(uint32_t b) {
  float f;
  std::memcpy(&f, &b, sizeof(f));
  return f;
}

// Smallest non-negative fp32 (by bit pattern, which orders them) for which
// pred holds; pred must be monotone and hold at `hi`.
template <class Pred>
float smallest_float(Pred pred, uint32_t hi) {
  uint32_t lo = 0;
  if (pred(float_of_bits(0))) return 0.0f;
  while (hi - lo > 1) {
    const uint32_t mid = lo + (hi - lo) / 2;
    if (pred(float_of_bits(mid))) hi = mid;
    else lo = mid;
  }
  return float_of_bits(hi);
}

// Per dimension: the first fp32 at or above L, then the first fp32 of cells
// 1 .. n-1 (the face tables of k_cells).
std::vector<float> face_tables(const Plan& pl) {
  std::vector<float> out;
  for (int d = 0; d < 3; ++d) {
    const double L = pl.box[d];
    const int n = pl.dims[d];
    const float limit = smallest_float([&](float x) { return static_cast<double>(x) >= L; }, 0x7f800000u);
    out.push_back(limit);
    uint32_t limit_bits;
    std::memcpy(&limit_bits, &limit, sizeof(limit_bits));
    for (int c = 1; c < n; ++c)
      out.push_back(smallest_float([&](float x) { return home_cell(x, n, L) >= c; }, limit_bits));
  }
  return out;
}

void cell_of(const Plan& pl, int r, int c[3]) {
  c[0] = r % pl.dims[0];
  c[1] = (r / pl.dims[0]) % pl.dims[1];
  c[2] = r / (pl.dims[0] * pl.dims[1]);
}

int domain_of(const Plan& pl, const int c[3]) { return c[0] + pl.dims[0] * (c[1] + pl.dims[1] * c[2]); }

int neighbour(const Plan& pl, int r, int d, int step) {
  int c[3];
  cell_of(pl, r, c);
  c[d] = ((c[d] + step) % pl.dims[d] + pl.dims[d]) % pl.dims[d];
  return domain_of(pl, c);
}

}  // namespace

struct hx_ctx {
  Plan pl;
  int device = 0;
  unsigned flags = 0;
  unsigned long long timeout_ns = 0;
  int sm_count = 0;

  bool built = false;
  int64_t n_atoms = 0;
  int64_t total_slots = 0;
  int64_t total_entries = 0;
  std::vector<int64_t> dom_offset;
  std::vector<int32_t> home, halo;
  // per (pulse p, sender r), index p * ndom + r
  std::vector<int64_t> t_map_off;
  std::vector<int32_t> t_size, t_recv, t_off, t_shift, t_split;

  int32_t* d_maps = nullptr;
  int32_t* d_home_ids = nullptr;
  Chunk* d_chunks[2] = {nullptr, nullptr};   // fused coordinate / force chunk lists
  Wait* d_waits[2] = {nullptr, nullptr};
  Chunk* d_uchunks = nullptr;                // unfused per-pulse chunk list
  unsigned long long* d_flags = nullptr;     // [2][n_items]
  unsigned int* d_blk = nullptr;             // [2][n_items]
  Ctrl* d_ctrl = nullptr;                    // [2]
  int n_chunks[2] = {0, 0};
  int grid[2] = {0, 0};
  size_t n_flags = 1;                        // flags (and election counters) per direction
  int family[2] = {0, 0};                    // kernel family of each direction's fused path (Family)
  TileUnit* d_units[2] = {nullptr, nullptr};
  TileSeg* d_segs[2] = {nullptr, nullptr};
  Wait* d_twaits[2] = {nullptr, nullptr};
  int n_units[2] = {0, 0};
  std::vector<int> u_begin;                  // per pulse, first unfused chunk (P + 1 entries)
  std::vector<GraphEntry> graphs;
  ResSeg* d_res_segs = nullptr;              // resolved mode: halo segments
  uint32_t* d_res_om = nullptr;              // ... origin and shift mask per halo slot
  int4* d_res_recs = nullptr;                // ... force trees: pairs and quads, general ones apart
  TreeRec* d_res_trees = nullptr;
  int64_t n_res_halo = 0, n_res_segs = 0, n_res_pairs = 0, n_res_quads = 0, n_res_trees = 0;
  CopyChunk* d_home_chunks = nullptr;        // host-buffer calls: every domain's home range
  CopyChunk* d_halo_chunks = nullptr;        // ... and halo range, in pieces of one block each
  int n_home_chunks = 0, n_halo_chunks = 0;
};

namespace {

void drop_graphs(hx_ctx* h) {
  for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
  h->graphs.clear();
}

void free_tables(hx_ctx* h) {
  drop_graphs(h);
  dev_free(h->d_maps);
  dev_free(h->d_home_ids);
  for (int k = 0; k < 2; ++k) {
    dev_free(h->d_chunks[k]);
    dev_free(h->d_waits[k]);
  }
  dev_free(h->d_uchunks);
  dev_free(h->d_res_segs);
  dev_free(h->d_res_om);
  dev_free(h->d_res_recs);
  dev_free(h->d_res_trees);
  h->n_res_halo = h->n_res_segs = h->n_res_pairs = h->n_res_quads = h->n_res_trees = 0;
  dev_free(h->d_home_chunks);
  dev_free(h->d_halo_chunks);
  h->n_home_chunks = h->n_halo_chunks = 0;
  for (int k = 0; k < 2; ++k) {
    dev_free(h->d_units[k]);
    dev_free(h->d_segs[k]);
    dev_free(h->d_twaits[k]);
    h->n_units[k] = 0;
  }
  dev_free(h->d_flags);
  dev_free(h->d_blk);
  dev_free(h->d_ctrl);
  h->built = false;
}

#define HX_CUDA(call)                       \
  do {                                      \
    cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return HX_ERR_CUDA; \
  } while (0)

int to_err(cudaError_t e) {
  if (e == cudaSuccess) return HX_OK;
  if (e == cudaErrorMemoryAllocation) return HX_ERR_NOMEM;
  return HX_ERR_CUDA;
}

DirParams dir_params(hx_ctx* h, int dir) {
  DirParams P;
  std::memset(&P, 0, sizeof(P));
  const size_t n_items = h->n_flags;
  P.chunks = h->d_chunks[dir];
  P.waits = h->d_waits[dir];
  P.maps = h->d_maps;
  P.flags = h->d_flags + dir * n_items;
  P.arrivals = h->d_blk + dir * n_items;
  P.ctrl = h->d_ctrl + dir;
  P.n_chunks = static_cast<unsigned long long>(h->n_chunks[dir]);
  P.direction = dir;
  P.timeout_ns = h->timeout_ns;
  return P;
}

const void* kernel_for(hx_ctx* h, int kind) {
  const int mode = (h->flags & HX_FLAG_FINE_WAITS) ? kChunkFlag
                   : (h->flags & HX_FLAG_COUNTER_SIGNAL) ? kCounter : kLastArrival;
  if (kind == 0) return coords_kernel(mode, (h->flags & HX_FLAG_BULK_STORE) != 0);
  if (kind == 1) return forces_kernel(mode, !(h->flags & HX_FLAG_UNORDERED_FORCES));
  return noop_kernel();
}

// Launch a fused exchange (kind 0/1) or the no-op (kind 2): directly, or via
// a cached single-node graph keyed by (kind, buffer pointer).
TileParams tile_params(hx_ctx* h, int dir) {
  TileParams P;
  std::memset(&P, 0, sizeof(P));
  P.units = h->d_units[dir];
  P.extra = h->d_segs[dir];
  P.waits = h->d_twaits[dir];
  P.maps = h->d_maps;
  P.flags = h->d_flags + static_cast<size_t>(dir) * h->n_flags;
  P.ctrl = h->d_ctrl + dir;
  P.n_units = static_cast<unsigned long long>(h->n_units[dir]);
  P.direction = dir;
  P.timeout_ns = h->timeout_ns;
  return P;
}

// Work items of the fused list of direction `dir`: units or chunks.
int work_items(const hx_ctx* h, int dir) {
  if (h->family[dir] == kFamCluster) return h->u_begin.empty() ? 0 : h->u_begin.back();
  if (h->family[dir] == kFamResolved)
    return static_cast<int>(dir == 0 ? h->n_res_halo : h->n_res_pairs + h->n_res_quads + h->n_res_trees);
  return h->family[dir] == kFamChunks ? h->n_chunks[dir] : h->n_units[dir];
}

// Launch shape of a direction's fused kernel.
const void* fused_kernel(hx_ctx* h, int dir) {
  if (h->family[dir] == kFamTiles) return tiles_kernel(dir);
  if (h->family[dir] == kFamSweep) return sweep_kernel(dir);
  if (h->family[dir] == kFamCluster) return cluster_kernel(dir);
  if (h->family[dir] == kFamResolved) return resolved_kernel(dir);
  return kernel_for(h, dir);
}
unsigned fused_threads(const hx_ctx* h, int dir) {
  if (h->family[dir] == kFamCluster) return kClusterThreads;
  if (h->family[dir] == kFamResolved) return kResThreads;
  return h->family[dir] == kFamTiles ? kTileThreads : kThreads;
}

// Blocks of kResThreads threads that hold n items at `per` items a thread.
int64_t resolved_blocks(int64_t n, int per) { return (n + int64_t{kResThreads} * per - 1) / (int64_t{kResThreads} * per); }

// Trees a thread of one class takes: several (more loads in flight per
// thread) only when even then the class fills the GPU several times over
// (four waves of four blocks per SM); small decompositions keep one a thread.
int resolved_per_thread(const hx_ctx* h, int64_t n, int most) {
  const int64_t wave = int64_t{4} * std::max(h->sm_count, 1) * kResThreads;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(most, n / (4 * wave))));
}

ResolvedParams resolved_params(hx_ctx* h) {
  ResolvedParams P;
  std::memset(&P, 0, sizeof(P));
  P.segs = h->d_res_segs;
  P.origin_mask = h->d_res_om;
  P.recs = h->d_res_recs;
  P.trees = h->d_res_trees;
  P.n_segs = h->n_res_segs;
  P.n_recs = h->n_res_pairs + h->n_res_quads;
  P.n_trees = h->n_res_trees;
  P.trees_per_thread = resolved_per_thread(h, P.n_recs, kResTreesPerThread);
  P.rec_blocks = static_cast<int32_t>(resolved_blocks(P.n_recs, P.trees_per_thread));
  for (int d = 0; d < 3; ++d) P.box[d] = h->pl.boxf[d];
  return P;
}

ClusterParams cluster_params(hx_ctx* h) {
  ClusterParams P;
  std::memset(&P, 0, sizeof(P));
  P.chunks = h->d_uchunks;
  P.maps = h->d_maps;
  P.n_pulses = h->pl.n_pulses;
  for (int p = 0; p <= h->pl.n_pulses; ++p) P.begin[p] = h->u_begin[p];
  return P;
}
size_t fused_smem(const hx_ctx* h, int dir) {
  if (h->family[dir] == kFamTiles) return tiles_smem_bytes(dir);
  if (h->family[dir] == kFamSweep) return sweep_smem_bytes(dir);
  return 0;
}

int launch(hx_ctx* h, int kind, float* buf, cudaStream_t s) {
  DirParams P;
  TileParams TP;
  ClusterParams CP;
  ResolvedParams RP;
  void* args2[2];
  void** args = nullptr;
  dim3 grid(1), block(kind == 2 ? 1 : kThreads);
  size_t smem = 0;
  const void* fn = kernel_for(h, kind);
  if (kind != 2 && h->family[kind] == kFamResolved) {
    RP = resolved_params(h);
    args2[0] = &buf;
    args2[1] = &RP;
    args = args2;
    grid = dim3(static_cast<unsigned>(h->grid[kind]));
    block = dim3(kResThreads);
    fn = resolved_kernel(kind);
  } else if (kind != 2 && h->family[kind] == kFamCluster) {
    CP = cluster_params(h);
    args2[0] = &buf;
    args2[1] = &CP;
    args = args2;
    grid = dim3(kClusterCtas);
    block = dim3(kClusterThreads);
    fn = cluster_kernel(kind);
  } else if (kind != 2 && h->family[kind] != kFamChunks) {
    TP = tile_params(h, kind);
    args2[0] = &buf;
    args2[1] = &TP;
    args = args2;
    grid = dim3(static_cast<unsigned>(h->grid[kind]));
    block = dim3(fused_threads(h, kind));
    smem = fused_smem(h, kind);
    fn = fused_kernel(h, kind);
  } else if (kind != 2) {
    P = dir_params(h, kind);
    args2[0] = &buf;
    args2[1] = &P;
    args = args2;
    grid = dim3(static_cast<unsigned>(h->grid[kind]));
  }
  if (kind != 2 && h->family[kind] == kFamResolved && (h->flags & HX_FLAG_PDL)) {
    // direct launch that may start while the stream's previous kernel finishes;
    // the resolved kernels wait for it (griddepcontrol.wait) before touching data
    cudaLaunchAttribute attr[1];
    std::memset(attr, 0, sizeof(attr));
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return to_err(cudaLaunchKernelExC(&cfg, fn, args));
  }
  if (h->flags & HX_FLAG_NO_GRAPH) return to_err(cudaLaunchKernel(fn, grid, block, args, smem, s));
  for (auto& g : h->graphs)
    if (g.kind == kind && g.ptr == buf) return to_err(cudaGraphLaunch(g.exec, s));
  cudaGraph_t graph;
  HX_CUDA(cudaGraphCreate(&graph, 0));
  cudaKernelNodeParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.func = const_cast<void*>(fn);
  kp.gridDim = grid;
  kp.blockDim = block;
  kp.sharedMemBytes = static_cast<unsigned>(smem);
  kp.kernelParams = args;
  cudaGraphNode_t node;
  cudaError_t e = cudaGraphAddKernelNode(&node, graph, nullptr, 0, &kp);
  cudaGraphExec_t exec = nullptr;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return to_err(e);
  if (static_cast<int>(h->graphs.size()) >= kGraphCache) {
    cudaGraphExecDestroy(h->graphs.front().exec);
    h->graphs.erase(h->graphs.begin());
  }
  h->graphs.push_back({kind, buf, exec});
  return to_err(cudaGraphLaunch(exec, s));
}

int reset_signals(hx_ctx* h, cudaStream_t s) {
  const size_t n_items = h->n_flags;
  HX_CUDA(cudaMemsetAsync(h->d_flags, 0, sizeof(unsigned long long) * 2 * n_items, s));
  HX_CUDA(cudaMemsetAsync(h->d_blk, 0, sizeof(unsigned int) * 2 * n_items, s));
  Ctrl c[2];
  std::memset(c, 0, sizeof(c));
  c[0].drop_item = c[1].drop_item = -1;
  HX_CUDA(cudaMemcpyAsync(h->d_ctrl, c, sizeof(c), cudaMemcpyHostToDevice, s));
  HX_CUDA(cudaStreamSynchronize(s));
  return HX_OK;
}

// ---------------------------------------------------------------- work tables
//
// Every (sender, pulse) item is cut into warp chunks of up to kChunk entries
// (a coordinate item into its independent prefix and its forwarded tail).
// Each chunk gets the list of what it must wait for:
//   coarse (the pages' rule): a forwarded coordinate chunk waits for every
//     earlier pulse into its sender; a force chunk of pulse p waits for every
//     later pulse of its receiver (the slots it reads) and of its sender (the
//     targets it adds into) - per-item signals;
//   fine: the exact producer chunks - the chunks that stored the slots a
//     forwarded coordinate chunk reads, the later-pulse chunks that add into
//     the slots a force chunk reads or into the targets it adds into - each
//     with its own signal.
// Chunks are then listed in a topological order of those waits (Kahn's
// algorithm, so a warp only ever waits for chunks handed out before its own)
// that follows a priority: domains in a folded order where the neighbours a
// pulse depends on sit close together, a domain's pulses together, and a
// consumer one resident-warp window behind its producers. A domain's slots
// are then fetched into L2 about once per launch, and a waiting chunk finds
// its producers mostly done.

// Runs body(i) for i in [0, n) on the host's cores (iterations must be
// independent).
template <class Body>
void parallel_for(size_t n, Body body, size_t grain = 256) {
  const size_t hw = std::max<size_t>(1, std::min<size_t>(16, std::thread::hardware_concurrency()));
  const size_t workers = std::min(hw, std::max<size_t>(1, n / grain));
  if (workers <= 1) {
    for (size_t i = 0; i < n; ++i) body(i);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(workers);
  for (size_t w = 0; w < workers; ++w)
    pool.emplace_back([&, w] {
      for (size_t i = w; i < n; i += workers) body(i);
    });
  for (auto& t : pool) t.join();
}

struct ItemInfo {
  int r, p, q;           // sender, pulse, receiver
  int64_t src, dst, map; // slot of sender base, slot of receive-range start, first map entry
  int size, split, dim, shift_flag;
};

struct Rec {             // one chunk before ordering
  int item;
  int begin, end;        // entry range within the item's map
  int halo_src;
  int stage;             // position of the chunk's pulse in the launch's dependency order
  long long key;         // priority (smaller first)
  std::vector<int> deps;   // chunk records that must be listed earlier
  std::vector<int> wait;   // coarse: items to wait for; fine: chunk records to wait for
};

// Position of cell c in the folded ring order 0, n-1, 1, n-2, ...: cells that
// are neighbours on the periodic ring are at most two positions apart.
int fold(int c, int n) { return (2 * c < n) ? 2 * c : 2 * (n - 1 - c) + 1; }

int64_t domain_rank(const Plan& pl, int r) {
  int c[3];
  cell_of(pl, r, c);
  // the first-communicating dimension (Z) varies fastest, X slowest
  return fold(c[2], pl.dims[2]) + static_cast<int64_t>(pl.dims[2]) *
                                      (fold(c[1], pl.dims[1]) + static_cast<int64_t>(pl.dims[1]) * fold(c[0], pl.dims[0]));
}

// Kahn's algorithm over chunk records by ascending key.
// Kahn's algorithm: a topological order of n records whose dependency lists
// deps(i) name earlier-done records, taking among the ready ones the smallest
// key(i) (ties by index). Users are kept in one flat list.
template <class Deps, class Key>
std::vector<int> kahn_order(int n, Deps deps, Key key) {
  std::vector<int> first(n + 1, 0), unmet(n, 0);
  for (int i = 0; i < n; ++i) {
    const auto& d = deps(i);
    unmet[i] = static_cast<int>(d.size());
    for (int x : d) ++first[x + 1];
  }
  for (int i = 0; i < n; ++i) first[i + 1] += first[i];
  std::vector<int> users(first[n]), fill(first.begin(), first.end() - 1);
  for (int i = 0; i < n; ++i)
    for (int x : deps(i)) users[fill[x]++] = i;
  auto cmp = [&](int a, int b) {
    const long long ka = key(a), kb = key(b);
    return ka != kb ? ka > kb : a > b;
  };
  std::vector<int> heap;
  for (int i = 0; i < n; ++i)
    if (unmet[i] == 0) heap.push_back(i);
  std::make_heap(heap.begin(), heap.end(), cmp);
  std::vector<int> order;
  order.reserve(n);
  while (!heap.empty()) {
    std::pop_heap(heap.begin(), heap.end(), cmp);
    const int i = heap.back();
    heap.pop_back();
    order.push_back(i);
    for (int k = first[i]; k < first[i + 1]; ++k)
      if (--unmet[users[k]] == 0) {
        heap.push_back(users[k]);
        std::push_heap(heap.begin(), heap.end(), cmp);
      }
  }
  return order;   // shorter than n only if the waits had a cycle (they cannot)
}

std::vector<int> order_chunks(const std::vector<Rec>& recs) {
  return kahn_order(
      static_cast<int>(recs.size()), [&](int i) -> const std::vector<int>& { return recs[i].deps; },
      [&](int i) { return recs[i].key; });
}

// ---------------------------------------------------------------- tile tables
//
// Each domain's array is cut into ranges (home, then the slots received in
// each pulse) and each range into tiles of up to kTile slots. A tile gets
// one segment per (sender, pulse) map that has entries inside it: for
// coordinates the maps it is a source of, for forces the maps it is a target
// of (segments last pulse first). Dependencies:
//   coordinates: a tile of received slots waits for the tiles of the sending
//     domain that stored those slots;
//   forces: a tile waits for the tiles of its receivers that hold the slots
//     it reads, when those tiles are themselves targets of later pulses.
// Tiles are listed by Kahn's algorithm with the same priority as the chunk
// lists (folded domain order, dependency depth, a lag of one resident window
// per depth).

struct TRec {
  int r;              // domain
  int range;          // -1 home, else the pulse whose received slots the tile holds
  int a, n;           // local index of the first slot, slot count
  std::vector<TileSeg> segs;
  std::vector<int> seg_pulse;
  std::vector<int> deps;   // TRec indices
  int stage = 0;
  long long key = 0;
};

int build_tile_tables(hx_ctx* h, const std::vector<ItemInfo>& items, const std::vector<int32_t>& maps,
                      const std::vector<int64_t>& rank, int max_slots, int max_entries, long long lag,
                      int tile_bytes, int map_bytes, int src_bytes, int dir) {
  const Plan& pl = h->pl;
  const int P = pl.n_pulses, nd = pl.ndom;
  auto upper = [&](int r, int q) { return neighbour(pl, r, pl.pulse_dim[q], +1); };
  {
    // tiles of each domain, cut on all host cores, then listed domain after domain;
    // by_range: per (domain, range) the tiles' indices in slot order
    std::vector<std::vector<TRec>> per(nd);
    std::vector<std::vector<std::vector<int>>> by_range(nd, std::vector<std::vector<int>>(P + 1));
    parallel_for(nd, [&](size_t ri) {
      const int r = static_cast<int>(ri);
      for (int rg = -1; rg < P; ++rg) {
        int lo, len;
        if (rg < 0) {
          lo = 0;
          len = h->home[r];
        } else {
          const int tu = rg * nd + upper(r, rg);
          lo = h->t_off[tu];
          len = h->t_size[tu];
        }
        // entries of every map of r that fall in slots [a, b)
        auto entries_in = [&](int a, int b) {
          int e = 0;
          for (int p = 0; p < P; ++p) {
            const ItemInfo& it = items[p * nd + r];
            if (it.size == 0) continue;
            const int32_t* m = maps.data() + it.map;
            e += static_cast<int>(std::lower_bound(m, m + it.size, b) - std::lower_bound(m, m + it.size, a));
          }
          return e;
        };
        for (int a = lo, b = lo; a < lo + len; a = b) {
          // at most kTile slots and kTileEntries entries (a slot has at most one entry per pulse)
          b = std::min(lo + len, a + max_slots);
          if (entries_in(a, b) > max_entries) {
            int good = a + 1, bad = b;
            while (bad - good > 1) {
              const int mid = good + (bad - good) / 2;
              if (entries_in(a, mid) <= max_entries) good = mid;
              else bad = mid;
            }
            b = good;
          }
          TRec t;
          t.r = r;
          t.range = rg;
          t.a = a;
          t.n = b - a;
          for (int k = 0; k < P; ++k) {
            const int p = dir == 0 ? k : P - 1 - k;
            const ItemInfo& it = items[p * nd + r];
            if (it.size == 0) continue;
            const int32_t* m = maps.data() + it.map;
            const int i1 = static_cast<int>(std::lower_bound(m, m + it.size, t.a) - m);
            const int i2 = static_cast<int>(std::lower_bound(m, m + it.size, t.a + t.n) - m);
            if (i2 <= i1) continue;
            TileSeg sg;
            std::memset(&sg, 0, sizeof(sg));
            sg.map = it.map + i1;
            sg.other = it.dst + i1;
            sg.n = i2 - i1;
            sg.dim = it.dim;
            sg.shift = pl.boxf[it.dim];
            sg.do_shift = (dir == 0) ? it.shift_flag : 0;
            t.segs.push_back(sg);
            t.seg_pulse.push_back(p);
          }
          if (t.segs.empty()) continue;
          by_range[r][rg + 1].push_back(static_cast<int>(per[r].size()));
          per[r].push_back(std::move(t));
        }
      }
    }, 1);
    std::vector<TRec> recs;
    for (int r = 0; r < nd; ++r) {
      const int base = static_cast<int>(recs.size());
      for (auto& lst : by_range[r])
        for (int& i : lst) i += base;
      for (TRec& t : per[r]) recs.push_back(std::move(t));
    }
    per.clear();
    // dependencies, one unit per task
    parallel_for(recs.size(), [&](size_t i) {
      TRec& t = recs[i];
      if (dir == 0) {
        if (t.range < 0) return;
        // slots [a, a+n) of r's range `p0` are entries [a - off, a - off + n) of the map (u, p0)
        const int p0 = t.range, u = upper(t.r, p0);
        const int64_t e0 = t.a - h->t_off[p0 * nd + u], e1 = e0 + t.n;
        for (int rg = 0; rg <= P; ++rg)
          for (int j : by_range[u][rg]) {
            const TRec& s = recs[j];
            for (size_t k = 0; k < s.segs.size(); ++k) {
              if (s.seg_pulse[k] != p0) continue;
              const int64_t b0 = s.segs[k].map - items[p0 * nd + u].map, b1 = b0 + s.segs[k].n;
              if (b0 < e1 && e0 < b1) t.deps.push_back(j);
            }
          }
      } else {
        // the slots read by segment (r, p) are q's slots [other, other + n) in q's range p
        for (size_t k = 0; k < t.segs.size(); ++k) {
          const int p = t.seg_pulse[k];
          const int q = items[p * nd + t.r].q;
          const int64_t s0 = t.segs[k].other - h->dom_offset[q], s1 = s0 + t.segs[k].n;
          for (int j : by_range[q][p + 1]) {
            const TRec& s = recs[j];
            if (s.a < s1 && s0 < s.a + s.n) t.deps.push_back(j);
          }
        }
      }
      std::sort(t.deps.begin(), t.deps.end());
      t.deps.erase(std::unique(t.deps.begin(), t.deps.end()), t.deps.end());
    }, 64);
    // dependency depth, then priority: base order + one resident window per depth
    {
      const int n = static_cast<int>(recs.size());
      auto deps_of = [&](int i) -> const std::vector<int>& { return recs[i].deps; };
      std::vector<int> topo = kahn_order(n, deps_of, [](int) { return 0ll; });   // any topological order
      if (topo.size() != recs.size()) return HX_ERR_STATE;
      for (int i : topo)
        for (int d : recs[i].deps) recs[i].stage = std::max(recs[i].stage, recs[d].stage + 1);
      std::vector<int> base(recs.size());
      for (size_t i = 0; i < recs.size(); ++i) base[i] = static_cast<int>(i);
      std::sort(base.begin(), base.end(), [&](int x, int y) {
        const TRec& a = recs[x];
        const TRec& b = recs[y];
        if (rank[a.r] != rank[b.r]) return rank[a.r] < rank[b.r];
        if (a.stage != b.stage) return a.stage < b.stage;
        if (a.range != b.range) return a.range < b.range;
        return a.a < b.a;
      });
      for (size_t k = 0; k < base.size(); ++k)
        recs[base[k]].key = static_cast<long long>(k) + lag * recs[base[k]].stage;
      std::vector<int> order = kahn_order(n, deps_of, [&](int i) { return recs[i].key; });
      if (order.size() != recs.size()) return HX_ERR_STATE;
      std::vector<int> pos(recs.size());
      for (size_t k = 0; k < order.size(); ++k) pos[order[k]] = static_cast<int>(k);
      std::vector<char> waited(recs.size(), 0);
      for (auto& t : recs)
        for (int d : t.deps) waited[d] = 1;
      std::vector<TileUnit> units;
      std::vector<TileSeg> segs;   // segments past kInlineSegs
      std::vector<Wait> waits;
      for (int i : order) {
        const TRec& t = recs[i];
        TileUnit u;
        std::memset(&u, 0, sizeof(u));
        u.base = h->dom_offset[t.r] + t.a;
        u.n = t.n;
        u.local_a = t.a;
        u.seg_cnt = static_cast<int32_t>(t.segs.size());
        u.extra_off = static_cast<int32_t>(segs.size());
        // stage regions: each run's region starts on a 16-byte boundary and is 16 bytes longer than the run
        int moff = tile_bytes, soff = tile_bytes + map_bytes;
        for (size_t k = 0; k < t.segs.size(); ++k) {
          TileSeg sg = t.segs[k];
          sg.map_off = moff;
          sg.src_off = dir == 1 ? soff : 0;
          moff += ((4 * sg.n + 15) & ~15) + 16;
          soff += ((12 * sg.n + 15) & ~15) + 16;
          if (static_cast<int>(k) < kInlineSegs) u.seg[k] = sg;
          else segs.push_back(sg);
        }
        // the stage regions must fit the kernel's buffer
        if (moff > tile_bytes + map_bytes || (dir == 1 && soff > tile_bytes + map_bytes + src_bytes))
          return HX_ERR_STATE;
        u.wait_off = static_cast<int32_t>(waits.size());
        u.wait_cnt = static_cast<int32_t>(t.deps.size());
        for (int d : t.deps) waits.push_back({pos[d], 1});
        u.flags = (waited[i] ? kSignal : 0) | (dir == 0 && t.range >= 0 ? kHaloSrc : 0);
        u.item = t.seg_pulse[0] * nd + t.r;
        for (const TileSeg& sg : t.segs) u.entries += sg.n;
        units.push_back(u);
      }
      h->n_units[dir] = static_cast<int>(units.size());
      HX_CUDA(dev_alloc(&h->d_units[dir], units.size()));
      HX_CUDA(dev_alloc(&h->d_segs[dir], segs.size()));
      HX_CUDA(dev_alloc(&h->d_twaits[dir], waits.size()));
      if (!units.empty())
        HX_CUDA(cudaMemcpy(h->d_units[dir], units.data(), sizeof(TileUnit) * units.size(), cudaMemcpyHostToDevice));
      if (!segs.empty())
        HX_CUDA(cudaMemcpy(h->d_segs[dir], segs.data(), sizeof(TileSeg) * segs.size(), cudaMemcpyHostToDevice));
      if (!waits.empty())
        HX_CUDA(cudaMemcpy(h->d_twaits[dir], waits.data(), sizeof(Wait) * waits.size(), cudaMemcpyHostToDevice));
    }
  }
  return HX_OK;
}

// Resolved tables: every halo slot's origin and shift mask (pulses in order,
// each received slot inheriting from the slot it was sent from), in halo
// order (domain after domain) with one segment record per block; and one
// tree per home atom that has copies, its adds sorted by descending pulse,
// numbered in home-slot order: pairs and quads as 16-byte records, the
// other trees as general records, each list in root order.
int build_resolved_tables(hx_ctx* h, const std::vector<ItemInfo>& items, const std::vector<int32_t>& maps,
                          cudaStream_t s) {
  const Plan& pl = h->pl;
  const int P = pl.n_pulses, nd = pl.ndom;
  // origins share a word with the shift mask; other slots are int32 in the records
  if (h->total_slots >= (int64_t{1} << kResOriginBits)) return HX_ERR_CAPACITY;
  std::vector<int64_t> hbase(nd + 1, 0), home_base(nd + 1, 0);
  for (int r = 0; r < nd; ++r) {
    hbase[r + 1] = hbase[r] + h->halo[r];
    home_base[r + 1] = home_base[r] + h->home[r];
  }
  const int64_t H = hbase[nd];
  std::vector<int32_t> origin_home(H), origin_slot(H), parent_h(H), root_dom(H);
  std::vector<uint8_t> mask(H), pulse(H);
  for (int p = 0; p < P; ++p)   // senders of one pulse write disjoint slots and read earlier pulses
    parallel_for(nd, [&](size_t ri) {
      const int r = static_cast<int>(ri);
      const ItemInfo& it = items[p * nd + r];
      const int64_t d0 = hbase[it.q] + (it.dst - h->dom_offset[it.q] - h->home[it.q]);
      for (int i = 0; i < it.size; ++i) {
        const int32_t mv = maps[it.map + i];
        const int64_t k = d0 + i;
        if (mv < h->home[r]) {
          origin_home[k] = static_cast<int32_t>(home_base[r] + mv);
          origin_slot[k] = static_cast<int32_t>(it.src + mv);
          root_dom[k] = r;
          mask[k] = 0;
          parent_h[k] = -1;
        } else {
          const int64_t sh = hbase[r] + (mv - h->home[r]);
          origin_home[k] = origin_home[sh];
          origin_slot[k] = origin_slot[sh];
          root_dom[k] = root_dom[sh];
          mask[k] = mask[sh];
          parent_h[k] = static_cast<int32_t>(sh);
        }
        if (it.shift_flag) mask[k] = static_cast<uint8_t>(mask[k] | (1 << it.dim));
        pulse[k] = static_cast<uint8_t>(p);
      }
    }, 1);
  // coordinates: origin and shift mask packed per halo slot, segments per domain
  std::vector<uint32_t> om(H);
  for (int64_t k = 0; k < H; ++k)
    om[k] = static_cast<uint32_t>(origin_slot[k]) | (static_cast<uint32_t>(mask[k]) << kResOriginBits);
  std::vector<ResSeg> segs;
  const int64_t seg_len = int64_t{kResThreads} * resolved_per_thread(h, H, kResSlotsPerThread);
  for (int r = 0; r < nd; ++r)
    for (int64_t k = hbase[r]; k < hbase[r + 1]; k += seg_len) {
      ResSeg sg;
      sg.k = static_cast<int32_t>(k);
      sg.slot = static_cast<int32_t>(h->dom_offset[r] + h->home[r] + (k - hbase[r]));
      sg.n = static_cast<int32_t>(std::min<int64_t>(seg_len, hbase[r + 1] - k));
      sg.pad = 0;
      segs.push_back(sg);
    }
  // trees: one per home atom that has copies, numbered in home-slot order.
  // A tree lies in its root's domain (every copy descends from the root), so
  // the halo slots are grouped by root domain (stably: halo order kept) and
  // each root domain's trees are built by one task, in a local array.
  std::vector<int64_t> by_root_begin(nd + 1, 0);
  for (int64_t k = 0; k < H; ++k) ++by_root_begin[root_dom[k] + 1];
  for (int r = 0; r < nd; ++r) by_root_begin[r + 1] += by_root_begin[r];
  std::vector<int32_t> by_root(H);
  {
    std::vector<int64_t> fill(by_root_begin.begin(), by_root_begin.end() - 1);
    for (int64_t k = 0; k < H; ++k) by_root[fill[root_dom[k]]++] = static_cast<int32_t>(k);
  }
  std::vector<uint8_t> node_idx(H);
  std::vector<std::vector<int4>> recs_of(nd);
  std::vector<std::vector<TreeRec>> general_of(nd);
  std::vector<int64_t> pairs_of(nd, 0), quads_of(nd, 0);
  std::vector<char> overflow(nd, 0);
  auto slot_of_halo = [&](int64_t k) {   // the global slot of halo index k
    const int r = static_cast<int>(std::upper_bound(hbase.begin(), hbase.end(), k) - hbase.begin()) - 1;
    return static_cast<int32_t>(h->dom_offset[r] + h->home[r] + (k - hbase[r]));
  };
  parallel_for(nd, [&](size_t ri) {
    const int r0 = static_cast<int>(ri);
    const int32_t* ks = by_root.data() + by_root_begin[r0];
    const int64_t nk = by_root_begin[r0 + 1] - by_root_begin[r0];
    std::vector<int32_t> tree_of(h->home[r0], -1);   // per home atom of r0
    for (int64_t i = 0; i < nk; ++i) tree_of[origin_home[ks[i]] - home_base[r0]] = 0;   // marks the roots
    int32_t n_trees = 0;
    for (auto& t : tree_of)
      if (t == 0) t = n_trees++;
    std::vector<TreeRec> trees(static_cast<size_t>(n_trees));   // zero-filled
    std::vector<uint8_t> add_pulse(trees.size() * kTreeNodes, 0);
    for (int64_t i = 0; i < nk; ++i) {   // nodes: the root, then its copies in halo order
      const int64_t k = ks[i];
      TreeRec& rec = trees[tree_of[origin_home[k] - home_base[r0]]];
      if (rec.n_nodes == 0) {
        rec.node[0] = origin_slot[k];
        rec.n_nodes = 1;
      }
      if (rec.n_nodes >= kTreeNodes) {   // more copies than a tree record holds
        overflow[r0] = 1;
        return;
      }
      node_idx[k] = static_cast<uint8_t>(rec.n_nodes);
      rec.node[rec.n_nodes++] = slot_of_halo(k);
    }
    for (int64_t i = 0; i < nk; ++i) {   // adds: copy j (node j > 0) into its parent (same tree)
      const int64_t k = ks[i];
      const size_t t = static_cast<size_t>(tree_of[origin_home[k] - home_base[r0]]);
      const int j = node_idx[k];
      const int tg = parent_h[k] < 0 ? 0 : node_idx[parent_h[k]];
      trees[t].ev[j - 1] = static_cast<uint8_t>(tg | (j << 4));
      add_pulse[t * kTreeNodes + j - 1] = pulse[k];
    }
    std::vector<int4>& recs = recs_of[r0];
    std::vector<TreeRec>& general = general_of[r0];
    recs.reserve(trees.size());
    for (size_t t = 0; t < trees.size(); ++t) {
      TreeRec& rec = trees[t];
      uint8_t* pu = add_pulse.data() + t * kTreeNodes;
      const int m = rec.n_nodes - 1;
      for (int a = 1; a < m; ++a)   // stable insertion sort by descending pulse
        for (int b = a; b > 0 && pu[b] > pu[b - 1]; --b) {
          std::swap(pu[b], pu[b - 1]);
          std::swap(rec.ev[b], rec.ev[b - 1]);
        }
      // records in root order. A four-node tree is a quad when its last add
      // (lowest pulse) is some copy u into the root and the two adds before
      // it are one copy into the root and one copy into u: then the fixed
      // order root += c, u += d, root += u is the staged order.
      if (rec.n_nodes == 2) {
        recs.push_back(make_int4(rec.node[0], rec.node[1], -1, -1));
        ++pairs_of[r0];
        continue;
      }
      if (rec.n_nodes == 4) {
        const int tg2 = rec.ev[2] & 15, u = rec.ev[2] >> 4;
        const int tg0 = rec.ev[0] & 15, s0 = rec.ev[0] >> 4, tg1 = rec.ev[1] & 15, s1 = rec.ev[1] >> 4;
        if (tg2 == 0 && u != 0 && ((tg0 == 0 && tg1 == u) || (tg0 == u && tg1 == 0))) {
          const int c = tg0 == 0 ? s0 : s1, d = tg0 == 0 ? s1 : s0;
          recs.push_back(make_int4(rec.node[0], rec.node[u], rec.node[c], rec.node[d]));
          ++quads_of[r0];
          continue;
        }
      }
      general.push_back(rec);
    }
  }, 1);
  for (int r = 0; r < nd; ++r)
    if (overflow[r]) return HX_ERR_PULSES;
  std::vector<int4> recs;
  std::vector<TreeRec> general;
  int64_t n_pairs = 0, n_quads = 0;
  for (int r = 0; r < nd; ++r) {   // domain after domain: root order overall
    recs.insert(recs.end(), recs_of[r].begin(), recs_of[r].end());
    general.insert(general.end(), general_of[r].begin(), general_of[r].end());
    n_pairs += pairs_of[r];
    n_quads += quads_of[r];
  }
  h->n_res_halo = H;
  h->n_res_segs = static_cast<int64_t>(segs.size());
  h->n_res_pairs = n_pairs;
  h->n_res_quads = n_quads;
  h->n_res_trees = static_cast<int64_t>(general.size());
  HX_CUDA(dev_alloc(&h->d_res_om, om.size()));
  HX_CUDA(dev_alloc(&h->d_res_segs, segs.size()));
  HX_CUDA(dev_alloc(&h->d_res_recs, recs.size()));
  HX_CUDA(dev_alloc(&h->d_res_trees, general.size()));
  if (H > 0) {
    HX_CUDA(cudaMemcpyAsync(h->d_res_om, om.data(), sizeof(uint32_t) * om.size(), cudaMemcpyHostToDevice, s));
    HX_CUDA(cudaMemcpyAsync(h->d_res_segs, segs.data(), sizeof(ResSeg) * segs.size(), cudaMemcpyHostToDevice, s));
  }
  if (!recs.empty())
    HX_CUDA(cudaMemcpyAsync(h->d_res_recs, recs.data(), sizeof(int4) * recs.size(), cudaMemcpyHostToDevice, s));
  if (!general.empty())
    HX_CUDA(cudaMemcpyAsync(h->d_res_trees, general.data(), sizeof(TreeRec) * general.size(),
                            cudaMemcpyHostToDevice, s));
  HX_CUDA(cudaStreamSynchronize(s));   // the host vectors go out of scope
  return HX_OK;
}

// Range pieces of the host-buffer calls: every domain's home slots and halo
// slots, cut into pieces of at most kCopyChunkWords words.
int build_copy_chunks(hx_ctx* h) {
  std::vector<CopyChunk> home, halo;
  auto cut = [](std::vector<CopyChunk>& out, int64_t first_slot, int64_t slots) {
    for (int64_t w = 0; w < 3 * slots; w += kCopyChunkWords) {
      CopyChunk c;
      c.word = 3 * first_slot + w;
      c.n = static_cast<int32_t>(std::min<int64_t>(kCopyChunkWords, 3 * slots - w));
      c.pad = 0;
      out.push_back(c);
    }
  };
  for (int r = 0; r < h->pl.ndom; ++r) {
    cut(home, h->dom_offset[r], h->home[r]);
    cut(halo, h->dom_offset[r] + h->home[r], h->halo[r]);
  }
  h->n_home_chunks = static_cast<int>(home.size());
  h->n_halo_chunks = static_cast<int>(halo.size());
  HX_CUDA(dev_alloc(&h->d_home_chunks, home.size()));
  HX_CUDA(dev_alloc(&h->d_halo_chunks, halo.size()));
  if (!home.empty())
    HX_CUDA(cudaMemcpy(h->d_home_chunks, home.data(), sizeof(CopyChunk) * home.size(), cudaMemcpyHostToDevice));
  if (!halo.empty())
    HX_CUDA(cudaMemcpy(h->d_halo_chunks, halo.data(), sizeof(CopyChunk) * halo.size(), cudaMemcpyHostToDevice));
  return HX_OK;
}

// Work tables of the fused and unfused kernels from the host copy of the plan.
int build_tables(hx_ctx* h, cudaStream_t s) {
  const Plan& pl = h->pl;
  const int P = pl.n_pulses, nd = pl.ndom;
  const int n_items = P * nd;
  if (const int rc = build_copy_chunks(h); rc != HX_OK) return rc;
  const bool fine = (h->flags & HX_FLAG_FINE_WAITS) != 0;
  const bool ordered = !(h->flags & HX_FLAG_UNORDERED_FORCES);
  std::vector<ItemInfo> items(std::max(n_items, 1));
  for (int p = 0; p < P; ++p)
    for (int r = 0; r < nd; ++r) {
      const int t = p * nd + r;
      ItemInfo& it = items[t];
      it.r = r;
      it.p = p;
      it.q = h->t_recv[t];
      it.src = h->dom_offset[r];
      it.dst = h->dom_offset[it.q] + h->t_off[t];
      it.map = h->t_map_off[t];
      it.size = h->t_size[t];
      it.split = h->t_split[t];
      it.dim = pl.pulse_dim[p];
      it.shift_flag = h->t_shift[t];
    }
  std::vector<int32_t> maps;
  if ((fine || (h->flags & (HX_FLAG_TILES | HX_FLAG_SWEEP | HX_FLAG_SWEEP_FORCES | HX_FLAG_RESOLVED))) &&
      h->total_entries > 0) {   // fine waits, units and resolved tables read the maps
    maps.resize(h->total_entries);
    // the maps were assembled on `s`, which need not synchronise with the legacy stream
    HX_CUDA(cudaMemcpyAsync(maps.data(), h->d_maps, sizeof(int32_t) * h->total_entries, cudaMemcpyDeviceToHost, s));
    HX_CUDA(cudaStreamSynchronize(s));
  }
  std::vector<int> upper_tab(static_cast<size_t>(nd) * std::max(P, 1));
  for (int r = 0; r < nd; ++r)
    for (int q = 0; q < P; ++q) upper_tab[static_cast<size_t>(r) * P + q] = neighbour(pl, r, pl.pulse_dim[q], +1);
  auto upper = [&](int r, int q) { return upper_tab[static_cast<size_t>(r) * P + q]; };
  std::vector<int64_t> rank(nd);
  for (int r = 0; r < nd; ++r) rank[r] = domain_rank(pl, r);
  h->family[0] = (h->flags & HX_FLAG_TILES)     ? kFamTiles
                 : (h->flags & HX_FLAG_SWEEP)   ? kFamSweep
                 : (h->flags & HX_FLAG_CLUSTER) ? kFamCluster
                 : (h->flags & HX_FLAG_RESOLVED) ? kFamResolved
                                                : kFamChunks;
  h->family[1] = (h->flags & (HX_FLAG_SWEEP | HX_FLAG_SWEEP_FORCES)) ? kFamSweep : h->family[0];
  for (int k = 0; k < 2; ++k) {
    const int per_sm = std::max(1, h->family[k] == kFamTiles     ? tiles_blocks_per_sm(k)
                                   : h->family[k] == kFamSweep   ? sweep_blocks_per_sm(k)
                                   : h->family[k] == kFamCluster ? 1
                                   : h->family[k] == kFamResolved ? 1
                                                                 : max_blocks_per_sm(kernel_for(h, k)));
    h->grid[k] = per_sm * h->sm_count;   // upper bound; trimmed to the work count below
  }
  // Unit lists. A dependent unit is placed a few resident windows after the
  // units it waits for: tile mode three stages per block, sweep eight units
  // per resident warp (measured on the 12M-atom workload: lags of 2, 3, 4, 6
  // and 10 windows gave forces in 112.6, 100.5, 94.2, 92.2 and 92.2 us).
  for (int dir = 0; dir < 2; ++dir) {
    int rc = HX_OK;
    if (h->family[dir] == kFamTiles) {
      rc = build_tile_tables(h, items, maps, rank, kTile, kTileEntries, 3ll * h->grid[dir], kTile * 12 + 16,
                             kTileEntries * 4 + 32 * kTileSegs, kTileEntries * 12 + 32 * kTileSegs, dir);
    } else if (h->family[dir] == kFamSweep) {
      if (P > kSweepSegs) return HX_ERR_PULSES;   // a unit's runs must fit one warp's stage
      rc = build_tile_tables(h, items, maps, rank, kSweepSlots, kSweepEntries, 8ll * h->grid[dir] * kWarps,
                             kSweepTileBytes, kSweepMapBytes, kSweepSrcBytes, dir);
    }
    if (rc != HX_OK) return rc;
  }

  for (int dir = 0; dir < 2; ++dir) {
    if (h->family[dir] != kFamChunks) continue;
    std::vector<Rec> recs;
    std::vector<std::vector<int>> item_recs(std::max(n_items, 1));   // chunk records of each item, in entry order
    auto add_part = [&](int t, int begin, int end, int halo_src, int stage, bool keep_empty) {
      if (end <= begin && !keep_empty) return;
      for (int b = begin;; b += kChunk) {
        Rec rc;
        rc.item = t;
        rc.begin = b;
        rc.end = std::min(end, b + kChunk);
        rc.halo_src = halo_src;
        rc.stage = stage;
        rc.key = 0;
        item_recs[t].push_back(static_cast<int>(recs.size()));
        recs.push_back(std::move(rc));
        if (b + kChunk >= end) break;
      }
    };
    // chunk record of item t holding entry e (item_recs are in entry order)
    auto rec_of_entry = [&](int t, int e) {
      const std::vector<int>& v = item_recs[t];
      int lo = 0, hi = static_cast<int>(v.size()) - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (recs[v[mid]].begin <= e) lo = mid;
        else hi = mid - 1;
      }
      return v[lo];
    };
    // Coarse waits may name empty items: those keep one empty chunk to signal.
    std::vector<char> coarse_waited(std::max(n_items, 1), 0);
    if (!fine) {
      if (dir == 0) {
        for (int p = 0; p < P; ++p)
          for (int r = 0; r < nd; ++r)
            if (items[p * nd + r].split < items[p * nd + r].size)
              for (int q = 0; q < p; ++q) coarse_waited[q * nd + upper(r, q)] = 1;
      } else {
        for (int p = 0; p < P; ++p)
          for (int r = 0; r < nd; ++r)
            for (int pp = p + 1; pp < P; ++pp) {
              coarse_waited[pp * nd + items[p * nd + r].q] = 1;
              if (ordered) coarse_waited[pp * nd + r] = 1;
            }
      }
    }
    for (int p = 0; p < P; ++p)
      for (int r = 0; r < nd; ++r) {
        const int t = p * nd + r;
        const ItemInfo& it = items[t];
        if (dir == 0) {
          add_part(t, 0, it.split, 0, 0, it.size == 0 && coarse_waited[t]);
          add_part(t, it.split, it.size, 1, p, false);
        } else {
          add_part(t, 0, it.size, 1, P - 1 - p, it.size == 0 && coarse_waited[t]);
        }
      }
    // waits (records are independent: spread over the host's cores)
    parallel_for(recs.size(), [&](size_t ci) {
      Rec& rc = recs[ci];
      const ItemInfo& it = items[rc.item];
      const int r = it.r, p = it.p;
      if (dir == 0) {
        if (!rc.halo_src) return;
        if (!fine) {
          for (int q = 0; q < p; ++q) rc.wait.push_back(q * nd + upper(r, q));
          return;
        }
        // producers: chunks of (upper(r, q), q) that stored the slots read
        // here. The entries ascend, r's receive ranges follow pulse order, and
        // an item's records follow entry order, so both cursors only move on.
        const int32_t* m = maps.data() + it.map;
        int q = 0, k = 0;
        for (int i = rc.begin; i < rc.end; ++i) {
          while (q < p) {
            const int tq = q * nd + upper(r, q);
            if (m[i] < h->t_off[tq] + items[tq].size) break;
            ++q;
            k = 0;
          }
          if (q >= p) break;
          const int tq = q * nd + upper(r, q);
          const int64_t e = m[i] - h->t_off[tq];
          if (e < 0) continue;   // a home slot (cannot occur in a forwarded tail)
          const std::vector<int>& v = item_recs[tq];
          while (k + 1 < static_cast<int>(v.size()) && recs[v[k + 1]].begin <= e) ++k;
          if (rc.wait.empty() || rc.wait.back() != v[k]) rc.wait.push_back(v[k]);
        }
      } else {
        if (!fine) {
          for (int pp = p + 1; pp < P; ++pp) {
            rc.wait.push_back(pp * nd + it.q);
            if (ordered && it.q != r) rc.wait.push_back(pp * nd + r);
          }
          std::sort(rc.wait.begin(), rc.wait.end());
          rc.wait.erase(std::unique(rc.wait.begin(), rc.wait.end()), rc.wait.end());
          return;
        }
        if (rc.end <= rc.begin) return;
        const int32_t* m = maps.data() + it.map;
        const int64_t slot_lo = h->t_off[rc.item] + rc.begin, slot_hi = h->t_off[rc.item] + rc.end;
        for (int pp = p + 1; pp < P; ++pp) {
          // later-pulse chunks of the receiver that add into the slots read here
          const int tq = pp * nd + it.q;
          const int32_t* mq = maps.data() + items[tq].map;
          const int nq = items[tq].size;
          const int i1 = static_cast<int>(std::lower_bound(mq, mq + nq, static_cast<int32_t>(slot_lo)) - mq);
          const int i2 = static_cast<int>(std::lower_bound(mq, mq + nq, static_cast<int32_t>(slot_hi)) - mq);
          if (i1 < i2) {
            const int c1 = rec_of_entry(tq, i1), c2 = rec_of_entry(tq, i2 - 1);
            for (int c = c1; c <= c2; ++c) rc.wait.push_back(c);   // records of one item are consecutive
          }
          if (!ordered) continue;
          // later-pulse chunks of the sender that add into the same targets
          const int tr = pp * nd + r;
          const int32_t* mr = maps.data() + items[tr].map;
          const int nr = items[tr].size;
          int k = static_cast<int>(std::lower_bound(mr, mr + nr, m[rc.begin]) - mr);
          if (k >= nr) continue;
          const std::vector<int>& v = item_recs[tr];
          int rec = 0;
          const int first = rec_of_entry(tr, k);
          while (v[rec] != first) ++rec;
          for (int i = rc.begin; i < rc.end && k < nr; ++i) {
            while (k < nr && mr[k] < m[i]) ++k;
            if (k < nr && mr[k] == m[i]) {
              while (rec + 1 < static_cast<int>(v.size()) && recs[v[rec + 1]].begin <= k) ++rec;
              if (rc.wait.empty() || rc.wait.back() != v[rec]) rc.wait.push_back(v[rec]);
            }
          }
        }
      }
      std::sort(rc.wait.begin(), rc.wait.end());
      rc.wait.erase(std::unique(rc.wait.begin(), rc.wait.end()), rc.wait.end());
    });
    // listing dependencies (chunk records) and who gets signalled
    std::vector<char> rec_waited(recs.size(), 0), item_waited(std::max(n_items, 1), 0);
    for (auto& rc : recs) {
      if (fine) {
        rc.deps = rc.wait;
        for (int d : rc.wait) rec_waited[d] = 1;
      } else {
        for (int t : rc.wait) {
          item_waited[t] = 1;
          rc.deps.insert(rc.deps.end(), item_recs[t].begin(), item_recs[t].end());
        }
      }
    }
    // priority: base order (domain rank, stage, pulse, entry), then a lag of
    // one resident-warp window per stage
    {
      std::vector<int> base(recs.size());
      for (size_t i = 0; i < recs.size(); ++i) base[i] = static_cast<int>(i);
      std::sort(base.begin(), base.end(), [&](int a, int b) {
        const Rec& x = recs[a];
        const Rec& y = recs[b];
        const ItemInfo& ix = items[x.item];
        const ItemInfo& iy = items[y.item];
        if (rank[ix.r] != rank[iy.r]) return rank[ix.r] < rank[iy.r];
        if (x.stage != y.stage) return x.stage < y.stage;
        if (ix.p != iy.p) return ix.p < iy.p;
        return x.begin < y.begin;
      });
      const long long window = static_cast<long long>(h->grid[dir]) * kWarps;
      for (size_t k = 0; k < base.size(); ++k)
        recs[base[k]].key = static_cast<long long>(k) + window * recs[base[k]].stage;
    }
    std::vector<int> order = order_chunks(recs);
    if (order.size() != recs.size()) return HX_ERR_STATE;
    std::vector<int> pos(recs.size());
    for (size_t k = 0; k < order.size(); ++k) pos[order[k]] = static_cast<int>(k);
    std::vector<int> item_chunks(std::max(n_items, 1), 0);
    for (auto& rc : recs) item_chunks[rc.item] += 1;
    std::vector<Chunk> chunks;
    std::vector<Wait> waits;
    chunks.reserve(order.size());
    for (int ri : order) {
      const Rec& rc = recs[ri];
      const ItemInfo& it = items[rc.item];
      Chunk ch;
      std::memset(&ch, 0, sizeof(ch));
      ch.src = it.src;
      ch.dst = it.dst + rc.begin;
      ch.map = it.map + rc.begin;
      ch.n = rc.end - rc.begin;
      ch.item = rc.item;
      ch.item_chunks = item_chunks[rc.item];
      ch.wait_off = static_cast<int32_t>(waits.size());
      ch.wait_cnt = static_cast<int32_t>(rc.wait.size());
      for (int w : rc.wait) waits.push_back(fine ? Wait{pos[w], 1} : Wait{w, 0});
      const bool sig = fine ? rec_waited[ri] != 0 : item_waited[rc.item] != 0;
      ch.flags = (rc.halo_src ? kHaloSrc : 0) | (sig ? kSignal : 0) | (dir == 0 && it.shift_flag ? kShift : 0);
      ch.dim = it.dim;
      ch.shift = pl.boxf[it.dim];
      chunks.push_back(ch);
    }
    if (!fine)
      for (auto& w : waits) w.chunks = item_chunks[w.item];
    h->n_chunks[dir] = static_cast<int>(chunks.size());
    HX_CUDA(dev_alloc(&h->d_chunks[dir], chunks.size()));
    HX_CUDA(dev_alloc(&h->d_waits[dir], waits.size()));
    if (!chunks.empty())
      HX_CUDA(cudaMemcpy(h->d_chunks[dir], chunks.data(), sizeof(Chunk) * chunks.size(), cudaMemcpyHostToDevice));
    if (!waits.empty())
      HX_CUDA(cudaMemcpy(h->d_waits[dir], waits.data(), sizeof(Wait) * waits.size(), cudaMemcpyHostToDevice));
  }

  if (h->family[0] == kFamResolved) {
    const int rc = build_resolved_tables(h, items, maps, s);
    if (rc != HX_OK) return rc;
  }

  // Unfused: per pulse, every item's entries in sender order, no waits or signals.
  std::vector<Chunk> uch;
  h->u_begin.assign(P + 1, 0);
  for (int p = 0; p < P; ++p) {
    h->u_begin[p] = static_cast<int>(uch.size());
    for (int r = 0; r < nd; ++r) {
      const ItemInfo& it = items[p * nd + r];
      for (int cb = 0; cb < it.size; cb += kChunk) {
        Chunk ch;
        std::memset(&ch, 0, sizeof(ch));
        ch.src = it.src;
        ch.dst = it.dst + cb;
        ch.map = it.map + cb;
        ch.n = std::min(it.size - cb, kChunk);
        ch.item = p * nd + r;
        ch.flags = kHaloSrc | (it.shift_flag ? kShift : 0);
        ch.dim = it.dim;
        ch.shift = pl.boxf[it.dim];
        uch.push_back(ch);
      }
    }
  }
  h->u_begin[P] = static_cast<int>(uch.size());
  HX_CUDA(dev_alloc(&h->d_uchunks, uch.size()));
  if (!uch.empty())
    HX_CUDA(cudaMemcpy(h->d_uchunks, uch.data(), sizeof(Chunk) * uch.size(), cudaMemcpyHostToDevice));

  // one flag (and one election counter) per item or per chunk, per direction
  h->n_flags = std::max<size_t>({static_cast<size_t>(std::max(n_items, 1)), static_cast<size_t>(h->n_chunks[0]),
                                 static_cast<size_t>(h->n_chunks[1]), static_cast<size_t>(h->n_units[0]),
                                 static_cast<size_t>(h->n_units[1])});
  HX_CUDA(dev_alloc(&h->d_flags, 2 * h->n_flags));
  HX_CUDA(dev_alloc(&h->d_blk, 2 * h->n_flags));
  HX_CUDA(dev_alloc(&h->d_ctrl, 2));
  // Persistent grid: every warp (tile mode: every block) co-resident, and no
  // more of them than there is work.
  for (int k = 0; k < 2; ++k) {
    if (h->family[k] == kFamResolved) {
      // coordinates: one block per halo segment; forces: general blocks, then record blocks
      const int64_t n = h->n_res_pairs + h->n_res_quads;
      const int64_t fb = resolved_blocks(n, resolved_per_thread(h, n, kResTreesPerThread)) +
                         resolved_blocks(h->n_res_trees, 1);
      h->grid[k] = static_cast<int>(std::max<int64_t>(1, k == 0 ? h->n_res_segs : fb));
    } else if (h->family[k] == kFamCluster) {
      h->grid[k] = kClusterCtas;   // exactly one cluster
    } else if (h->family[k] == kFamTiles) {
      h->grid[k] = std::max(1, std::min(h->n_units[k], h->grid[k]));
    } else if (h->family[k] == kFamSweep) {   // one warp per batch of units
      const int warps = std::max(1, std::min((h->n_units[k] + kSweepBatch - 1) / kSweepBatch, h->grid[k] * kWarps));
      h->grid[k] = (warps + kWarps - 1) / kWarps;
    } else {
      const int warps = std::max(1, std::min(h->n_chunks[k], h->grid[k] * kWarps));
      h->grid[k] = (warps + kWarps - 1) / kWarps;
    }
  }
  return reset_signals(h, s);
}

struct BuildScratch {
  int32_t* dom_id = nullptr;
  float* faces = nullptr;
  int32_t* hist = nullptr;
  int32_t* hist_scan = nullptr;
  int* err = nullptr;
  float* home_xyz = nullptr;
  int32_t* home_dom = nullptr;
  int64_t* home_start = nullptr;
  int64_t* dom_off = nullptr;
  BuildTile* tiles = nullptr;
  int32_t* tile_cnt = nullptr;
  int32_t* tile_off = nullptr;
  const float** bufs = nullptr;
  std::vector<float*> recv;     // per pulse: received coordinates, sender-major
  std::vector<int32_t*> maps;   // per pulse: maps, sender-major
  ~BuildScratch() {
    dev_free(dom_id); dev_free(faces); dev_free(hist); dev_free(hist_scan); dev_free(err); dev_free(home_xyz);
    dev_free(home_dom); dev_free(home_start); dev_free(dom_off); dev_free(tiles); dev_free(tile_cnt);
    dev_free(tile_off); dev_free(bufs);
    for (auto* p : recv) dev_free(p);
    for (auto* p : maps) dev_free(p);
  }
};

int build(hx_ctx* h, const float* pos, int64_t n, float* coords, int64_t capacity, cudaStream_t s) {
  const Plan& pl = h->pl;
  const int nd = pl.ndom, P = pl.n_pulses;
  BuildScratch b;
  // 1. home cells and stable partition
  const int ntiles = static_cast<int>((n + kPartTile - 1) / kPartTile);
  HX_CUDA(dev_alloc(&b.dom_id, n));
  HX_CUDA(dev_alloc(&b.hist, static_cast<size_t>(nd) * std::max(ntiles, 1)));
  HX_CUDA(dev_alloc(&b.hist_scan, static_cast<size_t>(nd) * std::max(ntiles, 1)));
  HX_CUDA(dev_alloc(&b.err, 1));
  HX_CUDA(dev_alloc(&b.home_xyz, 3 * static_cast<size_t>(n)));
  HX_CUDA(dev_alloc(&b.home_dom, n));
  HX_CUDA(dev_alloc(&h->d_home_ids, n));
  HX_CUDA(cudaMemsetAsync(b.err, 0, sizeof(int), s));
  const std::vector<float> faces = face_tables(pl);
  HX_CUDA(dev_alloc(&b.faces, faces.size()));
  HX_CUDA(cudaMemcpyAsync(b.faces, faces.data(), sizeof(float) * faces.size(), cudaMemcpyHostToDevice, s));
  HX_CUDA(launch_cells(pos, n, pl.dims, b.faces, nd, b.dom_id, b.hist, ntiles, b.err, s));
  HX_CUDA(scan_exclusive(b.hist, b.hist_scan, static_cast<int64_t>(nd) * ntiles, s));
  std::vector<int32_t> first(nd, 0);
  if (ntiles > 0)
    HX_CUDA(cudaMemcpy2DAsync(first.data(), sizeof(int32_t), b.hist_scan, sizeof(int32_t) * ntiles,
                              sizeof(int32_t), nd, cudaMemcpyDeviceToHost, s));
  int err_host = 0;
  HX_CUDA(cudaMemcpyAsync(&err_host, b.err, sizeof(int), cudaMemcpyDeviceToHost, s));
  HX_CUDA(cudaStreamSynchronize(s));
  if (err_host) return HX_ERR_RANGE;
  std::vector<int64_t> home_start(nd);
  h->home.assign(nd, 0);
  for (int r = 0; r < nd; ++r) {
    home_start[r] = first[r];
    const int64_t next = (r + 1 < nd) ? first[r + 1] : n;
    h->home[r] = static_cast<int32_t>(next - first[r]);
  }
  HX_CUDA(launch_scatter_home(pos, n, nd, b.dom_id, b.hist_scan, ntiles, h->d_home_ids, b.home_xyz, b.home_dom,
                              s));

  // 2. pulses in global order
  std::vector<int64_t> len(nd);
  for (int r = 0; r < nd; ++r) len[r] = h->home[r];
  std::vector<int64_t> off(static_cast<size_t>(nd) * std::max(P, 1), 0), rcv(off.size(), 0);
  std::vector<int64_t> sender_prefix(off.size(), 0);   // [p * nd + r] position of r's map in pulse p
  std::vector<int64_t> pulse_total(std::max(P, 1), 0);
  h->t_map_off.assign(static_cast<size_t>(nd) * P, 0);
  h->t_size.assign(static_cast<size_t>(nd) * P, 0);
  h->t_recv.assign(static_cast<size_t>(nd) * P, 0);
  h->t_off.assign(static_cast<size_t>(nd) * P, 0);
  h->t_shift.assign(static_cast<size_t>(nd) * P, 0);
  h->t_split.assign(static_cast<size_t>(nd) * P, 0);
  HX_CUDA(dev_alloc(&b.bufs, 1 + P));
  std::vector<const float*> bufs_host(1 + P, nullptr);
  bufs_host[0] = b.home_xyz;
  b.recv.assign(P, nullptr);
  b.maps.assign(P, nullptr);
  for (int p = 0; p < P; ++p) {
    const int d = pl.pulse_dim[p];
    const int k = pl.pulse_k[p];
    std::vector<BuildTile> tiles;
    std::vector<int> tile_home(0);   // 1 when the tile lies in the sender's home range
    std::vector<int> first_tile(nd + 1, 0);
    for (int r = 0; r < nd; ++r) {
      first_tile[r] = static_cast<int>(tiles.size());
      int c[3];
      cell_of(pl, r, c);
      auto add_segment = [&](int buf, int64_t elem_begin, int64_t local_begin, int64_t count, int is_home) {
        for (int64_t e = 0; e < count; e += kSelTile) {
          BuildTile t;
          std::memset(&t, 0, sizeof(t));
          t.sender = r;
          t.local_begin = static_cast<int32_t>(local_begin + e);
          t.n = static_cast<int32_t>(std::min<int64_t>(kSelTile, count - e));
          t.buf = buf;
          t.elem_begin = elem_begin + e;
          t.lo = pl.lo[d][c[d]];
          t.shift = pl.boxf[d];
          t.do_shift = (c[d] == 0);
          tiles.push_back(t);
          tile_home.push_back(is_home);
        }
      };
      if (k == 0) {
        add_segment(0, home_start[r], 0, h->home[r], 1);
        for (int q = 0; q < p; ++q) {
          const int up = neighbour(pl, r, pl.pulse_dim[q], +1);   // the domain that sent into r in pulse q
          add_segment(1 + q, sender_prefix[static_cast<size_t>(q) * nd + up], off[static_cast<size_t>(r) * P + q],
                      rcv[static_cast<size_t>(r) * P + q], 0);
        }
      } else {
        const int q = p - 1;
        const int up = neighbour(pl, r, pl.pulse_dim[q], +1);
        add_segment(1 + q, sender_prefix[static_cast<size_t>(q) * nd + up], off[static_cast<size_t>(r) * P + q],
                    rcv[static_cast<size_t>(r) * P + q], 0);
      }
    }
    first_tile[nd] = static_cast<int>(tiles.size());
    const int nt = static_cast<int>(tiles.size());
    dev_free(b.tiles);
    dev_free(b.tile_cnt);
    dev_free(b.tile_off);
    HX_CUDA(dev_alloc(&b.tiles, nt));
    HX_CUDA(dev_alloc(&b.tile_cnt, nt));
    HX_CUDA(dev_alloc(&b.tile_off, nt));
    if (nt > 0)
      HX_CUDA(cudaMemcpyAsync(b.tiles, tiles.data(), sizeof(BuildTile) * nt, cudaMemcpyHostToDevice, s));
    HX_CUDA(cudaMemcpyAsync(b.bufs, bufs_host.data(), sizeof(float*) * bufs_host.size(), cudaMemcpyHostToDevice, s));
    HX_CUDA(launch_select_count(b.tiles, nt, b.bufs, d, pl.rcf, b.tile_cnt, s));
    HX_CUDA(scan_exclusive(b.tile_cnt, b.tile_off, nt, s));
    std::vector<int32_t> cnt(std::max(nt, 1)), toff(std::max(nt, 1));
    if (nt > 0) {
      HX_CUDA(cudaMemcpyAsync(cnt.data(), b.tile_cnt, sizeof(int32_t) * nt, cudaMemcpyDeviceToHost, s));
      HX_CUDA(cudaMemcpyAsync(toff.data(), b.tile_off, sizeof(int32_t) * nt, cudaMemcpyDeviceToHost, s));
    }
    HX_CUDA(cudaStreamSynchronize(s));
    int64_t total = 0;
    for (int r = 0; r < nd; ++r) {
      int64_t S = 0, split = 0;
      for (int t = first_tile[r]; t < first_tile[r + 1]; ++t) {
        S += cnt[t];
        if (tile_home[t]) split += cnt[t];
      }
      const size_t idx = static_cast<size_t>(p) * nd + r;
      sender_prefix[idx] = total;
      if (first_tile[r] < first_tile[r + 1] && toff[first_tile[r]] != total) return HX_ERR_CUDA;
      h->t_size[idx] = static_cast<int32_t>(S);
      h->t_split[idx] = static_cast<int32_t>(split);
      int c[3];
      cell_of(pl, r, c);
      h->t_shift[idx] = (c[d] == 0);
      total += S;
    }
    pulse_total[p] = total;
    HX_CUDA(dev_alloc(&b.recv[p], 3 * static_cast<size_t>(total)));
    HX_CUDA(dev_alloc(&b.maps[p], static_cast<size_t>(total)));
    bufs_host[1 + p] = b.recv[p];
    HX_CUDA(launch_select_write(b.tiles, nt, b.bufs, d, pl.rcf, b.tile_off, b.maps[p], b.recv[p], s));
    // receivers: each domain receives exactly one range per pulse
    std::vector<int64_t> len_before = len;
    for (int r = 0; r < nd; ++r) {
      const size_t idx = static_cast<size_t>(p) * nd + r;
      const int q = neighbour(pl, r, d, -1);
      h->t_recv[idx] = q;
      h->t_off[idx] = static_cast<int32_t>(len_before[q]);
      off[static_cast<size_t>(q) * P + p] = len_before[q];
      rcv[static_cast<size_t>(q) * P + p] = h->t_size[idx];
      len[q] += h->t_size[idx];
    }
    for (int r = 0; r < nd; ++r)
      if (len[r] > INT32_MAX) return HX_ERR_CAPACITY;
  }

  // 3. layout and concatenated maps (pulse-major, sender-minor)
  h->dom_offset.assign(nd, 0);
  h->halo.assign(nd, 0);
  int64_t slots = 0;
  for (int r = 0; r < nd; ++r) {
    h->dom_offset[r] = slots;
    h->halo[r] = static_cast<int32_t>(len[r] - h->home[r]);
    slots += len[r];
  }
  h->total_slots = slots;
  int64_t entries = 0;
  for (int p = 0; p < P; ++p) entries += pulse_total[p];
  h->total_entries = entries;
  HX_CUDA(dev_alloc(&h->d_maps, entries));
  int64_t base = 0;
  for (int p = 0; p < P; ++p) {
    if (pulse_total[p] > 0)
      HX_CUDA(cudaMemcpyAsync(h->d_maps + base, b.maps[p], sizeof(int32_t) * pulse_total[p],
                              cudaMemcpyDeviceToDevice, s));
    for (int r = 0; r < nd; ++r) {
      const size_t idx = static_cast<size_t>(p) * nd + r;
      h->t_map_off[idx] = base + sender_prefix[idx];
    }
    base += pulse_total[p];
  }
  // keep what placing the home coordinates needs
  HX_CUDA(dev_alloc(&b.home_start, nd));
  HX_CUDA(dev_alloc(&b.dom_off, nd));
  HX_CUDA(cudaMemcpyAsync(b.home_start, home_start.data(), sizeof(int64_t) * nd, cudaMemcpyHostToDevice, s));
  HX_CUDA(cudaMemcpyAsync(b.dom_off, h->dom_offset.data(), sizeof(int64_t) * nd, cudaMemcpyHostToDevice, s));
  int rc = build_tables(h, s);
  if (rc != HX_OK) return rc;
  h->n_atoms = n;
  h->built = true;
  if (!coords) return HX_OK;
  if (capacity < h->total_slots) return HX_ERR_CAPACITY;
  // 4. fill the caller's array: home coordinates, then one coordinate exchange
  HX_CUDA(launch_place_home(b.home_xyz, b.home_dom, b.home_start, b.dom_off, n, coords, s));
  if (P > 0 && work_items(h, 0) > 0) {
    rc = launch(h, 0, coords, s);
    if (rc != HX_OK) return rc;
  }
  HX_CUDA(cudaStreamSynchronize(s));
  return HX_OK;
}

}  // namespace

// ------------------------------------------------------------------ scratch-free launch

int hx::handle_device(const hx_ctx* h) { return h->device; }

int hx::launch_coords_with_scratch(hx_ctx* h, float* coords, cudaStream_t s, Ctrl* ctrl,
                                   unsigned long long* flags, unsigned int* arrivals, size_t max_flags) {
  if (!h->built) return HX_ERR_STATE;
  if (!coords && h->total_slots > 0) return HX_ERR_ARG;
  const int work = work_items(h, 0);
  if (h->pl.n_pulses == 0 || work == 0) return HX_OK;
  if (h->family[0] == kFamResolved) {   // no dependencies, no scratch at all
    ResolvedParams RP = resolved_params(h);
    void* rargs[2] = {&coords, &RP};
    return to_err(
        cudaLaunchKernel(resolved_kernel(0), dim3(static_cast<unsigned>(h->grid[0])), dim3(kResThreads), rargs, 0, s));
  }
  if (h->family[0] == kFamCluster) {   // cluster barriers, no scratch at all
    ClusterParams CP = cluster_params(h);
    void* cargs[2] = {&coords, &CP};
    return to_err(cudaLaunchKernel(cluster_kernel(0), dim3(kClusterCtas), dim3(kClusterThreads), cargs, 0, s));
  }
  // flags are indexed by item (pulse signals) or by list position (chunk / tile signals)
  const size_t need = std::max<size_t>(static_cast<size_t>(h->pl.n_pulses) * h->pl.ndom, static_cast<size_t>(work));
  if (need > max_flags) return HX_ERR_CAPACITY;
  HX_CUDA(cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), s));
  HX_CUDA(cudaMemsetAsync(&ctrl->drop_item, 0xff, sizeof(int), s));   // -1: no fault injection
  HX_CUDA(cudaMemsetAsync(flags, 0, sizeof(unsigned long long) * need, s));
  HX_CUDA(cudaMemsetAsync(arrivals, 0, sizeof(unsigned int) * need, s));
  void* args[2];
  DirParams P;
  TileParams TP;
  const void* fn;
  size_t smem = 0;
  args[0] = &coords;
  if (h->family[0] != kFamChunks) {
    TP = tile_params(h, 0);
    TP.flags = flags;
    TP.ctrl = ctrl;
    args[1] = &TP;
    fn = fused_kernel(h, 0);
    smem = fused_smem(h, 0);
  } else {
    P = dir_params(h, 0);
    P.flags = flags;
    P.arrivals = arrivals;
    P.ctrl = ctrl;
    args[1] = &P;
    fn = kernel_for(h, 0);
  }
  return to_err(cudaLaunchKernel(fn, dim3(static_cast<unsigned>(h->grid[0])), dim3(fused_threads(h, 0)),
                                args, smem, s));
}

// ------------------------------------------------------------------ C ABI

extern "C" {

const char* hx_error_string(int code) {
  switch (code) {
    case HX_OK: return "ok";
    case HX_ERR_ARG: return "invalid argument";
    case HX_ERR_PULSES: return "too many pulses: the cutoff spans the whole periodic dimension";
    case HX_ERR_RANGE: return "position outside [0, L)";
    case HX_ERR_CAPACITY: return "buffer smaller than the layout";
    case HX_ERR_CUDA: return "CUDA error";
    case HX_ERR_TIMEOUT: return "device wait for a pulse signal timed out";
    case HX_ERR_STATE: return "exchange before a successful build";
    case HX_ERR_NOMEM: return "out of memory";
    default: return "unknown error";
  }
}

int hx_query_plan(const double box[3], const int dims[3], double cutoff, int* n_pulses, int32_t* pulse_dim,
                  int32_t* pulse_k) {
  Plan pl;
  const int rc = make_plan(box, dims, cutoff, &pl);
  if (rc != HX_OK) return rc;
  if (n_pulses) *n_pulses = pl.n_pulses;
  for (int p = 0; p < pl.n_pulses; ++p) {
    if (pulse_dim) pulse_dim[p] = pl.pulse_dim[p];
    if (pulse_k) pulse_k[p] = pl.pulse_k[p];
  }
  return HX_OK;
}

int hx_init(hx_handle* out, const double box[3], const int dims[3], double cutoff, int device, unsigned flags,
            unsigned timeout_us) {
  if (!out) return HX_ERR_ARG;
  *out = nullptr;
  Plan pl;
  int rc = make_plan(box, dims, cutoff, &pl);
  if (rc != HX_OK) return rc;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return HX_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return HX_ERR_CUDA;
  hx_ctx* h = new (std::nothrow) hx_ctx();
  if (!h) return HX_ERR_NOMEM;
  h->pl = pl;
  h->device = device;
  // at most one kernel family for the coordinates (forces follow it), and
  // HX_FLAG_SWEEP_FORCES only over the chunk or resolved coordinate kernels
  const unsigned families = flags & (HX_FLAG_TILES | HX_FLAG_SWEEP | HX_FLAG_CLUSTER | HX_FLAG_RESOLVED);
  const bool sweep_forces_clash =
      (flags & HX_FLAG_SWEEP_FORCES) && (flags & (HX_FLAG_TILES | HX_FLAG_SWEEP | HX_FLAG_CLUSTER));
  if ((families & (families - 1)) || sweep_forces_clash) {
    delete h;
    return HX_ERR_ARG;
  }
  h->flags = flags;
  h->timeout_ns = 1000ull * (timeout_us ? timeout_us : 1000000u);
  if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete h;
    return HX_ERR_CUDA;
  }
  *out = h;
  return HX_OK;
}

int hx_build_maps(hx_handle h, const float* pos_in, int64_t n_atoms, float* coords, int64_t capacity,
                  int64_t* needed, void* stream) {
  if (!h || n_atoms < 0 || n_atoms > INT32_MAX || (n_atoms > 0 && !pos_in)) return HX_ERR_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return HX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  free_tables(h);
  const int rc = build(h, pos_in, n_atoms, coords, capacity, s);
  if (rc == HX_OK || rc == HX_ERR_CAPACITY) {
    if (needed) *needed = h->total_slots;
    return rc;
  }
  free_tables(h);
  return rc;
}

namespace {

int ensure_device(hx_ctx* h) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return HX_ERR_CUDA;
  if (cur != h->device && cudaSetDevice(h->device) != cudaSuccess) return HX_ERR_CUDA;
  return HX_OK;
}

int exchange(hx_handle h, float* buf, void* stream, int kind) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (!buf && h->total_slots > 0) return HX_ERR_ARG;   // an empty layout touches no memory
  if (h->pl.n_pulses == 0 || work_items(h, kind) == 0) return HX_OK;   // nothing moves
  const int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  return launch(h, kind, buf, static_cast<cudaStream_t>(stream));
}

}  // namespace

int hx_exchange_coords(hx_handle h, float* coords, void* stream) { return exchange(h, coords, stream, 0); }

int hx_exchange_forces(hx_handle h, float* forces, void* stream) { return exchange(h, forces, stream, 1); }

namespace {

// Device address of a page-locked, mapped host buffer (HX_ERR_ARG otherwise).
int device_view(float* host, float** out) {
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, host, 0) != cudaSuccess || d == nullptr) {
    cudaGetLastError();   // not sticky; clear it for the caller's next check
    return HX_ERR_ARG;
  }
  *out = static_cast<float*>(d);
  return HX_OK;
}

int exchange_host(hx_handle h, float* host, float* dev, void* stream, int kind) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (h->total_slots == 0) return HX_OK;
  if (!host || !dev) return HX_ERR_ARG;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  float* hv = nullptr;
  if ((rc = device_view(host, &hv)) != HX_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == 0) {   // home coordinates in, halo coordinates out
    HX_CUDA(launch_copy_chunks(hv, dev, h->d_home_chunks, h->n_home_chunks, s));
    if ((rc = exchange(h, dev, stream, 0)) != HX_OK) return rc;
    HX_CUDA(launch_copy_chunks(dev, hv, h->d_halo_chunks, h->n_halo_chunks, s));
  } else {           // every slot's force in, home forces out
    HX_CUDA(cudaMemcpyAsync(dev, host, sizeof(float) * 3 * h->total_slots, cudaMemcpyHostToDevice, s));
    if ((rc = exchange(h, dev, stream, 1)) != HX_OK) return rc;
    HX_CUDA(launch_copy_chunks(dev, hv, h->d_home_chunks, h->n_home_chunks, s));
  }
  return HX_OK;
}

}  // namespace

int hx_exchange_coords_host(hx_handle h, float* coords_host, float* coords_dev, void* stream) {
  return exchange_host(h, coords_host, coords_dev, stream, 0);
}

int hx_exchange_forces_host(hx_handle h, float* forces_host, float* forces_dev, void* stream) {
  return exchange_host(h, forces_host, forces_dev, stream, 1);
}

int hx_exchange_coords_unfused(hx_handle h, float* coords, void* stream) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (!coords && h->total_slots > 0) return HX_ERR_ARG;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int p = 0; p < h->pl.n_pulses; ++p) {
    PulseParams pp{h->d_uchunks, h->d_maps, h->u_begin[p], h->u_begin[p + 1] - h->u_begin[p]};
    rc = to_err(launch_pack_pulse(coords, pp, s));
    if (rc != HX_OK) return rc;
  }
  return HX_OK;
}

int hx_exchange_forces_unfused(hx_handle h, float* forces, void* stream) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (!forces && h->total_slots > 0) return HX_ERR_ARG;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int p = h->pl.n_pulses - 1; p >= 0; --p) {
    PulseParams pp{h->d_uchunks, h->d_maps, h->u_begin[p], h->u_begin[p + 1] - h->u_begin[p]};
    rc = to_err(launch_unpack_pulse(forces, pp, s));
    if (rc != HX_OK) return rc;
  }
  return HX_OK;
}

int hx_noop(hx_handle h, void* stream) {
  if (!h) return HX_ERR_ARG;
  const int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  return launch(h, 2, nullptr, static_cast<cudaStream_t>(stream));
}

int hx_get_counts(hx_handle h, int* n_domains, int* n_pulses, int64_t* total_slots, int64_t* total_entries) {
  if (!h) return HX_ERR_ARG;
  if (n_domains) *n_domains = h->pl.ndom;
  if (n_pulses) *n_pulses = h->pl.n_pulses;
  if (!h->built) return HX_ERR_STATE;
  if (total_slots) *total_slots = h->total_slots;
  if (total_entries) *total_entries = h->total_entries;
  return HX_OK;
}

int hx_get_resolved_counts(hx_handle h, int64_t* n_pairs, int64_t* n_quads, int64_t* n_general) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (n_pairs) *n_pairs = h->n_res_pairs;
  if (n_quads) *n_quads = h->n_res_quads;
  if (n_general) *n_general = h->n_res_trees;
  return HX_OK;
}

int hx_get_layout(hx_handle h, int64_t* dom_offset, int32_t* home_count, int32_t* halo_count) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  for (int r = 0; r < h->pl.ndom; ++r) {
    if (dom_offset) dom_offset[r] = h->dom_offset[r];
    if (home_count) home_count[r] = h->home[r];
    if (halo_count) halo_count[r] = h->halo[r];
  }
  return HX_OK;
}

int hx_get_home_ids(hx_handle h, int32_t* home_ids, void* stream) {
  if (!h || (!home_ids && h->n_atoms > 0)) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (h->n_atoms == 0) return HX_OK;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  return to_err(cudaMemcpyAsync(home_ids, h->d_home_ids, sizeof(int32_t) * h->n_atoms, cudaMemcpyDeviceToDevice,
                                static_cast<cudaStream_t>(stream)));
}

int hx_get_maps(hx_handle h, int32_t* maps_host, int64_t cap, int64_t* table_host) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  if (maps_host) {
    if (cap < h->total_entries) return HX_ERR_CAPACITY;
    if (h->total_entries > 0 &&
        cudaMemcpy(maps_host, h->d_maps, sizeof(int32_t) * h->total_entries, cudaMemcpyDeviceToHost) != cudaSuccess)
      return HX_ERR_CUDA;
  }
  if (table_host) {
    const size_t n = static_cast<size_t>(h->pl.n_pulses) * h->pl.ndom;
    for (size_t t = 0; t < n; ++t) {
      table_host[6 * t + 0] = h->t_map_off[t];
      table_host[6 * t + 1] = h->t_size[t];
      table_host[6 * t + 2] = h->t_recv[t];
      table_host[6 * t + 3] = h->t_off[t];
      table_host[6 * t + 4] = h->t_shift[t];
      table_host[6 * t + 5] = h->t_split[t];
    }
  }
  return HX_OK;
}

int hx_status(hx_handle h, void* stream, int* detail) {
  if (detail) *detail = -1;
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_OK;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HX_ERR_CUDA;
  Ctrl c[2];
  if (cudaMemcpy(c, h->d_ctrl, sizeof(c), cudaMemcpyDeviceToHost) != cudaSuccess) return HX_ERR_CUDA;
  for (int k = 0; k < 2; ++k) {
    if (c[k].status != 0) {
      if (detail) *detail = c[k].detail;
      return c[k].status;
    }
  }
  return HX_OK;
}

int hx_clear_status(hx_handle h, void* stream) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_OK;
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HX_ERR_CUDA;
  return reset_signals(h, s);
}

int hx_debug_drop_signal(hx_handle h, int direction, int domain, int pulse) {
  if (!h || direction < 0 || direction > 1) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  int item = -1;
  if (domain >= 0) {
    if (domain >= h->pl.ndom || pulse < 0 || pulse >= h->pl.n_pulses) return HX_ERR_ARG;
    item = pulse * h->pl.ndom + domain;
  }
  int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return HX_ERR_CUDA;
  Ctrl* c = h->d_ctrl + direction;
  if (cudaMemcpy(&c->drop_item, &item, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return HX_ERR_CUDA;
  return HX_OK;
}

void hx_destroy(hx_handle h) {
  if (!h) return;
  if (ensure_device(h) == HX_OK) cudaDeviceSynchronize();
  free_tables(h);
  delete h;
}

}  // extern "C"
