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
#include <vector>

#include "../../include/hx.h"
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
  std::vector<int> u_begin;                  // per pulse, first unfused chunk (P + 1 entries)
  std::vector<GraphEntry> graphs;
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
  const size_t n_items = static_cast<size_t>(std::max(h->pl.n_pulses * h->pl.ndom, 1));
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
  const int mode = (h->flags & HX_FLAG_COUNTER_SIGNAL) ? kCounter : kLastArrival;
  if (kind == 0) return coords_kernel(mode);
  if (kind == 1) return forces_kernel(mode, !(h->flags & HX_FLAG_UNORDERED_FORCES));
  return noop_kernel();
}

// Launch a fused exchange (kind 0/1) or the no-op (kind 2): directly, or via
// a cached single-node graph keyed by (kind, buffer pointer).
int launch(hx_ctx* h, int kind, float* buf, cudaStream_t s) {
  DirParams P;
  void* args2[2];
  void** args = nullptr;
  dim3 grid(1), block(kind == 2 ? 1 : kThreads);
  if (kind != 2) {
    P = dir_params(h, kind);
    args2[0] = &buf;
    args2[1] = &P;
    args = args2;
    grid = dim3(static_cast<unsigned>(h->grid[kind]));
  }
  const void* fn = kernel_for(h, kind);
  if (h->flags & HX_FLAG_NO_GRAPH) return to_err(cudaLaunchKernel(fn, grid, block, args, 0, s));
  for (auto& g : h->graphs)
    if (g.kind == kind && g.ptr == buf) return to_err(cudaGraphLaunch(g.exec, s));
  cudaGraph_t graph;
  HX_CUDA(cudaGraphCreate(&graph, 0));
  cudaKernelNodeParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.func = const_cast<void*>(fn);
  kp.gridDim = grid;
  kp.blockDim = block;
  kp.sharedMemBytes = 0;
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
  const size_t n_items = static_cast<size_t>(std::max(h->pl.n_pulses * h->pl.ndom, 1));
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
// A "part" is a run of entries of one item that is listed as a unit: the
// independent prefix and the forwarded tail of a coordinate item, or a whole
// force item. Parts are emitted in a topological order of their waits
// (Kahn's algorithm) that prefers the lowest (domain, pulse) key, so the
// chunks of one domain's pulses sit close together in the list and run
// close together in time: the domain's slots are fetched into L2 once per
// launch instead of once per pulse.

struct Part {
  int item;
  int begin, end;       // entry range within the item's map
  int halo_src;
  long long key;        // emission priority (smaller first)
  std::vector<int> deps;          // items that must be complete before this part
  std::vector<std::vector<int>> chunk_waits;  // per chunk (fine waits) or one shared list
};

struct ItemInfo {
  int r, p, q;           // sender, pulse, receiver
  int64_t src, dst, map; // slot of sender base, slot of receive-range start, first map entry
  int size, split, dim, shift_flag;
};

// Sorted-array helpers for the fine waits.
bool any_in_range(const int32_t* a, int n, int64_t lo, int64_t hi) {   // any a[i] in [lo, hi)
  const int32_t* it = std::lower_bound(a, a + n, static_cast<int32_t>(std::min<int64_t>(lo, INT32_MAX)));
  return it != a + n && *it < hi;
}

bool sorted_intersect(const int32_t* a, int na, const int32_t* b, int nb) {
  int i = 0, k = 0;
  while (i < na && k < nb) {
    if (a[i] == b[k]) return true;
    if (a[i] < b[k]) ++i;
    else ++k;
  }
  return false;
}

// Emits parts in a locality-preferring topological order; returns the order.
std::vector<int> order_parts(const std::vector<Part>& parts, int n_items, std::vector<int>* item_parts_left) {
  std::vector<std::vector<int>> waiters(n_items);
  std::vector<int> unmet(parts.size(), 0);
  for (size_t i = 0; i < parts.size(); ++i) {
    unmet[i] = static_cast<int>(parts[i].deps.size());
    for (int it : parts[i].deps) waiters[it].push_back(static_cast<int>(i));
  }
  auto cmp = [&](int a, int b) { return parts[a].key > parts[b].key; };
  std::vector<int> heap;
  for (size_t i = 0; i < parts.size(); ++i)
    if (unmet[i] == 0) heap.push_back(static_cast<int>(i));
  std::make_heap(heap.begin(), heap.end(), cmp);
  std::vector<int> order;
  order.reserve(parts.size());
  while (!heap.empty()) {
    std::pop_heap(heap.begin(), heap.end(), cmp);
    const int i = heap.back();
    heap.pop_back();
    order.push_back(i);
    const int it = parts[i].item;
    if (--(*item_parts_left)[it] == 0) {
      for (int w : waiters[it]) {
        if (--unmet[w] == 0) {
          heap.push_back(w);
          std::push_heap(heap.begin(), heap.end(), cmp);
        }
      }
    }
  }
  return order;   // shorter than parts only if the waits had a cycle (they cannot)
}

// Work tables of the fused and unfused kernels from the host copy of the plan.
int build_tables(hx_ctx* h, cudaStream_t s) {
  const Plan& pl = h->pl;
  const int P = pl.n_pulses, nd = pl.ndom;
  const int n_items = P * nd;
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
  if (fine && h->total_entries > 0) {
    maps.resize(h->total_entries);
    HX_CUDA(cudaMemcpy(maps.data(), h->d_maps, sizeof(int32_t) * h->total_entries, cudaMemcpyDeviceToHost));
  }
  // upper_q(r): the domain that sends into r in pulse q
  auto upper = [&](int r, int q) { return neighbour(pl, r, pl.pulse_dim[q], +1); };

  for (int dir = 0; dir < 2; ++dir) {
    std::vector<Part> parts;
    auto chunks_of = [](int begin, int end) { return std::max(1, (end - begin + kChunk - 1) / kChunk); };
    if (dir == 0) {
      for (int p = 0; p < P; ++p)
        for (int r = 0; r < nd; ++r) {
          const int t = p * nd + r;
          const ItemInfo& it = items[t];
          if (it.split > 0 || it.size == 0) {
            Part a;
            a.item = t;
            a.begin = 0;
            a.end = it.split;
            a.halo_src = 0;
            a.key = (static_cast<long long>(r) * P + p) * 2;
            parts.push_back(std::move(a));
          }
          if (it.split < it.size) {
            Part b;
            b.item = t;
            b.begin = it.split;
            b.end = it.size;
            b.halo_src = 1;
            b.key = (static_cast<long long>(r) * P + p) * 2 + 1;
            // forwarded entries read r's receive ranges of pulses q < p
            const int nch = chunks_of(b.begin, b.end);
            std::vector<int> all;
            for (int q = 0; q < p; ++q) all.push_back(q * nd + upper(r, q));
            for (int c = 0; c < nch; ++c) {
              const int cb = b.begin + c * kChunk, ce = std::min(b.end, cb + kChunk);
              if (!fine) {
                b.chunk_waits.push_back(all);
                continue;
              }
              std::vector<int> w;
              const int32_t* m = maps.data() + it.map + cb;
              for (int q = 0; q < p; ++q) {
                const int64_t lo = h->t_off[q * nd + upper(r, q)];
                const int64_t hi = lo + h->t_size[q * nd + upper(r, q)];
                if (any_in_range(m, ce - cb, lo, hi)) w.push_back(q * nd + upper(r, q));
              }
              b.chunk_waits.push_back(w);
            }
            parts.push_back(std::move(b));
          }
        }
    } else {
      for (int p = P - 1; p >= 0; --p)
        for (int r = 0; r < nd; ++r) {
          const int t = p * nd + r;
          const ItemInfo& it = items[t];
          Part a;
          a.item = t;
          a.begin = 0;
          a.end = it.size;
          a.halo_src = 1;
          a.key = static_cast<long long>(r) * P + (P - 1 - p);
          const int nch = chunks_of(a.begin, a.end);
          std::vector<int> all;
          for (int pp = p + 1; pp < P; ++pp) {
            all.push_back(pp * nd + it.q);                       // writes of the slots read here
            if (ordered && it.q != r) all.push_back(pp * nd + r); // earlier adds into the same targets
          }
          for (int c = 0; c < nch; ++c) {
            const int cb = c * kChunk, ce = std::min(it.size, cb + kChunk);
            if (!fine) {
              a.chunk_waits.push_back(all);
              continue;
            }
            std::vector<int> w;
            const int64_t slot_lo = h->t_off[t] + cb, slot_hi = h->t_off[t] + ce;
            for (int pp = p + 1; pp < P; ++pp) {
              const int tq = pp * nd + it.q, tr = pp * nd + r;
              // q forwards some of the slots this chunk reads in pulse pp
              const bool need_q = any_in_range(maps.data() + items[tq].map, items[tq].size, slot_lo, slot_hi);
              // r adds into some of this chunk's targets in pulse pp
              const bool need_r = ordered && sorted_intersect(maps.data() + items[tr].map, items[tr].size,
                                                              maps.data() + it.map + cb, ce - cb);
              if (tq == tr) {
                if (need_q || need_r) w.push_back(tq);
              } else {
                if (need_q) w.push_back(tq);
                if (need_r) w.push_back(tr);
              }
            }
            a.chunk_waits.push_back(w);
          }
          parts.push_back(std::move(a));
        }
    }
    // deps per part; which items anybody waits for; drop unneeded empty parts
    std::vector<char> waited(std::max(n_items, 1), 0);
    for (auto& pt : parts) {
      std::vector<int> d;
      for (auto& w : pt.chunk_waits) d.insert(d.end(), w.begin(), w.end());
      std::sort(d.begin(), d.end());
      d.erase(std::unique(d.begin(), d.end()), d.end());
      pt.deps = d;
      for (int it : d) waited[it] = 1;
    }
    std::vector<Part> kept;
    for (auto& pt : parts)
      if (pt.end > pt.begin || waited[pt.item]) kept.push_back(std::move(pt));
    parts.swap(kept);
    std::vector<int> item_chunks(std::max(n_items, 1), 0), parts_left(std::max(n_items, 1), 0);
    for (auto& pt : parts) {
      item_chunks[pt.item] += chunks_of(pt.begin, pt.end);
      parts_left[pt.item] += 1;
    }
    std::vector<int> order = order_parts(parts, std::max(n_items, 1), &parts_left);
    if (order.size() != parts.size()) return HX_ERR_STATE;
    std::vector<Chunk> chunks;
    std::vector<Wait> waits;
    for (int pi : order) {
      const Part& pt = parts[pi];
      const ItemInfo& it = items[pt.item];
      const int nch = chunks_of(pt.begin, pt.end);
      for (int c = 0; c < nch; ++c) {
        const int cb = pt.begin + c * kChunk, ce = std::min(pt.end, cb + kChunk);
        Chunk ch;
        std::memset(&ch, 0, sizeof(ch));
        ch.src = it.src;
        ch.dst = it.dst + cb;
        ch.map = it.map + cb;
        ch.n = ce - cb;
        ch.item = pt.item;
        ch.item_chunks = item_chunks[pt.item];
        const std::vector<int>& w = pt.chunk_waits.empty() ? std::vector<int>() : pt.chunk_waits[c];
        ch.wait_off = static_cast<int32_t>(waits.size());
        ch.wait_cnt = static_cast<int32_t>(w.size());
        for (int x : w) waits.push_back({x, 0});
        ch.flags = (pt.halo_src ? kHaloSrc : 0) | (waited[pt.item] ? kSignal : 0) |
                   (dir == 0 && it.shift_flag ? kShift : 0);
        ch.dim = it.dim;
        ch.shift = pl.boxf[it.dim];
        chunks.push_back(ch);
      }
    }
    for (auto& w : waits) w.chunks = item_chunks[w.item];
    h->n_chunks[dir] = static_cast<int>(chunks.size());
    HX_CUDA(dev_alloc(&h->d_chunks[dir], chunks.size()));
    HX_CUDA(dev_alloc(&h->d_waits[dir], waits.size()));
    if (!chunks.empty())
      HX_CUDA(cudaMemcpy(h->d_chunks[dir], chunks.data(), sizeof(Chunk) * chunks.size(), cudaMemcpyHostToDevice));
    if (!waits.empty())
      HX_CUDA(cudaMemcpy(h->d_waits[dir], waits.data(), sizeof(Wait) * waits.size(), cudaMemcpyHostToDevice));
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

  const size_t n_flags = 2 * static_cast<size_t>(std::max(n_items, 1));
  HX_CUDA(dev_alloc(&h->d_flags, n_flags));
  HX_CUDA(dev_alloc(&h->d_blk, n_flags));
  HX_CUDA(dev_alloc(&h->d_ctrl, 2));
  // Persistent grid: every warp co-resident, one warp per chunk at most.
  for (int k = 0; k < 2; ++k) {
    const int per_sm = std::max(1, max_blocks_per_sm(kernel_for(h, k)));
    const int warps = std::max(1, std::min(h->n_chunks[k], per_sm * h->sm_count * kWarps));
    h->grid[k] = (warps + kWarps - 1) / kWarps;
  }
  return reset_signals(h, s);
}

struct BuildScratch {
  int32_t* dom_id = nullptr;
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
    dev_free(dom_id); dev_free(hist); dev_free(hist_scan); dev_free(err); dev_free(home_xyz);
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
  HX_CUDA(launch_cells(pos, n, pl.dims, pl.box, nd, b.dom_id, b.hist, ntiles, b.err, s));
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
  if (P > 0 && h->n_chunks[0] > 0) {
    rc = launch(h, 0, coords, s);
    if (rc != HX_OK) return rc;
  }
  HX_CUDA(cudaStreamSynchronize(s));
  return HX_OK;
}

}  // namespace

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
  if (h->pl.n_pulses == 0 || h->n_chunks[kind] == 0) return HX_OK;   // nothing moves
  const int rc = ensure_device(h);
  if (rc != HX_OK) return rc;
  return launch(h, kind, buf, static_cast<cudaStream_t>(stream));
}

}  // namespace

int hx_exchange_coords(hx_handle h, float* coords, void* stream) { return exchange(h, coords, stream, 0); }

int hx_exchange_forces(hx_handle h, float* forces, void* stream) { return exchange(h, forces, stream, 1); }

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
