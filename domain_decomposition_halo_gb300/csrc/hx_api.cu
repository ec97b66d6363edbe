// Host runtime and C-ABI of libhx: decomposition plan, map-build driver,
// launch parameters, CUDA-graph launch cache, status. The work tables the
// build derives from the maps are in hx_tables.cu.
//
// The plan follows "A Practical Guide to GPU-Initiated Communication for
// Molecular Dynamics at Scale": pulses numbered globally Z -> Y -> X
// (section "Dependency-aware packing"); a dependent tail that waits for every
// earlier pulse into its sender; forces in reverse pulse order (section
// "Force halo exchange: Reversing the dependency chain").
#include "hx_runtime.h"

namespace hx_rt {

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
  dev_free(h->d_pack);
  h->pack_slots = 0;
  for (int k = 0; k < 2; ++k) {
    dev_free(h->d_units[k]);
    dev_free(h->d_segs[k]);
    dev_free(h->d_twaits[k]);
    h->n_units[k] = 0;
  }
  dev_free(h->d_flags);
  dev_free(h->d_blk);
  dev_free(h->d_ctrl);
  dev_free(h->d_status);
  h->built = false;
}


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
  // The slot sweep's persistent grid must be wholly resident. Scheduled
  // while the coordinate blocks still run, some SMs were measured to take
  // only two of its three blocks per SM once those blocks had gone (18-22 of
  // 456 blocks on the 12M-atom workload started only after other sweep
  // blocks finished, and waits on their units ran out). Scheduled as the
  // coordinate blocks exit, it lands on empty SMs.
  P.late_dependents = (dir == 0 && h->family[1] == kFamSweep) ? 1 : 0;
  P.timeout_ns = h->timeout_ns;
  return P;
}

const void* kernel_for(hx_ctx* h, int kind) {
  const int mode = (h->flags & HX_FLAG_FINE_WAITS) ? kChunkFlag : kLastArrival;
  if (kind == 0) return coords_kernel(mode, (h->flags & HX_FLAG_BULK_STORE) != 0);
  if (kind == 1) return forces_kernel(mode, !(h->flags & HX_FLAG_UNORDERED_FORCES));
  return noop_kernel();
}

UnitParams unit_params(hx_ctx* h, int dir) {
  UnitParams P;
  std::memset(&P, 0, sizeof(P));
  P.units = h->d_units[dir];
  P.extra = h->d_segs[dir];
  P.waits = h->d_twaits[dir];
  P.maps = h->d_maps;
  P.flags = h->d_flags + static_cast<size_t>(dir) * h->n_flags;
  P.ctrl = h->d_ctrl + dir;
  P.n_units = static_cast<unsigned long long>(h->n_units[dir]);
  P.direction = dir;
  // Segment-by-segment waits where each warp has few units, so that the
  // pulse chain bounds the launch; whole-unit waits where each warp has many
  // and its producers are mostly done by the time it reaches a dependent unit.
  // Measured on one GB300 (forces back to back): 8 domains 11.0 -> 9.2 us and
  // 64 domains 18.1 -> 15.7 us with segment waits (about 1.6 units a warp);
  // 256 domains (16 units a warp) 78.2 -> 79.2 us, so it keeps unit waits.
  P.seg_waits = h->sweep_waits == 1   ? 1
                : h->sweep_waits == 2 ? 0
                                      : (h->n_units[dir] <= kSegWaitUnitsPerWarp * h->grid[dir] * kWarps ? 1 : 0);
  P.timeout_ns = h->timeout_ns;
  return P;
}

// Work items of the fused list of direction `dir`: units or chunks.
int work_items(const hx_ctx* h, int dir) {
  if (h->family[dir] == kFamResolved)
    return static_cast<int>(dir == 0 ? h->n_res_halo : h->n_res_pairs + h->n_res_quads + h->n_res_trees);
  return h->family[dir] == kFamChunks ? h->n_chunks[dir] : h->n_units[dir];
}

// Launch shape of a direction's fused kernel.
const void* fused_kernel(hx_ctx* h, int dir) {
  if (h->family[dir] == kFamSweep) return sweep_kernel(dir);
  if (h->family[dir] == kFamResolved) return resolved_kernel(dir);
  return kernel_for(h, dir);
}
unsigned fused_threads(const hx_ctx* h, int dir) {
  if (h->family[dir] == kFamResolved) return kResThreads;
  return kThreads;
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

size_t fused_smem(const hx_ctx* h, int dir) {
  if (h->family[dir] == kFamSweep) return sweep_smem_bytes(dir);
  if (h->family[dir] == kFamChunks) return chunk_smem_bytes(dir, dir == 0 && (h->flags & HX_FLAG_BULK_STORE));
  return 0;
}

// Launch a fused exchange (kind 0/1) or the no-op (kind 2): directly, or via
// a cached single-node graph keyed by (kind, buffer pointer).
int launch(hx_ctx* h, int kind, float* buf, cudaStream_t s) {
  DirParams P;
  UnitParams TP;
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
  } else if (kind != 2 && h->family[kind] != kFamChunks) {
    TP = unit_params(h, kind);
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
    smem = fused_smem(h, kind);
  }
  if (h->flags & HX_FLAG_PDL) {
    // Direct launch that may start while the stream's previous kernel
    // finishes; every exchange kernel waits for it (griddepcontrol.wait)
    // before touching data. The empty kernel (kind 2) is launched the same
    // way, so that launch floors are measured like the exchanges.
    cudaLaunchAttribute attr[1];
    std::memset(attr, 0, sizeof(attr));
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const unsigned n_attr = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
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

}  // namespace hx_rt

// ------------------------------------------------------------------ scratch-free launch

const void* hx::static_kernel(const hx_ctx* h) {
  if (!h->built || h->pl.n_pulses == 0) return nullptr;
  hx_ctx* m = const_cast<hx_ctx*>(h);
  if (h->family[0] == kFamResolved) return resolved_kernel(0);
  return kernel_for(m, 0);
}

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
  // flags are indexed by item (pulse signals) or by list position (chunk signals)
  const size_t need = std::max<size_t>(static_cast<size_t>(h->pl.n_pulses) * h->pl.ndom, static_cast<size_t>(work));
  if (need > max_flags) return HX_ERR_CAPACITY;
  HX_CUDA(cudaMemsetAsync(ctrl, 0, sizeof(Ctrl), s));
  // the handle's fault-injection item (hx_debug_drop_signal; -1: none), device to device
  HX_CUDA(cudaMemcpyAsync(&ctrl->drop_item, &h->d_ctrl[0].drop_item, sizeof(int), cudaMemcpyDeviceToDevice, s));
  HX_CUDA(cudaMemsetAsync(flags, 0, sizeof(unsigned long long) * need, s));
  HX_CUDA(cudaMemsetAsync(arrivals, 0, sizeof(unsigned int) * need, s));
  DirParams P = dir_params(h, 0);   // the chunk kernel, on the given scratch
  P.flags = flags;
  P.arrivals = arrivals;
  P.ctrl = ctrl;
  void* args[2] = {&coords, &P};
  return to_err(cudaLaunchKernel(kernel_for(h, 0), dim3(static_cast<unsigned>(h->grid[0])), dim3(kThreads), args,
                                fused_smem(h, 0), s));
}

// ------------------------------------------------------------------ C ABI

namespace {

// hx_status_async: the first direction's sticky status that is not HX_OK
// (else HX_OK) and its detail, for one copy to the host in stream order.
__global__ void k_status(const Ctrl* c, int* out) {
  int st = 0, det = -1;
  for (int k = 0; k < 2; ++k)
    if (st == 0 && c[k].status != 0) {
      st = c[k].status;
      det = c[k].detail;
    }
  out[0] = st;
  out[1] = det;
}

}  // namespace

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
  if (flags & ~HX_FLAGS_ALL) return HX_ERR_ARG;
  Plan pl;
  int rc = make_plan(box, dims, cutoff, &pl);
  if (rc != HX_OK) return rc;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return HX_ERR_CUDA;
  DeviceGuard guard(device);
  if (!guard.ok()) return HX_ERR_CUDA;
  hx_ctx* h = new (std::nothrow) hx_ctx();
  if (!h) return HX_ERR_NOMEM;
  h->pl = pl;
  h->device = device;
  // the slot sweep serves the forces of the chunk modes; resolved mode has its own force pass
  if ((flags & HX_FLAG_SWEEP_FORCES) && (flags & HX_FLAG_RESOLVED)) {
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  free_tables(h);
  const int rc = build(h, pos_in, n_atoms, coords, capacity, s);
  if (rc == HX_OK || rc == HX_ERR_CAPACITY) {
    if (needed) *needed = h->total_slots;
    static_prepare(h);   // on failure the static call reports HX_ERR_CUDA; the regular path is unaffected
    return rc;
  }
  free_tables(h);
  return rc;
}

namespace {

int exchange(hx_handle h, float* buf, void* stream, int kind) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (!buf && h->total_slots > 0) return HX_ERR_ARG;   // an empty layout touches no memory
  if (h->pl.n_pulses == 0 || work_items(h, kind) == 0) return HX_OK;   // nothing moves
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  int rc = HX_OK;
  float* hv = nullptr;
  if ((rc = device_view(host, &hv)) != HX_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == 0) {   // home coordinates in, halo coordinates out
    HX_CUDA(launch_copy_chunks(hv, dev, h->d_home_chunks, h->n_home_chunks, kCopySame, s));
    if ((rc = exchange(h, dev, stream, 0)) != HX_OK) return rc;
    HX_CUDA(launch_copy_chunks(dev, hv, h->d_halo_chunks, h->n_halo_chunks, kCopySame, s));
  } else {           // every slot's force in, home forces out
    HX_CUDA(cudaMemcpyAsync(dev, host, sizeof(float) * 3 * h->total_slots, cudaMemcpyHostToDevice, s));
    if ((rc = exchange(h, dev, stream, 1)) != HX_OK) return rc;
    HX_CUDA(launch_copy_chunks(dev, hv, h->d_home_chunks, h->n_home_chunks, kCopySame, s));
  }
  return HX_OK;
}

// The packed form: one copy-engine transfer each way over the host link, the
// scatter into the layout and the gather out of it as range copies in HBM
// through the handle's packing buffer.
int exchange_host_packed(hx_handle h, const float* in, float* out, float* dev, void* stream, int kind) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (h->total_slots == 0) return HX_OK;
  const int64_t n_home = h->n_atoms, n_halo = h->total_slots - h->n_atoms;
  if (!dev || (!in && (kind == 1 || n_home > 0)) || (!out && (kind == 1 ? n_home > 0 : n_halo > 0)))
    return HX_ERR_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  const int64_t need = std::max<int64_t>(1, std::max(n_home, n_halo));
  if (h->pack_slots < need) {
    // The first packed call after a build allocates the buffer; it is kept
    // until the next build or hx_destroy.
    dev_free(h->d_pack);
    h->pack_slots = 0;
    if (dev_alloc(&h->d_pack, 3 * need) != cudaSuccess) {
      cudaGetLastError();
      return HX_ERR_NOMEM;
    }
    h->pack_slots = need;
  }
  int rc = HX_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == 0) {   // packed home coordinates in, packed halo coordinates out
    if (n_home > 0) {
      HX_CUDA(cudaMemcpyAsync(h->d_pack, in, sizeof(float) * 3 * n_home, cudaMemcpyHostToDevice, s));
      HX_CUDA(launch_copy_chunks(h->d_pack, dev, h->d_home_chunks, h->n_home_chunks, kCopyUnpack, s));
    }
    if ((rc = exchange(h, dev, stream, 0)) != HX_OK) return rc;
    if (n_halo > 0) {
      HX_CUDA(launch_copy_chunks(dev, h->d_pack, h->d_halo_chunks, h->n_halo_chunks, kCopyPack, s));
      HX_CUDA(cudaMemcpyAsync(out, h->d_pack, sizeof(float) * 3 * n_halo, cudaMemcpyDeviceToHost, s));
    }
  } else {           // every slot's force in (the layout), packed home forces out
    HX_CUDA(cudaMemcpyAsync(dev, in, sizeof(float) * 3 * h->total_slots, cudaMemcpyHostToDevice, s));
    if ((rc = exchange(h, dev, stream, 1)) != HX_OK) return rc;
    if (n_home > 0) {
      HX_CUDA(launch_copy_chunks(dev, h->d_pack, h->d_home_chunks, h->n_home_chunks, kCopyPack, s));
      HX_CUDA(cudaMemcpyAsync(out, h->d_pack, sizeof(float) * 3 * n_home, cudaMemcpyDeviceToHost, s));
    }
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

int hx_exchange_coords_host_packed(hx_handle h, const float* home_host, float* halo_host, float* coords_dev,
                                   void* stream) {
  return exchange_host_packed(h, home_host, halo_host, coords_dev, stream, 0);
}

int hx_exchange_forces_host_packed(hx_handle h, const float* forces_host, float* home_forces_host, float* forces_dev,
                                   void* stream) {
  return exchange_host_packed(h, forces_host, home_forces_host, forces_dev, stream, 1);
}

int hx_exchange_coords_unfused(hx_handle h, float* coords, void* stream) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  if (!coords && h->total_slots > 0) return HX_ERR_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  int rc = HX_OK;
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  int rc = HX_OK;
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  return to_err(cudaMemcpyAsync(home_ids, h->d_home_ids, sizeof(int32_t) * h->n_atoms, cudaMemcpyDeviceToDevice,
                                static_cast<cudaStream_t>(stream)));
}

int hx_get_maps(hx_handle h, int32_t* maps_host, int64_t cap, int64_t* table_host) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_ERR_STATE;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
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
  int st = 0, det = -1;   // the handle's last call of hx_exchange_coords_static, if it is the device's last
  if (static_status(h, &st, &det) != HX_OK) return HX_ERR_CUDA;
  if (st != 0 && detail) *detail = det;
  return st;
}

int hx_status_async(hx_handle h, int* status_host, void* stream) {
  if (!h || !status_host) return HX_ERR_ARG;
  if (!h->built) {
    status_host[0] = HX_OK;
    status_host[1] = -1;
    return HX_OK;
  }
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_status<<<1, 1, 0, s>>>(h->d_ctrl, h->d_status);
  HX_CUDA(cudaGetLastError());
  HX_CUDA(cudaMemcpyAsync(status_host, h->d_status, 2 * sizeof(int), cudaMemcpyDeviceToHost, s));
  return HX_OK;
}

int hx_clear_status(hx_handle h, void* stream) {
  if (!h) return HX_ERR_ARG;
  if (!h->built) return HX_OK;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HX_ERR_CUDA;
  if (static_clear(h, s) != HX_OK) return HX_ERR_CUDA;
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
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return HX_ERR_CUDA;
  Ctrl* c = h->d_ctrl + direction;
  if (cudaMemcpy(&c->drop_item, &item, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return HX_ERR_CUDA;
  return HX_OK;
}

int hx_debug_sweep_waits(hx_handle h, int mode) {
  if (!h || mode < 0 || mode > 2) return HX_ERR_ARG;
  DeviceGuard guard(h->device);
  if (!guard.ok()) return HX_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return HX_ERR_CUDA;
  h->sweep_waits = mode;
  drop_graphs(h);   // cached graphs hold the launch parameters of the previous choice
  return HX_OK;
}

void hx_destroy(hx_handle h) {
  if (!h) return;
  DeviceGuard guard(h->device);
  if (guard.ok()) cudaDeviceSynchronize();
  static_forget(h);
  free_tables(h);
  delete h;
}

}  // extern "C"
