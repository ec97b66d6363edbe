// Work tables of libhx, built on the host from the maps at map-build time:
// the fused kernels' chunk and unit lists with their waits, the per-pulse
// chunk lists of the unfused baseline, the resolved-mode tables and the
// range pieces of the host-buffer calls.
#include "hx_runtime.h"

#include <atomic>
#include <memory>

namespace hx_rt {

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

// The records in ascending key (ties by index) when that order is
// topological, else Kahn's order by the same keys (which then differs only
// where a record's key is below one of its producers'). A key that grows by
// a lag of whole resident windows per dependency stage makes the first case
// the usual one, and the keys span a small range: a counting sort, then one
// check of every dependency.
template <class Deps, class Key>
std::vector<int> key_order(int n, Deps deps, Key key) {
  std::vector<int> order(n);
  if (n == 0) return order;
  long long lo = key(0), hi = key(0);
  for (int i = 1; i < n; ++i) {
    lo = std::min(lo, key(i));
    hi = std::max(hi, key(i));
  }
  if (hi - lo > 4ll * n + (1ll << 20)) return kahn_order(n, deps, key);
  std::vector<int> first(static_cast<size_t>(hi - lo) + 2, 0);
  for (int i = 0; i < n; ++i) ++first[static_cast<size_t>(key(i) - lo) + 1];
  for (size_t k = 1; k < first.size(); ++k) first[k] += first[k - 1];
  for (int i = 0; i < n; ++i) order[first[static_cast<size_t>(key(i) - lo)]++] = i;   // stable: ties by index
  std::vector<int> pos(n);
  for (int k = 0; k < n; ++k) pos[order[k]] = k;
  for (int i = 0; i < n; ++i)
    for (int d : deps(i))
      if (pos[d] >= pos[i]) return kahn_order(n, deps, key);
  return order;
}

std::vector<int> order_chunks(const std::vector<Rec>& recs) {
  return key_order(
      static_cast<int>(recs.size()), [&](int i) -> const std::vector<int>& { return recs[i].deps; },
      [&](int i) { return recs[i].key; });
}

// An array of n records left uninitialised: the parallel fill that follows
// writes every byte of each record, and is also its first touch.
template <class T>
struct RecordArray {
  std::unique_ptr<T[]> p;
  size_t n;
  explicit RecordArray(size_t count) : p(new T[count ? count : 1]), n(count) {}
  T& operator[](size_t i) { return p[i]; }
  T* data() { return p.get(); }
  size_t size() const { return n; }
  bool empty() const { return n == 0; }
};

// Dependency depth of every record: 0 without producers, else one more than
// its deepest producer. Relaxation passes over all records: the depths settle
// within as many passes as the longest chain has links. False if they still
// change after `max_passes` (a cycle, which the waits cannot form).
template <class Deps>
bool dependency_depths(int n, Deps deps, std::vector<int>& depth, int max_passes) {
  depth.assign(n, 0);
  for (int pass = 0; pass <= max_passes; ++pass) {
    bool changed = false;
    for (int i = 0; i < n; ++i) {
      int v = 0;
      for (int d : deps(i)) v = std::max(v, depth[d] + 1);
      if (v != depth[i]) {
        depth[i] = v;
        changed = true;
      }
    }
    if (!changed) return true;
  }
  return false;
}

// ---------------------------------------------------------------- unit tables
//
// Each domain's array is cut into ranges (home, then the slots received in
// each pulse) and each range into units of up to max_slots slots. A unit gets
// one segment per (sender, pulse) map whose targets fall inside it, last
// pulse first. A unit waits for the units of its receivers that hold the
// slots it reads, when those units are themselves targets of later pulses.
// Units are listed with the same priority as the chunk lists (folded domain
// order, dependency depth, a lag of `lag` list positions per depth).

// The dependencies of a unit: a run of the unit list's dependency pool.
struct IntSpan {
  const int* b;
  const int* e;
  const int* begin() const { return b; }
  const int* end() const { return e; }
  size_t size() const { return static_cast<size_t>(e - b); }
};

struct TRec {
  int r;              // domain
  int range;          // -1 home, else the pulse whose received slots the unit holds
  int a, n;           // local index of the first slot, slot count
  int seg_begin, seg_cnt;   // its segments in the domain's segment pool (each with its pulse in `pad`)
  int64_t dep_begin;  // its dependencies (unit indices) in the dependency pool, segment by segment
  int dep_cnt;
  int stage = 0;
  long long key = 0;
};

int build_unit_tables(hx_ctx* h, const std::vector<ItemInfo>& items, const std::vector<int32_t>& maps,
                      const std::vector<int64_t>& rank, int max_slots, int max_entries, long long lag,
                      int slot_bytes, int map_bytes, int src_bytes, int dir) {
  const Plan& pl = h->pl;
  const int P = pl.n_pulses, nd = pl.ndom;
  if (dir != 1) return HX_ERR_STATE;   // the sweep serves the force exchange
  auto upper = [&](int r, int q) { return neighbour(pl, r, pl.pulse_dim[q], +1); };
  std::vector<std::vector<UnitSeg>> seg_pool;
  {
    // units of each domain, cut on all host cores, then listed domain after domain;
    // by_range: per (domain, range) the units' indices in slot order
    std::vector<std::vector<TRec>> per(nd);
    std::vector<std::vector<std::vector<int>>> by_range(nd, std::vector<std::vector<int>>(P + 1));
    // one pool of segments per domain (a unit refers to a run of its domain's
    // pool), so that cutting tens of thousands of units allocates per domain
    seg_pool.assign(nd, std::vector<UnitSeg>());
    parallel_for(nd, [&](size_t ri) {
      const int r = static_cast<int>(ri);
      {
        size_t est = 0;   // units before any split by entries
        for (int rg = -1; rg < P; ++rg) {
          const int len = rg < 0 ? h->home[r] : h->t_size[rg * nd + upper(r, rg)];
          est += static_cast<size_t>((len + max_slots - 1) / max_slots);
        }
        per[r].reserve(est + 1);
        seg_pool[r].reserve(est * static_cast<size_t>(P) + 1);
      }
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
        // Per pulse, the first map entry at or past slot a: the units of a
        // range advance through every map, so each unit costs one search per
        // pulse (for its end) from where the previous one ended.
        int cur[HX_MAX_PULSES], end[HX_MAX_PULSES];
        for (int p = 0; p < P; ++p) {
          const ItemInfo& it = items[p * nd + r];
          const int32_t* m = maps.data() + it.map;
          cur[p] = static_cast<int>(std::lower_bound(m, m + it.size, lo) - m);
        }
        // entries of every map of r in slots [a, b), with end[p] the first entry at or past b
        auto entries_to = [&](int b) {
          int e = 0;
          for (int p = 0; p < P; ++p) {
            const ItemInfo& it = items[p * nd + r];
            const int32_t* m = maps.data() + it.map;
            end[p] = static_cast<int>(std::lower_bound(m + cur[p], m + it.size, b) - m);
            e += end[p] - cur[p];
          }
          return e;
        };
        for (int a = lo, b = lo; a < lo + len; a = b) {
          // at most max_slots slots and max_entries entries (a slot has at most one entry per pulse)
          b = std::min(lo + len, a + max_slots);
          if (entries_to(b) > max_entries) {
            int good = a + 1, bad = b;
            while (bad - good > 1) {
              const int mid = good + (bad - good) / 2;
              if (entries_to(mid) <= max_entries) good = mid;
              else bad = mid;
            }
            b = good;
            entries_to(b);
          }
          TRec t;
          t.r = r;
          t.range = rg;
          t.a = a;
          t.n = b - a;
          t.seg_begin = static_cast<int>(seg_pool[r].size());
          t.seg_cnt = 0;
          for (int k = 0; k < P; ++k) {
            const int p = P - 1 - k;
            const ItemInfo& it = items[p * nd + r];
            if (it.size == 0) continue;
            const int i1 = cur[p], i2 = end[p];
            if (i2 <= i1) continue;
            UnitSeg sg;
            std::memset(&sg, 0, sizeof(sg));
            sg.map = it.map + i1;
            sg.other = it.dst + i1;
            sg.n = i2 - i1;
            sg.dim = it.dim;
            sg.shift = pl.boxf[it.dim];
            sg.do_shift = 0;
            sg.pad = p;   // the segment's pulse while the tables are built (cleared in the records)
            seg_pool[r].push_back(sg);
            ++t.seg_cnt;
          }
          for (int p = 0; p < P; ++p) cur[p] = end[p];
          if (t.seg_cnt == 0) continue;
          by_range[r][rg + 1].push_back(static_cast<int>(per[r].size()));
          per[r].push_back(std::move(t));
        }
      }
    }, 1);
    std::vector<TRec> recs;
    {
      size_t total = 0;
      for (int r = 0; r < nd; ++r) total += per[r].size();
      recs.reserve(total);
    }
    auto seg = [&](const TRec& t, int k) -> UnitSeg& { return seg_pool[t.r][static_cast<size_t>(t.seg_begin + k)]; };
    for (int r = 0; r < nd; ++r) {
      const int base = static_cast<int>(recs.size());
      for (auto& lst : by_range[r])
        for (int& i : lst) i += base;
      for (TRec& t : per[r]) recs.push_back(std::move(t));
    }
    per.clear();
    // Dependencies. The slots read by segment (r, p) are q's slots [other,
    // other + n) in q's range p; the units of q's range p that overlap them
    // are its producers. They are listed segment by segment (segments of one
    // unit read different ranges, so their producers differ), each segment
    // records how many are its own, and all units' lists share one pool:
    // counted on the host's cores, laid out by a prefix sum, then filled.
    auto producers = [&](const TRec& t, const UnitSeg& sk) {
      const int q = items[sk.pad * nd + t.r].q;
      const int64_t s0 = sk.other - h->dom_offset[q], s1 = s0 + sk.n;
      // q's units of range p, in slot order: the first one that ends past s0, then on while they start before s1
      const std::vector<int>& in_range = by_range[q][sk.pad + 1];
      auto lo_j = std::partition_point(in_range.begin(), in_range.end(),
                                       [&](int j) { return recs[j].a + recs[j].n <= s0; });
      auto hi_j = lo_j;
      while (hi_j != in_range.end() && recs[*hi_j].a < s1) ++hi_j;
      return std::make_pair(lo_j, hi_j);
    };
    parallel_for(recs.size(), [&](size_t i) {
      TRec& t = recs[i];
      t.dep_cnt = 0;
      for (int k = 0; k < t.seg_cnt; ++k) {
        UnitSeg& sk = seg(t, k);
        const auto range = producers(t, sk);
        sk.dep = static_cast<int32_t>(range.second - range.first);
        t.dep_cnt += sk.dep;
      }
    }, 64);
    std::vector<int> dep_pool;
    {
      int64_t total = 0;
      for (TRec& t : recs) {
        t.dep_begin = total;
        total += t.dep_cnt;
      }
      dep_pool.resize(static_cast<size_t>(total));
    }
    parallel_for(recs.size(), [&](size_t i) {
      const TRec& t = recs[i];
      int64_t w = t.dep_begin;
      for (int k = 0; k < t.seg_cnt; ++k) {
        const auto range = producers(t, seg(t, k));
        for (auto j = range.first; j != range.second; ++j) dep_pool[static_cast<size_t>(w++)] = *j;
      }
    }, 64);
    // dependency depth, then priority: base order + one resident window per depth
    {
      const int n = static_cast<int>(recs.size());
      auto deps_of = [&](int i) {
        const int* b = dep_pool.data() + recs[i].dep_begin;
        return IntSpan{b, b + recs[i].dep_cnt};
      };
      std::vector<int> depth;
      if (!dependency_depths(n, deps_of, depth, P + 1)) return HX_ERR_STATE;
      for (int i = 0; i < n; ++i) recs[i].stage = depth[i];
      // Base order: domains by rank, a domain's units by stage, then as they
      // were cut (range, then first slot), which is their order in `recs`.
      std::vector<int> doms(nd);
      for (int r = 0; r < nd; ++r) doms[r] = r;
      std::sort(doms.begin(), doms.end(), [&](int x, int y) { return rank[x] != rank[y] ? rank[x] < rank[y] : x < y; });
      std::vector<int> dom_first(nd + 1, 0);
      for (const TRec& t : recs) ++dom_first[t.r + 1];
      for (int r = 0; r < nd; ++r) dom_first[r + 1] += dom_first[r];
      long long k = 0;
      int max_stage = 0;
      for (const TRec& t : recs) max_stage = std::max(max_stage, t.stage);
      for (int r : doms)
        for (int st = 0; st <= max_stage; ++st)
          for (int i = dom_first[r]; i < dom_first[r + 1]; ++i)
            if (recs[i].stage == st) recs[i].key = k++ + lag * st;
      std::vector<int> order = key_order(n, deps_of, [&](int i) { return recs[i].key; });
      if (order.size() != recs.size()) return HX_ERR_STATE;
      std::vector<int> pos(recs.size());
      for (size_t q = 0; q < order.size(); ++q) pos[order[q]] = static_cast<int>(q);
      std::vector<char> waited(recs.size(), 0);
      for (int d : dep_pool) waited[d] = 1;
      // records in list order, filled on the host's cores: each one's share of
      // the overflow segments and of the wait list comes from prefix sums
      std::vector<int64_t> seg_at(n + 1, 0), wait_at(n + 1, 0);
      for (int q = 0; q < n; ++q) {
        const TRec& t = recs[order[q]];
        seg_at[q + 1] = seg_at[q] + std::max<int64_t>(0, static_cast<int64_t>(t.seg_cnt) - kInlineSegs);
        wait_at[q + 1] = wait_at[q] + t.dep_cnt;
      }
      RecordArray<Unit> units(n);
      std::vector<UnitSeg> segs(seg_at[n]);   // segments past kInlineSegs
      std::vector<Wait> waits(wait_at[n]);
      std::atomic<bool> fits{true};
      parallel_for(static_cast<size_t>(n), [&](size_t q) {
        const int i = order[q];
        const TRec& t = recs[i];
        Unit& u = units[q];
        std::memset(&u, 0, sizeof(u));
        u.base = h->dom_offset[t.r] + t.a;
        u.n = t.n;
        u.local_a = t.a;
        u.seg_cnt = static_cast<int32_t>(t.seg_cnt);
        u.extra_off = static_cast<int32_t>(seg_at[q]);
        // stage regions: each run's region starts on a 16-byte boundary and is 16 bytes longer than the run
        int moff = slot_bytes, soff = slot_bytes + map_bytes;
        for (int g = 0; g < t.seg_cnt; ++g) {
          UnitSeg sg = seg(t, g);
          sg.pad = 0;
          sg.map_off = moff;
          sg.src_off = soff;
          moff += ((4 * sg.n + 15) & ~15) + 16;
          soff += ((12 * sg.n + 15) & ~15) + 16;
          if (static_cast<int>(g) < kInlineSegs) u.seg[g] = sg;
          else segs[u.extra_off + g - kInlineSegs] = sg;
        }
        // the stage regions must fit the kernel's buffer
        if (moff > slot_bytes + map_bytes || soff > slot_bytes + map_bytes + src_bytes)
          fits.store(false, std::memory_order_relaxed);
        u.wait_off = static_cast<int32_t>(wait_at[q]);
        u.wait_cnt = static_cast<int32_t>(t.dep_cnt);
        const int* deps = dep_pool.data() + t.dep_begin;
        for (int w = 0; w < u.wait_cnt; ++w) waits[u.wait_off + w] = {pos[deps[w]], 1};
        for (int w = 0; w < std::min(u.wait_cnt, kInlineWaits); ++w) u.wait_inline[w] = waits[u.wait_off + w];
        u.flags = waited[i] ? kSignal : 0;
        u.item = seg(t, 0).pad * nd + t.r;
        for (int g = 0; g < t.seg_cnt; ++g) u.entries += seg(t, g).n;
      }, 64);
      if (!fits.load()) return HX_ERR_STATE;
      h->n_units[dir] = static_cast<int>(units.size());
      HX_CUDA(dev_alloc(&h->d_units[dir], units.size()));
      HX_CUDA(dev_alloc(&h->d_segs[dir], segs.size()));
      HX_CUDA(dev_alloc(&h->d_twaits[dir], waits.size()));
      if (!units.empty())
        HX_CUDA(cudaMemcpy(h->d_units[dir], units.data(), sizeof(Unit) * units.size(), cudaMemcpyHostToDevice));
      if (!segs.empty())
        HX_CUDA(cudaMemcpy(h->d_segs[dir], segs.data(), sizeof(UnitSeg) * segs.size(), cudaMemcpyHostToDevice));
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
  int64_t packed_home = 0, packed_halo = 0;   // words of each table's ranges laid end to end so far
  auto cut = [](std::vector<CopyChunk>& out, int64_t& packed, int64_t first_slot, int64_t slots) {
    for (int64_t w = 0; w < 3 * slots; w += kCopyChunkWords) {
      CopyChunk c;
      c.word = 3 * first_slot + w;
      c.packed = packed + w;
      c.n = static_cast<int32_t>(std::min<int64_t>(kCopyChunkWords, 3 * slots - w));
      c.pad = 0;
      out.push_back(c);
    }
    packed += 3 * slots;
  };
  for (int r = 0; r < h->pl.ndom; ++r) {
    cut(home, packed_home, h->dom_offset[r], h->home[r]);
    cut(halo, packed_halo, h->dom_offset[r] + h->home[r], h->halo[r]);
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

#ifndef HX_SWEEP_LAG_WINDOWS
#define HX_SWEEP_LAG_WINDOWS 8
#endif
constexpr long long kSweepLagWindows = HX_SWEEP_LAG_WINDOWS;   // resident-warp windows per dependency stage

#ifndef HX_CHUNK_LAG_WINDOWS
#define HX_CHUNK_LAG_WINDOWS 1
#endif
// Resident-warp windows by which a chunk of dependency stage s is placed
// after stage s - 1 in the chunk list (its priority key grows by that many
// windows per stage).
constexpr long long kChunkLagWindows = HX_CHUNK_LAG_WINDOWS;

#ifndef HX_FUSED_CHUNK
#define HX_FUSED_CHUNK 0   // 0: chosen per direction from the work (below)
#endif
// Entries per chunk of the fused chunk kernels of direction dir: the
// smallest power of two from 32 to kChunk with which the resident warps
// hold every coordinate chunk at once, or every force chunk two deep. A
// chunk issues all its gathers before any store, so one chunk per warp
// beats two half chunks in sequence; a force chunk waits for the later-pulse
// chunks that add into its slots, and halving it halves what it waits for.
// Measured on one GB300 (us per step back to back, chunks with programmatic
// launch): 31.7k entries on 8 domains 18.4 at 256 entries, 15.2 at 32;
// 0.83M entries on 64 domains 31.8 at 256, 27.9 at 128, 55 at 32.
static int fused_chunk_entries(const hx_ctx* h, int dir) {
  if (HX_FUSED_CHUNK > 0) return std::min(HX_FUSED_CHUNK, kChunk);
  const int64_t warps = std::max<int64_t>(1, static_cast<int64_t>(h->grid[dir]) * kWarps) * (dir == 0 ? 1 : 2);
  const int64_t per_warp = (h->total_entries + warps - 1) / warps;
  int n = 32;
  while (n < kChunk && n < per_warp) n *= 2;
  return n;
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
  if (h->total_entries > 0) {   // chunk records carry their map runs; fine waits, units and resolved tables read them
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
  h->family[0] = (h->flags & HX_FLAG_RESOLVED) ? kFamResolved
                                                : kFamChunks;
  h->family[1] = (h->flags & HX_FLAG_SWEEP_FORCES) ? kFamSweep : h->family[0];
  for (int k = 0; k < 2; ++k) {
    const int per_sm = std::max(1, h->family[k] == kFamSweep   ? sweep_blocks_per_sm(k)
                                   : h->family[k] == kFamResolved ? 1
                                                                 : max_blocks_per_sm(kernel_for(h, k), fused_smem(h, k)));
    h->grid[k] = per_sm * h->sm_count;   // upper bound; trimmed to the work count below
  }
  // Unit lists. A dependent unit is placed a few resident windows after the
  // units it waits for: eight units per resident warp (measured on the
  // 12M-atom workload with an earlier sweep: lags of 2, 3, 4, 6 and 10
  // windows gave forces in 112.6, 100.5, 94.2, 92.2 and 92.2 us; with the
  // current one, 2 and 4 windows 81.7 and 79.5 us against 78.5 at 8).
  for (int dir = 0; dir < 2; ++dir) {
    int rc = HX_OK;
    if (h->family[dir] == kFamSweep) {
      if (P > kSweepSegs) return HX_ERR_PULSES;   // a unit's runs must fit one warp's stage
      rc = build_unit_tables(h, items, maps, rank, kSweepSlots, kSweepEntries,
                             kSweepLagWindows * h->grid[dir] * kWarps,
                             kSweepSlotBytes, kSweepMapBytes, kSweepSrcBytes, dir);
    }
    if (rc != HX_OK) return rc;
  }

  for (int dir = 0; dir < 2; ++dir) {
    if (h->family[dir] != kFamChunks) continue;
    std::vector<Rec> recs;
    std::vector<std::vector<int>> item_recs(std::max(n_items, 1));   // chunk records of each item, in entry order
    const int cut = fused_chunk_entries(h, dir);
    auto add_part = [&](int t, int begin, int end, int halo_src, int stage, bool keep_empty) {
      if (end <= begin && !keep_empty) return;
      for (int b = begin;; b += cut) {
        Rec rc;
        rc.item = t;
        rc.begin = b;
        rc.end = std::min(end, b + cut);
        rc.halo_src = halo_src;
        rc.stage = stage;
        rc.key = 0;
        item_recs[t].push_back(static_cast<int>(recs.size()));
        recs.push_back(std::move(rc));
        if (b + cut >= end) break;
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
      // Records were cut pulse by pulse, each pulse domain by domain, so a
      // domain's records of one stage are already in (pulse, entry) order: a
      // counting sort by (domain rank, stage) keeps that order.
      std::vector<int> dom_pos(nd);
      {
        std::vector<int> doms(nd);
        for (int r = 0; r < nd; ++r) doms[r] = r;
        std::sort(doms.begin(), doms.end(),
                  [&](int x, int y) { return rank[x] != rank[y] ? rank[x] < rank[y] : x < y; });
        for (int q = 0; q < nd; ++q) dom_pos[doms[q]] = q;
      }
      int n_stages = 1;
      for (const Rec& rc : recs) n_stages = std::max(n_stages, rc.stage + 1);
      std::vector<int> first(static_cast<size_t>(nd) * n_stages + 1, 0);
      auto bucket = [&](const Rec& rc) { return static_cast<size_t>(dom_pos[items[rc.item].r]) * n_stages + rc.stage; };
      for (const Rec& rc : recs) ++first[bucket(rc) + 1];
      for (size_t q = 1; q < first.size(); ++q) first[q] += first[q - 1];
      std::vector<int> base(recs.size());
      for (size_t i = 0; i < recs.size(); ++i) base[first[bucket(recs[i])]++] = static_cast<int>(i);
      const long long window = static_cast<long long>(h->grid[dir]) * kWarps * kChunkLagWindows;
      for (size_t k = 0; k < base.size(); ++k)
        recs[base[k]].key = static_cast<long long>(k) + window * recs[base[k]].stage;
    }
    std::vector<int> order = order_chunks(recs);
    if (order.size() != recs.size()) return HX_ERR_STATE;
    std::vector<int> pos(recs.size());
    for (size_t k = 0; k < order.size(); ++k) pos[order[k]] = static_cast<int>(k);
    std::vector<int> item_chunks(std::max(n_items, 1), 0);
    for (auto& rc : recs) item_chunks[rc.item] += 1;
    // records in list order, filled on the host's cores (wait-list offsets from a prefix sum)
    const size_t nc = order.size();
    std::vector<int64_t> wait_at(nc + 1, 0);
    for (size_t k = 0; k < nc; ++k) wait_at[k + 1] = wait_at[k] + static_cast<int64_t>(recs[order[k]].wait.size());
    RecordArray<ChunkSlot> chunks(nc);
    std::vector<Wait> waits(wait_at[nc]);
    parallel_for(nc, [&](size_t k) {
      const int ri = order[k];
      const Rec& rc = recs[ri];
      const ItemInfo& it = items[rc.item];
      ChunkSlot& slot = chunks[k];
      std::memset(&slot, 0, sizeof(slot));
      Chunk& ch = slot.rec;
      ch.src = it.src;
      ch.dst = it.dst + rc.begin;
      ch.map = it.map + rc.begin;
      ch.n = rc.end - rc.begin;
      ch.item = rc.item;
      ch.item_chunks = item_chunks[rc.item];
      ch.wait_off = static_cast<int32_t>(wait_at[k]);
      ch.wait_cnt = static_cast<int32_t>(rc.wait.size());
      for (int w = 0; w < ch.wait_cnt; ++w) {
        const int x = rc.wait[w];
        waits[ch.wait_off + w] = fine ? Wait{pos[x], 1} : Wait{x, item_chunks[x]};
      }
      const bool sig = fine ? rec_waited[ri] != 0 : item_waited[rc.item] != 0;
      ch.flags = (rc.halo_src ? kHaloSrc : 0) | (sig ? kSignal : 0) | (dir == 0 && it.shift_flag ? kShift : 0);
      ch.dim = it.dim;
      ch.shift = pl.boxf[it.dim];
      if (ch.n > 0) std::memcpy(slot.map, maps.data() + ch.map, sizeof(int32_t) * ch.n);
      // the first waits of the chunk inside its record
      for (int w = 0; w < std::min(ch.wait_cnt, kWaitSlots); ++w) slot.waits[w] = waits[ch.wait_off + w];
    }, 64);
    h->n_chunks[dir] = static_cast<int>(chunks.size());
    HX_CUDA(dev_alloc(&h->d_chunks[dir], chunks.size()));
    HX_CUDA(dev_alloc(&h->d_waits[dir], waits.size()));
    if (!chunks.empty())
      HX_CUDA(cudaMemcpy(h->d_chunks[dir], chunks.data(), sizeof(ChunkSlot) * chunks.size(), cudaMemcpyHostToDevice));
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
  HX_CUDA(dev_alloc(&h->d_status, 2));
  // Persistent grid: every warp co-resident, and no more of them than there
  // is work.
  for (int k = 0; k < 2; ++k) {
    if (h->family[k] == kFamResolved) {
      // coordinates: one block per halo segment; forces: general blocks, then record blocks
      const int64_t n = h->n_res_pairs + h->n_res_quads;
      const int64_t fb = resolved_blocks(n, resolved_per_thread(h, n, kResTreesPerThread)) +
                         resolved_blocks(h->n_res_trees, 1);
      h->grid[k] = static_cast<int>(std::max<int64_t>(1, k == 0 ? h->n_res_segs : fb));
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

}  // namespace hx_rt
