// Launch-time tile schedule for the persistent attention kernels.
//
// A kernel launch runs min(tiles, SMs) CTAs, each walking a fixed list of
// work tiles, so the launch lasts as long as its busiest CTA.  A tile of n
// blocks costs 8n + 12 (in eighths of a block: about one and a half blocks
// of per-tile work).  Two assignments are built: the greedy one (each tile,
// longest first, to the CTA with the least work so far) and MULTIFIT
// (Coffman, Garey and Johnson, "An application of bin-packing to
// multiprocessor scheduling", 1978): the smallest CTA capacity, found by
// bisection, under which first-fit decreasing places every tile.  The
// greedy one is kept unless MULTIFIT's maximum is at least 3% lower: its
// waves of similar tiles (the same rows of the heads of a KV group at the
// same time) share K/V and Q/dO through L2, and with many tiles per CTA it
// balances within about 1%.  With few tiles per CTA and a few sizes
// repeated (the dK/dV tiles of a causal mask: every key block once per KV
// head) it leaves the busiest CTAs ~7% above the mean, and MULTIFIT ~0.4%.
// Each CTA walks its tiles longest first.  Built schedules are kept per
// (row lengths, row order, configuration) for the process, so a mask
// compiled again (every training step) finds its schedule built.
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <iterator>
#include <list>
#include <mutex>

#include "internal.h"

namespace bsa {

namespace {

// A work tile: {row, blocks, b * n_g + g, split}.
struct Tile {
  int32_t i, n, bg, sp;
};

// First-fit decreasing of the tiles (already longest first) into `grid`
// CTAs of capacity `cap`: each tile to the lowest-numbered CTA it fits in,
// found in a segment tree of the CTAs' loads (minimum per node).  False if
// some tile fits nowhere; else the owners and the largest load.
bool first_fit(const std::vector<Tile>& tiles, int32_t grid, int64_t cap, std::vector<int32_t>* owner, int64_t* mx) {
  int32_t leaves = 1;
  while (leaves < grid) leaves <<= 1;
  const int64_t kFull = INT64_MAX / 4;
  std::vector<int64_t> tree(2 * static_cast<size_t>(leaves), kFull);
  for (int32_t c = 0; c < grid; ++c) tree[static_cast<size_t>(leaves + c)] = 0;
  for (int32_t v = leaves - 1; v >= 1; --v) tree[v] = std::min(tree[2 * v], tree[2 * v + 1]);
  int64_t top = 0;
  for (size_t k = 0; k < tiles.size(); ++k) {
    const int64_t w = 8 * static_cast<int64_t>(tiles[k].n) + 12;
    if (tree[1] > cap - w) return false;
    int32_t v = 1;
    while (v < leaves) v = tree[2 * v] <= cap - w ? 2 * v : 2 * v + 1;
    tree[v] += w;
    top = std::max(top, tree[v]);
    (*owner)[k] = v - leaves;
    for (v >>= 1; v >= 1; v >>= 1) tree[v] = std::min(tree[2 * v], tree[2 * v + 1]);
  }
  *mx = top;
  return true;
}

}  // namespace

bsa_status schedule_lists(const int32_t* row_len, const int32_t* row_order, int32_t rows, int32_t heads,
                          int32_t n_b, int32_t n_g, int32_t group, int32_t splits, int32_t grid,
                          std::vector<int4>* flat, int32_t* stride) {
  if (grid <= 0 || rows <= 0 || n_b <= 0 || n_g <= 0 || group <= 0 || splits <= 0 || group % splits)
    return fail(BSA_ERR_INVALID_ARG, "empty tile schedule");
  const int32_t gs = group / splits;  // mask heads of one split
  // tiles in longest-first order
  std::vector<Tile> tiles;
  tiles.reserve(static_cast<size_t>(rows) * n_b * n_g);
  if (heads == 1) {
    // rows by decreasing length (row_order), each for every (b, g)
    for (int32_t rank = 0; rank < rows; ++rank) {
      const int32_t i = row_order[rank];
      const int32_t n = row_len[i] * gs;
      for (int32_t bg = 0; bg < n_b * n_g; ++bg)
        for (int32_t sp = 0; sp < splits; ++sp) tiles.push_back({i, n, bg, sp});
    }
  } else {
    // per-head masks: tile (b, g, i, split) covers mask heads
    // g*group + split*gs .. + gs - 1 of row i
    for (int32_t g = 0; g < n_g; ++g)
      for (int32_t i = 0; i < rows; ++i)
        for (int32_t sp = 0; sp < splits; ++sp) {
          int32_t n = 0;
          for (int32_t gh = sp * gs; gh < (sp + 1) * gs; ++gh)
            n += row_len[static_cast<size_t>(g * group + gh) * rows + i];
          for (int32_t b = 0; b < n_b; ++b) tiles.push_back({i, n, b * n_g + g, sp});
        }
    std::stable_sort(tiles.begin(), tiles.end(), [](const Tile& x, const Tile& y) { return x.n > y.n; });
  }
  // the greedy assignment.  The CTAs are kept sorted by key = (work so far)
  // << 16 | CTA, so the smallest key is the least-loaded CTA, ties going to
  // the lower index.  The tiles come in runs of equal size (longest first);
  // within a run the keys taken out grow, so the updated keys form a second
  // sorted list, merged back when the run ends: linear work per run instead
  // of a heap operation per tile, with the same assignment.
  if (grid > 0xFFFF) return fail(BSA_ERR_UNSUPPORTED, "tile schedule grid above 65535");
  std::vector<uint64_t> keys(static_cast<size_t>(grid)), upd, merged;
  for (int32_t c = 0; c < grid; ++c) keys[static_cast<size_t>(c)] = static_cast<uint64_t>(c);
  upd.reserve(static_cast<size_t>(grid));
  merged.reserve(static_cast<size_t>(grid));
  std::vector<int32_t> owner(tiles.size()), slot(tiles.size()), count(static_cast<size_t>(grid), 0);
  for (size_t k = 0; k < tiles.size();) {
    const int32_t n = tiles[k].n;
    const uint64_t add = static_cast<uint64_t>(8 * static_cast<int64_t>(n) + 12) << 16;
    size_t ki = 0, ui = 0;
    upd.clear();
    for (; k < tiles.size() && tiles[k].n == n; ++k) {
      const bool from_keys = ki < keys.size() && (ui == upd.size() || keys[ki] < upd[ui]);
      const uint64_t top = from_keys ? keys[ki++] : upd[ui++];
      const int32_t c = static_cast<int32_t>(top & 0xFFFFu);
      owner[k] = c;
      slot[k] = count[static_cast<size_t>(c)]++;
      upd.push_back(top + add);
    }
    if (upd.size() - ui <= 4) {  // a short run: insert its few keys
      keys.erase(keys.begin(), keys.begin() + static_cast<std::ptrdiff_t>(ki));
      for (size_t j = ui; j < upd.size(); ++j) keys.insert(std::upper_bound(keys.begin(), keys.end(), upd[j]), upd[j]);
    } else {
      merged.clear();
      std::merge(keys.begin() + static_cast<std::ptrdiff_t>(ki), keys.end(),
                 upd.begin() + static_cast<std::ptrdiff_t>(ui), upd.end(), std::back_inserter(merged));
      keys.swap(merged);
    }
  }
  // MULTIFIT: the smallest capacity (bisection between the mean and the
  // greedy's maximum) under which first-fit decreasing places every tile;
  // kept when its maximum is at least 3% below the greedy's (the greedy's
  // waves of similar tiles share K/V and Q/dO through L2, which is worth a
  // few percent of balance)
  {
    std::vector<int64_t> gload(static_cast<size_t>(grid), 0);
    int64_t total = 0, biggest = 0;
    for (size_t k = 0; k < tiles.size(); ++k) {
      const int64_t w = 8 * static_cast<int64_t>(tiles[k].n) + 12;
      gload[static_cast<size_t>(owner[k])] += w;
      total += w;
      biggest = std::max(biggest, w);
    }
    const int64_t greedy_max = *std::max_element(gload.begin(), gload.end());
    int64_t lo = std::max(biggest, (total + grid - 1) / grid), hi = greedy_max - 1;
    // no assignment goes below lo: when even that is not 3% under the
    // greedy's maximum, skip the search (many tiles per CTA)
    if (100 * (greedy_max - lo) < 3 * greedy_max) hi = lo - 1;
    std::vector<int32_t> ff_owner(tiles.size()), best_owner;
    int64_t best_max = greedy_max;
    while (lo <= hi) {
      const int64_t cap = lo + (hi - lo) / 2;
      int64_t mx = 0;
      if (first_fit(tiles, grid, cap, &ff_owner, &mx)) {
        best_owner = ff_owner;
        best_max = mx;
        hi = std::min(cap, mx) - 1;
      } else {
        lo = cap + 1;
      }
    }
    if (!best_owner.empty() && 100 * (greedy_max - best_max) >= 3 * greedy_max) {
      std::fill(count.begin(), count.end(), 0);
      for (size_t k = 0; k < tiles.size(); ++k) {
        owner[k] = best_owner[k];
        slot[k] = count[static_cast<size_t>(owner[k])]++;
      }
    }
  }
  int32_t longest = 0;
  for (int32_t c : count) longest = std::max(longest, c);
  const int32_t st = longest + 1;  // room for the end mark
  flat->assign(static_cast<size_t>(grid) * st, make_int4(0, -1, 0, 0));
  for (size_t k = 0; k < tiles.size(); ++k)
    (*flat)[static_cast<size_t>(owner[k]) * st + static_cast<size_t>(slot[k])] =
        make_int4(tiles[k].i, tiles[k].n, tiles[k].bg, tiles[k].sp);
  *stride = st;
  return BSA_OK;
}

namespace {

// A piece of a tile schedule carried in a kernel's parameters (a launch
// takes up to 32,764 bytes of them).  The launch path brings it to the
// device, not a copy engine, so the upload does not wait behind large
// host<->device copies that other streams have in flight (a pageable copy
// of more than 64 KiB does, holding the calling thread until they end).
constexpr int kPutInt4s = 1900;
struct PutChunk {
  int4 v[kPutInt4s];
  int32_t n;
};

__global__ void __launch_bounds__(256) put_int4s(int4* __restrict__ dst, const __grid_constant__ PutChunk c) {
  for (int i = threadIdx.x; i < c.n; i += blockDim.x) dst[i] = c.v[i];
  __threadfence();
}

// Built schedules of the process, most recently used first: the host side
// of a schedule depends only on the row lengths, the row order and the
// launch configuration, which a mask compiled again repeats.
struct ListsEntry {
  std::vector<int32_t> row_len, row_order;
  int32_t rows, heads, n_b, n_g, group, splits, grid;
  std::vector<int4> flat;
  int32_t stride;
};
constexpr size_t kListsCache = 32;
std::mutex g_lists_mu;
std::list<ListsEntry> g_lists;

bsa_status cached_schedule_lists(const bsa_mask_info* info, int32_t n_b, int32_t n_g, int32_t group, int32_t splits,
                                 int32_t grid, std::vector<int4>* flat, int32_t* stride) {
  const size_t n = static_cast<size_t>(info->heads) * static_cast<size_t>(info->rows);
  if (info->row_len_h.size() < n || info->row_order_h.size() < n)
    return fail(BSA_ERR_INVALID_ARG, "MaskInfo without its host row arrays");
  std::lock_guard<std::mutex> lk(g_lists_mu);
  for (auto it = g_lists.begin(); it != g_lists.end(); ++it)
    if (it->rows == info->rows && it->heads == info->heads && it->n_b == n_b && it->n_g == n_g &&
        it->group == group && it->splits == splits && it->grid == grid &&
        std::equal(it->row_len.begin(), it->row_len.end(), info->row_len_h.begin()) &&
        std::equal(it->row_order.begin(), it->row_order.end(), info->row_order_h.begin())) {
      *flat = it->flat;
      *stride = it->stride;
      g_lists.splice(g_lists.begin(), g_lists, it);
      return BSA_OK;
    }
  const bsa_status ls = schedule_lists(info->row_len_h.data(), info->row_order_h.data(), info->rows, info->heads, n_b,
                                       n_g, group, splits, grid, flat, stride);
  if (ls != BSA_OK) return ls;
  if (flat->size() * sizeof(int4) > (size_t(4) << 20)) return BSA_OK;  // (not kept: over 4 MiB)
  ListsEntry e;
  e.row_len.assign(info->row_len_h.begin(), info->row_len_h.begin() + static_cast<std::ptrdiff_t>(n));
  e.row_order.assign(info->row_order_h.begin(), info->row_order_h.begin() + static_cast<std::ptrdiff_t>(n));
  e.rows = info->rows;
  e.heads = info->heads;
  e.n_b = n_b;
  e.n_g = n_g;
  e.group = group;
  e.splits = splits;
  e.grid = grid;
  e.flat = *flat;
  e.stride = *stride;
  g_lists.push_front(std::move(e));
  if (g_lists.size() > kListsCache) g_lists.pop_back();
  return BSA_OK;
}

}  // namespace

bsa_status tile_schedule(const bsa_mask_info* info, int32_t n_b, int32_t n_g, int32_t group, int32_t splits,
                         int32_t grid, cudaStream_t stream, const int4** out, int32_t* stride) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(info->sched_mu);
  for (const auto& sc : info->schedules)
    if (sc.n_b == n_b && sc.n_g == n_g && sc.group == group && sc.splits == splits && sc.grid == grid &&
        sc.device == dev) {
      e = cudaStreamWaitEvent(stream, sc.ready, 0);
      if (e != cudaSuccess) return cuda_fail(e, "wait for the tile schedule upload");
      *out = sc.dev;
      *stride = sc.stride;
      return BSA_OK;
    }
  std::vector<int4> flat;
  int32_t st = 0;
  {
    const bsa_status ls = cached_schedule_lists(info, n_b, n_g, group, splits, grid, &flat, &st);
    if (ls != BSA_OK) return ls;
  }
  // stream-ordered upload (no synchronisation with earlier work on the
  // device) in kernel parameters; the host copy lives as long as the schedule
  bsa_mask_info::Schedule sc;
  sc.host = std::move(flat);
  void* dv = nullptr;
  bsa_status bs = pool_alloc(&dv, sc.host.size() * sizeof(int4), stream);
  if (bs != BSA_OK) return bs;
  int4* d = static_cast<int4*>(dv);
  e = cudaSuccess;
  for (size_t off = 0; e == cudaSuccess && off < sc.host.size(); off += kPutInt4s) {
    PutChunk c;
    c.n = static_cast<int32_t>(std::min<size_t>(kPutInt4s, sc.host.size() - off));
    std::copy(sc.host.begin() + static_cast<std::ptrdiff_t>(off),
              sc.host.begin() + static_cast<std::ptrdiff_t>(off) + c.n, c.v);
    put_int4s<<<1, 256, 0, stream>>>(d + off, c);
    e = cudaGetLastError();
  }
  // (the event between the upload and the launch that reads the schedule
  // also orders them fully: that launch's early start covers only its own
  // predecessor kernel, and the forward's walker reads the schedule at once)
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sc.ready, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventRecord(sc.ready, stream);
  if (e != cudaSuccess) {
    if (sc.ready) cudaEventDestroy(sc.ready);
    pool_free(d, stream);
    return cuda_fail(e, "upload tile schedule");
  }
  sc.n_b = n_b;
  sc.n_g = n_g;
  sc.group = group;
  sc.splits = splits;
  sc.grid = grid;
  sc.device = dev;
  sc.stride = st;
  sc.dev = d;
  info->schedules.push_back(std::move(sc));
  *out = d;
  *stride = st;
  return BSA_OK;
}

}  // namespace bsa
