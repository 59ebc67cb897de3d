// Launch-time tile schedule for the persistent attention kernels.
//
// A kernel launch runs min(tiles, SMs) CTAs, each walking a fixed list of
// work tiles.  Handing tiles out round-robin in longest-first order leaves
// the last round partly empty when the tile count is not a multiple of the
// CTA count; the greedy assignment here (each tile, longest first, to the
// CTA with the least work so far) evens the CTAs' totals out, so short
// tiles fill the gaps left by the long ones.
#include <algorithm>
#include <cstddef>
#include <iterator>

#include "internal.h"

namespace bsa {

bsa_status schedule_lists(const int32_t* row_len, const int32_t* row_order, int32_t rows, int32_t heads,
                          int32_t n_b, int32_t n_g, int32_t group, int32_t splits, int32_t grid,
                          std::vector<int4>* flat, int32_t* stride) {
  if (grid <= 0 || rows <= 0 || n_b <= 0 || n_g <= 0 || group <= 0 || splits <= 0 || group % splits)
    return fail(BSA_ERR_INVALID_ARG, "empty tile schedule");
  const int32_t gs = group / splits;  // mask heads of one split
  // tiles in longest-first order: {row, blocks, b * n_g + g, split}
  struct T {
    int32_t i, n, bg, sp;
  };
  std::vector<T> tiles;
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
    std::stable_sort(tiles.begin(), tiles.end(), [](const T& x, const T& y) { return x.n > y.n; });
  }
  // greedy; cost in eighths of a block, with a per-tile overhead of about
  // one and a half blocks.  The CTAs are kept sorted by key = (work so far)
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
    const bsa_status ls = schedule_lists(info->row_len_h.data(), info->row_order_h.data(), info->rows, info->heads,
                                         n_b, n_g, group, splits, grid, &flat, &st);
    if (ls != BSA_OK) return ls;
  }
  // stream-ordered upload (no synchronisation with earlier work on the
  // device), from a host copy that lives as long as the schedule
  bsa_mask_info::Schedule sc;
  sc.host = std::move(flat);
  void* dv = nullptr;
  bsa_status bs = pool_alloc(&dv, sc.host.size() * sizeof(int4), stream);
  if (bs != BSA_OK) return bs;
  int4* d = static_cast<int4*>(dv);
  e = cudaMemcpyAsync(d, sc.host.data(), sc.host.size() * sizeof(int4), cudaMemcpyHostToDevice, stream);
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
