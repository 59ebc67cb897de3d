// Launch-time tile schedule for the persistent attention kernels.
//
// A kernel launch runs min(tiles, SMs) CTAs, each walking a fixed list of
// work tiles.  Handing tiles out round-robin in longest-first order leaves
// the last round partly empty when the tile count is not a multiple of the
// CTA count; the greedy assignment here (each tile, longest first, to the
// CTA with the least work so far) evens the CTAs' totals out, so short
// tiles fill the gaps left by the long ones.
#include <algorithm>
#include <functional>
#include <queue>
#include <utility>

#include "internal.h"

namespace bsa {

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
  const int32_t rows = info->rows;
  if (grid <= 0 || rows <= 0 || n_b <= 0 || n_g <= 0 || group <= 0 || splits <= 0 || group % splits)
    return fail(BSA_ERR_INVALID_ARG, "empty tile schedule");
  const int32_t gs = group / splits;  // mask heads of one split
  // tiles in longest-first order: {row, blocks, b * n_g + g, split}
  struct T {
    int32_t i, n, bg, sp;
  };
  std::vector<T> tiles;
  tiles.reserve(static_cast<size_t>(rows) * n_b * n_g);
  if (info->heads == 1) {
    // rows by decreasing length (row_order), each for every (b, g)
    for (int32_t rank = 0; rank < rows; ++rank) {
      const int32_t i = info->row_order_h[static_cast<size_t>(rank)];
      const int32_t n = info->row_len_h[static_cast<size_t>(i)] * gs;
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
            n += info->row_len_h[static_cast<size_t>((g * group + gh) * rows + i)];
          for (int32_t b = 0; b < n_b; ++b) tiles.push_back({i, n, b * n_g + g, sp});
        }
    std::stable_sort(tiles.begin(), tiles.end(), [](const T& x, const T& y) { return x.n > y.n; });
  }
  // greedy; cost in eighths of a block, with a per-tile overhead of about
  // one and a half blocks
  std::vector<std::vector<int4>> lists(static_cast<size_t>(grid));
  using Load = std::pair<int64_t, int32_t>;  // (work so far, CTA): ties go to the lower CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int32_t c = 0; c < grid; ++c) heap.push({0, c});
  for (const T& t : tiles) {
    Load top = heap.top();
    heap.pop();
    lists[static_cast<size_t>(top.second)].push_back(make_int4(t.i, t.n, t.bg, t.sp));
    top.first += 8 * static_cast<int64_t>(t.n) + 12;
    heap.push(top);
  }
  size_t longest = 0;
  for (const auto& l : lists) longest = std::max(longest, l.size());
  const int32_t st = static_cast<int32_t>(longest) + 1;  // room for the end mark
  std::vector<int4> flat(static_cast<size_t>(grid) * st, make_int4(0, -1, 0, 0));
  for (int32_t c = 0; c < grid; ++c)
    std::copy(lists[static_cast<size_t>(c)].begin(), lists[static_cast<size_t>(c)].end(),
              flat.begin() + static_cast<size_t>(c) * st);
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
