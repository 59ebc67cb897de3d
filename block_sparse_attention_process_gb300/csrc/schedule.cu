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

bsa_status tile_schedule(const bsa_mask_info* info, int64_t units, int32_t hq, int32_t grid, const int4** out,
                         int32_t* stride) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(info->sched_mu);
  for (const auto& sc : info->schedules)
    if (sc.units == units && sc.hq == hq && sc.grid == grid && sc.device == dev) {
      *out = sc.dev;
      *stride = sc.stride;
      return BSA_OK;
    }
  const int64_t n_rows = static_cast<int64_t>(info->row_order_h.size());
  const int64_t n_tiles = n_rows * units;
  if (grid <= 0 || n_tiles <= 0) return fail(BSA_ERR_INVALID_ARG, "empty tile schedule");
  // greedy over tiles in longest-first order; cost in eighths of a block,
  // with a per-tile overhead of about one and a half blocks
  std::vector<std::vector<int4>> lists(static_cast<size_t>(grid));
  using Load = std::pair<int64_t, int32_t>;  // (work so far, CTA): ties go to the lower CTA
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int32_t c = 0; c < grid; ++c) heap.push({0, c});
  for (int64_t rank = 0; rank < n_rows; ++rank) {
    const int32_t row = info->row_order_h[static_cast<size_t>(rank)];
    const int32_t n = info->row_len_h[static_cast<size_t>(row)];
    const int32_t i = row % info->rows;
    const int32_t hm = row / info->rows;
    for (int64_t u = 0; u < units; ++u) {
      // shared mask: u = b * Hq + hq; per-head masks: u = b and hq = the mask head
      const int32_t bh = info->heads == 1 ? static_cast<int32_t>(u) : static_cast<int32_t>(u) * hq + hm;
      Load top = heap.top();
      heap.pop();
      lists[static_cast<size_t>(top.second)].push_back(make_int4(row, n, bh, i));
      top.first += 8 * static_cast<int64_t>(n) + 12;
      heap.push(top);
    }
  }
  size_t longest = 0;
  for (const auto& l : lists) longest = std::max(longest, l.size());
  const int32_t st = static_cast<int32_t>(longest) + 1;  // room for the end mark
  std::vector<int4> flat(static_cast<size_t>(grid) * st, make_int4(0, -1, 0, 0));
  for (int32_t c = 0; c < grid; ++c)
    std::copy(lists[static_cast<size_t>(c)].begin(), lists[static_cast<size_t>(c)].end(),
              flat.begin() + static_cast<size_t>(c) * st);
  int4* d = nullptr;
  e = cudaMalloc(&d, flat.size() * sizeof(int4));
  if (e != cudaSuccess) return cuda_fail(e, "alloc tile schedule");
  e = cudaMemcpy(d, flat.data(), flat.size() * sizeof(int4), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(d);
    return cuda_fail(e, "upload tile schedule");
  }
  bsa_mask_info::Schedule sc;
  sc.units = units;
  sc.hq = hq;
  sc.grid = grid;
  sc.device = dev;
  sc.stride = st;
  sc.dev = d;
  info->schedules.push_back(sc);
  *out = d;
  *stride = st;
  return BSA_OK;
}

}  // namespace bsa
