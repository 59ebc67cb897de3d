// Internal declarations shared by the host side of the library.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include "bsa.h"

// Compiled mask, owned by the library.
struct bsa_mask_info {
  int32_t kind = 0, orientation = 0, shrink = 1;
  int32_t heads = 0, rows = 0, cols = 0, width = 0;
  int64_t q_len = 0, kv_len = 0;
  int64_t num_partial = 0, n_empty = 0, n_partial = 0, n_full = 0;
  int32_t data_next_bytes = 1, mask_next_bytes = 0;
  // mask parameters, kept so the kernels can recompute computable masks
  int64_t local_left = -1, local_right = -1, chunk = 0;
  // device storage (one allocation each)
  int8_t* block_mask = nullptr;      // [heads, rows, width]
  void* data_next = nullptr;         // [heads, rows, width]
  void* mask_next = nullptr;         // [heads, rows, width] or null
  uint8_t* partial = nullptr;        // [num_partial, 128, 128] or null
  // the same blocks as bits (internal, for the kernels): word w of row r of
  // block b, bit j = partial[b, r, 32 w + j]; [num_partial, 128, 4] or null
  uint32_t* partial_bits = nullptr;
  int32_t* q_sequence = nullptr;     // [q_len]
  int32_t* row_len = nullptr;        // [heads, rows] non-empty blocks per row (internal)
  int32_t* row_order = nullptr;      // [heads * rows] rows sorted by decreasing row_len (internal)
  // host copies of row_len / row_order, for the launch-time tile schedules
  std::vector<int32_t> row_len_h, row_order_h;
  // tile schedules built so far (device memory from the library's pool,
  // freed with the handle).  The upload is stream-ordered on the launch
  // that built it; `ready` marks its end for launches on other streams, and
  // `host` keeps the source alive.
  struct Schedule {
    int32_t n_b = 0, n_g = 0, group = 0, splits = 0, grid = 0, device = -1, stride = 0;
    int4* dev = nullptr;
    cudaEvent_t ready = nullptr;
    std::vector<int4> host;
  };
  mutable std::vector<Schedule> schedules;
  mutable std::mutex sched_mu;
};

namespace bsa {

constexpr int kBlock = 128;

void set_last_error(const std::string& msg);
bsa_status fail(bsa_status s, const std::string& msg);
bsa_status cuda_fail(cudaError_t e, const char* what);
uint32_t* device_error_word();          // per-device error word (lazily allocated)
uint64_t wait_limit_ns();

// Launchers implemented in the .cu files (argument checking is done by the caller).
bsa_status mask_compile_impl(const bsa_mask_spec* spec, const bsa_mask_opts* opts, cudaStream_t stream,
                             bsa_mask_info** out);
bsa_status fwd_launch(const bsa_fwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream);
bsa_status fwd_partial_launch(const bsa_fwd_partial_args* a, const bsa_mask_info* info, float scale,
                              cudaStream_t stream);
bsa_status merge_launch(const bsa_merge_args* a, cudaStream_t stream);
bsa_status rowsum_launch(const bsa_bwd_args* a, cudaStream_t stream);
// `err` (optional) replaces the library's device error word for this launch;
// `schedule` false hands tiles out round-robin instead of building (and
// allocating) a tile schedule.
bsa_status dkv_launch(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream,
                      uint32_t* err = nullptr, bool schedule = true);
bsa_status dq_launch(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream,
                     uint32_t* err = nullptr, bool schedule = true);
bsa_status debug_wait_timeout_launch(cudaStream_t stream);
bsa_status debug_selfcheck_launch(cudaStream_t stream);

int num_sms();

// Raises `func`'s dynamic shared-memory limit to `smem` bytes on the current
// device, once per (device, kernel): the attribute is per device, so a
// process that launches on several GPUs sets it on each.
bsa_status ensure_smem_attr(const void* func, size_t smem, const char* what);

// Host-side checks of a backward call's arguments (shapes, pointers and
// their alignment, score transforms); `need_dsum` false for the entry point
// that keeps the rowsum in its own scratch.
bsa_status check_bwd_args(const bsa_bwd_args* a, bool need_dsum);

// The allocation-free backward's device error word on the current device,
// or null when no call there has set it up yet.
uint32_t* noalloc_error_word_if_set();

// Work tiles of a launch: (b, g, MaskInfo row i, split) for b < n_b, g < n_g
// and split < splits, each covering group / splits mask heads (the q heads
// of a KV group in the dK/dV launch, split over `splits` CTAs when the
// group is large; 1 head, 1 split in the forward and dQ launches), handed
// to `grid` persistent CTAs greedily, longest first: each tile goes to the
// CTA with the least work so far (blocks plus a per-tile overhead).  CTA
// c's tiles are entries [c * stride, c * stride + stride) of *out, in
// order, each {i, blocks, b * n_g + g, split}, ended early by blocks = -1.
// Built on the first launch of a (n_b, n_g, group, splits, grid, device)
// and cached in the MaskInfo; `stream` (the launch's) is ordered after its
// upload.
// The host part of a tile schedule: CTA c's entries {row, blocks, b*n_g + g,
// split} at flat[c*stride ..], each list closed by an entry with blocks -1.
bsa_status schedule_lists(const int32_t* row_len, const int32_t* row_order, int32_t rows, int32_t heads,
                          int32_t n_b, int32_t n_g, int32_t group, int32_t splits, int32_t grid,
                          std::vector<int4>* flat, int32_t* stride);
bsa_status tile_schedule(const bsa_mask_info* info, int32_t n_b, int32_t n_g, int32_t group, int32_t splits,
                         int32_t grid, cudaStream_t stream, const int4** out, int32_t* stride);

// Stream-ordered device memory from the library's pool on the current
// device (kept cached by the pool between calls).
bsa_status pool_alloc(void** p, size_t bytes, cudaStream_t stream);
bsa_status pool_free(void* p, cudaStream_t stream);

// Programmatic dependent launch: a kernel launched this way may start (its
// set-up: barriers, tensor memory, descriptor prefetch) while the previous
// kernel in the stream finishes; it waits (griddepcontrol.wait) before it
// touches global memory.  Off when the environment sets BSA_PDL=0.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace bsa
