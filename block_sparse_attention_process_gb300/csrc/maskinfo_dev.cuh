// Device-side view of a compiled MaskInfo, and the element predicates of the
// computable masks, shared by the attention kernels.
#pragma once
#include <cstdint>

#include "bsa.h"
#include "internal.h"
#include "ptx.cuh"

namespace bsa {

// The mask kind an attention kernel instantiation is compiled for: one whose
// partial blocks are computed from each row's visible interval, one whose
// partial blocks are read as bits from the stack, or either (decided at run
// time; used by the instantiations with the logit transforms).
enum MaskMode : int { kComputableMask = 0, kDenseMask = 1, kAnyMask = 2 };

template <int kM>
__device__ __forceinline__ bool dense_mask(int kind) {
  return kM == kDenseMask || (kM == kAnyMask && kind == BSA_MASK_DENSE);
}

struct MaskInfoDev {
  const int8_t* block_mask;   // [heads, rows, width]
  const void* data_next;      // [heads, rows, width]
  const void* mask_next;      // [heads, rows, width] or null
  const uint8_t* partial;     // [P, 128, 128] or null
  const uint32_t* partial_bits;  // [P, 128, 4]: bit j of word w = partial[., row, 32 w + j]
  const int32_t* q_sequence;  // [q_len]
  const int32_t* row_len;     // [heads, rows]
  const int32_t* row_order;   // [heads * rows]
  int32_t heads, rows, width, cols;
  int32_t dn_bytes, mn_bytes;
  int32_t kind, orientation;
  int64_t num_partial;
  int64_t left, right, chunk;
};

inline MaskInfoDev mask_info_dev(const bsa_mask_info* info) {
  MaskInfoDev m{};
  m.block_mask = info->block_mask;
  m.data_next = info->data_next;
  m.mask_next = info->mask_next;
  m.partial = info->partial;
  m.partial_bits = info->partial_bits;
  m.q_sequence = info->q_sequence;
  m.row_len = info->row_len;
  m.row_order = info->row_order;
  m.heads = info->heads;
  m.rows = info->rows;
  m.width = info->width;
  m.cols = info->cols;
  m.dn_bytes = info->data_next_bytes;
  m.mn_bytes = info->mask_next_bytes;
  m.kind = info->kind;
  m.orientation = info->orientation;
  m.num_partial = info->num_partial;
  m.left = info->local_left;
  m.right = info->local_right;
  m.chunk = info->chunk;
  return m;
}

__device__ __forceinline__ int32_t load_idx(const void* base, int bytes, int64_t i) {
  if (bytes == 1) return static_cast<const int8_t*>(base)[i];
  if (bytes == 2) return static_cast<const int16_t*>(base)[i];
  return static_cast<const int32_t*>(base)[i];
}

// One grid position of a MaskInfo row, with its indices checked.
struct BlockRef {
  int32_t label;  // 0, 1, 2
  int32_t col;    // key block (fwd orientation) / query block (dkv orientation)
  int32_t slot;   // stack slot for dense label-1 blocks, else 0
};

// Unchecked entry as loaded (so that the load can be issued ahead of use).
struct RawRef {
  int32_t label, col, slot;
};

__device__ __forceinline__ RawRef load_block(const MaskInfoDev& m, int64_t row_base, int t) {
  RawRef r;
  r.label = m.block_mask[row_base + t];
  r.col = load_idx(m.data_next, m.dn_bytes, row_base + t);
  r.slot = m.mask_next ? load_idx(m.mask_next, m.mn_bytes, row_base + t) : 0;
  return r;
}

__device__ __forceinline__ BlockRef check_block(const MaskInfoDev& m, const RawRef& raw, uint32_t* err) {
  BlockRef r;
  r.label = raw.label;
  r.col = raw.col;
  r.slot = raw.slot;
  bool bad = r.label < 0 || r.label > 2 || r.col < 0 || r.col >= m.cols;
  if (m.mask_next && r.label == 1) bad |= r.slot < 0 || r.slot >= m.num_partial;
  if (bad) {
    if (err) atomicOr(err, DEV_ERR_BOUNDS);
    r.label = 0;  // treated as empty: nothing is fetched or computed for it
    r.col = 0;
    r.slot = 0;
  }
  return r;
}

__device__ __forceinline__ BlockRef read_block(const MaskInfoDev& m, int64_t row_base, int t, uint32_t* err) {
  return check_block(m, load_block(m, row_base, t), err);
}

constexpr int64_t kMaskInf = int64_t(1) << 40;

// Visible interval [lo, hi] of key indices for query index q (computable
// masks): causal k <= q; local q-left <= k <= q+right; chunked
// q/c == k/c and k <= q; full: everything.
__device__ __forceinline__ void key_interval(int kind, int64_t left, int64_t right, int64_t chunk, int64_t q,
                                             int64_t& lo, int64_t& hi) {
  lo = -kMaskInf;
  hi = kMaskInf;
  if (kind == BSA_MASK_CAUSAL) {
    hi = q;
  } else if (kind == BSA_MASK_LOCAL) {
    if (left >= 0) lo = q - left;
    if (right >= 0) hi = q + right;
  } else if (kind == BSA_MASK_CHUNKED_CAUSAL) {
    lo = (q / chunk) * chunk;
    hi = q;
  }
}

// Visible interval [lo, hi] of query indices for key index k.
__device__ __forceinline__ void query_interval(int kind, int64_t left, int64_t right, int64_t chunk, int64_t k,
                                               int64_t& lo, int64_t& hi) {
  lo = -kMaskInf;
  hi = kMaskInf;
  if (kind == BSA_MASK_CAUSAL) {
    lo = k;
  } else if (kind == BSA_MASK_LOCAL) {
    if (right >= 0) lo = k - right;
    if (left >= 0) hi = k + left;
  } else if (kind == BSA_MASK_CHUNKED_CAUSAL) {
    lo = k;
    hi = (k / chunk) * chunk + chunk - 1;
  }
}

}  // namespace bsa
