// GPU mask compiler: mask -> MaskInfo.
//
// Follows "Splash Attention: When the Mask Stops Being Arithmetic and Becomes
// the Loop":
//   * "What is splash attention and how is it different from flash
//     attention?" / "Does splash attention make every sparse mask faster?":
//     every 128x128 block is labelled by asking any() and all() of it
//     (0 = all zeros, 1 = mixed, 2 = all ones)            -> classify_*
//   * "What is MaskInfo in splash attention?": the mixed blocks of a dense
//     mask go into a deduplicated stack pointed at by mask_next; data_next
//     names the key/value block to hold at each grid position; the integer
//     arrays are downcast to the smallest type their largest value fits;
//     computable masks (causal, local, chunked causal) carry no stack
//                                                         -> dedup_*, write_rows
//   * "What does grid shrinking do in splash attention?": each block row
//     keeps only its non-empty columns, padded to the widest row
//                                                         -> write_rows
//
// Contract where the page is silent: stack slots in order of first
// occurrence walking (head, row, column); data_next at an empty cell is the
// next non-empty column to the right, else the last one to the left, else
// 0; mask_next is 0 at label-0/2 cells; shrink padding is label 0 with the
// row's last real column and mask_next 0; signed downcast (<=127 int8,
// <=32767 int16, else int32).  The dkv orientation is the same on the
// transposed mask.
#include <algorithm>
#include <vector>

#include "internal.h"

namespace bsa {
namespace {

constexpr int B = kBlock;

struct MaskParams {
  int32_t kind, orient, heads;
  int32_t nR, nC;  // block rows / columns in this orientation
  int64_t q_len, kv_len, left, right, chunk;
  const uint8_t* dense;
};

struct Stats {
  unsigned long long n_empty, n_partial, n_full;
  int32_t width;    // max non-empty blocks in a row
  int32_t max_col;  // largest non-empty column index (0 if none)
  int32_t n1;       // number of label-1 cells
  int32_t P;        // stack depth
};

constexpr int64_t kInf = int64_t(1) << 40;

// Visible interval [lo, hi] of the column coordinate for logical row `r`
// (a query index in the fwd orientation, a key index in the dkv one).
__device__ __forceinline__ void row_interval(const MaskParams& p, int64_t r, int64_t& lo, int64_t& hi) {
  lo = -kInf;
  hi = kInf;
  const bool fwd = p.orient == BSA_ORIENT_FWD;
  switch (p.kind) {
    case BSA_MASK_CAUSAL:  // k <= q
      if (fwd) hi = r; else lo = r;
      break;
    case BSA_MASK_LOCAL:  // q - left <= k <= q + right
      if (fwd) {
        if (p.left >= 0) lo = r - p.left;
        if (p.right >= 0) hi = r + p.right;
      } else {
        if (p.right >= 0) lo = r - p.right;
        if (p.left >= 0) hi = r + p.left;
      }
      break;
    case BSA_MASK_CHUNKED_CAUSAL:  // q / c == k / c and k <= q
      if (fwd) {
        lo = (r / p.chunk) * p.chunk;
        hi = r;
      } else {
        lo = r;
        hi = (r / p.chunk) * p.chunk + p.chunk - 1;
      }
      break;
    default:
      break;
  }
}

// Each block row of a computable mask allows one interval per element row,
// so counting the overlap of that interval with the block's columns decides
// any()/all() exactly.  One CTA (128 threads, one per element row) per cell.
__global__ void classify_computable(MaskParams p, int8_t* __restrict__ labels, int64_t n_cells) {
  for (int64_t cell = blockIdx.x; cell < n_cells; cell += gridDim.x) {
    const int c = static_cast<int>(cell % p.nC);
    const int r = static_cast<int>((cell / p.nC) % p.nR);
    const int64_t row = static_cast<int64_t>(r) * B + threadIdx.x;
    int64_t lo, hi;
    row_interval(p, row, lo, hi);
    const int64_t c0 = static_cast<int64_t>(c) * B, c1 = c0 + B - 1;
    const int64_t a = lo > c0 ? lo : c0, b = hi < c1 ? hi : c1;
    const int64_t cnt = b >= a ? b - a + 1 : 0;
    const int any = __syncthreads_or(cnt > 0);
    const int all = __syncthreads_and(cnt == B);
    if (threadIdx.x == 0) labels[cell] = all ? 2 : (any ? 1 : 0);
  }
}

// Byte-wise "is nonzero" of a 32-bit word: 0x01 in every nonzero byte.
__device__ __forceinline__ uint32_t nz_bytes(uint32_t x) {
  const uint32_t y = ((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x;
  return (y >> 7) & 0x01010101u;
}

// SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", 2014).
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Address of element row `row` (0..127) of the ORIGINAL (query-major) dense
// block behind logical cell (h, r, c).
__device__ __forceinline__ const uint8_t* dense_block_row(const MaskParams& p, int h, int r, int c, int row) {
  const int qb = p.orient == BSA_ORIENT_FWD ? r : c;
  const int kb = p.orient == BSA_ORIENT_FWD ? c : r;
  return p.dense + (static_cast<size_t>(h) * p.q_len + static_cast<size_t>(qb) * B + row) * p.kv_len +
         static_cast<size_t>(kb) * B;
}

// Dense classifier: one CTA (256 threads) per cell reads the 16 KiB block,
// answers any()/all() and hashes the normalised 0/1 bytes (order-free sum of
// per-word hashes, so every thread layout gives the same value).
__global__ void __launch_bounds__(256) classify_dense(MaskParams p, int8_t* __restrict__ labels,
                                                     uint64_t* __restrict__ hashes, int64_t n_cells) {
  __shared__ uint64_t red[8];
  for (int64_t cell = blockIdx.x; cell < n_cells; cell += gridDim.x) {
    const int c = static_cast<int>(cell % p.nC);
    const int r = static_cast<int>((cell / p.nC) % p.nR);
    const int h = static_cast<int>(cell / (static_cast<int64_t>(p.nC) * p.nR));
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    const uint4* src = reinterpret_cast<const uint4*>(dense_block_row(p, h, r, c, row) + half * 64);
    bool any = false, all = true;
    uint64_t hsum = 0;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 w = __ldg(src + v);
      const uint32_t n0 = nz_bytes(w.x), n1 = nz_bytes(w.y), n2 = nz_bytes(w.z), n3 = nz_bytes(w.w);
      any |= (n0 | n1 | n2 | n3) != 0u;
      all &= (n0 & n1 & n2 & n3) == 0x01010101u;
      const uint64_t e = static_cast<uint64_t>(row) * 16 + half * 8 + v * 2;  // 8-byte word index
      hsum += mix64((static_cast<uint64_t>(n1) << 32 | n0) ^ (e * 0x9E3779B97F4A7C15ull));
      hsum += mix64((static_cast<uint64_t>(n3) << 32 | n2) ^ ((e + 1) * 0x9E3779B97F4A7C15ull));
    }
    for (int o = 16; o > 0; o >>= 1) hsum += __shfl_xor_sync(0xffffffffu, hsum, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = hsum;
    const int a = __syncthreads_or(any);
    const int l = __syncthreads_and(all);
    if (threadIdx.x == 0) {
      uint64_t t = 0;
      for (int i = 0; i < 8; ++i) t += red[i];
      labels[cell] = l ? 2 : (a ? 1 : 0);
      hashes[cell] = t;
    }
    __syncthreads();
  }
}

// Per block row: number of non-empty blocks, plus grid-wide counts.
__global__ void row_pass(const int8_t* __restrict__ labels, int32_t nC, int64_t n_rows, int32_t* row_len,
                         Stats* st) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= n_rows) return;
  const int8_t* L = labels + row * nC;
  int n = 0, last = -1;
  unsigned long long e = 0, pa = 0, f = 0;
  for (int c = 0; c < nC; ++c) {
    const int8_t v = L[c];
    if (v == 0) {
      ++e;
    } else {
      ++n;
      last = c;
      if (v == 1) ++pa; else ++f;
    }
  }
  row_len[row] = n;
  atomicMax(&st->width, n);
  if (last >= 0) atomicMax(&st->max_col, last);
  atomicAdd(&st->n_empty, e);
  atomicAdd(&st->n_partial, pa);
  atomicAdd(&st->n_full, f);
}

// Block-wide exclusive scan of one int per thread (1024 threads).
__device__ __forceinline__ int block_excl_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = warp_sums[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const int before = wid ? warp_sums[wid - 1] : 0;
  *total = warp_sums[31];
  __syncthreads();
  return before + x - v;
}

// List of label-1 cells in (head, row, column) order.  One CTA of 1024.
__global__ void __launch_bounds__(1024) compact_partial(const int8_t* __restrict__ labels, int64_t n_cells,
                                                        int32_t* __restrict__ list, Stats* st) {
  int base_out = 0;
  for (int64_t base = 0; base < n_cells; base += 1024) {
    const int64_t i = base + threadIdx.x;
    const int f = (i < n_cells && labels[i] == 1) ? 1 : 0;
    int total;
    const int ex = block_excl_scan(f, &total);
    if (f) list[base_out + ex] = static_cast<int32_t>(i);
    base_out += total;
  }
  if (threadIdx.x == 0) st->n1 = base_out;
}

__device__ __forceinline__ bool blocks_equal(const MaskParams& p, int64_t cell_a, int64_t cell_b, int lane) {
  const int64_t per_head = static_cast<int64_t>(p.nC) * p.nR;
  const int ha = static_cast<int>(cell_a / per_head), hb = static_cast<int>(cell_b / per_head);
  const int ra = static_cast<int>((cell_a / p.nC) % p.nR), rb = static_cast<int>((cell_b / p.nC) % p.nR);
  const int ca = static_cast<int>(cell_a % p.nC), cb = static_cast<int>(cell_b % p.nC);
  bool eq = true;
  // 128 rows x 8 uint4 per row = 1024 uint4; 32 per lane
  for (int i = lane; i < B * 8; i += 32) {
    const int row = i >> 3, v = i & 7;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(dense_block_row(p, ha, ra, ca, row)) + v);
    const uint4 y = __ldg(reinterpret_cast<const uint4*>(dense_block_row(p, hb, rb, cb, row)) + v);
    eq &= nz_bytes(x.x) == nz_bytes(y.x) && nz_bytes(x.y) == nz_bytes(y.y) && nz_bytes(x.z) == nz_bytes(y.z) &&
          nz_bytes(x.w) == nz_bytes(y.w);
  }
  return __all_sync(0xffffffffu, eq);
}

// For each label-1 cell k of the list, the first list entry with the same
// bytes (possibly k itself).  One warp per entry; hashes filter, a full byte
// compare decides.
__global__ void find_first_equal(MaskParams p, const int32_t* __restrict__ list, int32_t n1,
                                 const uint64_t* __restrict__ hashes, int32_t* __restrict__ rep) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t k = warp_global; k < n1; k += nwarps) {
    const int32_t cell = list[k];
    const uint64_t hk = hashes[cell];
    int32_t found = -1;
    for (int64_t base = 0; base <= k && found < 0; base += 32) {
      const int64_t j = base + lane;
      const bool cand = j <= k && hashes[list[j]] == hk;
      uint32_t m = __ballot_sync(0xffffffffu, cand);
      while (m && found < 0) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        const int64_t jj = base + b;
        if (jj == k || blocks_equal(p, list[jj], cell, lane)) found = static_cast<int32_t>(jj);
      }
    }
    if (lane == 0) rep[k] = found;
  }
}

// Stack slots: new entries numbered in list order; duplicates take their
// first occurrence's slot.  One CTA of 1024.
__global__ void __launch_bounds__(1024) assign_slots(const int32_t* __restrict__ rep, int32_t n1,
                                                     int32_t* __restrict__ new_id, Stats* st) {
  int base_out = 0;
  for (int base = 0; base < n1; base += 1024) {
    const int k = base + threadIdx.x;
    const int f = (k < n1 && rep[k] == k) ? 1 : 0;
    int total;
    const int ex = block_excl_scan(f, &total);
    if (k < n1) new_id[k] = f ? base_out + ex : -1;
    base_out += total;
  }
  if (threadIdx.x == 0) st->P = base_out;
}

__global__ void scatter_slots(const int32_t* __restrict__ list, const int32_t* __restrict__ rep,
                              const int32_t* __restrict__ new_id, int32_t n1, int32_t* __restrict__ slot_of_cell) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k >= n1) return;
  slot_of_cell[list[k]] = new_id[rep[k]];
}

// The stacked blocks as bits for the attention kernels: one thread per
// 32 columns of a row, bit j of the word = byte j of those columns.
__global__ void __launch_bounds__(256) pack_stack_bits(const uint8_t* __restrict__ stack, int64_t n_words,
                                                       uint32_t* __restrict__ bits) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(stack + i * 32);
    const uint4 a = src[0], b = src[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) out |= ((w[j >> 2] >> ((j & 3) * 8)) & 0xFFu) ? (1u << j) : 0u;
    bits[i] = out;
  }
}

// Copy each new partial block into its stack slot as 0/1 bytes (transposed
// for the dkv orientation).  One CTA of 256 threads per list entry.
__global__ void __launch_bounds__(256) copy_stack(MaskParams p, const int32_t* __restrict__ list,
                                                  const int32_t* __restrict__ new_id, int32_t n1,
                                                  uint8_t* __restrict__ stack) {
  __shared__ uint8_t tile[B][B + 4];
  for (int64_t k = blockIdx.x; k < n1; k += gridDim.x) {
    const int32_t slot = new_id[k];
    if (slot < 0) continue;  // uniform across the CTA
    const int64_t cell = list[k];
    const int64_t per_head = static_cast<int64_t>(p.nC) * p.nR;
    const int h = static_cast<int>(cell / per_head);
    const int r = static_cast<int>((cell / p.nC) % p.nR);
    const int c = static_cast<int>(cell % p.nC);
    uint8_t* dst = stack + static_cast<size_t>(slot) * B * B;
    if (p.orient == BSA_ORIENT_FWD) {
      for (int i = threadIdx.x; i < B * 8; i += blockDim.x) {
        const int row = i >> 3, v = i & 7;
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(dense_block_row(p, h, r, c, row)) + v);
        const uint4 y = make_uint4(nz_bytes(x.x), nz_bytes(x.y), nz_bytes(x.z), nz_bytes(x.w));
        reinterpret_cast<uint4*>(dst + row * B)[v] = y;
      }
    } else {
      for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int row = i >> 7, col = i & 127;
        tile[row][col] = dense_block_row(p, h, r, c, row)[col] != 0 ? 1 : 0;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < B * B; i += blockDim.x) {
        const int row = i >> 7, col = i & 127;
        dst[row * B + col] = tile[col][row];
      }
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void store_idx(void* base, int bytes, int64_t i, int32_t v) {
  if (bytes == 1) static_cast<int8_t*>(base)[i] = static_cast<int8_t>(v);
  else if (bytes == 2) static_cast<int16_t*>(base)[i] = static_cast<int16_t>(v);
  else static_cast<int32_t*>(base)[i] = v;
}

// Final MaskInfo rows: one thread per block row writes block_mask,
// data_next and mask_next (shrunk or not) in their final integer types.
__global__ void write_rows(const int8_t* __restrict__ labels, const int32_t* __restrict__ slot_of_cell,
                           int32_t nC, int64_t n_rows, int32_t width, int32_t shrink, int8_t* __restrict__ bm,
                           void* dn, int dn_bytes, void* mn, int mn_bytes) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= n_rows) return;
  const int8_t* L = labels + row * nC;
  const int64_t out0 = row * width;
  if (shrink) {
    int t = 0, last = 0;
    for (int c = 0; c < nC; ++c) {
      const int8_t v = L[c];
      if (v == 0) continue;
      bm[out0 + t] = v;
      store_idx(dn, dn_bytes, out0 + t, c);
      if (mn) store_idx(mn, mn_bytes, out0 + t, v == 1 ? slot_of_cell[row * nC + c] : 0);
      last = c;
      ++t;
    }
    for (; t < width; ++t) {
      bm[out0 + t] = 0;
      store_idx(dn, dn_bytes, out0 + t, last);
      if (mn) store_idx(mn, mn_bytes, out0 + t, 0);
    }
  } else {
    int last = -1;
    for (int c = 0; c < nC; ++c)
      if (L[c] != 0) last = c;
    int nxt = -1;
    for (int c = nC - 1; c >= 0; --c) {
      const int8_t v = L[c];
      int d;
      if (v != 0) {
        nxt = c;
        d = c;
      } else {
        d = nxt >= 0 ? nxt : (last >= 0 ? last : 0);
      }
      bm[out0 + c] = v;
      store_idx(dn, dn_bytes, out0 + c, d);
      if (mn) store_idx(mn, mn_bytes, out0 + c, v == 1 ? slot_of_cell[row * nC + c] : 0);
    }
  }
}

__global__ void iota_i32(int32_t* __restrict__ out, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) out[i] = static_cast<int32_t>(i);
}

// Rows ordered by decreasing number of non-empty blocks (stable), for a
// longest-first work order.  Counting sort in one CTA of 1024.
__global__ void __launch_bounds__(1024) order_rows(const int32_t* __restrict__ row_len, int32_t n_rows,
                                                   int32_t max_len, int32_t* __restrict__ hist,
                                                   int32_t* __restrict__ order) {
  for (int i = threadIdx.x; i <= max_len; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n_rows; i += blockDim.x) atomicAdd(&hist[max_len - row_len[i]], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i <= max_len; ++i) {
      const int c = hist[i];
      hist[i] = run;
      run += c;
    }
  }
  __syncthreads();
  // stable placement: one thread walks the rows in order
  if (threadIdx.x == 0) {
    for (int i = 0; i < n_rows; ++i) order[hist[max_len - row_len[i]]++] = i;
  }
}

int idx_bytes(int64_t max_value) {
  if (max_value <= 127) return 1;
  if (max_value <= 32767) return 2;
  return 4;
}

// Scratch memory of one compile, from the library's stream-ordered pool
// (no device-wide synchronisation on release, unlike cudaFree).
struct DevBuf {
  cudaStream_t s;
  void* p = nullptr;
  explicit DevBuf(cudaStream_t st) : s(st) {}
  ~DevBuf() {
    if (p) pool_free(p, s);
  }
};

}  // namespace

bsa_status mask_compile_impl(const bsa_mask_spec* spec, const bsa_mask_opts* opts, cudaStream_t stream,
                             bsa_mask_info** out) {
  MaskParams p{};
  p.kind = spec->kind;
  p.orient = opts->orientation;
  p.heads = spec->mask_heads;
  p.q_len = spec->q_len;
  p.kv_len = spec->kv_len;
  p.left = spec->local_left;
  p.right = spec->local_right;
  p.chunk = spec->chunk;
  p.dense = spec->dense;
  const int nq = static_cast<int>(spec->q_len / B), nk = static_cast<int>(spec->kv_len / B);
  p.nR = p.orient == BSA_ORIENT_FWD ? nq : nk;
  p.nC = p.orient == BSA_ORIENT_FWD ? nk : nq;
  const int64_t n_rows = static_cast<int64_t>(p.heads) * p.nR;
  const int64_t n_cells = n_rows * p.nC;
  if (n_cells > (int64_t(1) << 30)) return fail(BSA_ERR_UNSUPPORTED, "block grid too large");
  const bool dense = p.kind == BSA_MASK_DENSE;

  DevBuf labels(stream), hashes(stream), stats(stream), list(stream), rep(stream), new_id(stream),
      slot_of_cell(stream), hist(stream);
  cudaError_t e;
#define BSA_CK(x, what)                         \
  do {                                          \
    e = (x);                                    \
    if (e != cudaSuccess) return cuda_fail(e, what); \
  } while (0)
  // all device memory of a compile, scratch and MaskInfo arrays alike, comes
  // from the stream-ordered pool; the final stream synchronisation makes the
  // arrays usable from any stream
#define BSA_ALLOC(ptr, bytes)                                          \
  do {                                                                 \
    void* q_ = nullptr;                                                \
    const bsa_status s_ = pool_alloc(&q_, (bytes), stream);            \
    if (s_ != BSA_OK) return s_;                                       \
    (ptr) = static_cast<decltype(ptr)>(q_);                            \
  } while (0)

  BSA_ALLOC(labels.p, n_cells);
  BSA_ALLOC(stats.p, sizeof(Stats));
  BSA_CK(cudaMemsetAsync(stats.p, 0, sizeof(Stats), stream), "clear stats");

  auto* info = new bsa_mask_info();
  struct Guard {
    bsa_mask_info*& i;
    bool keep = false;
    ~Guard() {
      if (!keep) bsa_mask_info_destroy(i);
    }
  } guard{info};
  info->kind = p.kind;
  info->orientation = p.orient;
  info->shrink = opts->shrink;
  info->heads = p.heads;
  info->rows = p.nR;
  info->cols = p.nC;
  info->q_len = p.q_len;
  info->kv_len = p.kv_len;
  info->local_left = p.left;
  info->local_right = p.right;
  info->chunk = p.chunk;
  BSA_ALLOC(info->row_len, n_rows * sizeof(int32_t));
  BSA_ALLOC(info->row_order, n_rows * sizeof(int32_t));
  BSA_ALLOC(info->q_sequence, p.q_len * sizeof(int32_t));

  const int grid_cells = static_cast<int>(std::min<int64_t>(n_cells, 152 * 64));
  Stats* st = static_cast<Stats*>(stats.p);
  if (dense) {
    BSA_ALLOC(hashes.p, n_cells * sizeof(uint64_t));
    classify_dense<<<grid_cells, 256, 0, stream>>>(p, static_cast<int8_t*>(labels.p),
                                                  static_cast<uint64_t*>(hashes.p), n_cells);
  } else {
    classify_computable<<<grid_cells, B, 0, stream>>>(p, static_cast<int8_t*>(labels.p), n_cells);
  }
  BSA_CK(cudaGetLastError(), "classify launch");
  row_pass<<<static_cast<unsigned>((n_rows + 127) / 128), 128, 0, stream>>>(
      static_cast<int8_t*>(labels.p), p.nC, n_rows, info->row_len, st);
  BSA_CK(cudaGetLastError(), "row_pass launch");
  if (dense) {
    BSA_ALLOC(list.p, n_cells * sizeof(int32_t));
    compact_partial<<<1, 1024, 0, stream>>>(static_cast<int8_t*>(labels.p), n_cells,
                                            static_cast<int32_t*>(list.p), st);
    BSA_CK(cudaGetLastError(), "compact launch");
  }
  Stats hs{};
  BSA_CK(cudaMemcpyAsync(&hs, st, sizeof(Stats), cudaMemcpyDeviceToHost, stream), "read stats");
  BSA_CK(cudaStreamSynchronize(stream), "mask compile sync");

  if (dense && hs.n1 > 0) {
    BSA_ALLOC(rep.p, hs.n1 * sizeof(int32_t));
    BSA_ALLOC(new_id.p, hs.n1 * sizeof(int32_t));
    BSA_ALLOC(slot_of_cell.p, n_cells * sizeof(int32_t));
    const int warps_per_cta = 8;
    const int ctas = static_cast<int>(std::min<int64_t>((hs.n1 + warps_per_cta - 1) / warps_per_cta, 152 * 16));
    find_first_equal<<<ctas, 32 * warps_per_cta, 0, stream>>>(p, static_cast<int32_t*>(list.p), hs.n1,
                                                              static_cast<uint64_t*>(hashes.p),
                                                              static_cast<int32_t*>(rep.p));
    BSA_CK(cudaGetLastError(), "dedup launch");
    assign_slots<<<1, 1024, 0, stream>>>(static_cast<int32_t*>(rep.p), hs.n1, static_cast<int32_t*>(new_id.p), st);
    BSA_CK(cudaGetLastError(), "slots launch");
    scatter_slots<<<(hs.n1 + 255) / 256, 256, 0, stream>>>(static_cast<int32_t*>(list.p),
                                                           static_cast<int32_t*>(rep.p),
                                                           static_cast<int32_t*>(new_id.p), hs.n1,
                                                           static_cast<int32_t*>(slot_of_cell.p));
    BSA_CK(cudaGetLastError(), "scatter launch");
    BSA_CK(cudaMemcpyAsync(&hs.P, &st->P, sizeof(int32_t), cudaMemcpyDeviceToHost, stream), "read P");
    BSA_CK(cudaStreamSynchronize(stream), "mask compile sync");
    BSA_ALLOC(info->partial, static_cast<size_t>(hs.P) * B * B);
    copy_stack<<<static_cast<unsigned>(std::min<int64_t>(hs.n1, 152 * 16)), 256, 0, stream>>>(
        p, static_cast<int32_t*>(list.p), static_cast<int32_t*>(new_id.p), hs.n1, info->partial);
    BSA_CK(cudaGetLastError(), "stack copy launch");
    const int64_t n_words = static_cast<int64_t>(hs.P) * B * (B / 32);
    BSA_ALLOC(info->partial_bits, n_words * sizeof(uint32_t));
    pack_stack_bits<<<static_cast<unsigned>(std::min<int64_t>((n_words + 255) / 256, 152 * 16)), 256, 0, stream>>>(
        info->partial, n_words, info->partial_bits);
    BSA_CK(cudaGetLastError(), "stack bits launch");
  } else if (dense) {
    hs.P = 0;
    BSA_ALLOC(info->partial, 16);
    BSA_ALLOC(info->partial_bits, 16);
  }

  const int32_t width = opts->shrink ? hs.width : p.nC;
  info->width = width;
  info->n_empty = static_cast<int64_t>(hs.n_empty);
  info->n_partial = static_cast<int64_t>(hs.n_partial);
  info->n_full = static_cast<int64_t>(hs.n_full);
  info->num_partial = dense ? hs.P : 0;
  info->data_next_bytes = idx_bytes(hs.max_col);
  info->mask_next_bytes = dense ? idx_bytes(hs.P > 0 ? hs.P - 1 : 0) : 0;
  const size_t n_out = static_cast<size_t>(n_rows) * width;
  const size_t alloc_n = n_out ? n_out : 1;
  BSA_ALLOC(info->block_mask, alloc_n);
  BSA_ALLOC(info->data_next, alloc_n * info->data_next_bytes);
  if (dense) BSA_ALLOC(info->mask_next, alloc_n * info->mask_next_bytes);
  if (dense && !slot_of_cell.p) {
    BSA_ALLOC(slot_of_cell.p, n_cells * sizeof(int32_t));
    BSA_CK(cudaMemsetAsync(slot_of_cell.p, 0, n_cells * sizeof(int32_t), stream), "clear slots");
  }
  if (n_out) {
    write_rows<<<static_cast<unsigned>((n_rows + 127) / 128), 128, 0, stream>>>(
        static_cast<int8_t*>(labels.p), static_cast<int32_t*>(slot_of_cell.p), p.nC, n_rows, width, opts->shrink,
        info->block_mask, info->data_next, info->data_next_bytes, info->mask_next, info->mask_next_bytes);
    BSA_CK(cudaGetLastError(), "write_rows launch");
  }
  iota_i32<<<static_cast<unsigned>((p.q_len + 255) / 256), 256, 0, stream>>>(info->q_sequence, p.q_len);
  BSA_CK(cudaGetLastError(), "iota launch");
  BSA_ALLOC(hist.p, (p.nC + 1) * sizeof(int32_t));
  order_rows<<<1, 1024, 0, stream>>>(info->row_len, static_cast<int32_t>(n_rows), p.nC,
                                     static_cast<int32_t*>(hist.p), info->row_order);
  BSA_CK(cudaGetLastError(), "order_rows launch");
  // host copies of the row lengths and order (for launch-time tile
  // schedules), in stream order, then one synchronisation: a returned
  // MaskInfo is complete
  info->row_len_h.resize(static_cast<size_t>(n_rows));
  info->row_order_h.resize(static_cast<size_t>(n_rows));
  BSA_CK(cudaMemcpyAsync(info->row_len_h.data(), info->row_len, n_rows * sizeof(int32_t), cudaMemcpyDeviceToHost,
                         stream),
         "copy row_len");
  BSA_CK(cudaMemcpyAsync(info->row_order_h.data(), info->row_order, n_rows * sizeof(int32_t),
                         cudaMemcpyDeviceToHost, stream),
         "copy row_order");
  BSA_CK(cudaStreamSynchronize(stream), "mask compile sync");
#undef BSA_ALLOC
#undef BSA_CK
  guard.keep = true;
  *out = info;
  return BSA_OK;
}

}  // namespace bsa
