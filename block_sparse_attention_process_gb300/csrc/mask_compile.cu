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
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
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
  uint64_t hash_mask;  // bits of the block hash kept (all; fewer only to test the dedup's collision path)
};

struct Stats {
  unsigned long long n_empty, n_partial, n_full;
  int32_t width;    // max non-empty blocks in a row
  int32_t max_col;  // largest non-empty column index (0 if none)
  int32_t n1;       // number of label-1 cells
  int32_t P;        // stack depth
};
static_assert(sizeof(Stats) % 4 == 0, "Stats is read back as 32-bit words");

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
// The same launch clears the grid-wide counts (which the row pass, the next
// launch, accumulates) and writes q_sequence (the identity).
__global__ void classify_computable(MaskParams p, int8_t* __restrict__ labels, int64_t n_cells, Stats* st,
                                    int32_t* __restrict__ q_sequence) {
  if (blockIdx.x == 0 && threadIdx.x == 0) *st = Stats{};
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.q_len;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    q_sequence[i] = static_cast<int32_t>(i);
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

// The 64 visibility bits of 64 mask bytes (one bit per byte, nonzero =
// visible): bytes that are all 0/1 skip the normalisation; the multiply
// gathers the low bits of a word's four 0/1 bytes into one nibble.
__device__ __forceinline__ uint64_t visibility_bits(const uint4 (&w)[4]) {
  uint32_t x[16] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w,
                    w[2].x, w[2].y, w[2].z, w[2].w, w[3].x, w[3].y, w[3].z, w[3].w};
  uint32_t high = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) high |= x[i];
  if (high & 0xFEFEFEFEu) {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = nz_bytes(x[i]);
  }
  uint64_t bits = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) bits |= static_cast<uint64_t>((x[i] * 0x08040201u) >> 24) << (4 * i);
  return bits;
}

// Dense classifier: each CTA (256 threads) takes two cells at a time, every
// thread loading 64 bytes (half an element row) of both before using any,
// so that 32 KiB per CTA are in flight.  A thread reduces its bytes to 64
// visibility bits: any() / all() of the block are warp votes on them, and
// the block's hash is an order-free sum of mix64(bits ^ position) over the
// threads (the same value for every thread layout).  One barrier per pair
// of cells: every warp writes its own partials, in one of two buffers by
// iteration parity, and two threads combine them after the barrier.
__global__ void __launch_bounds__(256, 4) classify_dense(MaskParams p, int8_t* __restrict__ labels,
                                                        uint64_t* __restrict__ hashes, int64_t n_cells) {
  __shared__ uint64_t red[2][2][8];    // [buffer][cell][warp] hash partial sums
  __shared__ uint32_t vote[2][2][8];   // [buffer][cell][warp] bit 0 any, bit 1 all
  const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t pos_key = static_cast<uint64_t>(threadIdx.x + 1) * 0x9E3779B97F4A7C15ull;
  int buf = 0;
  for (int64_t cell0 = static_cast<int64_t>(blockIdx.x) * 2; cell0 < n_cells;
       cell0 += static_cast<int64_t>(gridDim.x) * 2, buf ^= 1) {
    uint4 w[2][4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t cell = cell0 + k < n_cells ? cell0 + k : cell0;
      const int c = static_cast<int>(cell % p.nC);
      const int r = static_cast<int>((cell / p.nC) % p.nR);
      const int h = static_cast<int>(cell / (static_cast<int64_t>(p.nC) * p.nR));
      const uint4* src = reinterpret_cast<const uint4*>(dense_block_row(p, h, r, c, row) + half * 64);
#pragma unroll
      for (int v = 0; v < 4; ++v) w[k][v] = __ldg(src + v);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint64_t bits = visibility_bits(w[k]);
      uint64_t hs = mix64(bits ^ pos_key);
      for (int o = 16; o > 0; o >>= 1) hs += __shfl_xor_sync(0xffffffffu, hs, o);
      const bool any = __any_sync(0xffffffffu, bits != 0);
      const bool all = __all_sync(0xffffffffu, bits == ~0ull);
      if (lane == 0) {
        red[buf][k][warp] = hs;
        vote[buf][k][warp] = (any ? 1u : 0u) | (all ? 2u : 0u);
      }
    }
    __syncthreads();
    if (threadIdx.x < 2 && cell0 + threadIdx.x < n_cells) {
      const int k = threadIdx.x;
      uint64_t t = 0;
      uint32_t any = 0, all = 2;
      for (int i = 0; i < 8; ++i) {
        t += red[buf][k][i];
        any |= vote[buf][k][i] & 1u;
        all &= vote[buf][k][i] & 2u;
      }
      labels[cell0 + k] = all ? 2 : (any ? 1 : 0);
      hashes[cell0 + k] = t & p.hash_mask;
    }
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

// ---------------------------------------------------------------- scans
// Device-wide exclusive prefix sums in three launches: per-chunk totals
// (chunk_sums, many CTAs), an exclusive scan of the chunk totals
// (scan_chunk_sums, one CTA: n / 1024 values), then each chunk's own scan
// plus its offset (chunk_write, many CTAs).  The number of elements may
// live in device memory (an earlier kernel's count), so nothing waits for
// the host.
constexpr int kChunk = 1024;

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

// Element count of a scan: a host value, or one read from device memory.
struct Count {
  int64_t host;
  const int32_t* dev;
  __device__ __forceinline__ int64_t get() const { return dev ? static_cast<int64_t>(*dev) : host; }
};

template <class V>
__global__ void __launch_bounds__(kChunk) chunk_sums(V val, Count cnt, int64_t n_chunks, int32_t* __restrict__ sums) {
  const int64_t n = cnt.get();
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const int64_t i = c * kChunk + threadIdx.x;
    const int v = i < n ? val(i) : 0;
    int total;
    (void)block_excl_scan(v, &total);
    if (threadIdx.x == 0) sums[c] = total;
  }
}

// Exclusive scan of `n` chunk totals in place (one CTA of 1024); the grand
// total goes to *total when it is not null.
__global__ void __launch_bounds__(kChunk) scan_chunk_sums(int32_t* __restrict__ sums, int64_t n,
                                                         int32_t* __restrict__ total) {
  int run = 0;
  for (int64_t base = 0; base < n; base += kChunk) {
    const int64_t i = base + threadIdx.x;
    const int v = i < n ? sums[i] : 0;
    int t;
    const int ex = block_excl_scan(v, &t);
    if (i < n) sums[i] = run + ex;
    run += t;
  }
  if (threadIdx.x == 0 && total) *total = run;
}

// Calls out(i, v, position) for every element, position = the exclusive
// prefix sum of the values before i.
template <class V, class W>
__global__ void __launch_bounds__(kChunk) chunk_write(V val, W out, Count cnt, int64_t n_chunks,
                                                     const int32_t* __restrict__ offs) {
  const int64_t n = cnt.get();
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const int64_t i = c * kChunk + threadIdx.x;
    const int v = i < n ? val(i) : 0;
    int total;
    const int ex = block_excl_scan(v, &total);
    if (i < n) out(i, v, offs[c] + ex);
  }
}

// ---------------------------------------------------------------- dedup
// Value / output functors of the scans.
struct IsPartial {  // label-1 cells
  const int8_t* labels;
  __device__ __forceinline__ int operator()(int64_t i) const { return labels[i] == 1 ? 1 : 0; }
};
struct ListOut {  // the list of label-1 cells, in (head, row, column) order
  int32_t* list;
  __device__ __forceinline__ void operator()(int64_t i, int v, int pos) const {
    if (v) list[pos] = static_cast<int32_t>(i);
  }
};
struct IsNew {  // a list entry that is its own first occurrence
  const int32_t* rep;
  __device__ __forceinline__ int operator()(int64_t k) const { return rep[k] == k ? 1 : 0; }
};
struct SlotOut {  // stack slots numbered in list order
  int32_t* new_id;
  __device__ __forceinline__ void operator()(int64_t k, int v, int pos) const { new_id[k] = v ? pos : -1; }
};

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

// Open-addressing table from a block's hash to the smallest list index
// holding that hash.  An entry whose hash is the empty marker is stored
// under hash ^ 1: keys only select candidates, equality is always decided
// by comparing the bytes.
struct HashSlot {
  unsigned long long key;
  unsigned int min_k;
  unsigned int pad;
};
constexpr unsigned long long kEmptyKey = ~0ull;

__device__ __forceinline__ unsigned long long table_key(uint64_t h) { return h == kEmptyKey ? h ^ 1ull : h; }

__global__ void hash_insert(const int32_t* __restrict__ list, const uint64_t* __restrict__ hashes,
                            const int32_t* __restrict__ n1_dev, HashSlot* __restrict__ tab, uint64_t mask) {
  const int64_t n1 = *n1_dev;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n1;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const unsigned long long key = table_key(hashes[list[k]]);
    uint64_t slot = (key >> 20) & mask;
    for (uint64_t probe = 0; probe <= mask; ++probe) {  // the table has more slots than entries
      const unsigned long long prev = atomicCAS(&tab[slot].key, kEmptyKey, key);
      if (prev == kEmptyKey || prev == key) {
        atomicMin(&tab[slot].min_k, static_cast<unsigned int>(k));
        break;
      }
      slot = (slot + 1) & mask;
    }
  }
}

// For each list entry k, the first list entry with the same bytes (possibly
// k itself): the table's smallest index with k's hash, confirmed by a byte
// compare; a hash shared by different blocks falls back to a scan of the
// earlier entries.  One warp per entry.
__global__ void hash_resolve(MaskParams p, const int32_t* __restrict__ list, const uint64_t* __restrict__ hashes,
                             const int32_t* __restrict__ n1_dev, const HashSlot* __restrict__ tab, uint64_t mask,
                             int32_t* __restrict__ rep) {
  const int lane = threadIdx.x & 31;
  const int64_t n1 = *n1_dev;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t k = warp_global; k < n1; k += nwarps) {
    const int32_t cell = list[k];
    const uint64_t hk = hashes[cell];
    const unsigned long long key = table_key(hk);
    uint64_t slot = (key >> 20) & mask;
    int64_t cand = k;
    for (uint64_t probe = 0; probe <= mask; ++probe) {
      const unsigned long long t = tab[slot].key;
      if (t == key) {
        cand = tab[slot].min_k;
        break;
      }
      if (t == kEmptyKey) break;  // not reached: every entry was inserted
      slot = (slot + 1) & mask;
    }
    int64_t found = -1;
    if (cand >= k) {
      found = k;
    } else if (blocks_equal(p, list[cand], cell, lane)) {
      found = cand;
    } else {
      // two different blocks with one hash: the first equal earlier entry
      for (int64_t base = cand + 1; base <= k && found < 0; base += 32) {
        const int64_t j = base + lane;
        const bool c = j <= k && hashes[list[j]] == hk;
        uint32_t m = __ballot_sync(0xffffffffu, c);
        while (m && found < 0) {
          const int b = __ffs(m) - 1;
          m &= m - 1;
          const int64_t jj = base + b;
          if (jj == k || blocks_equal(p, list[jj], cell, lane)) found = jj;
        }
      }
    }
    if (lane == 0) rep[k] = static_cast<int32_t>(found);
  }
}

__global__ void scatter_slots(const int32_t* __restrict__ list, const int32_t* __restrict__ rep,
                              const int32_t* __restrict__ new_id, const int32_t* __restrict__ n1_dev,
                              int32_t* __restrict__ slot_of_cell) {
  const int64_t n1 = *n1_dev;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n1;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x)
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

// Rows ordered by decreasing number of non-empty blocks, ties by row index
// (a stable counting sort, for a longest-first work order): bucket
// b = max_len - row_len.  order_count counts rows per (bucket, chunk of
// 1024 rows); an exclusive scan of those counts, bucket-major, gives each
// (bucket, chunk) its first output position; order_place ranks each chunk's
// rows within their bucket by a bitonic sort of (bucket, row) in shared
// memory and writes them out.
__global__ void order_count(const int32_t* __restrict__ row_len, int64_t n_rows, int32_t max_len, int64_t n_chunks,
                            int32_t* __restrict__ cnt) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_rows;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    atomicAdd(&cnt[static_cast<int64_t>(max_len - row_len[i]) * n_chunks + i / kChunk], 1);
}

struct ArrayVal {
  const int32_t* a;
  __device__ __forceinline__ int operator()(int64_t i) const { return a[i]; }
};
struct ArrayOut {  // exclusive prefix sums in place of the values
  int32_t* a;
  __device__ __forceinline__ void operator()(int64_t i, int, int pos) const { a[i] = pos; }
};

// Ascending bitonic sort of kChunk keys in shared memory, one per thread.
__device__ __forceinline__ void bitonic_sort(unsigned long long* key, int t) {
  __syncthreads();
  for (int k = 2; k <= kChunk; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int partner = t ^ j;
      if (partner > t) {
        const unsigned long long a = key[t], b = key[partner];
        const bool up = (t & k) == 0;
        if ((a > b) == up) {
          key[t] = b;
          key[partner] = a;
        }
      }
      __syncthreads();
    }
}

__global__ void __launch_bounds__(kChunk) order_place(const int32_t* __restrict__ row_len, int64_t n_rows,
                                                     int32_t max_len, int64_t n_chunks,
                                                     const int32_t* __restrict__ offs, int32_t* __restrict__ order) {
  __shared__ unsigned long long key[kChunk];
  __shared__ int start[kChunk];
  const int t = threadIdx.x;
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const int64_t i = c * kChunk + t;
    key[t] = i < n_rows ? (static_cast<unsigned long long>(max_len - row_len[i]) << 32) | static_cast<unsigned>(t)
                        : ~0ull;
    bitonic_sort(key, t);
    const unsigned long long me = key[t];
    const uint32_t bucket = static_cast<uint32_t>(me >> 32);
    start[t] = (t == 0 || static_cast<uint32_t>(key[t - 1] >> 32) != bucket) ? t : 0;
    __syncthreads();
    // inclusive max-scan: the first position of each thread's bucket
    for (int o = 1; o < kChunk; o <<= 1) {
      const int v = t >= o ? start[t - o] : 0;
      __syncthreads();
      if (v > start[t]) start[t] = v;
      __syncthreads();
    }
    if (me != ~0ull)
      order[offs[static_cast<int64_t>(bucket) * n_chunks + c] + (t - start[t])] =
          static_cast<int32_t>(c * kChunk + static_cast<int64_t>(me & 0xFFFFFFFFull));
    __syncthreads();
  }
}

// The same order for at most kChunk rows in one CTA: sorted by (bucket,
// row), a row's place in the sorted keys is its place in the order.
__global__ void __launch_bounds__(kChunk) order_small(const int32_t* __restrict__ row_len, int32_t n_rows,
                                                     int32_t max_len, int32_t* __restrict__ order) {
  __shared__ unsigned long long key[kChunk];
  const int t = threadIdx.x;
  key[t] = t < n_rows ? (static_cast<unsigned long long>(max_len - row_len[t]) << 32) | static_cast<unsigned>(t)
                      : ~0ull;
  bitonic_sort(key, t);
  if (t < n_rows) order[t] = static_cast<int32_t>(key[t] & 0xFFFFFFFFull);
}

// BSA_DEDUP_HASH_BITS=n (0..63) keeps only the low n bits of every block
// hash, so that different blocks share hashes and the dedup has to settle
// them by comparing bytes (for testing that path; the default keeps all 64).
uint64_t dedup_hash_mask() {
  static const uint64_t m = [] {
    const char* e = std::getenv("BSA_DEDUP_HASH_BITS");
    if (!e || !*e) return ~0ull;
    const int n = std::atoi(e);
    return n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1));
  }();
  return m;
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

// Small read-backs (the counts and the row arrays) are written by a kernel
// straight into mapped, pinned host memory.  A device-to-host copy is a
// copy-engine transfer, and while other streams keep large host<->device
// copies in flight it waits on them; stores from a kernel do not.  One
// staging buffer for the process, grown on demand (an outgrown one stays
// allocated: releasing pinned memory can synchronise the device), used
// under a lock from the copy kernel's launch to the host's read.
struct ReadBack {
  void* host;
  const void* dev;
  size_t bytes;  // a multiple of 4
};

std::mutex g_stage_mu;
uint32_t* g_stage = nullptr;
size_t g_stage_words = 0;

constexpr int kMaxReadBack = 2;
struct WordCopies {
  uint32_t* dst[kMaxReadBack];
  const uint32_t* src[kMaxReadBack];
  int64_t n[kMaxReadBack];
  int count;
};

__global__ void words_to_host(WordCopies w) {
  for (int k = 0; k < w.count; ++k)
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < w.n[k];
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
      w.dst[k][i] = w.src[k][i];
}

bsa_status read_back(cudaStream_t stream, std::initializer_list<ReadBack> parts) {
  if (parts.size() > static_cast<size_t>(kMaxReadBack)) return fail(BSA_ERR_UNSUPPORTED, "too many read-back parts");
  size_t words = 0;
  for (const ReadBack& r : parts) words += r.bytes / 4;
  std::lock_guard<std::mutex> lk(g_stage_mu);
  cudaError_t e;
  if (words > g_stage_words) {
    const size_t cap = std::max<size_t>(std::max<size_t>(words, 2 * g_stage_words), 16384);
    void* h = nullptr;
    e = cudaHostAlloc(&h, cap * 4, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_fail(e, "allocate the read-back buffer");
    g_stage = static_cast<uint32_t*>(h);
    g_stage_words = cap;
  }
  void* d = nullptr;
  e = cudaHostGetDevicePointer(&d, g_stage, 0);
  if (e != cudaSuccess) return cuda_fail(e, "map the read-back buffer");
  // one launch copies every part
  WordCopies w{};
  size_t off = 0;
  int64_t most = 0;
  for (const ReadBack& r : parts) {
    w.dst[w.count] = static_cast<uint32_t*>(d) + off;
    w.src[w.count] = static_cast<const uint32_t*>(r.dev);
    w.n[w.count] = static_cast<int64_t>(r.bytes / 4);
    most = std::max(most, w.n[w.count]);
    off += r.bytes / 4;
    ++w.count;
  }
  if (most > 0)
    words_to_host<<<static_cast<unsigned>(std::min<int64_t>((most + 255) / 256, 152 * 4)), 256, 0, stream>>>(w);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "mask compile read-back");
  off = 0;
  for (const ReadBack& r : parts) {
    if (r.bytes) std::memcpy(r.host, g_stage + off, r.bytes);
    off += r.bytes / 4;
  }
  return BSA_OK;
}

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
  p.hash_mask = dedup_hash_mask();
  const int nq = static_cast<int>(spec->q_len / B), nk = static_cast<int>(spec->kv_len / B);
  p.nR = p.orient == BSA_ORIENT_FWD ? nq : nk;
  p.nC = p.orient == BSA_ORIENT_FWD ? nk : nq;
  const int64_t n_rows = static_cast<int64_t>(p.heads) * p.nR;
  const int64_t n_cells = n_rows * p.nC;
  if (n_cells > (int64_t(1) << 30)) return fail(BSA_ERR_UNSUPPORTED, "block grid too large");
  const bool dense = p.kind == BSA_MASK_DENSE;

  DevBuf labels(stream), hashes(stream), stats(stream), list(stream), rep(stream), new_id(stream),
      slot_of_cell(stream), hist(stream), csum(stream), csum2(stream), table(stream);
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
  // (a computable mask's classifier clears the counts itself)
  if (dense) BSA_CK(cudaMemsetAsync(stats.p, 0, sizeof(Stats), stream), "clear stats");

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
    classify_computable<<<grid_cells, B, 0, stream>>>(p, static_cast<int8_t*>(labels.p), n_cells, st,
                                                       info->q_sequence);
  }
  BSA_CK(cudaGetLastError(), "classify launch");
  row_pass<<<static_cast<unsigned>((n_rows + 127) / 128), 128, 0, stream>>>(
      static_cast<int8_t*>(labels.p), p.nC, n_rows, info->row_len, st);
  BSA_CK(cudaGetLastError(), "row_pass launch");
  const int64_t n_chunks = (n_cells + kChunk - 1) / kChunk;
  const unsigned scan_grid = static_cast<unsigned>(std::min<int64_t>(n_chunks, 152 * 8));
  if (dense) {
    // list of the label-1 cells (its length n1 stays on the device)
    BSA_ALLOC(list.p, n_cells * sizeof(int32_t));
    BSA_ALLOC(csum.p, n_chunks * sizeof(int32_t));
    int32_t* lst = static_cast<int32_t*>(list.p);
    int32_t* cs = static_cast<int32_t*>(csum.p);
    const IsPartial is_partial{static_cast<int8_t*>(labels.p)};
    const Count all_cells{n_cells, nullptr};
    chunk_sums<<<scan_grid, kChunk, 0, stream>>>(is_partial, all_cells, n_chunks, cs);
    scan_chunk_sums<<<1, kChunk, 0, stream>>>(cs, n_chunks, &st->n1);
    chunk_write<<<scan_grid, kChunk, 0, stream>>>(is_partial, ListOut{lst}, all_cells, n_chunks, cs);
    BSA_CK(cudaGetLastError(), "compact launch");
    // first occurrence of each partial block: hash table, then byte compare
    uint64_t tab_n = 64;
    while (tab_n < 2 * static_cast<uint64_t>(n_cells)) tab_n <<= 1;
    BSA_ALLOC(table.p, tab_n * sizeof(HashSlot));
    BSA_CK(cudaMemsetAsync(table.p, 0xFF, tab_n * sizeof(HashSlot), stream), "clear hash table");
    BSA_ALLOC(rep.p, n_cells * sizeof(int32_t));
    BSA_ALLOC(new_id.p, n_cells * sizeof(int32_t));
    BSA_ALLOC(slot_of_cell.p, n_cells * sizeof(int32_t));
    const int32_t* n1_dev = &st->n1;
    const uint64_t* hsh = static_cast<uint64_t*>(hashes.p);
    HashSlot* tab = static_cast<HashSlot*>(table.p);
    int32_t* rp = static_cast<int32_t*>(rep.p);
    int32_t* nid = static_cast<int32_t*>(new_id.p);
    hash_insert<<<static_cast<unsigned>(std::min<int64_t>((n_cells + 255) / 256, 152 * 16)), 256, 0, stream>>>(
        lst, hsh, n1_dev, tab, tab_n - 1);
    hash_resolve<<<static_cast<unsigned>(std::min<int64_t>((n_cells + 7) / 8, 152 * 16)), 256, 0, stream>>>(
        p, lst, hsh, n1_dev, tab, tab_n - 1, rp);
    BSA_CK(cudaGetLastError(), "dedup launch");
    // stack slots: new blocks numbered in list order, duplicates take their
    // first occurrence's slot
    const IsNew is_new{rp};
    const Count n1_count{0, n1_dev};
    chunk_sums<<<scan_grid, kChunk, 0, stream>>>(is_new, n1_count, n_chunks, cs);
    scan_chunk_sums<<<1, kChunk, 0, stream>>>(cs, n_chunks, &st->P);
    chunk_write<<<scan_grid, kChunk, 0, stream>>>(is_new, SlotOut{nid}, n1_count, n_chunks, cs);
    scatter_slots<<<static_cast<unsigned>(std::min<int64_t>((n_cells + 255) / 256, 152 * 16)), 256, 0, stream>>>(
        lst, rp, nid, n1_dev, static_cast<int32_t*>(slot_of_cell.p));
    BSA_CK(cudaGetLastError(), "slots launch");
  }
  // one synchronisation: the grid width, the largest column, the counts
  // and the stack depth size the MaskInfo arrays
  Stats hs{};
  {
    const bsa_status rs = read_back(stream, {{&hs, st, sizeof(Stats)}});
    if (rs != BSA_OK) return rs;
  }

  if (dense && hs.n1 > 0) {
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
  if (n_out) {
    write_rows<<<static_cast<unsigned>((n_rows + 127) / 128), 128, 0, stream>>>(
        static_cast<int8_t*>(labels.p), static_cast<int32_t*>(slot_of_cell.p), p.nC, n_rows, width, opts->shrink,
        info->block_mask, info->data_next, info->data_next_bytes, info->mask_next, info->mask_next_bytes);
    BSA_CK(cudaGetLastError(), "write_rows launch");
  }
  if (dense) {
    iota_i32<<<static_cast<unsigned>((p.q_len + 255) / 256), 256, 0, stream>>>(info->q_sequence, p.q_len);
    BSA_CK(cudaGetLastError(), "iota launch");
  }
  // rows by decreasing length (stable counting sort; up to kChunk rows, one
  // CTA sorting (bucket, row) keys)
  if (n_rows <= kChunk) {
    order_small<<<1, kChunk, 0, stream>>>(info->row_len, static_cast<int32_t>(n_rows), p.nC, info->row_order);
    BSA_CK(cudaGetLastError(), "row order launch");
  } else {
    const int64_t r_chunks = (n_rows + kChunk - 1) / kChunk;
    const int64_t n_cnt = static_cast<int64_t>(p.nC + 1) * r_chunks;
    BSA_ALLOC(hist.p, n_cnt * sizeof(int32_t));
    int32_t* cnt = static_cast<int32_t*>(hist.p);
    BSA_CK(cudaMemsetAsync(cnt, 0, n_cnt * sizeof(int32_t), stream), "clear row counts");
    order_count<<<static_cast<unsigned>(std::min<int64_t>((n_rows + 255) / 256, 152 * 16)), 256, 0, stream>>>(
        info->row_len, n_rows, p.nC, r_chunks, cnt);
    const int64_t c_chunks = (n_cnt + kChunk - 1) / kChunk;
    BSA_ALLOC(csum2.p, c_chunks * sizeof(int32_t));
    int32_t* cs2 = static_cast<int32_t*>(csum2.p);
    const unsigned g2 = static_cast<unsigned>(std::min<int64_t>(c_chunks, 152 * 8));
    chunk_sums<<<g2, kChunk, 0, stream>>>(ArrayVal{cnt}, Count{n_cnt, nullptr}, c_chunks, cs2);
    scan_chunk_sums<<<1, kChunk, 0, stream>>>(cs2, c_chunks, nullptr);
    chunk_write<<<g2, kChunk, 0, stream>>>(ArrayVal{cnt}, ArrayOut{cnt}, Count{n_cnt, nullptr}, c_chunks, cs2);
    order_place<<<static_cast<unsigned>(std::min<int64_t>(r_chunks, 152 * 8)), kChunk, 0, stream>>>(
        info->row_len, n_rows, p.nC, r_chunks, cnt, info->row_order);
    BSA_CK(cudaGetLastError(), "row order launch");
  }
  // host copies of the row lengths and order (for launch-time tile
  // schedules), in stream order, then one synchronisation: a returned
  // MaskInfo is complete
  info->row_len_h.resize(static_cast<size_t>(n_rows));
  info->row_order_h.resize(static_cast<size_t>(n_rows));
  {
    const size_t nb = static_cast<size_t>(n_rows) * sizeof(int32_t);
    const bsa_status rs = read_back(stream, {{info->row_len_h.data(), info->row_len, nb},
                                             {info->row_order_h.data(), info->row_order, nb}});
    if (rs != BSA_OK) return rs;
  }
#undef BSA_ALLOC
#undef BSA_CK
  guard.keep = true;
  *out = info;
  return BSA_OK;
}

}  // namespace bsa
