// Block-sparse backward attention for sm_103a: the dK/dV launch and the dQ
// launch.
//
// Method: "Flash Attention on a TPU, Line by Line".  "Why does the TPU flash
// attention backward pass run two kernels instead of one?": a key block's
// gradient sums over query blocks (queries innermost) and a query block's
// over key blocks (keys innermost), so there are two grids and the scores
// are rebuilt in each.  "What does the TPU flash attention kernel save for
// the backward pass?": the scores are rebuilt from Q, K and the saved row
// statistics (here one logsumexp per row) and rowsum(dO*O) comes in
// precomputed.  The block walk is MaskInfo's, as in the forward ("Splash
// Attention: When the Mask Stops Being Arithmetic and Becomes the Loop"):
// label-0 blocks are never fetched, label-2 blocks are not masked.
//
// Per block, with P = exp(scale*S - LSE) and dS = P * (dP - Dsum):
//   dK/dV launch (grid: batch, kv head, key block; inner: q heads of the
//   group x query blocks of the dkv MaskInfo row):
//       S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q
//   dQ launch (grid: batch, q head, query block; inner: key blocks):
//       S = Q K^T, dP = dO V^T, dQ += dS K
// dK and dQ take the softmax scale at the end.
//
// GB300 design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer; also the only reader of MaskInfo: it publishes
//               each block's descriptor into a shared-memory ring
//   warp 1      tcgen05 issuer, warp-converged, one elected lane issues
//   warp 2      second TMA producer (V blocks of the dQ launch)
//   warps 4-    kParts elementwise warpgroups (4 for D = 128, 2 for D = 64),
//               one (tile row, 128 / kParts of the score columns) per
//               thread: rebuild P and dS from the scores in TMEM and write
//               them back to TMEM as bf16, where they are the A operand of
//               the accumulating MMAs; each part writes inside its own
//               column range, so the parts never race, and the MMA reads the
//               A operand in per-part pieces.  The dK/dV launch publishes
//               P^T in two halves per thread, so that dV starts on the first
//               half.  At a tile's end the same warps run the epilogue: bf16
//               dK/dV through shared memory and tensor stores, dQ with
//               32-byte stores.
// The dK/dV launch keeps each item's Q in three shared-memory stages and
// its (dO, LSE, Dsum) in two: Q is what the next items need first (their
// S^T), and with two stages its load had only the time of two GEMMs to
// land.  All MMAs are 128 x 128 (full rate on sm_103a).
#include <cmath>

#include "internal.h"
#include "maskinfo_dev.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace bsa {
namespace {

// Both gradient launches split their elementwise work over kParts
// warpgroups, each taking 128 / kParts of the score columns (and D / kParts
// of the output columns at the epilogue), beside one warpgroup of role
// warps (producers, MMA issuer).
template <int D>
struct EwShape {
  static constexpr int kParts = D == 128 ? 4 : 2;
  static constexpr int kCols = 128 / kParts;
  static constexpr int kThreads = 128 + 128 * kParts;
};
template <int D>
using DkvShape = EwShape<D>;
template <int D>
using DqShape = EwShape<D>;
constexpr uint32_t kTmemCols = 512;
constexpr int kInfoRing = 16;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int32_t B, Hq, Hkv, nQ, nK;
  int64_t Sq, Skv;
  float scale, scale_log2;
  // soft cap c (off when cap_scale == 0): scaled score -> c*tanh(s/c), in
  // log2 units cap_log2 * tanh(raw * cap_scale) with cap_scale = scale / c;
  // dS then also carries the factor 1 - tanh^2
  float cap_log2, cap_scale;
  const float* lse;
  const float* dsum;
  void* dq;
  void* dk;
  void* dv;
  const void* kp;  // K and V (for L2 prefetch)
  const void* vp;
  int32_t grad_fp32;
  MaskInfoDev mi;
  int32_t n_tiles;
  // this launch's tile lists (sched_stride entries per CTA), or null for
  // round-robin tiles in longest-first order
  const int4* sched;
  int32_t sched_stride;
  // dK/dV launch with the q heads of a group split over kv_splits CTAs:
  // each writes fp32 partial sums at row split * part_rows + key row of
  // part_dk / part_dv, summed afterwards (kv_splits == 1: direct output)
  int32_t kv_splits;
  int64_t part_rows;
  float* part_dk;
  float* part_dv;
  uint32_t* err;
  uint64_t wait_ns;
};

// One row of 32 fp32 values times `mul`, as bf16, into row `r` of a
// [32 rows, 64 bytes] staging box in the 64-byte swizzle of its tensor map
// (conflict-free: the 8 rows of a quarter warp cover all 32 banks).
__device__ __forceinline__ void stage_row_sw64(uint8_t* box, int r, const uint32_t* v, float mul) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 o;
    o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * mul, __uint_as_float(v[8 * j + 1]) * mul);
    o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * mul, __uint_as_float(v[8 * j + 3]) * mul);
    o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * mul, __uint_as_float(v[8 * j + 5]) * mul);
    o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * mul, __uint_as_float(v[8 * j + 7]) * mul);
    *reinterpret_cast<uint4*>(box + r * 64 + ((j ^ ((r >> 1) & 3)) * 16)) = o;
  }
}

__device__ __forceinline__ void store_row(void* base, int fp32, int64_t row, int D, const uint32_t* v, int c0,
                                          float mul) {
  // 32 consecutive fp32 accumulator values of one row -> output columns [c0, c0+32)
  if (fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + row * D + c0);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      dst[e] = make_float4(__uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                           __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row * D + c0);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint4 o;
      o.x = pack_bf16x2(__uint_as_float(v[8 * e + 0]) * mul, __uint_as_float(v[8 * e + 1]) * mul);
      o.y = pack_bf16x2(__uint_as_float(v[8 * e + 2]) * mul, __uint_as_float(v[8 * e + 3]) * mul);
      o.z = pack_bf16x2(__uint_as_float(v[8 * e + 4]) * mul, __uint_as_float(v[8 * e + 5]) * mul);
      o.w = pack_bf16x2(__uint_as_float(v[8 * e + 6]) * mul, __uint_as_float(v[8 * e + 7]) * mul);
      dst[e] = o;
    }
  }
}

// store_row with 32-byte stores (half the store instructions of the
// row-per-thread pattern) where the output is 32-byte aligned.
__device__ __forceinline__ void store_row_wide(void* base, int fp32, int64_t row, int D, const uint32_t* v, int c0,
                                               float mul) {
  if ((reinterpret_cast<uintptr_t>(base) & 31u) != 0) {
    store_row(base, fp32, row, D, v, c0, mul);
    return;
  }
  if (fp32) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<float*>(base) + row * D + c0);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(__uint_as_float(v[8 * e + i]) * mul);
      st_global_v8(dst + 8 * e, w);
    }
  } else {
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(base) + row * D + c0);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = pack_bf16x2(__uint_as_float(v[16 * e + 2 * i]) * mul, __uint_as_float(v[16 * e + 2 * i + 1]) * mul);
      st_global_v8(dst + 8 * e, w);
    }
  }
}

__device__ __forceinline__ void store_zero_cols(void* base, int fp32, int64_t row, int D, int c0, int n) {
  if (fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + row * D + c0);
    for (int e = 0; e < n / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row * D + c0);
    for (int e = 0; e < n / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
  }
}

// TMEM column of 16-bit A-operand k-step kk when the operand is split into
// parts of kCols columns, each part's kCols/2 packed words at the start of
// its own kCols-column range.
template <int kCols>
__device__ __forceinline__ uint32_t part_a_col(int kk) {
  constexpr int kSteps = kCols / 16;  // k-steps (16 elements = 8 columns) per part
  return static_cast<uint32_t>((kk / kSteps) * kCols + (kk % kSteps) * 8);
}

// Store N (16 or 32) consecutive TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t* r) {
  if constexpr (N == 32) tmem_st32(taddr, r);
  else if constexpr (N == 16) tmem_st16(taddr, r);
  else tmem_st8(taddr, r);
}

// Visibility bits of N (32 or 64) consecutive columns of one row of a stacked block.
template <int N>
__device__ __forceinline__ uint64_t dense_bits(const uint32_t* row_bits, uint32_t c0) {
  // row_bits: the block row's 4 words of visibility bits (c0 a multiple of N)
  if constexpr (N == 64) return __ldg(reinterpret_cast<const unsigned long long*>(row_bits) + (c0 >> 6));
  else return static_cast<uint64_t>(__ldg(row_bits + (c0 >> 5)));
}

// Bits of the columns [c0, c0+64) that lie inside [lo, hi].
__device__ __forceinline__ uint64_t interval_bits_64(int64_t c0, int64_t lo, int64_t hi) {
  const int64_t a = lo > c0 ? lo - c0 : 0;
  const int64_t b = hi < c0 + 63 ? hi - c0 : 63;
  if (b < a) return 0ull;
  const int n = static_cast<int>(b - a + 1);
  const uint64_t run = n >= 64 ? ~0ull : ((1ull << n) - 1ull);
  return run << a;
}

__device__ __forceinline__ uint32_t pack_info(int32_t col, int32_t label, bool first, bool last) {
  return static_cast<uint32_t>(col) | (static_cast<uint32_t>(label) << 16) | (first ? 1u << 20 : 0u) |
         (last ? 1u << 21 : 0u);
}

// ===========================================================================
// dQ launch
// ===========================================================================
constexpr int kDqStagesK = 3;   // S is issued two blocks ahead of the dQ MMA that frees its K
constexpr int kDqStagesV = 2;
constexpr uint32_t kDqColS = 0;     // two S buffers at 0 and 128
constexpr uint32_t kDqColDP = 256;  // dP, then dS (bf16) over it
constexpr uint32_t kDqColQ = 384;   // dQ accumulator

template <int D>
struct __align__(1024) DqSmem {
  static constexpr int kTile = 128 * D * 2;
  uint8_t q[kTile];
  uint8_t dout[kTile];
  uint8_t k[kDqStagesK][kTile];
  uint8_t v[kDqStagesV][kTile];
  uint64_t qo_full, qo_empty;
  uint64_t k_full[kDqStagesK], k_empty[kDqStagesK];
  uint64_t v_full[kDqStagesV], v_empty[kDqStagesV];
  uint64_t s_full[2], dp_full, ds_full;
  uint64_t acc_full, acc_empty, drain, stats_read;
  // per block: {col | label<<16 | first<<20 | last<<21, stack slot, q_sequence of the tile's first
  // query, (b*Hq + hq)*Sq + 128*i = row of the tile's first query}
  uint4 binfo[kInfoRing];
  float stats[2][128];  // LSE and Dsum of the tile's 128 query rows (loaded with Q and dO)
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct DqTile {
  int32_t b, hq, i, hm, n;
  int64_t row_base;
};

__device__ __forceinline__ DqTile dq_decode(const BwdParams& p, int32_t T) {
  DqTile t;
  if (p.mi.heads == 1) {
    const int32_t bh = T % (p.B * p.Hq);
    t.i = p.mi.row_order[T / (p.B * p.Hq)];
    t.b = bh / p.Hq;
    t.hq = bh % p.Hq;
    t.hm = 0;
  } else {
    t.b = T % p.B;
    const int32_t row = p.mi.row_order[T / p.B];
    t.hm = row / p.mi.rows;
    t.i = row % p.mi.rows;
    t.hq = t.hm;
  }
  t.n = p.mi.row_len[t.hm * p.mi.rows + t.i];
  t.row_base = (static_cast<int64_t>(t.hm) * p.mi.rows + t.i) * p.mi.width;
  return t;
}

// The k-th tile of this CTA, from the launch's schedule (or round-robin);
// false past the last one.
__device__ __forceinline__ bool dq_tile(const BwdParams& p, int32_t k, DqTile& t) {
  if (p.sched) {
    if (k >= p.sched_stride) return false;
    const int4 te = p.sched[static_cast<int64_t>(blockIdx.x) * p.sched_stride + k];
    if (te.y < 0) return false;
    t.i = te.x;
    t.n = te.y;
    t.b = te.z / p.Hq;
    t.hq = te.z % p.Hq;
    t.hm = p.mi.heads == 1 ? 0 : t.hq;
    t.row_base = (static_cast<int64_t>(t.hm) * p.mi.rows + t.i) * p.mi.width;
    return true;
  }
  const int64_t T = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(k) * gridDim.x;
  if (T >= p.n_tiles) return false;
  t = dq_decode(p, static_cast<int32_t>(T));
  return true;
}

// Cursor over the CTA's (tile, block) sequence of the dQ launch (tiles
// without blocks skipped; each tile yields exactly row_len blocks).
struct DqSeq {
  int32_t k, j, pos;
  DqTile t;
  RawRef ahead;
  bool valid;
  __device__ __forceinline__ void start_tile(const BwdParams& p) {
    while (true) {
      ++k;
      if (!dq_tile(p, k, t)) {
        valid = false;
        return;
      }
      if (t.n > 0) break;
    }
    j = 0;
    pos = 0;
    if (p.mi.width > 0) ahead = load_block(p.mi, t.row_base, 0);
    valid = true;
  }
  __device__ __forceinline__ void init(const BwdParams& p) {
    k = -1;
    start_tile(p);
  }
  __device__ __forceinline__ bool next(const BwdParams& p, BlockRef& br, bool& first, bool& last) {
    if (!valid) return false;
    bool found = false;
    while (pos < p.mi.width) {
      const RawRef cur = ahead;
      ++pos;
      if (pos < p.mi.width) ahead = load_block(p.mi, t.row_base, pos);
      br = check_block(p.mi, cur, p.err);
      if (br.label != 0) {
        found = true;
        break;
      }
    }
    if (!found) {
      if (p.err) atomicOr(p.err, DEV_ERR_BOUNDS);
      br.label = 2;
      br.col = 0;
      br.slot = 0;
    }
    first = j == 0;
    ++j;
    last = j == t.n;
    return true;
  }
};

// kCap: the logit soft cap is compiled in (a separate instantiation).
template <int D, bool kCap, int kM>
__global__ void __launch_bounds__(DqShape<D>::kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = DqSmem<D>;
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kTile = Smem::kTile;
  constexpr int kChunks = D / 64;
  const int warp = warp_id();
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.qo_full, 1);
    mbar_init(&s.qo_empty, 1);
    for (int i = 0; i < kDqStagesK; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < kDqStagesV; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(&s.s_full[0], 1);
    mbar_init(&s.s_full[1], 1);
    mbar_init(&s.dp_full, 1);
    mbar_init(&s.ds_full, 128 * DqShape<D>::kParts);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 128 * DqShape<D>::kParts);
    mbar_init(&s.drain, 1);
    mbar_init(&s.stats_read, 128 * DqShape<D>::kParts);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // broadcast from lane 0 so the compiler keeps it in a uniform register
  const uint32_t tmem = __shfl_sync(0xffffffffu, s.tmem_base, 0);
  const WaitCtl wc{p.err, &s.abort_flag, p.wait_ns};
  // set-up done: the next kernel may launch; this one waits for the previous
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------ Q/dO/LSE/Dsum (per tile) and K (per block); block ring
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t qo_loads = 0, k_loads = 0;
      bool ok = true;
      DqSeq sq;
      sq.init(p);
      BlockRef br;
      bool first, last;
      int64_t kv_base = 0;
      int32_t tile_q0 = 0, qrow = 0;
      while (ok && sq.next(p, br, first, last)) {
        if (first) {
          // the previous tile's Q/dO are free and its LSE/Dsum have been read
          if (qo_loads >= 1 && !mbar_wait(&s.qo_empty, (qo_loads - 1) & 1u, wc)) { ok = false; break; }
          if (qo_loads >= 1 && !mbar_wait(&s.stats_read, (qo_loads - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.qo_full, 2 * kTile + 1024);
          qrow = static_cast<int32_t>((static_cast<int64_t>(sq.t.b) * p.Hq + sq.t.hq) * p.Sq + sq.t.i * 128);
          tile_q0 = p.mi.q_sequence[sq.t.i * 128];
          for (int c = 0; c < kChunks; ++c) {
            tma_load_2d(s.q + c * 16384, &tm_q, &s.qo_full, c * 64, qrow, pol_q);
            tma_load_2d(s.dout + c * 16384, &tm_do, &s.qo_full, c * 64, qrow, pol_q);
          }
          bulk_load(s.stats[0], p.lse + qrow, 512, &s.qo_full);
          bulk_load(s.stats[1], p.dsum + qrow, 512, &s.qo_full);
          ++qo_loads;
          kv_base = (static_cast<int64_t>(sq.t.b) * p.Hkv + sq.t.hq / (p.Hq / p.Hkv)) * p.Skv;
        }
        const uint32_t ks = k_loads % kDqStagesK;
        if (k_loads >= kDqStagesK && !mbar_wait(&s.k_empty[ks], ((k_loads / kDqStagesK) - 1) & 1u, wc)) { ok = false; break; }
        s.binfo[k_loads % kInfoRing] = make_uint4(pack_info(br.col, br.label, first, last), static_cast<uint32_t>(br.slot),
                                                  static_cast<uint32_t>(tile_q0), static_cast<uint32_t>(qrow));
        mbar_arrive_expect_tx(&s.k_full[ks], kTile);
        const int32_t krow = static_cast<int32_t>(kv_base + br.col * 128);
        for (int c = 0; c < kChunks; ++c) tma_load_2d(s.k[ks] + c * 16384, &tm_k, &s.k_full[ks], c * 64, krow, pol_kv);
        ++k_loads;
        if (last) sq.start_tile(p);
      }
      if (!ok) {
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        if (qo_loads) (void)mbar_wait(&s.qo_full, (qo_loads - 1) & 1u, dw);
        for (uint32_t i = (k_loads > kDqStagesK ? k_loads - kDqStagesK : 0); i < k_loads; ++i)
          (void)mbar_wait(&s.k_full[i % kDqStagesK], (i / kDqStagesK) & 1u, dw);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------ V (per block)
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_kv = policy_evict_last();
      uint32_t v_loads = 0;
      bool ok = true;
      DqSeq sq;
      sq.init(p);
      BlockRef br;
      bool first, last;
      int64_t kv_base = 0;
      while (ok && sq.next(p, br, first, last)) {
        if (first) kv_base = (static_cast<int64_t>(sq.t.b) * p.Hkv + sq.t.hq / (p.Hq / p.Hkv)) * p.Skv;
        const uint32_t vs = v_loads % kDqStagesV;
        if (v_loads >= kDqStagesV && !mbar_wait(&s.v_empty[vs], ((v_loads / kDqStagesV) - 1) & 1u, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.v_full[vs], kTile);
        const int32_t krow = static_cast<int32_t>(kv_base + br.col * 128);
        for (int c = 0; c < kChunks; ++c) tma_load_2d(s.v[vs] + c * 16384, &tm_v, &s.v_full[vs], c * 64, krow, pol_kv);
        ++v_loads;
        if (last) sq.start_tile(p);
      }
      if (!ok) {
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        for (uint32_t i = (v_loads > kDqStagesV ? v_loads - kDqStagesV : 0); i < v_loads; ++i)
          (void)mbar_wait(&s.v_full[i % kDqStagesV], (i / kDqStagesV) & 1u, dw);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp)
    // order: S0 dP0 S1 | dQ0 dP1 S2 | dQ1 dP2 S3 | ...; at a tile's last block
    // L: ... dQ(L-1) dP(L) | dQ(L) S(L+1) dP(L+1) S(L+2) | ...
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
    constexpr uint64_t kTileDesc = kTile >> 4;
    const uint64_t qdesc = sdesc_sw128(smem_u32(s.q), 16, 1024);
    const uint64_t dodesc = sdesc_sw128(smem_u32(s.dout), 16, 1024);
    const uint64_t kdesc0 = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
    const uint64_t kmn0 = sdesc_sw128(smem_u32(s.k[0]), 16384, 1024);
    const uint64_t vdesc0 = sdesc_sw128(smem_u32(s.v[0]), 16, 1024);
    uint32_t total = 0;
    {
      DqTile t;
      for (int32_t kt = 0; dq_tile(p, kt, t); ++kt) total += static_cast<uint32_t>(t.n);
    }
    uint32_t s_cnt = 0, dp_cnt = 0, q_uses = 0, acc_uses = 0;
    bool ok = true;
    auto k_ready = [&](uint32_t n) -> bool {
      return mbar_wait_warp(&s.k_full[n % kDqStagesK], (n / kDqStagesK) & 1u, wc);
    };
    // S_n = Q K_n^T.  A tile's first S waits until the previous tile's last
    // dQ has been issued (allow_first false holds it back, s_cnt unchanged):
    // that dQ, and so the epilogue, then never waits for the next tile's
    // Q / dO load.
    auto issue_s = [&](bool allow_first) -> bool {
      const uint32_t n = s_cnt;
      if (!k_ready(n)) return false;
      const uint32_t info = __shfl_sync(0xffffffffu, s.binfo[n % kInfoRing].x, 0);
      if ((info >> 20) & 1u) {  // first block of a tile: wait for its Q/dO
        if (!allow_first) return true;
        if (!mbar_wait_warp(&s.qo_full, q_uses & 1u, wc)) return false;
        ++q_uses;
      }
      tc_fence_after();
      const uint64_t kd = kdesc0 + (n % kDqStagesK) * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        mma_ss_elect(BSA_TMEM(tmem + kDqColS + (n & 1u) * 128, 128u, p.err), qdesc + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&s.s_full[n & 1u]);
      ++s_cnt;
      return true;
    };
    auto issue_dp = [&]() -> bool {  // dP_n = dO V_n^T
      const uint32_t n = dp_cnt;
      const uint32_t vs = n % kDqStagesV;
      if (!mbar_wait_warp(&s.v_full[vs], (n / kDqStagesV) & 1u, wc)) return false;
      tc_fence_after();
      const uint64_t vd = vdesc0 + vs * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        mma_ss_elect(BSA_TMEM(tmem + kDqColDP, 128u, p.err), dodesc + off, vd + off, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&s.dp_full);
      mma_commit_elect(&s.v_empty[vs]);
      const uint32_t info = __shfl_sync(0xffffffffu, s.binfo[n % kInfoRing].x, 0);
      if ((info >> 21) & 1u) mma_commit_elect(&s.qo_empty);  // last S and dP of the tile are issued
      ++dp_cnt;
      return true;
    };
    if (total > 0) {
      ok = issue_s(true) && issue_dp();
      if (ok && total > 1) ok = issue_s(false);
    }
    for (uint32_t n = 0; ok && n < total; ++n) {
      const uint32_t info = __shfl_sync(0xffffffffu, s.binfo[n % kInfoRing].x, 0);
      const bool first = (info >> 20) & 1u, last = (info >> 21) & 1u;
      if (!mbar_wait_warp(&s.ds_full, n & 1u, wc)) { ok = false; break; }
      if (first && acc_uses > 0 && !mbar_wait_warp(&s.acc_empty, (acc_uses - 1) & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      // dQ += dS K_n  (dS in the dP buffer, K_n as an MN-major B operand)
      const uint64_t kmn = kmn0 + (n % kDqStagesK) * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_elect(BSA_TMEM(tmem + kDqColQ, 128u, p.err), BSA_TMEM(tmem + kDqColDP + part_a_col<DqShape<D>::kCols>(kk), 8u, p.err),
                     kmn + static_cast<uint64_t>(kk * 2048 >> 4),
                     idesc_acc, (first && kk == 0) ? 0u : 1u);
      mma_commit_elect(&s.k_empty[n % kDqStagesK]);
      if (last) {
        mma_commit_elect(&s.acc_full);
        ++acc_uses;
      }
      // a first S held back behind this dQ goes ahead of dP(n + 1)
      if (s_cnt == n + 1 && s_cnt < total && !issue_s(true)) { ok = false; break; }
      if (dp_cnt < total && !issue_dp()) { ok = false; break; }
      if (s_cnt < total && !issue_s(false)) { ok = false; break; }
    }
    mma_commit_elect(&s.drain);
    uint32_t dummy_abort = 0;
    WaitCtl dw{p.err, &dummy_abort, p.wait_ns};
    (void)mbar_wait(&s.drain, 0, dw);
  } else if (warp >= 4) {
    // ------------------------------------------------ P and dS (kParts warpgroups)
    constexpr int kParts = DqShape<D>::kParts;
    constexpr int kCols = DqShape<D>::kCols;  // key columns per thread
    constexpr int kPartD = D / kParts;        // dQ columns per thread at the epilogue
    const int part = (warp - 4) >> 2;
    const int quarter = (warp - 4) & 3;
    const int r = quarter * 32 + lane;  // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(part) * kCols;
    const float scale_log2 = p.scale_log2;
    uint32_t n = 0, acc_uses = 0;
    bool ok = true;
    uint32_t total = 0;
    {
      DqTile t;
      for (int32_t kt = 0; dq_tile(p, kt, t); ++kt) {
        total += static_cast<uint32_t>(t.n);
        if (t.n > 0) continue;
        const int64_t qrow = (static_cast<int64_t>(t.b) * p.Hq + t.hq) * p.Sq + static_cast<int64_t>(t.i) * 128 + r;
        store_zero_cols(p.dq, p.grad_fp32, qrow, D, part * kPartD, kPartD);
      }
    }
    float lse2 = 0.f, dsum_r = 0.f;
    int64_t lo = 0, hi = 0, qrow = 0;
    uint32_t tiles = 0;
    for (; ok && n < total; ++n) {
      const uint32_t sb = n & 1u;
      if (!mbar_wait_warp(&s.s_full[sb], (n >> 1) & 1u, wc)) { ok = false; break; }
      const uint4 bi = s.binfo[n % kInfoRing];
      const int32_t col = static_cast<int32_t>(bi.x & 0xFFFFu);
      const int32_t label = static_cast<int32_t>((bi.x >> 16) & 3u);
      const bool first = (bi.x >> 20) & 1u, last = (bi.x >> 21) & 1u;
      if (first) {
        // row statistics arrive with the tile's Q/dO; q_sequence is consecutive within a block
        qrow = BSA_RANGE(static_cast<int64_t>(bi.w) + r, int64_t(0), static_cast<int64_t>(p.B) * p.Hq * p.Sq, p.err);
        if (!dense_mask<kM>(p.mi.kind))
          key_interval(p.mi.kind, p.mi.left, p.mi.right, p.mi.chunk, static_cast<int64_t>(static_cast<int32_t>(bi.z)) + r,
                       lo, hi);
        if (!mbar_wait_warp(&s.qo_full, tiles & 1u, wc)) { ok = false; break; }
        lse2 = s.stats[0][r] * kLog2e;
        dsum_r = s.stats[1][r];
        mbar_arrive(&s.stats_read);
        ++tiles;
      }
      uint64_t allowed = ~0ull;
      if (label == 1) {
        if (dense_mask<kM>(p.mi.kind))
          allowed = dense_bits<kCols>(p.mi.partial_bits + (bi.y * 128u + static_cast<uint32_t>(r)) * 4u, col0);
        else
          allowed = interval_bits_64(static_cast<int64_t>(col) * 128 + col0, lo, hi);
      }
      // no branch joins while the loaded registers are in flight
      tc_fence_after();
      uint32_t sv[kCols];
#pragma unroll
      for (int c = 0; c < kCols; c += 32) tmem_ld32(BSA_TMEM(tmem + kDqColS + sb * 128 + col0 + c + lane_off, 32u, p.err), sv + c);
      tmem_wait_ld();
      reg_fence<kCols>(sv);
      // P = exp2(s * scale_log2 - lse2), packed pairs
      const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nl2 = f2_pack(-lse2, -lse2);
      float pv[kCols];
      if constexpr (!kCap) {
#pragma unroll
        for (int c = 0; c < kCols; c += 2) {
          float e0, e1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, nl2), e0, e1);
          pv[c] = ex2_approx(e0);
          pv[c + 1] = ex2_approx(e1);
        }
      } else {
        // soft cap: P = exp2(cap_log2 * t - lse2) with t = tanh(s * cap_scale);
        // dQ only needs dS, so the factor 1 - t^2 goes into P here
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const float t = tanh_fast(__uint_as_float(sv[c]) * p.cap_scale);
          pv[c] = ex2_approx(fmaf(t, p.cap_log2, -lse2)) * fmaf(-t, t, 1.f);
        }
      }
      if (label == 1) {
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (!((allowed >> c) & 1ull)) pv[c] = 0.f;
      }
      if (!mbar_wait_warp(&s.dp_full, n & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t dpv[kCols];
#pragma unroll
      for (int c = 0; c < kCols; c += 32) tmem_ld32(BSA_TMEM(tmem + kDqColDP + col0 + c + lane_off, 32u, p.err), dpv + c);
      tmem_wait_ld();
      reg_fence<kCols>(dpv);
      // dS = P * (dP - Dsum)
      const uint64_t nd2 = f2_pack(-dsum_r, -dsum_r);
      uint32_t dspk[kCols / 2];
#pragma unroll
      for (int c = 0; c < kCols / 2; ++c) {
        float d0, d1;
        f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dpv[2 * c]), __uint_as_float(dpv[2 * c + 1])), nd2),
                         f2_pack(pv[2 * c], pv[2 * c + 1])),
                  d0, d1);
        dspk[c] = pack_bf16x2(d0, d1);
      }
      tmem_st_cols<kCols / 2>(BSA_TMEM(tmem + kDqColDP + col0 + lane_off, static_cast<uint32_t>(kCols / 2), p.err), dspk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.ds_full);
      if (!last) continue;
      if (!mbar_wait_warp(&s.acc_full, acc_uses & 1u, wc)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kPartD / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(BSA_TMEM(tmem + kDqColQ + part * kPartD + c * 32 + lane_off, 32u, p.err), v);
        tmem_wait_ld();
        reg_fence32(v);
        store_row_wide(p.dq, p.grad_fp32, qrow, D, v, part * kPartD + c * 32, p.scale);
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty);
      ++acc_uses;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===========================================================================
// dK / dV launch
// ===========================================================================
constexpr int kDkvQStages = 3;       // Q of one query block
constexpr int kDkvDoStages = 2;      // (dO, LSE, Dsum) of one query block
constexpr int kDkvInfoRing = 8;      // item descriptors (written with an item's Q)
constexpr uint32_t kDkvColST = 0;    // S^T, then P^T (bf16) over it
constexpr uint32_t kDkvColDP = 128;  // dP^T, then dS^T (bf16) over it
constexpr uint32_t kDkvColDV = 256;
constexpr uint32_t kDkvColDK = 384;

template <int D>
struct __align__(1024) DkvSmem {
  static constexpr int kTile = 128 * D * 2;
  uint8_t k[kTile];
  uint8_t v[kTile];
  uint8_t q[kDkvQStages][kTile];
  uint8_t dout[kDkvDoStages][kTile];
  float lse[kDkvDoStages][128];
  float dsum[kDkvDoStages][128];
  uint64_t k_full, k_empty, v_full, v_empty;
  // An item's inputs in stages of their own: Q, read up to the item's dK
  // and needed first by the next items (three stages, so that a load has
  // two items' time to land), and (dO, LSE, Dsum), read up to the item's dV
  // and dS (two stages).  q_empty: the MMA warp's commit after the item's
  // dK plus one arrival per elementwise warp (from the MMA warp, except at a
  // tile's last item, where the elementwise warps arrive once their tensor
  // stores out of the item's Q buffer have read it); do_empty: the commit
  // after the item's dV plus one arrival per elementwise warp once it has
  // computed dS (or, at a tile's last item, once its stores out of the dO
  // buffer have read it).
  uint64_t q_full[kDkvQStages], q_empty[kDkvQStages];
  uint64_t do_full[kDkvDoStages], do_empty[kDkvDoStages];
  // p_full[h]: half h of every thread's query columns of P^T is in tensor
  // memory (dV takes those k-steps first)
  uint64_t st_full, dpt_full, p_full[2], ds_full;
  uint64_t acc_full, acc_empty, drain;
  // per item: {col | label<<16 | first<<20 | last<<21, stack slot (dense) or q_sequence of the
  // query block's first row (computable), 128*j = first key of the tile, row of that key in dK/dV}
  uint4 binfo[kDkvInfoRing];
  uint32_t tmem_base;
  uint32_t abort_flag;
};
// The layout starts on a 1024-byte boundary (128-byte swizzled tiles); the
// dynamic shared memory of a launch does (the kernel checks it), so no slack
// is requested and the three Q stages fit.
static_assert(sizeof(DkvSmem<128>) <= 232448, "dK/dV shared memory exceeds 227 KB per CTA");

struct DkvTile {
  int32_t b, g, j;
  int32_t total;  // non-empty blocks over the q heads of this tile's split of the group
  int32_t split;
};

__device__ __forceinline__ int32_t dkv_mask_head(const BwdParams& p, int32_t hq) {
  return p.mi.heads == 1 ? 0 : hq;
}

__device__ __forceinline__ DkvTile dkv_decode(const BwdParams& p, int32_t T) {
  DkvTile t;
  const int32_t G = p.Hq / p.Hkv;
  if (p.mi.heads == 1) {
    const int32_t bg = T % (p.B * p.Hkv);
    t.j = p.mi.row_order[T / (p.B * p.Hkv)];
    t.b = bg / p.Hkv;
    t.g = bg % p.Hkv;
    t.total = p.mi.row_len[t.j] * G;
    t.split = 0;
  } else {
    t.j = T % p.nK;
    const int32_t bg = T / p.nK;
    t.b = bg / p.Hkv;
    t.g = bg % p.Hkv;
    t.total = 0;
    t.split = 0;
    for (int32_t gh = 0; gh < G; ++gh) t.total += p.mi.row_len[(t.g * G + gh) * p.mi.rows + t.j];
  }
  return t;
}

// The k-th tile of this CTA, from the launch's schedule (or round-robin);
// false past the last one.
__device__ __forceinline__ bool dkv_tile(const BwdParams& p, int32_t k, DkvTile& t) {
  if (p.sched) {
    if (k >= p.sched_stride) return false;
    const int4 te = p.sched[static_cast<int64_t>(blockIdx.x) * p.sched_stride + k];
    if (te.y < 0) return false;
    t.j = te.x;
    t.total = te.y;
    t.b = te.z / p.Hkv;
    t.g = te.z % p.Hkv;
    t.split = te.w;
    return true;
  }
  const int64_t T = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(k) * gridDim.x;
  if (T >= p.n_tiles) return false;
  t = dkv_decode(p, static_cast<int32_t>(T));
  return true;
}

// Row of a tile's first key in the dK/dV output (or in the partial sums of
// its split).
__device__ __forceinline__ int64_t dkv_out_row(const BwdParams& p, const DkvTile& t, int64_t krow) {
  return p.kv_splits > 1 ? static_cast<int64_t>(t.split) * p.part_rows + krow : krow;
}

// Items of one dK/dV tile, in order: q heads of the group, then the
// non-empty query blocks of that head's MaskInfo row (each yields exactly
// row_len blocks; a malformed row is padded with flagged dummy blocks).
struct DkvItems {
  int32_t gh, gh_end, n, j, pos;
  int64_t row_base;
  RawRef ahead;
  __device__ __forceinline__ void start_head(const BwdParams& p, const DkvTile& t) {
    const int32_t G = p.Hq / p.Hkv;
    while (gh < gh_end) {
      const int32_t hm = dkv_mask_head(p, t.g * G + gh);
      row_base = (static_cast<int64_t>(hm) * p.mi.rows + t.j) * p.mi.width;
      n = p.mi.row_len[hm * p.mi.rows + t.j];
      if (n > 0) break;
      ++gh;
    }
    j = 0;
    pos = 0;
    if (gh < gh_end && p.mi.width > 0) ahead = load_block(p.mi, row_base, 0);
  }
  __device__ __forceinline__ void init(const BwdParams& p, const DkvTile& t) {
    const int32_t gs = p.Hq / p.Hkv / p.kv_splits;  // q heads of one split
    gh = t.split * gs;
    gh_end = gh + gs;
    start_head(p, t);
  }
  __device__ __forceinline__ bool next(const BwdParams& p, const DkvTile& t, int32_t& hq, BlockRef& br) {
    const int32_t G = p.Hq / p.Hkv;
    if (gh >= gh_end) return false;
    bool found = false;
    while (pos < p.mi.width) {
      const RawRef cur = ahead;
      ++pos;
      if (pos < p.mi.width) ahead = load_block(p.mi, row_base, pos);
      br = check_block(p.mi, cur, p.err);
      if (br.label != 0) {
        found = true;
        break;
      }
    }
    if (!found) {
      if (p.err) atomicOr(p.err, DEV_ERR_BOUNDS);
      br.label = 2;
      br.col = 0;
      br.slot = 0;
    }
    hq = t.g * G + gh;
    if (++j == n) {
      ++gh;
      start_head(p, t);
    }
    return true;
  }
};

// kCap: the logit soft cap is compiled in (a separate instantiation).
template <int D, bool kCap, int kM>
__global__ void __launch_bounds__(DkvShape<D>::kThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
               const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = DkvSmem<D>;
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  constexpr uint32_t kTile = Smem::kTile;
  constexpr int kChunks = D / 64;
  const int warp = warp_id();
  const int lane = threadIdx.x & 31;
  if (smem_u32(smem_raw) & 1023u) {  // (uniform over the CTA) nothing has been touched yet
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DEV_ERR_SMEM_ALIGN);
    return;
  }

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.k_full, 1);
    mbar_init(&s.k_empty, 1);
    mbar_init(&s.v_full, 1);
    mbar_init(&s.v_empty, 1);
    for (int i = 0; i < kDkvQStages; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1 + 4 * DkvShape<D>::kParts);
    }
    for (int i = 0; i < kDkvDoStages; ++i) {
      mbar_init(&s.do_full[i], 1);
      mbar_init(&s.do_empty[i], 1 + 4 * DkvShape<D>::kParts);
    }
    mbar_init(&s.st_full, 1);
    mbar_init(&s.dpt_full, 1);
    mbar_init(&s.p_full[0], 128 * DkvShape<D>::kParts);
    mbar_init(&s.p_full[1], 128 * DkvShape<D>::kParts);
    mbar_init(&s.ds_full, 128 * DkvShape<D>::kParts);
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 128 * DkvShape<D>::kParts);
    mbar_init(&s.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // broadcast from lane 0 so the compiler keeps it in a uniform register
  const uint32_t tmem = __shfl_sync(0xffffffffu, s.tmem_base, 0);
  const WaitCtl wc{p.err, &s.abort_flag, p.wait_ns};
  // set-up done: the next kernel may launch; this one waits for the previous
  griddep_launch_dependents();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------ K/V (per tile), Q/dO/LSE/Dsum (per item); item ring
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      uint32_t k_loads = 0, v_loads = 0, in_loads = 0, do_loads = 0;
      bool ok = true;
      DkvTile t;
      for (int32_t kt = 0; ok && dkv_tile(p, kt, t); ++kt) {
        if (t.total == 0) continue;
        const int32_t krow = static_cast<int32_t>((static_cast<int64_t>(t.b) * p.Hkv + t.g) * p.Skv + t.j * 128);
        DkvItems it;
        it.init(p, t);
        int32_t hq;
        BlockRef br;
        for (int32_t x = 0; x < t.total && ok; ++x) {
          it.next(p, t, hq, br);
          const int64_t qrow = (static_cast<int64_t>(t.b) * p.Hq + hq) * p.Sq + br.col * 128;
          // Q (needed first, by the item's S^T), then dO with LSE and Dsum
          const uint32_t qs = in_loads % kDkvQStages;
          if (in_loads >= kDkvQStages && !mbar_wait(&s.q_empty[qs], ((in_loads / kDkvQStages) - 1) & 1u, wc)) { ok = false; break; }
          const uint32_t extra = p.mi.kind == BSA_MASK_DENSE ? static_cast<uint32_t>(br.slot)
                                                             : static_cast<uint32_t>(p.mi.q_sequence[br.col * 128]);
          s.binfo[in_loads % kDkvInfoRing] = make_uint4(pack_info(br.col, br.label, x == 0, x == t.total - 1), extra,
                                                     static_cast<uint32_t>(t.j * 128),
                                                     static_cast<uint32_t>(dkv_out_row(p, t, krow)));
          mbar_arrive_expect_tx(&s.q_full[qs], kTile);
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(s.q[qs] + c * 16384, &tm_q, &s.q_full[qs], c * 64, static_cast<int32_t>(qrow), pol_q);
          ++in_loads;
          const uint32_t ds = do_loads % kDkvDoStages;
          if (do_loads >= kDkvDoStages && !mbar_wait(&s.do_empty[ds], ((do_loads / kDkvDoStages) - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.do_full[ds], kTile + 1024);
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(s.dout[ds] + c * 16384, &tm_do, &s.do_full[ds], c * 64, static_cast<int32_t>(qrow), pol_q);
          bulk_load(s.lse[ds], p.lse + qrow, 512, &s.do_full[ds]);
          bulk_load(s.dsum[ds], p.dsum + qrow, 512, &s.do_full[ds]);
          ++do_loads;
          if (x > 0) continue;
          // The tile's K and V follow its first query block, so that this
          // block's loads do not wait for the previous tile's last MMAs: K is
          // free once the previous tile's last S^T has completed, V once its
          // last dP^T has.
          if (k_loads >= 1 && !mbar_wait(&s.k_empty, (k_loads - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.k_full, kTile);
          for (int c = 0; c < kChunks; ++c) tma_load_2d(s.k + c * 16384, &tm_k, &s.k_full, c * 64, krow, pol_kv);
          ++k_loads;
          if (v_loads >= 1 && !mbar_wait(&s.v_empty, (v_loads - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.v_full, kTile);
          for (int c = 0; c < kChunks; ++c) tma_load_2d(s.v + c * 16384, &tm_v, &s.v_full, c * 64, krow, pol_kv);
          ++v_loads;
          // warm L2 with this CTA's next tile's K and V
          DkvTile t2;
          for (int32_t k2 = kt + 1; dkv_tile(p, k2, t2); ++k2) {
            if (t2.total == 0) continue;
            const int64_t row2 = (static_cast<int64_t>(t2.b) * p.Hkv + t2.g) * p.Skv + t2.j * 128;
            prefetch_l2(static_cast<const uint8_t*>(p.kp) + row2 * D * 2, 128 * D * 2);
            prefetch_l2(static_cast<const uint8_t*>(p.vp) + row2 * D * 2, 128 * D * 2);
            break;
          }
        }
      }
      if (!ok) {
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        if (k_loads) (void)mbar_wait(&s.k_full, (k_loads - 1) & 1u, dw);
        if (v_loads) (void)mbar_wait(&s.v_full, (v_loads - 1) & 1u, dw);
        for (uint32_t i = (in_loads > kDkvQStages ? in_loads - kDkvQStages : 0); i < in_loads; ++i)
          (void)mbar_wait(&s.q_full[i % kDkvQStages], (i / kDkvQStages) & 1u, dw);
        for (uint32_t i = (do_loads > kDkvDoStages ? do_loads - kDkvDoStages : 0); i < do_loads; ++i)
          (void)mbar_wait(&s.do_full[i % kDkvDoStages], (i / kDkvDoStages) & 1u, dw);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp)
    // per item n: S^T dP^T | (P ready) dV | (dS ready) dK
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
    constexpr uint64_t kTileDesc = kTile >> 4;
    const uint64_t kdesc = sdesc_sw128(smem_u32(s.k), 16, 1024);
    const uint64_t vdesc = sdesc_sw128(smem_u32(s.v), 16, 1024);
    const uint64_t qdesc0 = sdesc_sw128(smem_u32(s.q[0]), 16, 1024);
    const uint64_t qmn0 = sdesc_sw128(smem_u32(s.q[0]), 16384, 1024);
    const uint64_t dodesc0 = sdesc_sw128(smem_u32(s.dout[0]), 16, 1024);
    const uint64_t domn0 = sdesc_sw128(smem_u32(s.dout[0]), 16384, 1024);
    uint32_t total = 0;
    {
      DkvTile t;
      for (int32_t kt = 0; dkv_tile(p, kt, t); ++kt) total += static_cast<uint32_t>(t.total);
    }
    uint32_t k_uses = 0, v_uses = 0, acc_uses = 0;
    bool ok = true;
    // S^T(n+1) is issued right after dV(n) (which reads P^T(n) from the same
    // columns first), so the tensor cores compute the next scores while the
    // elementwise warps work on dS^T(n); dP^T(n+1) follows dK(n) likewise.
    // Order: S^T(0) dP^T(0) | dV(0) S^T(1) dK(0) dP^T(1) | dV(1) S^T(2) ...
    // At a tile's last item n, S^T(n+1) waits until after dK(n): the
    // accumulators go to the epilogue without waiting for the next tile's
    // loads.
    uint32_t flags = 0;  // first/last bits of items n and n+1, two per item
    auto item_flags = [&](uint32_t k) -> bool {
      if (!mbar_wait_warp(&s.q_full[k % kDkvQStages], (k / kDkvQStages) & 1u, wc)) return false;
      const uint32_t info = __shfl_sync(0xffffffffu, s.binfo[k % kDkvInfoRing].x, 0);
      const uint32_t sh = 2u * (k & 7u);
      flags = (flags & ~(3u << sh)) | (((info >> 20) & 3u) << sh);
      if ((info >> 20) & 1u) {  // first item of a tile: its K
        if (!mbar_wait_warp(&s.k_full, k_uses & 1u, wc)) return false;
        ++k_uses;
      }
      tc_fence_after();
      return true;
    };
    auto issue_st = [&](uint32_t k) {
      const uint64_t qd = qdesc0 + (k % kDkvQStages) * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        mma_ss_elect(BSA_TMEM(tmem + kDkvColST, 128u, p.err), kdesc + off, qd + off, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&s.st_full);
      // K is read by the S^T MMAs only
      if ((flags >> (2u * (k & 7u))) & 2u) mma_commit_elect(&s.k_empty);
    };
    auto issue_dpt = [&](uint32_t k) -> bool {
      if ((flags >> (2u * (k & 7u))) & 1u) {  // first item of a tile: its V
        if (!mbar_wait_warp(&s.v_full, v_uses & 1u, wc)) return false;
        ++v_uses;
      }
      if (!mbar_wait_warp(&s.do_full[k % kDkvDoStages], (k / kDkvDoStages) & 1u, wc)) return false;
      tc_fence_after();
      const uint64_t dod = dodesc0 + (k % kDkvDoStages) * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        mma_ss_elect(BSA_TMEM(tmem + kDkvColDP, 128u, p.err), vdesc + off, dod + off, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&s.dpt_full);
      // V is read by the dP^T MMAs only
      if ((flags >> (2u * (k & 7u))) & 2u) mma_commit_elect(&s.v_empty);
      return true;
    };
    if (total > 0) {
      ok = item_flags(0);
      if (ok) {
        issue_st(0);
        ok = issue_dpt(0);
      }
    }
    for (uint32_t n = 0; ok && n < total; ++n) {
      const uint32_t qs = n % kDkvQStages, ds = n % kDkvDoStages;
      const uint32_t fl = (flags >> (2u * (n & 7u))) & 3u;
      const bool first = fl & 1u, last = fl & 2u;
      const bool more = n + 1 < total;
      // dV += P^T dO, the k-steps of each half of the parts' columns as
      // soon as that half of P^T is in tensor memory
      if (!mbar_wait_warp(&s.p_full[0], n & 1u, wc)) { ok = false; break; }
      if (first && acc_uses > 0 && !mbar_wait_warp(&s.acc_empty, (acc_uses - 1) & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      const uint64_t domn = domn0 + ds * kTileDesc;
      {
        constexpr int kSteps = DkvShape<D>::kCols / 16;  // k-steps per part
        bool half_ok = true;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1) {
            half_ok = mbar_wait_warp(&s.p_full[1], n & 1u, wc);
            if (!half_ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            if ((kk % kSteps) / (kSteps / 2) != h) continue;
            mma_ts_elect(BSA_TMEM(tmem + kDkvColDV, 128u, p.err), BSA_TMEM(tmem + kDkvColST + part_a_col<DkvShape<D>::kCols>(kk), 8u, p.err),
                         domn + static_cast<uint64_t>(kk * 2048 >> 4), idesc_acc, (first && kk == 0) ? 0u : 1u);
          }
        }
        if (!half_ok) { ok = false; break; }
      }
      // dO is read by dP^T and dV only (the elementwise warps add their
      // arrivals once dS is computed)
      mma_commit_elect(&s.do_empty[ds]);
      // next item's S^T over the P^T columns the dV MMA has just read
      if (more && !last) {
        if (!item_flags(n + 1)) { ok = false; break; }
        issue_st(n + 1);
      }
      // dK += dS^T Q
      if (!mbar_wait_warp(&s.ds_full, n & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      const uint64_t qmn = qmn0 + qs * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_elect(BSA_TMEM(tmem + kDkvColDK, 128u, p.err), BSA_TMEM(tmem + kDkvColDP + part_a_col<DkvShape<D>::kCols>(kk), 8u, p.err),
                     qmn + static_cast<uint64_t>(kk * 2048 >> 4),
                     idesc_acc, (first && kk == 0) ? 0u : 1u);
      mma_commit_elect(&s.q_empty[qs]);
      if (last) {
        mma_commit_elect(&s.acc_full);
        ++acc_uses;
      } else {
        // the elementwise warps' share of q_empty (they hold the Q buffer
        // only at a tile's last item, for the epilogue's tensor stores)
        mbar_arrive_cnt_elect(&s.q_empty[qs], 4 * DkvShape<D>::kParts);
      }
      if (more) {
        if (last) {
          if (!item_flags(n + 1)) { ok = false; break; }
          issue_st(n + 1);
        }
        // next item's dP^T over the dS^T columns the dK MMA has just read
        if (!issue_dpt(n + 1)) { ok = false; break; }
      }
    }
    mma_commit_elect(&s.drain);
    uint32_t dummy_abort = 0;
    WaitCtl dw{p.err, &dummy_abort, p.wait_ns};
    (void)mbar_wait(&s.drain, 0, dw);
  } else if (warp >= 4) {
    // ------------------------------------------------ P^T and dS^T (kParts warpgroups)
    constexpr int kParts = DkvShape<D>::kParts;
    constexpr int kCols = DkvShape<D>::kCols;  // query columns per thread
    constexpr int kPartD = D / kParts;         // output columns per thread at the epilogue
    const int part = (warp - 4) >> 2;
    const int quarter = (warp - 4) & 3;
    const int r = quarter * 32 + lane;  // key row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(part) * kCols;  // query columns of this part
    bool ok = true;
    uint32_t total = 0;
    {
      DkvTile t;
      for (int32_t kt = 0; dkv_tile(p, kt, t); ++kt) {
        total += static_cast<uint32_t>(t.total);
        if (t.total > 0) continue;
        const int64_t krow =
            dkv_out_row(p, t, (static_cast<int64_t>(t.b) * p.Hkv + t.g) * p.Skv + static_cast<int64_t>(t.j) * 128) + r;
        const bool sp = p.kv_splits > 1;
        store_zero_cols(sp ? p.part_dk : p.dk, sp ? 1 : p.grad_fp32, krow, D, part * kPartD, kPartD);
        store_zero_cols(sp ? p.part_dv : p.dv, sp ? 1 : p.grad_fp32, krow, D, part * kPartD, kPartD);
      }
    }
    uint32_t acc_uses = 0;
    int64_t lo = 0, hi = 0, krow = 0;
    const uint64_t nsc2 = f2_pack(-p.scale, -p.scale), nl2e2 = f2_pack(-kLog2e, -kLog2e);
    for (uint32_t n = 0; ok && n < total; ++n) {
      const uint32_t st = n % kDkvDoStages;  // LSE and Dsum of this item
      if (!mbar_wait_warp(&s.do_full[st], (n / kDkvDoStages) & 1u, wc)) { ok = false; break; }
      const uint4 bi = s.binfo[n % kDkvInfoRing];
      const int32_t label = static_cast<int32_t>((bi.x >> 16) & 3u);
      const bool first = (bi.x >> 20) & 1u, last = (bi.x >> 21) & 1u;
      if (first) {
        krow = BSA_RANGE(static_cast<int64_t>(bi.w) + r, int64_t(0),
                         (p.kv_splits > 1 ? p.kv_splits : 1) * static_cast<int64_t>(p.B) * p.Hkv * p.Skv, p.err);
        if (!dense_mask<kM>(p.mi.kind))
          query_interval(p.mi.kind, p.mi.left, p.mi.right, p.mi.chunk, static_cast<int64_t>(bi.z) + r, lo, hi);
      }
      // the visibility bits (a dense mask's from memory) before the wait for the scores
      uint64_t allowed = ~0ull;
      if (label == 1) {
        if (dense_mask<kM>(p.mi.kind)) {
          allowed = dense_bits<kCols>(p.mi.partial_bits + (bi.y * 128u + static_cast<uint32_t>(r)) * 4u, col0);
        } else {
          // q_sequence is consecutive within a query block
          allowed = interval_bits_64(static_cast<int64_t>(static_cast<int32_t>(bi.y)) + col0, lo, hi);
        }
      }
      if (!mbar_wait_warp(&s.st_full, n & 1u, wc)) { ok = false; break; }
      // per-column statistics of this part's query rows
      const float4* lse4 = reinterpret_cast<const float4*>(&s.lse[st][col0]);
      // no branch joins while the loaded registers are in flight
      tc_fence_after();
      uint32_t sv[kCols];
#pragma unroll
      for (int c = 0; c < kCols; c += 32) tmem_ld32(BSA_TMEM(tmem + kDkvColST + col0 + c + lane_off, 32u, p.err), sv + c);
      tmem_wait_ld();
      reg_fence<kCols>(sv);
      // P = exp2((s*scale - LSE) * log2e): (LSE - s*scale) then times -log2e, packed pairs
      float pv[kCols];
      if constexpr (!kCap) {
        // two halves of the columns, each published as soon as it is in
        // tensor memory so that dV starts on it
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c4 = h * kCols / 8; c4 < (h + 1) * kCols / 8; ++c4) {
            const float4 l4 = lse4[c4];
            const int c = c4 * 4;
            float e0, e1, e2, e3;
            f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), nsc2,
                                    f2_pack(l4.x, l4.y)),
                             nl2e2),
                      e0, e1);
            f2_unpack(f2_mul(f2_fma(f2_pack(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), nsc2,
                                    f2_pack(l4.z, l4.w)),
                             nl2e2),
                      e2, e3);
            pv[c] = ex2_approx(e0);
            pv[c + 1] = ex2_approx(e1);
            pv[c + 2] = ex2_approx(e2);
            pv[c + 3] = ex2_approx(e3);
          }
          if (label == 1) {
#pragma unroll
            for (int c = h * kCols / 2; c < (h + 1) * kCols / 2; ++c)
              if (!((allowed >> c) & 1ull)) pv[c] = 0.f;
          }
          uint32_t ppk[kCols / 4];
#pragma unroll
          for (int c = 0; c < kCols / 4; ++c)
            ppk[c] = pack_bf16x2(pv[h * kCols / 2 + 2 * c], pv[h * kCols / 2 + 2 * c + 1]);
          tmem_st_cols<kCols / 4>(BSA_TMEM(tmem + kDkvColST + col0 + h * (kCols / 4) + lane_off, static_cast<uint32_t>(kCols / 4), p.err), ppk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&s.p_full[h]);
        }
      } else {
        // soft cap: P = exp2(cap_log2 * t - LSE * log2e), t = tanh(s * cap_scale);
        // P^T goes to tensor memory for dV, and pv keeps P (1 - t^2) for dS
        uint32_t ppk[kCols / 2];
#pragma unroll
        for (int c = 0; c < kCols; c += 2) {
          const float t0 = tanh_fast(__uint_as_float(sv[c]) * p.cap_scale);
          const float t1 = tanh_fast(__uint_as_float(sv[c + 1]) * p.cap_scale);
          float p0 = ex2_approx(fmaf(t0, p.cap_log2, -s.lse[st][col0 + c] * kLog2e));
          float p1 = ex2_approx(fmaf(t1, p.cap_log2, -s.lse[st][col0 + c + 1] * kLog2e));
          if (label == 1) {
            p0 = ((allowed >> c) & 1ull) ? p0 : 0.f;
            p1 = ((allowed >> (c + 1)) & 1ull) ? p1 : 0.f;
          }
          ppk[c / 2] = pack_bf16x2(p0, p1);
          pv[c] = p0 * fmaf(-t0, t0, 1.f);
          pv[c + 1] = p1 * fmaf(-t1, t1, 1.f);
        }
        tmem_st_cols<kCols / 2>(BSA_TMEM(tmem + kDkvColST + col0 + lane_off, static_cast<uint32_t>(kCols / 2), p.err), ppk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[0]);
        mbar_arrive(&s.p_full[1]);
      }
      if (!mbar_wait_warp(&s.dpt_full, n & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      const float4* ds4 = reinterpret_cast<const float4*>(&s.dsum[st][col0]);
      uint32_t dspk[kCols / 2];
#pragma unroll
      for (int h2 = 0; h2 < kCols / 32; ++h2) {  // 32 columns at a time to bound register use
        uint32_t dpv[32];
        tmem_ld32(BSA_TMEM(tmem + kDkvColDP + col0 + h2 * 32 + lane_off, 32u, p.err), dpv);
        tmem_wait_ld();
        reg_fence32(dpv);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 d4 = ds4[h2 * 8 + c4];
          const int c = h2 * 32 + c4 * 4, cl = c4 * 4;
          float a0, a1, a2, a3;
          // dS = P * (dP - Dsum)
          f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dpv[cl]), __uint_as_float(dpv[cl + 1])), f2_pack(-d4.x, -d4.y)),
                           f2_pack(pv[c], pv[c + 1])),
                    a0, a1);
          f2_unpack(f2_mul(f2_add(f2_pack(__uint_as_float(dpv[cl + 2]), __uint_as_float(dpv[cl + 3])), f2_pack(-d4.z, -d4.w)),
                           f2_pack(pv[c + 2], pv[c + 3])),
                    a2, a3);
          dspk[c / 2] = pack_bf16x2(a0, a1);
          dspk[c / 2 + 1] = pack_bf16x2(a2, a3);
        }
      }
      tmem_st_cols<kCols / 2>(BSA_TMEM(tmem + kDkvColDP + col0 + lane_off, static_cast<uint32_t>(kCols / 2), p.err), dspk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.ds_full);
      if (!last) {
        // done with this item's LSE and Dsum
        if (lane == 0) mbar_arrive(&s.do_empty[st]);
        continue;
      }
      if (!mbar_wait_warp(&s.acc_full, acc_uses & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      static_assert(kPartD == 32, "one 32-column slice of dK and dV per thread");
      const bool sp = p.kv_splits > 1;
      if (!sp && !p.grad_fp32) {
        // bf16 dV and dK through shared memory: the last item's dO and Q
        // buffers are free (its MMAs have completed) and stay the
        // elementwise warps' until each releases them on q_empty and do_empty.  A warp's
        // [32 keys, 32 columns] of each goes out in one tensor store.
        uint8_t* stv = s.dout[st] + (warp - 4) * 2048;
        uint8_t* stk = s.q[n % kDkvQStages] + (warp - 4) * 2048;
        uint32_t v[32];
        tmem_ld32(BSA_TMEM(tmem + kDkvColDV + part * kPartD + lane_off, 32u, p.err), v);
        tmem_wait_ld();
        reg_fence32(v);
        stage_row_sw64(stv, lane, v, 1.f);
        tmem_ld32(BSA_TMEM(tmem + kDkvColDK + part * kPartD + lane_off, 32u, p.err), v);
        tmem_wait_ld();
        reg_fence32(v);
        stage_row_sw64(stk, lane, v, p.scale);
        tc_fence_before();
        mbar_arrive(&s.acc_empty);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int32_t row0 = static_cast<int32_t>(krow - lane);  // key row of this warp's lane 0
          tma_store_2d(&tm_dv, stv, part * kPartD, row0);
          tma_store_2d(&tm_dk, stk, part * kPartD, row0);
          tma_store_commit();
          tma_store_wait_read();
          mbar_arrive(&s.q_empty[n % kDkvQStages]);
          mbar_arrive(&s.do_empty[st]);
        }
        __syncwarp();
      } else {
        uint32_t v[32];
        tmem_ld32(BSA_TMEM(tmem + kDkvColDV + part * kPartD + lane_off, 32u, p.err), v);
        tmem_wait_ld();
        reg_fence32(v);
        store_row(sp ? p.part_dv : p.dv, sp ? 1 : p.grad_fp32, krow, D, v, part * kPartD, 1.f);
        tmem_ld32(BSA_TMEM(tmem + kDkvColDK + part * kPartD + lane_off, 32u, p.err), v);
        tmem_wait_ld();
        reg_fence32(v);
        store_row(sp ? p.part_dk : p.dk, sp ? 1 : p.grad_fp32, krow, D, v, part * kPartD, p.scale);
        tc_fence_before();
        mbar_arrive(&s.acc_empty);
        if (lane == 0) {
          mbar_arrive(&s.q_empty[n % kDkvQStages]);
          mbar_arrive(&s.do_empty[st]);
        }
      }
      ++acc_uses;
    }
    // every tensor store has completed before the CTA exits
    if (lane == 0) tma_store_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// dK, dV = sums of the splits' fp32 partials (fixed order, so the result
// does not depend on timing).  HBM-bound: 4 floats per thread and pass.
__global__ void __launch_bounds__(256) dkv_reduce_kernel(const float4* __restrict__ pk, const float4* __restrict__ pv,
                                                         void* dk, void* dv, int64_t n4, int64_t part4, int32_t splits,
                                                         int32_t fp32) {
  griddep_launch_dependents();
  griddep_wait();  // the partials come from the dK/dV kernel
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = __ldcs(pk + i), b = __ldcs(pv + i);
    for (int32_t sp = 1; sp < splits; ++sp) {
      const float4 x = __ldcs(pk + sp * part4 + i), y = __ldcs(pv + sp * part4 + i);
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
    }
    if (fp32) {
      static_cast<float4*>(dk)[i] = a;
      static_cast<float4*>(dv)[i] = b;
    } else {
      static_cast<uint2*>(dk)[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
      static_cast<uint2*>(dv)[i] = make_uint2(pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
  }
}

bool make_maps(const bsa_bwd_args* a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tdo) {
  const uint64_t q_rows = static_cast<uint64_t>(a->B) * a->Hq * a->S_q;
  const uint64_t kv_rows = static_cast<uint64_t>(a->B) * a->Hkv * a->S_kv;
  const int D = a->D;
  return make_tmap_bf16_2d(tq, a->q, q_rows, D, D * 2, 128, 64) &&
         make_tmap_bf16_2d(tk, a->k, kv_rows, D, D * 2, 128, 64) &&
         make_tmap_bf16_2d(tv, a->v, kv_rows, D, D * 2, 128, 64) &&
         make_tmap_bf16_2d(tdo, a->do_, q_rows, D, D * 2, 128, 64);
}

BwdParams make_params(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, uint32_t* err) {
  BwdParams p{};
  p.kv_splits = 1;
  if (a->logits_soft_cap > 0.f) {
    p.cap_scale = scale / a->logits_soft_cap;
    p.cap_log2 = a->logits_soft_cap * 1.4426950408889634f;
  }
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.Sq = a->S_q;
  p.Skv = a->S_kv;
  p.nQ = static_cast<int32_t>(a->S_q / 128);
  p.nK = static_cast<int32_t>(a->S_kv / 128);
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.lse = a->lse;
  p.dsum = a->dsum;
  p.dq = a->dq;
  p.dk = a->dk;
  p.dv = a->dv;
  p.kp = a->k;
  p.vp = a->v;
  p.grad_fp32 = a->grad_fp32 ? 1 : 0;
  p.mi = mask_info_dev(info);
  p.err = err ? err : device_error_word();
  p.wait_ns = wait_limit_ns();
  return p;
}

template <int D>
bsa_status launch_dkv(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream,
                      uint32_t* err, bool schedule) {
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (!make_maps(a, &tq, &tk, &tv, &tdo)) return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor");
  BwdParams p = make_params(a, info, scale, err);
  if (!p.err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  p.n_tiles = a->B * a->Hkv * p.nK;
  const bool cap = p.cap_scale != 0.f;
  // instantiation: the soft cap (either mask kind), or none with the
  // computable or the dense mask compiled in
  const int variant = cap ? 2 : (info->kind == BSA_MASK_DENSE ? 1 : 0);
  auto kern = variant == 2 ? dkv_kernel<D, true, kAnyMask>
                           : (variant == 1 ? dkv_kernel<D, false, kDenseMask> : dkv_kernel<D, false, kComputableMask>);
  const size_t smem = sizeof(DkvSmem<D>);  // no alignment slack: see DkvSmem
  {
    bsa_status st = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, "set dkv smem size");
    if (st != BSA_OK) return st;
  }
  // With few KV tiles (MQA, short sequences) the q heads of a group are
  // split over several CTAs: the smallest divisor of the group that gives
  // two tiles per SM, whose fp32 partial sums are then added up.
  const int32_t G = a->Hq / a->Hkv;
  const int64_t part_rows = static_cast<int64_t>(a->B) * a->Hkv * a->S_kv;
  int32_t splits = 1;
  if (schedule && G > 1 && p.n_tiles < 2 * num_sms()) {
    splits = G;
    for (int32_t d = 2; d <= G; ++d)
      if (G % d == 0 && static_cast<int64_t>(p.n_tiles) * d >= 2 * num_sms()) {
        splits = d;
        break;
      }
    if (splits * part_rows > static_cast<int64_t>(INT32_MAX)) splits = 1;
  }
  p.kv_splits = splits;
  p.part_rows = part_rows;
  // bf16 dK / dV leave through tensor stores of [32 keys, 32 columns]; fp32
  // outputs and split partials use plain stores (the Q map stands in, unused)
  if (splits == 1 && !a->grad_fp32) {
    if (!make_tmap_bf16_2d_sw64(&tdk, a->dk, part_rows, D, D * 2, 32) ||
        !make_tmap_bf16_2d_sw64(&tdv, a->dv, part_rows, D, D * 2, 32))
      return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected the dK / dV description");
  } else {
    tdk = tq;
    tdv = tq;
  }
  const int grid = static_cast<int>(std::min<int64_t>(static_cast<int64_t>(p.n_tiles) * splits, num_sms()));
  if (schedule) {
    bsa_status st = tile_schedule(info, a->B, a->Hkv, G, splits, grid, stream, &p.sched, &p.sched_stride);
    if (st != BSA_OK) return st;
  }
  void* ws = nullptr;
  if (splits > 1) {
    bsa_status st = pool_alloc(&ws, 2 * static_cast<size_t>(splits) * part_rows * D * sizeof(float), stream);
    if (st != BSA_OK) return st;
    p.part_dk = static_cast<float*>(ws);
    p.part_dv = p.part_dk + static_cast<size_t>(splits) * part_rows * D;
  }
  cudaError_t e =
      launch_kernel(kern, dim3(grid), dim3(DkvShape<D>::kThreads), smem, stream, tq, tk, tv, tdo, tdk, tdv, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e == cudaSuccess && splits > 1) {
    const int64_t n4 = part_rows * D / 4;
    const int rgrid = static_cast<int>(std::min<int64_t>((n4 + 255) / 256, static_cast<int64_t>(num_sms()) * 8));
    e = launch_kernel(dkv_reduce_kernel, dim3(rgrid), dim3(256), 0, stream, reinterpret_cast<const float4*>(p.part_dk),
                      reinterpret_cast<const float4*>(p.part_dv), a->dk, a->dv, n4, n4, splits, a->grad_fp32);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  if (ws) {
    bsa_status st = pool_free(ws, stream);
    if (e == cudaSuccess && st != BSA_OK) return st;
  }
  if (e != cudaSuccess) return cuda_fail(e, "dkv launch");
  return BSA_OK;
}

template <int D>
bsa_status launch_dq(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream,
                     uint32_t* err, bool schedule) {
  CUtensorMap tq, tk, tv, tdo;
  if (!make_maps(a, &tq, &tk, &tv, &tdo)) return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor");
  BwdParams p = make_params(a, info, scale, err);
  if (!p.err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  p.n_tiles = a->B * a->Hq * p.nQ;
  const bool cap = p.cap_scale != 0.f;
  const int variant = cap ? 2 : (info->kind == BSA_MASK_DENSE ? 1 : 0);
  auto kern = variant == 2 ? dq_kernel<D, true, kAnyMask>
                           : (variant == 1 ? dq_kernel<D, false, kDenseMask> : dq_kernel<D, false, kComputableMask>);
  const size_t smem = sizeof(DqSmem<D>) + 1024;
  {
    bsa_status st = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, "set dq smem size");
    if (st != BSA_OK) return st;
  }
  const int grid = std::min(p.n_tiles, num_sms());
  if (schedule) {
    bsa_status st = tile_schedule(info, a->B, a->Hq, 1, 1, grid, stream, &p.sched, &p.sched_stride);
    if (st != BSA_OK) return st;
  }
  cudaError_t e = launch_kernel(kern, dim3(grid), dim3(DqShape<D>::kThreads), smem, stream, tq, tk, tv, tdo, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dq launch");
  return BSA_OK;
}

}  // namespace

bsa_status dkv_launch(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream,
                      uint32_t* err, bool schedule) {
  if (a->D == 128) return launch_dkv<128>(a, info, scale, stream, err, schedule);
  return launch_dkv<64>(a, info, scale, stream, err, schedule);
}

bsa_status dq_launch(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream,
                     uint32_t* err, bool schedule) {
  if (a->D == 128) return launch_dq<128>(a, info, scale, stream, err, schedule);
  return launch_dq<64>(a, info, scale, stream, err, schedule);
}

}  // namespace bsa
