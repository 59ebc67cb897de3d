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
// GB300 design: warp 0 loads by TMA, warp 1 issues tcgen05 MMAs, warps 4-7
// (one TMEM lane / tile row per thread) rebuild P and dS and write them to
// tensor memory as bf16, where they are the A operand of the accumulating
// MMAs.  The inner loop runs over 64-wide halves of each block so that the
// score buffers can be double-buffered next to the two 128-column
// accumulators (TMEM: S x2, dP x2 of 64 columns, then dV/dK or dQ): the
// MMAs of half n+1 overlap the elementwise work of half n.
#include <cmath>

#include "internal.h"
#include "maskinfo_dev.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace bsa {
namespace {

constexpr int kThreads = 256;
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;     // S (or S^T) halves at 0 and 64
constexpr uint32_t kColDP = 128;  // dP (or dP^T) halves at 128 and 192
constexpr uint32_t kColAcc = 256; // dV then dK (dK/dV launch), or dQ (dQ launch)
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int32_t B, Hq, Hkv, nQ, nK;
  int64_t Sq, Skv;
  float scale, scale_log2;
  const float* lse;
  const float* dsum;
  void* dq;
  void* dk;
  void* dv;
  int32_t grad_fp32;
  MaskInfoDev mi;
  int32_t n_tiles;
  uint32_t* err;
  uint64_t wait_ns;
};

// Walk of one MaskInfo row's non-empty positions (same for every role).
struct Walk {
  int32_t pos = 0, taken = 0;
  __device__ __forceinline__ bool next(const BwdParams& p, int64_t row_base, int32_t n, BlockRef& out) {
    while (taken < n && pos < p.mi.width) {
      const BlockRef r = read_block(p.mi, row_base, pos++, p.err);
      if (r.label != 0) {
        ++taken;
        out = r;
        return true;
      }
    }
    return false;
  }
};

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

__device__ __forceinline__ void store_zero_row(void* base, int fp32, int64_t row, int D) {
  if (fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + row * D);
    for (int e = 0; e < D / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row * D);
    for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
  }
}

// Elementwise core shared by both launches: for 64 columns of one row,
// P = exp2(S*scale_log2 - lse2) where visible (else 0), dS = P*(dP - dsum),
// packed to bf16 pairs.  `allowed` bit c says column c is visible.
template <bool kPerColumnStats>
__device__ __forceinline__ void p_ds_64(const uint32_t* s, const uint32_t* dp, uint64_t allowed, float scale_log2,
                                        float lse2_row, float dsum_row, const float* lse2_col,
                                        const float* dsum_col, uint32_t* p_pk, uint32_t* ds_pk) {
#pragma unroll
  for (int c = 0; c < 64; c += 2) {
    float pv[2], dv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int cc = c + e;
      const float l2 = kPerColumnStats ? lse2_col[cc] : lse2_row;
      const float ds_ = kPerColumnStats ? dsum_col[cc] : dsum_row;
      const float pe = ex2_approx(fmaf(__uint_as_float(s[cc]), scale_log2, -l2));
      const float pm = ((allowed >> cc) & 1ull) ? pe : 0.f;
      pv[e] = pm;
      dv[e] = pm * (__uint_as_float(dp[cc]) - ds_);
    }
    if (p_pk) p_pk[c >> 1] = pack_bf16x2(pv[0], pv[1]);
    ds_pk[c >> 1] = pack_bf16x2(dv[0], dv[1]);
  }
}

// Visibility bits of 64 consecutive columns for one row of a label-1 block.
__device__ __forceinline__ uint64_t dense_bits_64(const uint8_t* row64) {
  uint64_t bits = 0;
  const uint4* src = reinterpret_cast<const uint4*>(row64);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 w = __ldg(src + v);
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if ((wv[e >> 2] >> ((e & 3) * 8)) & 0xFFu) bits |= 1ull << (v * 16 + e);
  }
  return bits;
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

// ===========================================================================
// dK / dV
// ===========================================================================
template <int D>
struct __align__(1024) DkvSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kHalf = 64 * D * 2;
  uint8_t k[kTile];
  uint8_t v[kTile];
  uint8_t q[kStages][kHalf];
  uint8_t dout[kStages][kHalf];
  float lse[kStages][64];
  float dsum[kStages][64];
  uint64_t kv_full, kv_empty;
  uint64_t in_full[kStages], in_empty[kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_empty, drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct DkvTile {
  int32_t b, g, j;
  int32_t total;  // non-empty blocks over the group's q heads
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
  } else {
    t.j = T % p.nK;
    const int32_t bg = T / p.nK;
    t.b = bg / p.Hkv;
    t.g = bg % p.Hkv;
    t.total = 0;
    for (int32_t gh = 0; gh < G; ++gh) t.total += p.mi.row_len[(t.g * G + gh) * p.mi.rows + t.j];
  }
  return t;
}

// Iterates the items (q head of the group, non-empty block, half) of a
// dK/dV tile in a fixed order; every role walks them identically.
struct DkvItems {
  int32_t gh = -1, n = 0;
  int half = 2;
  int64_t row_base = 0;
  Walk w;
  BlockRef cur;
  __device__ __forceinline__ bool next(const BwdParams& p, const DkvTile& t, int32_t& hq, BlockRef& br, int& h) {
    const int32_t G = p.Hq / p.Hkv;
    if (half >= 2) {
      while (true) {
        if (gh >= 0 && gh < G && w.next(p, row_base, n, cur)) {
          half = 0;
          break;
        }
        if (gh >= G) return false;
        ++gh;
        if (gh >= G) return false;
        const int32_t hm = dkv_mask_head(p, t.g * G + gh);
        row_base = (static_cast<int64_t>(hm) * p.mi.rows + t.j) * p.mi.width;
        n = p.mi.row_len[hm * p.mi.rows + t.j];
        w = Walk();
      }
    }
    hq = t.g * G + gh;
    br = cur;
    h = half++;
    return true;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = DkvSmem<D>;
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kChunks = D / 64;
  const int warp = warp_id();
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.kv_full, 1);
    mbar_init(&s.kv_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.in_full[i], 1);
      mbar_init(&s.in_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 128);
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
  const uint32_t tmem = s.tmem_base;
  const WaitCtl wc{p.err, &s.abort_flag, p.wait_ns};
  const uint32_t colDV = kColAcc, colDK = kColAcc + D;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      uint32_t kv_loads = 0, in_loads = 0;
      bool ok = true;
      for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
        const DkvTile t = dkv_decode(p, T);
        if (t.total == 0) continue;
        if (kv_loads >= 1 && !mbar_wait(&s.kv_empty, (kv_loads - 1) & 1u, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.kv_full, 2 * Smem::kTile);
        const int32_t krow = static_cast<int32_t>((static_cast<int64_t>(t.b) * p.Hkv + t.g) * p.Skv + t.j * 128);
        for (int c = 0; c < kChunks; ++c)
          for (int rb = 0; rb < 2; ++rb) {
            tma_load_2d(s.k + c * 16384 + rb * 8192, &tm_k, &s.kv_full, c * 64, krow + rb * 64, pol_kv);
            tma_load_2d(s.v + c * 16384 + rb * 8192, &tm_v, &s.kv_full, c * 64, krow + rb * 64, pol_kv);
          }
        ++kv_loads;
        DkvItems it;
        int32_t hq;
        BlockRef br;
        int half;
        while (it.next(p, t, hq, br, half)) {
          const uint32_t st = in_loads % kStages;
          if (in_loads >= kStages && !mbar_wait(&s.in_empty[st], ((in_loads / kStages) - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.in_full[st], 2 * Smem::kHalf + 512);
          const int64_t qrow = (static_cast<int64_t>(t.b) * p.Hq + hq) * p.Sq + br.col * 128 + half * 64;
          for (int c = 0; c < kChunks; ++c) {
            tma_load_2d(s.q[st] + c * 8192, &tm_q, &s.in_full[st], c * 64, static_cast<int32_t>(qrow), pol_q);
            tma_load_2d(s.dout[st] + c * 8192, &tm_do, &s.in_full[st], c * 64, static_cast<int32_t>(qrow), pol_q);
          }
          bulk_load(s.lse[st], p.lse + qrow, 256, &s.in_full[st]);
          bulk_load(s.dsum[st], p.dsum + qrow, 256, &s.in_full[st]);
          ++in_loads;
        }
      }
      if (!ok) {
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        if (kv_loads) (void)mbar_wait(&s.kv_full, (kv_loads - 1) & 1u, dw);
        for (uint32_t i = (in_loads > kStages ? in_loads - kStages : 0); i < in_loads; ++i)
          (void)mbar_wait(&s.in_full[i % kStages], (i / kStages) & 1u, dw);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      uint32_t kv_uses = 0, in_uses = 0, items = 0, acc_uses = 0;
      uint32_t prev_stage = 0;
      bool ok = true;
      auto issue_acc = [&](uint32_t x, uint32_t stage, bool first) -> bool {
        const uint32_t b2 = x & 1u;
        if (!mbar_wait(&s.p_full[b2], (x >> 1) & 1u, wc)) return false;
        if (first && acc_uses > 0 && !mbar_wait(&s.acc_empty, (acc_uses - 1) & 1u, wc)) return false;
        tc_fence_after();
        const uint32_t dob = smem_u32(s.dout[stage]), qb = smem_u32(s.q[stage]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem + colDV, tmem + kColS + b2 * 64 + kk * 8, sdesc_sw128(dob + kk * 2048, 8192, 1024), idesc_acc,
                 (first && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem + colDK, tmem + kColDP + b2 * 64 + kk * 8, sdesc_sw128(qb + kk * 2048, 8192, 1024), idesc_acc,
                 (first && kk == 0) ? 0u : 1u);
        mma_commit(&s.in_empty[stage]);
        return true;
      };
      for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
        const DkvTile t = dkv_decode(p, T);
        if (t.total == 0) continue;
        if (!mbar_wait(&s.kv_full, kv_uses & 1u, wc)) { ok = false; break; }
        const uint32_t kb = smem_u32(s.k), vb = smem_u32(s.v);
        uint32_t local = 0;
        DkvItems it;
        int32_t hq;
        BlockRef br;
        int half;
        while (it.next(p, t, hq, br, half)) {
          const uint32_t st = in_uses % kStages;
          if (!mbar_wait(&s.in_full[st], (in_uses / kStages) & 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t b2 = items & 1u;
          const uint32_t qb = smem_u32(s.q[st]), dob = smem_u32(s.dout[st]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_ss(tmem + kColS + b2 * 64, sdesc_sw128(kb + ao, 16, 1024), sdesc_sw128(qb + bo, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_ss(tmem + kColDP + b2 * 64, sdesc_sw128(vb + ao, 16, 1024), sdesc_sw128(dob + bo, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(&s.s_full[b2]);
          if (local > 0 && !issue_acc(items - 1, prev_stage, local == 1)) { ok = false; break; }
          prev_stage = st;
          ++in_uses;
          ++items;
          ++local;
        }
        if (!ok) break;
        mma_commit(&s.kv_empty);
        ++kv_uses;
        if (local > 0) {
          if (!issue_acc(items - 1, prev_stage, local == 1)) { ok = false; break; }
          mma_commit(&s.acc_full);
          ++acc_uses;
        }
      }
      mma_commit(&s.drain);
      uint32_t dummy_abort = 0;
      WaitCtl dw{p.err, &dummy_abort, p.wait_ns};
      (void)mbar_wait(&s.drain, 0, dw);
    }
  } else if (warp >= 4) {
    const int r = static_cast<int>(threadIdx.x) - 128;  // key row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t in_uses = 0, items = 0, acc_uses = 0;
    bool ok = true;
    for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
      const DkvTile t = dkv_decode(p, T);
      const int64_t krow = (static_cast<int64_t>(t.b) * p.Hkv + t.g) * p.Skv + static_cast<int64_t>(t.j) * 128 + r;
      if (t.total == 0) {
        store_zero_row(p.dk, p.grad_fp32, krow, D);
        store_zero_row(p.dv, p.grad_fp32, krow, D);
        continue;
      }
      int64_t lo = 0, hi = 0;
      if (p.mi.kind != BSA_MASK_DENSE)
        query_interval(p.mi.kind, p.mi.left, p.mi.right, p.mi.chunk, static_cast<int64_t>(t.j) * 128 + r, lo, hi);
      uint32_t local = 0;
      DkvItems it;
      int32_t hq;
      BlockRef br;
      int half;
      while (it.next(p, t, hq, br, half)) {
        const uint32_t st = in_uses % kStages;
        const uint32_t b2 = items & 1u;
        if (!mbar_wait_warp(&s.in_full[st], (in_uses / kStages) & 1u, wc)) { ok = false; break; }
        if (!mbar_wait_warp(&s.s_full[b2], (items >> 1) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64], dpv[64];
        tmem_ld32(tmem + kColS + b2 * 64 + lane_off, sv);
        tmem_ld32(tmem + kColS + b2 * 64 + 32 + lane_off, sv + 32);
        tmem_ld32(tmem + kColDP + b2 * 64 + lane_off, dpv);
        tmem_ld32(tmem + kColDP + b2 * 64 + 32 + lane_off, dpv + 32);
        uint64_t allowed = ~0ull;
        if (br.label == 1) {
          if (p.mi.kind == BSA_MASK_DENSE) {
            allowed = dense_bits_64(p.mi.partial + (static_cast<int64_t>(br.slot) * 128 + r) * 128 + half * 64);
          } else {
            const int64_t q0 = p.mi.q_sequence[br.col * 128 + half * 64];
            allowed = interval_bits_64(q0, lo, hi);
          }
        }
        float lse2[64], dsc[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          lse2[c] = s.lse[st][c] * kLog2e;
          dsc[c] = s.dsum[st][c];
        }
        tmem_wait_ld();
        uint32_t ppk[32], dspk[32];
        p_ds_64<true>(sv, dpv, allowed, p.scale_log2, 0.f, 0.f, lse2, dsc, ppk, dspk);
        tmem_st32(tmem + kColS + b2 * 64 + lane_off, ppk);
        tmem_st32(tmem + kColDP + b2 * 64 + lane_off, dspk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[b2]);
        ++in_uses;
        ++items;
        ++local;
      }
      if (!ok) break;
      if (local > 0) {
        if (!mbar_wait_warp(&s.acc_full, acc_uses & 1u, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + colDV + c * 32 + lane_off, v);
          tmem_wait_ld();
          store_row(p.dv, p.grad_fp32, krow, D, v, c * 32, 1.f);
          tmem_ld32(tmem + colDK + c * 32 + lane_off, v);
          tmem_wait_ld();
          store_row(p.dk, p.grad_fp32, krow, D, v, c * 32, p.scale);
        }
        tc_fence_before();
        mbar_arrive(&s.acc_empty);
        ++acc_uses;
      } else {
        store_zero_row(p.dk, p.grad_fp32, krow, D);
        store_zero_row(p.dv, p.grad_fp32, krow, D);
      }
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
// dQ
// ===========================================================================
template <int D>
struct __align__(1024) DqSmem {
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kHalf = 64 * D * 2;
  uint8_t q[kTile];
  uint8_t dout[kTile];
  uint8_t k[kStages][kHalf];
  uint8_t v[kStages][kHalf];
  uint64_t qo_full, qo_empty;
  uint64_t in_full[kStages], in_empty[kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full, acc_empty, drain;
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

struct DqItems {
  int half = 2;
  Walk w;
  BlockRef cur;
  __device__ __forceinline__ bool next(const BwdParams& p, const DqTile& t, BlockRef& br, int& h) {
    if (half >= 2) {
      if (!w.next(p, t.row_base, t.n, cur)) return false;
      half = 0;
    }
    br = cur;
    h = half++;
    return true;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = DqSmem<D>;
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kChunks = D / 64;
  const int warp = warp_id();
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.qo_full, 1);
    mbar_init(&s.qo_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.in_full[i], 1);
      mbar_init(&s.in_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    mbar_init(&s.acc_full, 1);
    mbar_init(&s.acc_empty, 128);
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
  const uint32_t tmem = s.tmem_base;
  const WaitCtl wc{p.err, &s.abort_flag, p.wait_ns};

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t qo_loads = 0, in_loads = 0;
      bool ok = true;
      for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
        const DqTile t = dq_decode(p, T);
        if (t.n == 0) continue;
        if (qo_loads >= 1 && !mbar_wait(&s.qo_empty, (qo_loads - 1) & 1u, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.qo_full, 2 * Smem::kTile);
        const int32_t qrow = static_cast<int32_t>((static_cast<int64_t>(t.b) * p.Hq + t.hq) * p.Sq + t.i * 128);
        for (int c = 0; c < kChunks; ++c)
          for (int rb = 0; rb < 2; ++rb) {
            tma_load_2d(s.q + c * 16384 + rb * 8192, &tm_q, &s.qo_full, c * 64, qrow + rb * 64, pol_q);
            tma_load_2d(s.dout + c * 16384 + rb * 8192, &tm_do, &s.qo_full, c * 64, qrow + rb * 64, pol_q);
          }
        ++qo_loads;
        const int32_t g = t.hq / (p.Hq / p.Hkv);
        const int64_t kv_base = (static_cast<int64_t>(t.b) * p.Hkv + g) * p.Skv;
        DqItems it;
        BlockRef br;
        int half;
        while (it.next(p, t, br, half)) {
          const uint32_t st = in_loads % kStages;
          if (in_loads >= kStages && !mbar_wait(&s.in_empty[st], ((in_loads / kStages) - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.in_full[st], 2 * Smem::kHalf);
          const int32_t krow = static_cast<int32_t>(kv_base + br.col * 128 + half * 64);
          for (int c = 0; c < kChunks; ++c) {
            tma_load_2d(s.k[st] + c * 8192, &tm_k, &s.in_full[st], c * 64, krow, pol_kv);
            tma_load_2d(s.v[st] + c * 8192, &tm_v, &s.in_full[st], c * 64, krow, pol_kv);
          }
          ++in_loads;
        }
      }
      if (!ok) {
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        if (qo_loads) (void)mbar_wait(&s.qo_full, (qo_loads - 1) & 1u, dw);
        for (uint32_t i = (in_loads > kStages ? in_loads - kStages : 0); i < in_loads; ++i)
          (void)mbar_wait(&s.in_full[i % kStages], (i / kStages) & 1u, dw);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      uint32_t qo_uses = 0, in_uses = 0, items = 0, acc_uses = 0, prev_stage = 0;
      bool ok = true;
      auto issue_acc = [&](uint32_t x, uint32_t stage, bool first) -> bool {
        const uint32_t b2 = x & 1u;
        if (!mbar_wait(&s.p_full[b2], (x >> 1) & 1u, wc)) return false;
        if (first && acc_uses > 0 && !mbar_wait(&s.acc_empty, (acc_uses - 1) & 1u, wc)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(s.k[stage]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem + kColAcc, tmem + kColDP + b2 * 64 + kk * 8, sdesc_sw128(kb + kk * 2048, 8192, 1024), idesc_acc,
                 (first && kk == 0) ? 0u : 1u);
        mma_commit(&s.in_empty[stage]);
        return true;
      };
      for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
        const DqTile t = dq_decode(p, T);
        if (t.n == 0) continue;
        if (!mbar_wait(&s.qo_full, qo_uses & 1u, wc)) { ok = false; break; }
        const uint32_t qb = smem_u32(s.q), dob = smem_u32(s.dout);
        uint32_t local = 0;
        DqItems it;
        BlockRef br;
        int half;
        while (it.next(p, t, br, half)) {
          const uint32_t st = in_uses % kStages;
          if (!mbar_wait(&s.in_full[st], (in_uses / kStages) & 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t b2 = items & 1u;
          const uint32_t kb = smem_u32(s.k[st]), vb = smem_u32(s.v[st]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_ss(tmem + kColS + b2 * 64, sdesc_sw128(qb + ao, 16, 1024), sdesc_sw128(kb + bo, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ao = (kk >> 2) * 16384 + (kk & 3) * 32, bo = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_ss(tmem + kColDP + b2 * 64, sdesc_sw128(dob + ao, 16, 1024), sdesc_sw128(vb + bo, 16, 1024), idesc_s,
                   kk > 0 ? 1u : 0u);
          }
          mma_commit(&s.s_full[b2]);
          if (local > 0 && !issue_acc(items - 1, prev_stage, local == 1)) { ok = false; break; }
          prev_stage = st;
          ++in_uses;
          ++items;
          ++local;
        }
        if (!ok) break;
        mma_commit(&s.qo_empty);
        ++qo_uses;
        if (local > 0) {
          if (!issue_acc(items - 1, prev_stage, local == 1)) { ok = false; break; }
          mma_commit(&s.acc_full);
          ++acc_uses;
        }
      }
      mma_commit(&s.drain);
      uint32_t dummy_abort = 0;
      WaitCtl dw{p.err, &dummy_abort, p.wait_ns};
      (void)mbar_wait(&s.drain, 0, dw);
    }
  } else if (warp >= 4) {
    const int r = static_cast<int>(threadIdx.x) - 128;  // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t items = 0, acc_uses = 0;
    bool ok = true;
    for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
      const DqTile t = dq_decode(p, T);
      const int64_t qrow = (static_cast<int64_t>(t.b) * p.Hq + t.hq) * p.Sq + static_cast<int64_t>(t.i) * 128 + r;
      if (t.n == 0) {
        store_zero_row(p.dq, p.grad_fp32, qrow, D);
        continue;
      }
      const float lse2 = p.lse[qrow] * kLog2e;
      const float dsum_r = p.dsum[qrow];
      int64_t lo = 0, hi = 0;
      if (p.mi.kind != BSA_MASK_DENSE) {
        const int64_t qi = p.mi.q_sequence[t.i * 128 + r];
        key_interval(p.mi.kind, p.mi.left, p.mi.right, p.mi.chunk, qi, lo, hi);
      }
      uint32_t local = 0;
      DqItems it;
      BlockRef br;
      int half;
      while (it.next(p, t, br, half)) {
        const uint32_t b2 = items & 1u;
        if (!mbar_wait_warp(&s.s_full[b2], (items >> 1) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64], dpv[64];
        tmem_ld32(tmem + kColS + b2 * 64 + lane_off, sv);
        tmem_ld32(tmem + kColS + b2 * 64 + 32 + lane_off, sv + 32);
        tmem_ld32(tmem + kColDP + b2 * 64 + lane_off, dpv);
        tmem_ld32(tmem + kColDP + b2 * 64 + 32 + lane_off, dpv + 32);
        uint64_t allowed = ~0ull;
        if (br.label == 1) {
          if (p.mi.kind == BSA_MASK_DENSE)
            allowed = dense_bits_64(p.mi.partial + (static_cast<int64_t>(br.slot) * 128 + r) * 128 + half * 64);
          else
            allowed = interval_bits_64(static_cast<int64_t>(br.col) * 128 + half * 64, lo, hi);
        }
        tmem_wait_ld();
        uint32_t dspk[32];
        p_ds_64<false>(sv, dpv, allowed, p.scale_log2, lse2, dsum_r, nullptr, nullptr, nullptr, dspk);
        tmem_st32(tmem + kColDP + b2 * 64 + lane_off, dspk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[b2]);
        ++items;
        ++local;
      }
      if (!ok) break;
      if (local > 0) {
        if (!mbar_wait_warp(&s.acc_full, acc_uses & 1u, wc)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + kColAcc + c * 32 + lane_off, v);
          tmem_wait_ld();
          store_row(p.dq, p.grad_fp32, qrow, D, v, c * 32, p.scale);
        }
        tc_fence_before();
        mbar_arrive(&s.acc_empty);
        ++acc_uses;
      } else {
        store_zero_row(p.dq, p.grad_fp32, qrow, D);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool make_maps(const bsa_bwd_args* a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tdo) {
  const uint64_t q_rows = static_cast<uint64_t>(a->B) * a->Hq * a->S_q;
  const uint64_t kv_rows = static_cast<uint64_t>(a->B) * a->Hkv * a->S_kv;
  const int D = a->D;
  return make_tmap_bf16_2d(tq, a->q, q_rows, D, D * 2, 64, 64) &&
         make_tmap_bf16_2d(tk, a->k, kv_rows, D, D * 2, 64, 64) &&
         make_tmap_bf16_2d(tv, a->v, kv_rows, D, D * 2, 64, 64) &&
         make_tmap_bf16_2d(tdo, a->do_, q_rows, D, D * 2, 64, 64);
}

BwdParams make_params(const bsa_bwd_args* a, const bsa_mask_info* info, float scale) {
  BwdParams p{};
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
  p.grad_fp32 = a->grad_fp32 ? 1 : 0;
  p.mi = mask_info_dev(info);
  p.err = device_error_word();
  p.wait_ns = wait_limit_ns();
  return p;
}

template <int D>
bsa_status launch_dkv(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo;
  if (!make_maps(a, &tq, &tk, &tv, &tdo)) return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor");
  BwdParams p = make_params(a, info, scale);
  if (!p.err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  p.n_tiles = a->B * a->Hkv * p.nK;
  const size_t smem = sizeof(DkvSmem<D>) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dkv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "set dkv smem size");
    attr_set = true;
  }
  const int grid = std::min(p.n_tiles, num_sms());
  dkv_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tk, tv, tdo, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dkv launch");
  return BSA_OK;
}

template <int D>
bsa_status launch_dq(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo;
  if (!make_maps(a, &tq, &tk, &tv, &tdo)) return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a tensor");
  BwdParams p = make_params(a, info, scale);
  if (!p.err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  p.n_tiles = a->B * a->Hq * p.nQ;
  const size_t smem = sizeof(DqSmem<D>) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "set dq smem size");
    attr_set = true;
  }
  const int grid = std::min(p.n_tiles, num_sms());
  dq_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tk, tv, tdo, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dq launch");
  return BSA_OK;
}

}  // namespace

bsa_status dkv_launch(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  if (a->D == 128) return launch_dkv<128>(a, info, scale, stream);
  return launch_dkv<64>(a, info, scale, stream);
}

bsa_status dq_launch(const bsa_bwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  if (a->D == 128) return launch_dq<128>(a, info, scale, stream);
  return launch_dq<64>(a, info, scale, stream);
}

}  // namespace bsa
