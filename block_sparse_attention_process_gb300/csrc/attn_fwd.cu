// Block-sparse forward attention for sm_103a (TMA + tcgen05/TMEM).
//
// Method: "Splash Attention: When the Mask Stops Being Arithmetic and
// Becomes the Loop", section "What is splash attention and how is it
// different from flash attention?": the kernel reads each grid position's
// label from MaskInfo; label 0 means the body does not run and the K/V
// blocks are not fetched, label 2 skips the masking, only label 1 computes
// and masks.  The row walk follows MaskInfo's data_next ("What is MaskInfo
// in splash attention?"), and a shrunk MaskInfo has only the non-empty
// columns ("What does grid shrinking do in splash attention?").  The
// softmax is the online one of flash attention: a running row maximum and
// normaliser, a rescale of the accumulator when the maximum moves, and one
// divide at the end.
//
// GB300 design (one CTA per SM, persistent):
//   warp 0      TMA producer: Q tile (2 buffers), K and V blocks (2-stage rings)
//   warp 1      tcgen05 issuer: S = Q K^T into TMEM (2 buffers), O += P V
//               with P read from TMEM (aliases its S buffer as bf16)
//   warps 4-7   softmax (one query row per thread): mask, row max, exp2,
//               row sum, P to TMEM, lazy O rescale in TMEM, epilogue
// Work tiles are (batch, query head, query block), visited longest row
// first; consecutive tiles take consecutive heads of a KV group so
// concurrently running CTAs share K/V blocks through L2.
#include <cmath>

#include "internal.h"
#include "maskinfo_dev.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace bsa {
namespace {

constexpr int kStagesK = 2;
constexpr int kStagesV = 2;
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // two S/P buffers at columns 0 and 128
constexpr uint32_t kTmemO = 256;  // O accumulator
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by more

template <int D>
struct __align__(1024) FwdSmem {
  static constexpr int kTileBytes = 128 * D * 2;
  uint8_t q[2][kTileBytes];
  uint8_t k[kStagesK][kTileBytes];
  uint8_t v[kStagesV][kTileBytes];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_full, o_empty, drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
};

struct FwdParams {
  int32_t B, Hq, Hkv, nQ, nK;
  int64_t Sq, Skv;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  MaskInfoDev mi;
  int32_t n_tiles;
  uint32_t* err;
  uint64_t wait_ns;
};

struct Tile {
  int32_t b, hq, i, hm, n;
  int64_t row_base;
};

__device__ __forceinline__ Tile decode_tile(const FwdParams& p, int32_t T) {
  Tile t;
  if (p.mi.heads == 1) {
    const int32_t bh = T % (p.B * p.Hq);
    const int32_t rank = T / (p.B * p.Hq);
    t.i = p.mi.row_order[rank];
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

// Walks the non-empty positions of one MaskInfo row.  Every role walks the
// same row the same way, so all of them see the same block sequence.
struct RowWalk {
  int32_t pos = 0, taken = 0;
  __device__ __forceinline__ bool next(const FwdParams& p, const Tile& t, BlockRef& out) {
    while (taken < t.n && pos < p.mi.width) {
      const BlockRef r = read_block(p.mi, t.row_base, pos++, p.err);
      if (r.label != 0) {
        ++taken;
        out = r;
        return true;
      }
    }
    return false;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  using Smem = FwdSmem<D>;
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kTileBytes = Smem::kTileBytes;
  constexpr int kChunks = D / 64;  // 64-column (128-byte) swizzle chunks per tile row

  const int warp = warp_id();
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    for (int i = 0; i < kStagesK; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < kStagesV; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.o_full, 1);
    mbar_init(&s.o_empty, 128);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t q_loads = 0, k_loads = 0, v_loads = 0;
      bool ok = true;
      for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
        const Tile t = decode_tile(p, T);
        if (t.n == 0) continue;
        const uint32_t qb = q_loads & 1u;
        if (q_loads >= 2 && !mbar_wait(&s.q_empty[qb], ((q_loads >> 1) - 1) & 1u, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.q_full[qb], kTileBytes);
        const int32_t qrow = static_cast<int32_t>((static_cast<int64_t>(t.b) * p.Hq + t.hq) * p.Sq + t.i * 128);
        for (int c = 0; c < kChunks; ++c) tma_load_2d(s.q[qb] + c * 16384, &tm_q, &s.q_full[qb], c * 64, qrow, pol_q);
        ++q_loads;
        const int32_t g = t.hq / (p.Hq / p.Hkv);
        const int64_t kv_base = (static_cast<int64_t>(t.b) * p.Hkv + g) * p.Skv;
        RowWalk w;
        BlockRef br;
        while (w.next(p, t, br)) {
          const int32_t krow = static_cast<int32_t>(kv_base + br.col * 128);
          const uint32_t ks = k_loads % kStagesK;
          if (k_loads >= kStagesK && !mbar_wait(&s.k_empty[ks], ((k_loads / kStagesK) - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.k_full[ks], kTileBytes);
          for (int c = 0; c < kChunks; ++c) tma_load_2d(s.k[ks] + c * 16384, &tm_k, &s.k_full[ks], c * 64, krow, pol_kv);
          ++k_loads;
          const uint32_t vs = v_loads % kStagesV;
          if (v_loads >= kStagesV && !mbar_wait(&s.v_empty[vs], ((v_loads / kStagesV) - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.v_full[vs], kTileBytes);
          for (int c = 0; c < kChunks; ++c) tma_load_2d(s.v[vs] + c * 16384, &tm_v, &s.v_full[vs], c * 64, krow, pol_kv);
          ++v_loads;
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        for (uint32_t i = (q_loads > 2 ? q_loads - 2 : 0); i < q_loads; ++i) (void)mbar_wait(&s.q_full[i & 1u], (i >> 1) & 1u, dw);
        for (uint32_t i = (k_loads > kStagesK ? k_loads - kStagesK : 0); i < k_loads; ++i)
          (void)mbar_wait(&s.k_full[i % kStagesK], (i / kStagesK) & 1u, dw);
        for (uint32_t i = (v_loads > kStagesV ? v_loads - kStagesV : 0); i < v_loads; ++i)
          (void)mbar_wait(&s.v_full[i % kStagesV], (i / kStagesV) & 1u, dw);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      uint32_t q_uses = 0, k_uses = 0, v_uses = 0, s_uses = 0, o_uses = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t sidx, bool first) -> bool {
        const uint32_t pb = sidx & 1u;
        if (!mbar_wait(&s.p_full[pb], (sidx >> 1) & 1u, wc)) return false;
        if (first && o_uses > 0 && !mbar_wait(&s.o_empty, (o_uses - 1) & 1u, wc)) return false;
        const uint32_t vs = v_uses % kStagesV;
        if (!mbar_wait(&s.v_full[vs], (v_uses / kStagesV) & 1u, wc)) return false;
        tc_fence_after();
        const uint32_t vbase = smem_u32(s.v[vs]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bdesc = sdesc_sw128(vbase + kk * 2048, 16384, 1024);
          mma_ts(tmem + kTmemO, tmem + kTmemS + pb * 128 + kk * 8, bdesc, idesc_o, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(&s.v_empty[vs]);
        mma_commit(&s.pv_done);
        ++v_uses;
        return true;
      };
      for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
        const Tile t = decode_tile(p, T);
        if (t.n == 0) continue;
        const uint32_t qb = q_uses & 1u;
        if (!mbar_wait(&s.q_full[qb], (q_uses >> 1) & 1u, wc)) { ok = false; break; }
        const uint32_t qbase = smem_u32(s.q[qb]);
        uint32_t exec = 0;
        RowWalk w;
        BlockRef br;
        while (w.next(p, t, br)) {
          const uint32_t ks = k_uses % kStagesK;
          if (!mbar_wait(&s.k_full[ks], (k_uses / kStagesK) & 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kbase = smem_u32(s.k[ks]);
          const uint32_t sb = s_uses & 1u;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tmem + kTmemS + sb * 128, sdesc_sw128(qbase + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024),
                   idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s.s_full[sb]);
          mma_commit(&s.k_empty[ks]);
          ++k_uses;
          if (exec > 0 && !issue_pv(s_uses - 1, exec == 1)) { ok = false; break; }
          ++s_uses;
          ++exec;
        }
        if (!ok) break;
        mma_commit(&s.q_empty[qb]);
        ++q_uses;
        if (exec > 0) {
          if (!issue_pv(s_uses - 1, exec == 1)) { ok = false; break; }
          mma_commit(&s.o_full);
          ++o_uses;
        }
      }
      // Every MMA issued so far completes before tensor memory is released.
      mma_commit(&s.drain);
      uint32_t dummy_abort = 0;
      WaitCtl dw{p.err, &dummy_abort, p.wait_ns};
      (void)mbar_wait(&s.drain, 0, dw);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int r = static_cast<int>(threadIdx.x) - 128;         // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float scale_log2 = p.scale_log2;
    uint32_t s_uses = 0, o_uses = 0;
    bool ok = true;
    for (int32_t T = blockIdx.x; T < p.n_tiles && ok; T += gridDim.x) {
      const Tile t = decode_tile(p, T);
      const int64_t orow = (static_cast<int64_t>(t.b) * p.Hq + t.hq) * p.Sq + static_cast<int64_t>(t.i) * 128 + r;
      __nv_bfloat16* optr = p.o + orow * D;
      int64_t lo = 0, hi = 0;
      if (p.mi.kind != BSA_MASK_DENSE) {
        const int64_t q = p.mi.q_sequence[t.i * 128 + r];
        key_interval(p.mi.kind, p.mi.left, p.mi.right, p.mi.chunk, q, lo, hi);
      }
      float m = -INFINITY, l = 0.f;
      uint32_t exec = 0;
      RowWalk w;
      BlockRef br;
      while (t.n > 0 && w.next(p, t, br)) {
        const uint32_t sb = s_uses & 1u;
        if (!mbar_wait_warp(&s.s_full[sb], (s_uses >> 1) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        float x[128];
        {
          uint32_t xu[128];
          const uint32_t sa = tmem + kTmemS + sb * 128 + lane_off;
          tmem_ld32(sa + 0, xu + 0);
          tmem_ld32(sa + 32, xu + 32);
          tmem_ld32(sa + 64, xu + 64);
          tmem_ld32(sa + 96, xu + 96);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(xu[c]);
        }
        if (br.label == 1) {
          if (p.mi.kind == BSA_MASK_DENSE) {
            const uint4* mrow = reinterpret_cast<const uint4*>(p.mi.partial + (static_cast<int64_t>(br.slot) * 128 + r) * 128);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const uint4 mw = __ldg(mrow + v);
              const uint32_t wv[4] = {mw.x, mw.y, mw.z, mw.w};
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (((wv[e >> 2] >> ((e & 3) * 8)) & 0xFFu) == 0u) x[v * 16 + e] = -INFINITY;
            }
          } else {
            const int64_t k0 = static_cast<int64_t>(br.col) * 128;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const int64_t k = k0 + c;
              if (k < lo || k > hi) x[c] = -INFINITY;
            }
          }
        }
        float mx = x[0];
#pragma unroll
        for (int c = 1; c < 128; ++c) mx = fmaxf(mx, x[c]);
        const float m_blk = mx * scale_log2;
        const float m_cand = fmaxf(m, m_blk);
        bool switch_ref = m_cand > m + kRescaleThreshold;
        const bool warp_switch = __any_sync(0xffffffffu, switch_ref);
        float alpha = 1.f;
        if (warp_switch) {
          alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_cand);
          m = m_cand;
        }
        const float m_use = (m == -INFINITY) ? 0.f : m;
        float rs = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2_approx(fmaf(x[2 * c], scale_log2, -m_use));
          const float p1 = ex2_approx(fmaf(x[2 * c + 1], scale_log2, -m_use));
          rs += p0 + p1;
          pk[c] = pack_bf16x2(p0, p1);
        }
        l = l * alpha + rs;
        // O holds earlier blocks' sum only after the first block; rescale it
        // (after the previous P V has landed) when this warp moved its max.
        if (warp_switch && exec > 0) {
          if (!mbar_wait_warp(&s.pv_done, (s_uses - 1) & 1u, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            const uint32_t oa = tmem + kTmemO + c * 32 + lane_off;
            tmem_ld32(oa, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(oa, ov);
          }
        }
        {
          const uint32_t pa = tmem + kTmemS + sb * 128 + lane_off;
          tmem_st32(pa + 0, pk + 0);
          tmem_st32(pa + 32, pk + 32);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[sb]);
        ++s_uses;
        ++exec;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (exec > 0) {
        if (!mbar_wait_warp(&s.o_full, o_uses & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem + kTmemO + c * 32 + lane_off, ov);
          tmem_wait_ld();
          uint4* dst = reinterpret_cast<uint4*>(optr + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 o4;
            o4.x = pack_bf16x2(__uint_as_float(ov[8 * v + 0]) * inv_l, __uint_as_float(ov[8 * v + 1]) * inv_l);
            o4.y = pack_bf16x2(__uint_as_float(ov[8 * v + 2]) * inv_l, __uint_as_float(ov[8 * v + 3]) * inv_l);
            o4.z = pack_bf16x2(__uint_as_float(ov[8 * v + 4]) * inv_l, __uint_as_float(ov[8 * v + 5]) * inv_l);
            o4.w = pack_bf16x2(__uint_as_float(ov[8 * v + 6]) * inv_l, __uint_as_float(ov[8 * v + 7]) * inv_l);
            dst[v] = o4;
          }
        }
        tc_fence_before();
        mbar_arrive(&s.o_empty);
        ++o_uses;
        const float m_use = (m == -INFINITY) ? 0.f : m;
        p.lse[orow] = l > 0.f ? (m_use + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      } else {
        uint4* dst = reinterpret_cast<uint4*>(optr);
        for (int v = 0; v < D / 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
        p.lse[orow] = -INFINITY;
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

template <int D>
bsa_status launch_fwd(const bsa_fwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  const uint64_t q_rows = static_cast<uint64_t>(a->B) * a->Hq * a->S_q;
  const uint64_t kv_rows = static_cast<uint64_t>(a->B) * a->Hkv * a->S_kv;
  if (!make_tmap_bf16_2d(&tq, a->q, q_rows, D, D * 2, 128, 64) ||
      !make_tmap_bf16_2d(&tk, a->k, kv_rows, D, D * 2, 128, 64) ||
      !make_tmap_bf16_2d(&tv, a->v, kv_rows, D, D * 2, 128, 64))
    return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a Q/K/V description");
  FwdParams p{};
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.Sq = a->S_q;
  p.Skv = a->S_kv;
  p.nQ = static_cast<int32_t>(a->S_q / 128);
  p.nK = static_cast<int32_t>(a->S_kv / 128);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = static_cast<__nv_bfloat16*>(a->o);
  p.lse = a->lse;
  p.mi = mask_info_dev(info);
  p.n_tiles = a->B * a->Hq * p.nQ;
  p.err = device_error_word();
  p.wait_ns = wait_limit_ns();
  if (!p.err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "set forward smem size");
    attr_set = true;
  }
  const int grid = std::min(p.n_tiles, num_sms());
  fwd_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return BSA_OK;
}

}  // namespace

bsa_status fwd_launch(const bsa_fwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  if (a->D == 128) return launch_fwd<128>(a, info, scale, stream);
  return launch_fwd<64>(a, info, scale, stream);
}

}  // namespace bsa
