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
// GB300 design (one persistent CTA per SM, warp-specialised):
//   warp 0      TMA producer of Q tiles (2 buffers) and K blocks (2 stages)
//   warp 1      tcgen05 issuer, warp-converged (one elected lane issues):
//               S = Q K^T into one of two TMEM score buffers, a block ahead
//               of the softmax, and O_p += P_p V_p for each softmax part p,
//               P_p read from TMEM (bf16 over the part's own score columns)
//   warp 2      TMA producer of V blocks (2 stages)
//   warp 3      walker: follows the CTA's tile list and the MaskInfo rows
//               and publishes one descriptor per non-empty block
//   warps 4-11  softmax in two warpgroups (parts), one (row, half of the
//               columns) per thread, each part with its own running maximum
//               and sum: mask, row max, exp2, row sum, P to TMEM, lazy
//               rescale of the part's O in TMEM; at a tile's end the
//               statistics go to shared memory and the softmax moves on
//   warps 12-15 epilogue: combines the parts' (maximum, sum, O) into O / l
//               in bf16 (tensor stores) and the logsumexp, one row per
//               thread, while the next tile runs
// Each CTA walks one fixed sequence of (tile, block) pairs; every role
// walks it the same way, so the pipelines stay in step without sharing
// state.  Work tiles are (batch, query head, query block), longest rows
// first; consecutive tiles take consecutive heads of a KV group so that
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
constexpr int kSBufs = 2;         // score buffers in TMEM
static_assert(kStagesK == kSBufs && kStagesV == kSBufs, "K stage, V stage and score buffer of a block share its index");
constexpr int kInfoRing = 32;     // block descriptors published by the walker warp
// The softmax is split over kParts warpgroups, each taking kCols of the 128
// score columns of every row (and D / kParts of the O columns).
constexpr int kParts = 2;
constexpr int kCols = 128 / kParts;
constexpr int kSoftmaxWarps = 4 * kParts;
// 4 role warps + the softmax warps + one epilogue warpgroup
constexpr int kThreads = 128 + 32 * kSoftmaxWarps + 128;
constexpr int kEpiWarp0 = 4 + kSoftmaxWarps;  // first warp of the epilogue warpgroup
// Readers that release a block descriptor: the V producer and every softmax
// warp.  A softmax warp releases it once the block's scores are ready, by
// when the K producer and the MMA warp have read it too.
constexpr uint32_t kInfoReaders = 1 + kSoftmaxWarps;
// Flags in a block descriptor's first word, beside col (bits 0-15) and label (16-17).
constexpr uint32_t kFirst = 1u << 20;  // first block of its tile
constexpr uint32_t kLast = 1u << 21;   // last block of its tile
constexpr uint32_t kEnd = 1u << 22;    // no more blocks for this CTA
constexpr uint32_t kTmemCols = 512;
// One O accumulator per softmax part after the two 128-column score
// buffers: part p's running maximum is its own, so its P V goes to its own
// accumulator, and the epilogue combines the parts.
constexpr uint32_t kTmemO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by more

template <int D>
struct __align__(1024) FwdSmem {
  static constexpr int kTileBytes = 128 * D * 2;
  uint8_t q[2][kTileBytes];
  uint8_t k[kStagesK][kTileBytes];
  uint8_t v[kStagesV][kTileBytes];
  // bf16 output staging of the epilogue warps: 32 rows x 64 columns each
  // (128-byte swizzle, the layout of the output tensor map's box)
  uint8_t ostage[4][32 * 128];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  // s_full[b] also frees K stage b (the scores of a block are the only
  // reader of its K) and v_empty[b] marks block n's P V done for the
  // softmax's rescale (b = n mod 2 for both)
  uint64_t s_full[kSBufs], p_full[kSBufs];
  uint64_t o_full, o_empty, drain;
  uint64_t info_full[kInfoRing], info_empty[kInfoRing];
  // per block: {col | label<<16 | flags, stack slot, q_sequence of the tile's first query,
  // (b*Hq + hq)*Sq + 128*i = Q and output row of the tile's first query}
  uint4 binfo[kInfoRing];
  uint32_t bkrow[kInfoRing];  // K/V row of the block's first key
  // a finished tile's row statistics for the epilogue warpgroup, per [tile
  // parity][part]: the part's running maximum (log2 units) and row sum
  float tmax[2][kParts][128];
  float tsum[2][kParts][128];
  uint32_t trow[2];              // output row of the tile's first query
  uint64_t stats_full[2], stats_empty[2];
  uint32_t tmem_base;
  uint32_t abort_flag;
};

static_assert(sizeof(FwdSmem<128>) + 1024 <= 232448, "forward shared memory exceeds 227 KB per CTA");

struct FwdParams {
  int32_t B, Hq, Hkv, nQ, nK;
  int64_t Sq, Skv;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  MaskInfoDev mi;
  int32_t n_tiles;
  const int4* sched;     // this launch's tile lists, sched_stride entries per CTA
  int32_t sched_stride;
  // Key shard: only MaskInfo blocks with column in [kv_lo, kv_hi) are
  // visited, K/V row of column c = (c - kv_lo) * 128.  With `partial` the
  // epilogue writes the unnormalised accumulator, reference maximum
  // (natural-log units) and normaliser instead of O and LSE.
  int32_t kv_lo, kv_hi;
  int32_t partial;
  // soft cap c (off when cap_scale == 0): scaled score s -> c*tanh(s/c),
  // i.e. log2 units cap_log2 * tanh(raw * cap_scale), cap_scale = scale / c
  float cap_log2, cap_scale;
  // sinks: n_sinks logits per row in the normaliser; row sinks_kv ? kv head : 0
  const float* sinks;
  int32_t n_sinks, sinks_kv;
  float* o_acc;
  float* m_out;
  float* l_out;
  uint32_t* err;
  uint64_t wait_ns;
};

// kX: the logit soft cap and / or attention sinks are compiled in (a
// separate instantiation, so that the plain kernel keeps its code); kBits:
// a dense mask's partial blocks are read as bits (the instantiation for
// dense masks without the transforms; the others read the bytes).
template <int D, bool kX, bool kBits>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const __grid_constant__ FwdParams p) {
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
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 32 * kSoftmaxWarps);
    }
    for (int i = 0; i < kStagesK; ++i) {
      mbar_init(&s.k_full[i], 1);
    }
    for (int i = 0; i < kStagesV; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    for (int i = 0; i < kInfoRing; ++i) {
      mbar_init(&s.info_full[i], 1);
      mbar_init(&s.info_empty[i], kInfoReaders);
    }
    mbar_init(&s.o_full, 1);
    mbar_init(&s.o_empty, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.stats_full[i], 32 * kSoftmaxWarps);
      mbar_init(&s.stats_empty[i], 128);
    }
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
  // Set-up done: the next kernel may launch.  This one waits for the
  // previous kernel (griddep_wait) only in the roles that touch Q/K/V or
  // write O/LSE; MaskInfo is complete when its compile returns, so the
  // walker starts right away.
  griddep_launch_dependents();

  if (warp == 3) {
    // ------------------------------------------------------------ block walker
    // Every lane walks the same sequence (same loads, one transaction each);
    // lane 0 publishes.  Tiles with no block are written here directly.
    uint32_t n = 0;
    bool ok = true;
    auto publish = [&](uint32_t x, uint32_t y, uint32_t z, uint32_t w, uint32_t krow) -> bool {
      const uint32_t slot = n % kInfoRing;
      if (n >= static_cast<uint32_t>(kInfoRing) &&
          !mbar_wait_warp(&s.info_empty[slot], ((n / kInfoRing) - 1) & 1u, wc))
        return false;
      if (lane == 0) {
        s.binfo[slot] = make_uint4(x, y, z, w);
        s.bkrow[slot] = krow;
        mbar_arrive(&s.info_full[slot]);
      }
      __syncwarp();
      ++n;
      return true;
    };
    // this CTA's tiles: {query block, blocks, b * Hq + hq}, next one loaded ahead
    const int4* mine = p.sched + static_cast<int64_t>(blockIdx.x) * p.sched_stride;
    int4 ahead_tile = mine[0];
    for (int32_t k = 0; ok && k < p.sched_stride; ++k) {
      const int4 te = ahead_tile;
      if (te.y < 0) break;
      if (k + 1 < p.sched_stride) ahead_tile = mine[k + 1];
      const int32_t t_n = te.y, t_i = te.x;
      const int32_t t_b = te.z / p.Hq, t_hq = te.z % p.Hq;
      const int32_t t_hm = p.mi.heads == 1 ? 0 : t_hq;
      const int64_t t_row_base = (static_cast<int64_t>(t_hm) * p.mi.rows + t_i) * p.mi.width;
      const int64_t n_rows_q = static_cast<int64_t>(p.B) * p.Hq * p.Sq;
      const int64_t out_row =
          BSA_RANGE(static_cast<int64_t>(te.z) * p.Sq + static_cast<int64_t>(t_i) * 128, int64_t(0), n_rows_q - 127, p.err);
      // blocks of this launch's key range: the whole row, or (a key shard)
      // those found by a first pass over the row
      const bool ranged = p.kv_lo > 0 || p.kv_hi < p.mi.cols;
      int32_t n_in = t_n;
      if (ranged && t_n > 0) {
        n_in = 0;
        int32_t j = 0;
        for (int32_t pos = 0; pos < p.mi.width && j < t_n; ++pos) {
          const BlockRef br = read_block(p.mi, t_row_base, pos, lane == 0 ? p.err : nullptr);
          if (br.label == 0) continue;
          ++j;
          if (br.col >= p.kv_lo && br.col < p.kv_hi) ++n_in;
        }
      }
      if (n_in == 0) {
        // every key of the range masked for the whole query block:
        // O = 0, LSE = -inf (a shard: accumulator 0, maximum -inf, normaliser 0)
        griddep_wait();
        if (p.partial) {
          float4* dst = reinterpret_cast<float4*>(p.o_acc + out_row * D);
          for (int v = lane; v < 128 * D / 4; v += 32) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int r = lane; r < 128; r += 32) {
            p.m_out[out_row + r] = -INFINITY;
            p.l_out[out_row + r] = 0.f;
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(p.o + out_row * D);
          for (int v = lane; v < 128 * D / 8; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
          // only the sinks are left in the normaliser
          float lse0 = -INFINITY;
          if (kX && p.n_sinks > 0) {
            const float* z = p.sinks + (p.sinks_kv ? (t_hq / (p.Hq / p.Hkv)) * p.n_sinks : 0);
            float zm = -INFINITY, zs = 0.f;
            for (int j = 0; j < p.n_sinks; ++j) zm = fmaxf(zm, z[j]);
            for (int j = 0; j < p.n_sinks; ++j) zs += expf(z[j] - zm);
            lse0 = zm + logf(zs);
          }
          for (int r = lane; r < 128; r += 32) p.lse[out_row + r] = lse0;
        }
        continue;
      }
      const uint32_t q0 = static_cast<uint32_t>(p.mi.q_sequence[t_i * 128]);
      const int64_t kv_base = (static_cast<int64_t>(t_b) * p.Hkv + t_hq / (p.Hq / p.Hkv)) * p.Skv;
      int32_t j = 0, pub = 0;
      RawRef ahead = load_block(p.mi, t_row_base, 0);
      for (int32_t pos = 0; ok && pos < p.mi.width && j < t_n; ++pos) {
        const RawRef cur = ahead;
        if (pos + 1 < p.mi.width) ahead = load_block(p.mi, t_row_base, pos + 1);
        const BlockRef br = check_block(p.mi, cur, lane == 0 ? p.err : nullptr);
        if (br.label == 0) continue;
        ++j;
        if (br.col < p.kv_lo || br.col >= p.kv_hi) continue;
        const uint32_t x = static_cast<uint32_t>(br.col) | (static_cast<uint32_t>(br.label) << 16) |
                           (pub == 0 ? kFirst : 0u) | (pub + 1 == n_in ? kLast : 0u);
        ok = publish(x, static_cast<uint32_t>(br.slot), q0, static_cast<uint32_t>(out_row),
                     static_cast<uint32_t>(kv_base + static_cast<int64_t>(br.col - p.kv_lo) * 128));
        ++pub;
      }
      // a malformed row with fewer non-empty entries than expected: flagged
      // dummy blocks keep every role's count in step
      for (; ok && pub < n_in; ++pub) {
        if (lane == 0 && p.err) atomicOr(p.err, DEV_ERR_BOUNDS);
        ok = publish((2u << 16) | (pub == 0 ? kFirst : 0u) | (pub + 1 == n_in ? kLast : 0u), 0u, q0,
                     static_cast<uint32_t>(out_row), static_cast<uint32_t>(kv_base));
      }
    }
    if (ok) (void)publish(kEnd, 0u, 0u, 0u, 0u);
  } else if (warp == 0) {
    // ------------------------------------------------------------ Q and K producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      griddep_wait();
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t n = 0, q_loads = 0, k_loads = 0;
      bool ok = true;
      while (ok) {
        const uint32_t slot = n % kInfoRing;
        if (!mbar_wait(&s.info_full[slot], (n / kInfoRing) & 1u, wc)) { ok = false; break; }
        const uint32_t x = s.binfo[slot].x;
        const uint32_t qrow = s.binfo[slot].w;
        const uint32_t krow = s.bkrow[slot];
        const uint32_t ks = k_loads % kStagesK;
        // stage ks is free once the scores of the block two back are ready
        if (k_loads >= kStagesK && !mbar_wait(&s.s_full[ks], ((k_loads / kStagesK) - 1) & 1u, wc)) { ok = false; break; }
        if (x & kEnd) {
          // no more blocks: complete the stage without data so the MMA warp reads the end mark
          mbar_arrive(&s.k_full[ks]);
          break;
        }
        if (x & kFirst) {
          const uint32_t qb = q_loads & 1u;
          if (q_loads >= 2 && !mbar_wait(&s.q_empty[qb], ((q_loads >> 1) - 1) & 1u, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.q_full[qb], kTileBytes);
          for (int c = 0; c < kChunks; ++c)
            tma_load_2d(s.q[qb] + c * 16384, &tm_q, &s.q_full[qb], c * 64, static_cast<int32_t>(qrow), pol_q);
          ++q_loads;
        }
        mbar_arrive_expect_tx(&s.k_full[ks], kTileBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(s.k[ks] + c * 16384, &tm_k, &s.k_full[ks], c * 64, static_cast<int32_t>(krow), pol_kv);
        ++k_loads;
        ++n;
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        for (uint32_t i = (q_loads > 2 ? q_loads - 2 : 0); i < q_loads; ++i) (void)mbar_wait(&s.q_full[i & 1u], (i >> 1) & 1u, dw);
        for (uint32_t i = (k_loads > kStagesK ? k_loads - kStagesK : 0); i < k_loads; ++i)
          (void)mbar_wait(&s.k_full[i % kStagesK], (i / kStagesK) & 1u, dw);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      griddep_wait();
      const uint64_t pol_kv = policy_evict_last();
      uint32_t n = 0, v_loads = 0;
      bool ok = true;
      while (ok) {
        const uint32_t slot = n % kInfoRing;
        if (!mbar_wait(&s.info_full[slot], (n / kInfoRing) & 1u, wc)) { ok = false; break; }
        const uint32_t x = s.binfo[slot].x;
        const uint32_t krow = s.bkrow[slot];
        mbar_arrive(&s.info_empty[slot]);
        if (x & kEnd) break;
        const uint32_t vs = v_loads % kStagesV;
        if (v_loads >= kStagesV && !mbar_wait(&s.v_empty[vs], ((v_loads / kStagesV) - 1) & 1u, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.v_full[vs], kTileBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(s.v[vs] + c * 16384, &tm_v, &s.v_full[vs], c * 64, static_cast<int32_t>(krow), pol_kv);
        ++v_loads;
        ++n;
      }
      if (!ok) {
        uint32_t dummy_abort = 0;
        WaitCtl dw{nullptr, &dummy_abort, p.wait_ns};
        for (uint32_t i = (v_loads > kStagesV ? v_loads - kStagesV : 0); i < v_loads; ++i)
          (void)mbar_wait(&s.v_full[i % kStagesV], (i / kStagesV) & 1u, dw);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
    // descriptors of buffer 0; buffers of one kind are contiguous, kTileBytes apart
    const uint64_t qdesc0 = sdesc_sw128(smem_u32(s.q[0]), 16, 1024);
    const uint64_t kdesc0 = sdesc_sw128(smem_u32(s.k[0]), 16, 1024);
    const uint64_t vdesc0 = sdesc_sw128(smem_u32(s.v[0]), 16384, 1024);
    constexpr uint64_t kTileDesc = kTileBytes >> 4;
    uint32_t s_cnt = 0, pv_cnt = 0, q_uses = 0;
    uint32_t flags = 0;  // first/last bits of the blocks between P V and S, two per block
    uint64_t cur_q = qdesc0;
    bool ok = true, s_end = false;

    // The block descriptor is read after the K stage fills: the K producer
    // read it (after the walker published it) before filling the stage.
    auto issue_s = [&]() -> bool {
      const uint32_t ks = s_cnt % kStagesK;
      if (!mbar_wait_warp(&s.k_full[ks], (s_cnt / kStagesK) & 1u, wc)) return false;
      const uint32_t info = __shfl_sync(0xffffffffu, s.binfo[s_cnt % kInfoRing].x, 0);
      if (info & kEnd) {
        s_end = true;
        return true;
      }
      if (info & kFirst) {  // first block of a tile: its Q buffer
        const uint32_t qb = q_uses & 1u;
        if (!mbar_wait_warp(&s.q_full[qb], (q_uses >> 1) & 1u, wc)) return false;
        cur_q = qb ? qdesc0 + kTileDesc : qdesc0;
      }
      tc_fence_after();
      const uint32_t sb = s_cnt % kSBufs;
      const uint64_t kd = ks ? kdesc0 + kTileDesc : kdesc0;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
        mma_ss_elect(BSA_TMEM(tmem + sb * 128, 128u, p.err), cur_q + off, kd + off, idesc_s, kk > 0 ? 1u : 0u);
      }
      mma_commit_elect(&s.s_full[sb]);  // also frees K stage ks (== sb)
      if (info & kLast) {  // last block of the tile: its Q buffer is free after this S
        mma_commit_elect(&s.q_empty[q_uses & 1u]);
        ++q_uses;
      }
      const uint32_t sh = 2u * (s_cnt & 7u);
      flags = (flags & ~(3u << sh)) | (((info >> 20) & 3u) << sh);
      ++s_cnt;
      return true;
    };

    while (ok && !s_end && s_cnt < static_cast<uint32_t>(kSBufs)) ok = issue_s();
    uint32_t o_uses = 0;
    while (ok && pv_cnt < s_cnt) {
      const uint32_t fl = (flags >> (2u * (pv_cnt & 7u))) & 3u;
      const bool pv_first = fl & 1u, pv_last = fl & 2u;
      const uint32_t pb = pv_cnt % kSBufs;
      // V and the accumulator (usually long ready) first: the wait for P is
      // the one the tensor pipe idles on, and P V follows it directly
      const uint32_t vs = pv_cnt % kStagesV;
      if (!mbar_wait_warp(&s.v_full[vs], (pv_cnt / kStagesV) & 1u, wc)) { ok = false; break; }
      if (pv_first && o_uses > 0 && !mbar_wait_warp(&s.o_empty, (o_uses - 1) & 1u, wc)) { ok = false; break; }
      if (!mbar_wait_warp(&s.p_full[pb], (pv_cnt / kSBufs) & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      const uint64_t vd = vdesc0 + vs * kTileDesc;
      // part p's P (keys [64p, 64p + 64), words [64p, 64p + 32) of the
      // buffer) into part p's accumulator
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts_elect(BSA_TMEM(tmem + kTmemO + (kk >> 2) * 128, 128u, p.err), BSA_TMEM(tmem + pb * 128 + (kk >> 2) * 64 + (kk & 3) * 8, 8u, p.err),
                     vd + static_cast<uint64_t>(kk * 2048 >> 4), idesc_o, (pv_first && (kk & 3) == 0) ? 0u : 1u);
      mma_commit_elect(&s.v_empty[vs]);  // also: this P V done (vs == pb)
      if (pv_last) {
        mma_commit_elect(&s.o_full);
        ++o_uses;
      }
      ++pv_cnt;
      // S for the block kSBufs ahead reuses this P buffer: issued after this P V.
      if (!s_end) ok = issue_s();
    }
    // Every MMA issued so far completes before tensor memory is released.
    mma_commit_elect(&s.drain);
    uint32_t dummy_abort = 0;
    WaitCtl dw{p.err, &dummy_abort, p.wait_ns};
    (void)mbar_wait(&s.drain, 0, dw);
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue warpgroup
    // One query row per thread: waits for a tile's statistics and its final
    // accumulators, combines the parts' (maximum m_p, sum l_p, O_p) with the
    // weights w_p = 2^(m_p - M), M = max over the parts with l_p > 0:
    // O = sum w_p O_p / L, L = sum w_p l_p; reads O out of tensor memory
    // (then releases it for the next tile's P V) and writes O in bf16 and the
    // logsumexp M + log2 L (natural-log units).
    const int quarter = warp - kEpiWarp0;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t obase = tmem + kTmemO + lane_off;
    griddep_wait();
    bool ok = true;
    for (uint32_t t = 0; ok; ++t) {
      const uint32_t tp = t & 1u;
      if (!mbar_wait_warp(&s.stats_full[tp], (t >> 1) & 1u, wc)) { ok = false; break; }
      const uint32_t row0 = s.trow[tp];
      if (row0 == 0xFFFFFFFFu) break;  // end mark from the softmax warps
      static_assert(kParts == 2, "the epilogue combines two parts");
      const float m0 = s.tmax[tp][0][r], m1 = s.tmax[tp][1][r];
      const float l0 = s.tsum[tp][0][r], l1 = s.tsum[tp][1][r];
      mbar_arrive(&s.stats_empty[tp]);
      const float mrow = fmaxf(l0 > 0.f ? m0 : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
      const float w0 = l0 > 0.f ? ex2_approx(m0 - mrow) : 0.f;
      const float w1 = l1 > 0.f ? ex2_approx(m1 - mrow) : 0.f;
      const float l_row = l0 * w0 + l1 * w1;
      if (!mbar_wait_warp(&s.o_full, t & 1u, wc)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = l_row > 0.f ? 1.f / l_row : 0.f;
      // per-part factors of the output: normalised (bf16 O) or not (a shard's accumulator)
      const float c0 = p.partial ? w0 : w0 * inv_l, c1 = p.partial ? w1 : w1 * inv_l;
      const int64_t orow =
          BSA_RANGE(static_cast<int64_t>(row0) + r, int64_t(0), static_cast<int64_t>(p.B) * p.Hq * p.Sq, p.err);
      if (p.partial) {
        // (a key shard) the unnormalised fp32 accumulator w0 O_0 + w1 O_1 (for
        // the reference maximum M), 16 columns at a time
        float4* dst = reinterpret_cast<float4*>(p.o_acc + orow * D);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t va[16], vb[16];
          tmem_ld16(BSA_TMEM(obase + c * 16, 16u, p.err), va);
          tmem_ld16(BSA_TMEM(obase + 128 + c * 16, 16u, p.err), vb);
          tmem_wait_ld();
          reg_fence16(va);
          reg_fence16(vb);
          float o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = fmaf(__uint_as_float(va[j]), c0, __uint_as_float(vb[j]) * c1);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[c * 4 + e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
        }
        // (every load of this tile's O has completed by the last wait)
        tc_fence_before();
        mbar_arrive(&s.o_empty);
      } else {
        // O / l in bf16 through this warp's staging buffer and a TMA store of
        // [32 rows, 64 columns] per half: the stores are coalesced and off the
        // load/store unit.  The second half waits in registers while the first
        // one's store reads the buffer, and O is released to the next tile's
        // P V as soon as both halves are out of tensor memory.
        uint8_t* stage = s.ostage[quarter];
        const int32_t grow = static_cast<int32_t>(row0) + quarter * 32;  // global row of lane 0
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t va[16], vb[16];
            tmem_ld16(BSA_TMEM(obase + h * 64 + c * 16, 16u, p.err), va);
            tmem_ld16(BSA_TMEM(obase + 128 + h * 64 + c * 16, 16u, p.err), vb);
            tmem_wait_ld();
            reg_fence16(va);
            reg_fence16(vb);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              pk[c * 8 + j] = pack_bf16x2(fmaf(__uint_as_float(va[2 * j]), c0, __uint_as_float(vb[2 * j]) * c1),
                                          fmaf(__uint_as_float(va[2 * j + 1]), c0, __uint_as_float(vb[2 * j + 1]) * c1));
          }
          if (h == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(&s.o_empty);
          }
          // the previous store out of this buffer has finished reading it
          if (lane == 0) tma_store_wait_read();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((j ^ (lane & 7)) * 16)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tm_o, stage, h * 64, grow);
            tma_store_commit();
          }
        }
      }
      if (p.partial) {
        p.m_out[orow] = l_row > 0.f ? mrow * 0.69314718055994530942f : -INFINITY;
        p.l_out[orow] = l_row;
      } else {
        p.lse[orow] = l_row > 0.f ? (mrow + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
      }
    }
    // the staging buffers stay valid until every TMA store has read them
    if (lane == 0) tma_store_wait_all();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax (kParts warpgroups)
    // Warpgroup `part` takes score columns [kCols*part, kCols*part + kCols)
    // of every row with a running maximum and sum of its own (no exchange
    // between the parts); its P V goes to its own O accumulator, and the
    // epilogue combines the parts' (maximum, sum, O).
    const int part = (warp - 4) >> 2;
    const int quarter = (warp - 4) & 3;
    const int r = quarter * 32 + lane;  // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(part) * kCols;  // first score column of this part
    const uint32_t ocol0 = kTmemO + static_cast<uint32_t>(part) * 128;  // this part's O accumulator
    const float scale_log2 = p.scale_log2;
    uint32_t n = 0;
    bool ok = true;
    float m = -INFINITY, l = 0.f;  // this part's running maximum (log2 units) and row sum
    int64_t lo = 0, hi = 0;
    uint32_t exec = 0;
    uint32_t tiles = 0;
    // Hands a finished tile's row statistics to the epilogue warpgroup.
    auto finish_tile = [&](uint32_t row) -> bool {
      const uint32_t tp = tiles & 1u;
      if (tiles >= 2 && !mbar_wait_warp(&s.stats_empty[tp], ((tiles >> 1) - 1) & 1u, wc)) return false;
      s.tmax[tp][part][r] = m;
      s.tsum[tp][part][r] = l;
      if (r == 0 && part == 0) s.trow[tp] = row;
      mbar_arrive(&s.stats_full[tp]);
      ++tiles;
      return true;
    };
    // block descriptors from the walker (published long before their
    // scores); the next one's barrier is tested while a block is computed
    if (!mbar_wait_warp(&s.info_full[0], 0u, wc)) ok = false;
    while (ok) {
      const uint32_t slot = n % kInfoRing;
      const uint4 bi = s.binfo[slot];
      if (bi.x & kEnd) break;
      const uint32_t sb = n % kSBufs;
      // A dense mask's visibility bits come from memory: they are loaded
      // before the wait for the scores (they do not depend on them).  The
      // other instantiations wait first (measured faster for them).
      if constexpr (!kBits) {
        if (!mbar_wait_warp(&s.s_full[sb], (n / kSBufs) & 1u, wc)) { ok = false; break; }
      }
      const int32_t col = static_cast<int32_t>(bi.x & 0xFFFFu);
      const int32_t label = static_cast<int32_t>((bi.x >> 16) & 3u);
      const bool first = bi.x & kFirst, last = bi.x & kLast;
      if (first) {
        m = -INFINITY;
        l = 0.f;
        exec = 0;
        if (kX && p.n_sinks > 0) {
          // the sinks open the running maximum of both parts and the sum of part 0
          const int32_t hq = static_cast<int32_t>((static_cast<int64_t>(bi.w) / p.Sq) % p.Hq);
          const float* z = p.sinks + (p.sinks_kv ? (hq / (p.Hq / p.Hkv)) * p.n_sinks : 0);
          for (int j = 0; j < p.n_sinks; ++j) m = fmaxf(m, z[j] * 1.4426950408889634f);
          if (part == 0)
            for (int j = 0; j < p.n_sinks; ++j) l += ex2_approx(z[j] * 1.4426950408889634f - m);
        }
        // q_sequence is consecutive within a query block: row r has q_sequence[128 i] + r
        if (p.mi.kind != BSA_MASK_DENSE)
          key_interval(p.mi.kind, p.mi.left, p.mi.right, p.mi.chunk, static_cast<int64_t>(static_cast<int32_t>(bi.z)) + r,
                       lo, hi);
      }
      uint64_t mbits = ~0ull;  // visibility of this part's columns (label 1 only)
      if (label == 1) {
        if constexpr (kBits) {
          // this part's 64 visibility bits of the stacked block's row
          static_assert(kCols == 64, "one 64-bit word of mask bits per part");
          mbits = __ldg(reinterpret_cast<const unsigned long long*>(p.mi.partial_bits +
                                                                     (static_cast<int64_t>(bi.y) * 128 + r) * 4) +
                        part);
        } else if (p.mi.kind == BSA_MASK_DENSE) {
          const uint4* mrow = reinterpret_cast<const uint4*>(
              p.mi.partial + (static_cast<int64_t>(bi.y) * 128 + r) * 128 + col0);
          mbits = 0;
#pragma unroll
          for (int v = 0; v < kCols / 16; ++v) {
            const uint4 mw = __ldg(mrow + v);
            const uint32_t wv[4] = {mw.x, mw.y, mw.z, mw.w};
#pragma unroll
            for (int e = 0; e < 16; ++e)
              mbits |= static_cast<uint64_t>(((wv[e >> 2] >> ((e & 3) * 8)) & 0xFFu) != 0u ? 1u : 0u) << (v * 16 + e);
          }
        } else {
          // visible columns of this row form [a, b] inside this part
          const int64_t k0 = static_cast<int64_t>(col) * 128 + col0;
          const int64_t a64 = lo - k0, b64 = hi - k0;
          const int32_t a = a64 < 0 ? 0 : (a64 > kCols ? kCols : static_cast<int32_t>(a64));
          const int32_t b = b64 > kCols - 1 ? kCols - 1 : (b64 < -1 ? -1 : static_cast<int32_t>(b64));
          if (b < a) {
            mbits = 0;
          } else {
            const uint64_t upto = b >= 63 ? ~0ull : ((1ull << (b + 1)) - 1ull);
            mbits = upto & ~((1ull << a) - 1ull);
          }
        }
      }
      if constexpr (kBits) {
        if (!mbar_wait_warp(&s.s_full[sb], (n / kSBufs) & 1u, wc)) { ok = false; break; }
      }
      // Released only now: the scores being ready means the K producer and
      // the MMA warp have read this descriptor too.
      if (lane == 0) mbar_arrive(&s.info_empty[slot]);
      // no branch joins while the loaded registers are in flight
      tc_fence_after();
      uint32_t xu[kCols];
#pragma unroll
      for (int c = 0; c < kCols; c += 32) tmem_ld32(BSA_TMEM(tmem + sb * 128 + col0 + c + lane_off, 32u, p.err), xu + c);
      tmem_wait_ld();
      reg_fence<kCols>(xu);
      const uint32_t nslot = (n + 1) % kInfoRing;
      const bool next_ready = mbar_test_wait(smem_u32(&s.info_full[nslot]), ((n + 1) / kInfoRing) & 1u);
      if (label == 1) {
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (!((mbits >> c) & 1ull)) xu[c] = 0xFF800000u;  // -inf
      }
      // partial row max over this part: four chains of three-input maxima
      // (columns 0-3 start the chains, 4 .. kCols-5 in steps of eight, the
      // last four close two of them)
      static_assert(kCols % 8 == 0, "the max chains take columns eight at a time");
      float m0 = __uint_as_float(xu[0]), m1 = __uint_as_float(xu[1]);
      float m2 = __uint_as_float(xu[2]), m3 = __uint_as_float(xu[3]);
#pragma unroll
      for (int c = 4; c + 8 <= kCols - 4; c += 8) {
        m0 = fmax3(m0, __uint_as_float(xu[c + 0]), __uint_as_float(xu[c + 1]));
        m1 = fmax3(m1, __uint_as_float(xu[c + 2]), __uint_as_float(xu[c + 3]));
        m2 = fmax3(m2, __uint_as_float(xu[c + 4]), __uint_as_float(xu[c + 5]));
        m3 = fmax3(m3, __uint_as_float(xu[c + 6]), __uint_as_float(xu[c + 7]));
      }
      m0 = fmax3(m0, __uint_as_float(xu[kCols - 4]), __uint_as_float(xu[kCols - 3]));
      m1 = fmax3(m1, __uint_as_float(xu[kCols - 2]), __uint_as_float(xu[kCols - 1]));
      const float pm = fmax3(fmaxf(m0, m1), m2, m3);
      const float mx = pm;
      // tanh is increasing: the capped maximum is the cap of the maximum
      const float m_blk = (!kX || p.cap_scale == 0.f) ? mx * scale_log2
                          : (mx == -INFINITY ? -INFINITY : p.cap_log2 * tanh_fast(mx * p.cap_scale));
      const float m_cand = fmaxf(m, m_blk);
      const bool switch_ref = m_cand > m + kRescaleThreshold;
      const bool warp_switch = __any_sync(0xffffffffu, switch_ref);
      float alpha = 1.f;
      if (warp_switch) {
        alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - m_cand);
        m = m_cand;
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      // p = exp2(s * scale_log2 - m): packed FMA, four packed partial sums
      const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_use, -m_use);
      uint64_t acc[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[a] = f2_pack(0.f, 0.f);
      uint32_t pk[kCols / 2];
      if (!kX || p.cap_scale == 0.f) {
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) {
          const uint64_t e2 = f2_fma(f2_pack(__uint_as_float(xu[2 * c]), __uint_as_float(xu[2 * c + 1])), sc2, nm2);
          float e0, e1;
          f2_unpack(e2, e0, e1);
          const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
          acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
      } else {
        // soft cap: exp2(cap_log2 * tanh(s * cap_scale) - m); masked (-inf) scores stay at 0
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) {
          const float x0 = __uint_as_float(xu[2 * c]), x1 = __uint_as_float(xu[2 * c + 1]);
          float e0 = fmaf(tanh_fast(x0 * p.cap_scale), p.cap_log2, -m_use);
          float e1 = fmaf(tanh_fast(x1 * p.cap_scale), p.cap_log2, -m_use);
          e0 = x0 == -INFINITY ? -INFINITY : e0;
          e1 = x1 == -INFINITY ? -INFINITY : e1;
          const float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
          acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
      }
      const uint64_t acc01 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
      float rs0, rs1;
      f2_unpack(acc01, rs0, rs1);
      l = l * alpha + (rs0 + rs1);
      // P (bf16 pairs) over the first half of this part's own score columns:
      // words [part*kCols, part*kCols + kCols/2) of the buffer.
#pragma unroll
      for (int c = 0; c < kCols / 2; c += 16)
        tmem_st16(BSA_TMEM(tmem + sb * 128 + static_cast<uint32_t>(part) * kCols + c + lane_off, 16u, p.err), pk + c);
      // O holds earlier blocks' sum only after the first block; rescale this
      // part's accumulator (after the previous P V has landed) when its max moved.
      if (warp_switch && exec > 0) {
        const uint32_t prev = n - 1;
        if (!mbar_wait_warp(&s.v_empty[prev % kStagesV], (prev / kStagesV) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t ov[16];
          const uint32_t oa = tmem + ocol0 + c + lane_off;
          tmem_ld16(BSA_TMEM(oa, 16u, p.err), ov);
          tmem_wait_ld();
          reg_fence16(ov);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const uint64_t o2 = f2_mul(f2_pack(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])), al2);
            float a0, a1;
            f2_unpack(o2, a0, a1);
            ov[e] = __float_as_uint(a0);
            ov[e + 1] = __float_as_uint(a1);
          }
          tmem_st16(BSA_TMEM(oa, 16u, p.err), ov);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full[sb]);
      ++n;
      ++exec;
      if (last && !finish_tile(bi.w)) { ok = false; break; }
      if (!__all_sync(0xffffffffu, next_ready) && !mbar_wait_warp(&s.info_full[nslot], (n / kInfoRing) & 1u, wc)) {
        ok = false;
        break;
      }
    }
    // end mark for the epilogue warpgroup
    if (ok) {
      const uint32_t tp = tiles & 1u;
      if (tiles < 2 || mbar_wait_warp(&s.stats_empty[tp], ((tiles >> 1) - 1) & 1u, wc)) {
        if (r == 0 && part == 0) s.trow[tp] = 0xFFFFFFFFu;
        mbar_arrive(&s.stats_full[tp]);
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

// One forward launch: the whole key axis (O, LSE) or one key shard
// (accumulator, maximum, normaliser).
struct FwdCall {
  const void *q, *k, *v;
  int32_t B, Hq, Hkv;
  int64_t Sq, Skv;  // Skv: keys in k / v (the shard's length for a shard)
  __nv_bfloat16* o;
  float* lse;
  float *o_acc, *m, *l;
  int32_t kv_lo, kv_hi, partial;
  float cap;
  const float* sinks;
  int32_t n_sinks, sinks_kv;
};

template <int D>
bsa_status launch_fwd(const FwdCall& c, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  const uint64_t q_rows = static_cast<uint64_t>(c.B) * c.Hq * c.Sq;
  const uint64_t kv_rows = static_cast<uint64_t>(c.B) * c.Hkv * c.Skv;
  if (!make_tmap_bf16_2d(&tq, c.q, q_rows, D, D * 2, 128, 64) ||
      !make_tmap_bf16_2d(&tk, c.k, kv_rows, D, D * 2, 128, 64) ||
      !make_tmap_bf16_2d(&tv, c.v, kv_rows, D, D * 2, 128, 64))
    return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected a Q/K/V description");
  // the bf16 output, stored in [32 rows, 64 columns] boxes (a key shard
  // writes fp32 with plain stores: the Q map stands in, unused)
  if (c.partial) to = tq;
  else if (!make_tmap_bf16_2d(&to, c.o, q_rows, D, D * 2, 32, 64))
    return fail(BSA_ERR_CUDA, "cuTensorMapEncodeTiled rejected the output description");
  FwdParams p{};
  p.B = c.B;
  p.Hq = c.Hq;
  p.Hkv = c.Hkv;
  p.Sq = c.Sq;
  p.Skv = c.Skv;
  p.nQ = static_cast<int32_t>(c.Sq / 128);
  p.nK = static_cast<int32_t>(c.Skv / 128);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o = c.o;
  p.lse = c.lse;
  p.o_acc = c.o_acc;
  p.m_out = c.m;
  p.l_out = c.l;
  p.kv_lo = c.kv_lo;
  p.kv_hi = c.kv_hi;
  p.partial = c.partial;
  if (c.cap > 0.f) {
    p.cap_scale = scale / c.cap;
    p.cap_log2 = c.cap * 1.4426950408889634f;
  }
  p.sinks = c.sinks;
  p.n_sinks = c.n_sinks;
  p.sinks_kv = c.sinks_kv;
  p.mi = mask_info_dev(info);
  p.n_tiles = c.B * c.Hq * p.nQ;
  p.err = device_error_word();
  p.wait_ns = wait_limit_ns();
  if (!p.err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  const bool xform = p.cap_scale != 0.f || p.n_sinks > 0;
  // instantiation: the logit transforms, the dense mask read as bits, or neither
  const int variant = xform ? 2 : (info->kind == BSA_MASK_DENSE ? 1 : 0);
  auto kern = variant == 2 ? fwd_kernel<D, true, false>
                           : (variant == 1 ? fwd_kernel<D, false, true> : fwd_kernel<D, false, false>);
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  {
    bsa_status st = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem, "set forward smem size");
    if (st != BSA_OK) return st;
  }
  const int grid = std::min(p.n_tiles, num_sms());
  bsa_status st = tile_schedule(info, c.B, c.Hq, 1, 1, grid, stream, &p.sched, &p.sched_stride);
  if (st != BSA_OK) return st;
  cudaError_t e = launch_kernel(kern, dim3(grid), dim3(kThreads), smem, stream, tq, tk, tv, to, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return BSA_OK;
}

bsa_status dispatch(const FwdCall& c, int D, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  if (D == 128) return launch_fwd<128>(c, info, scale, stream);
  return launch_fwd<64>(c, info, scale, stream);
}

}  // namespace

bsa_status fwd_launch(const bsa_fwd_args* a, const bsa_mask_info* info, float scale, cudaStream_t stream) {
  FwdCall c{};
  c.q = a->q;
  c.k = a->k;
  c.v = a->v;
  c.B = a->B;
  c.Hq = a->Hq;
  c.Hkv = a->Hkv;
  c.Sq = a->S_q;
  c.Skv = a->S_kv;
  c.o = static_cast<__nv_bfloat16*>(a->o);
  c.lse = a->lse;
  c.kv_lo = 0;
  c.kv_hi = info->cols;
  c.partial = 0;
  c.cap = a->logits_soft_cap;
  c.sinks = a->num_sinks > 0 ? a->sinks : nullptr;
  c.n_sinks = a->num_sinks > 0 ? a->num_sinks : 0;
  c.sinks_kv = a->sinks_per_kv_head ? 1 : 0;
  return dispatch(c, a->D, info, scale, stream);
}

bsa_status fwd_partial_launch(const bsa_fwd_partial_args* a, const bsa_mask_info* info, float scale,
                              cudaStream_t stream) {
  FwdCall c{};
  c.q = a->q;
  c.k = a->k;
  c.v = a->v;
  c.B = a->B;
  c.Hq = a->Hq;
  c.Hkv = a->Hkv;
  c.Sq = a->S_q;
  c.Skv = a->S_kv_shard;
  c.o_acc = a->o_acc;
  c.m = a->m;
  c.l = a->l;
  c.kv_lo = static_cast<int32_t>(a->kv_offset / 128);
  c.kv_hi = static_cast<int32_t>((a->kv_offset + a->S_kv_shard) / 128);
  c.partial = 1;
  c.cap = a->logits_soft_cap;
  return dispatch(c, a->D, info, scale, stream);
}

}  // namespace bsa
