// C ABI entry points: argument checking, error plumbing, dispatch to the
// kernel launchers.  Nothing here computes attention or masks.
#include <cmath>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace bsa {

static thread_local std::string g_last_error;
static uint64_t g_wait_limit_ns = 2000000000ull;
static std::mutex g_err_mu;
static uint32_t* g_err_word[64] = {nullptr};

void set_last_error(const std::string& msg) { g_last_error = msg; }

bsa_status fail(bsa_status s, const std::string& msg) {
  set_last_error(msg);
  return s;
}

bsa_status cuda_fail(cudaError_t e, const char* what) {
  set_last_error(std::string(what) + ": " + cudaGetErrorString(e));
  return e == cudaErrorMemoryAllocation ? BSA_ERR_OOM : BSA_ERR_CUDA;
}

// The library's error word of the current device if a launch there has
// already allocated it (a reader need not allocate: no word, no error).
uint32_t* device_error_word_if_set() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  return g_err_word[dev];
}

uint32_t* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_word[dev]) {
    uint32_t* p = nullptr;
    if (cudaMalloc(&p, sizeof(uint32_t)) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, sizeof(uint32_t)) != cudaSuccess) return nullptr;
    g_err_word[dev] = p;
  }
  return g_err_word[dev];
}

uint64_t wait_limit_ns() { return g_wait_limit_ns; }

namespace {
std::mutex g_pool_mu;
cudaMemPool_t g_pools[64] = {};
}  // namespace

bsa_status pool_alloc(void** p, size_t bytes, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(BSA_ERR_UNSUPPORTED, "device index above 63");
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pools[dev]) {
      cudaMemPoolProps props{};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&g_pools[dev], &props);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
      uint64_t keep = UINT64_MAX;  // keep freed memory for the next call
      cudaMemPoolSetAttribute(g_pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
    }
    pool = g_pools[dev];
  }
  e = cudaMallocFromPoolAsync(p, bytes, pool, stream);
  if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? fail(BSA_ERR_OOM, "workspace allocation failed")
                                                              : cuda_fail(e, "cudaMallocFromPoolAsync");
  return BSA_OK;
}

bsa_status pool_free(void* p, cudaStream_t stream) {
  cudaError_t e = cudaFreeAsync(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync");
  return BSA_OK;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("BSA_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

bsa_status ensure_smem_attr(const void* func, size_t smem, const char* what) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({dev, func})) return BSA_OK;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, what);
  done.insert({dev, func});
  return BSA_OK;
}

int num_sms() {
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = n > 0 ? n : 1;
  }
  return sms[dev];
}

// One CTA waits on an mbarrier that nothing arrives at; the bounded wait
// must run out, record DEV_ERR_TIMEOUT and return.
__global__ void debug_wait_timeout_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtl w{err, &abort_flag, limit_ns};
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, w);
}

// Out-of-range indices passed through the range checks (and used for
// nothing else): the range-checked build records DEV_ERR_DEBUG with the
// line of the first; the release build compiles the checks away.
__global__ void debug_selfcheck_kernel(uint32_t* err, uint32_t col, int64_t row) {
  (void)BSA_TMEM(col, 32u, err);
  (void)BSA_RANGE(row, int64_t(0), int64_t(16), err);
}

bsa_status debug_selfcheck_launch(cudaStream_t stream) {
  uint32_t* err = device_error_word();
  if (!err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  debug_selfcheck_kernel<<<1, 1, 0, stream>>>(err, 500u, int64_t(-1));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "debug_selfcheck launch");
  return BSA_OK;
}

bsa_status debug_wait_timeout_launch(cudaStream_t stream) {
  uint32_t* err = device_error_word();
  if (!err) return fail(BSA_ERR_CUDA, "could not allocate the device error word");
  debug_wait_timeout_kernel<<<1, 32, 0, stream>>>(err, g_wait_limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "debug_wait_timeout launch");
  return BSA_OK;
}

}  // namespace bsa

using namespace bsa;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bsa_status check_shapes(int32_t B, int32_t Hq, int32_t Hkv, int64_t Sq, int64_t Skv, int32_t D) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0) return fail(BSA_ERR_INVALID_ARG, "B, Hq and Hkv must be positive");
  if (Hq % Hkv != 0) return fail(BSA_ERR_INVALID_ARG, "Hq must be a multiple of Hkv");
  if (Sq <= 0 || Skv <= 0) return fail(BSA_ERR_INVALID_ARG, "sequence lengths must be positive");
  if (Sq % kBlock || Skv % kBlock) return fail(BSA_ERR_INVALID_ARG, "sequence lengths must be multiples of 128");
  if (D != 64 && D != 128) return fail(BSA_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if ((int64_t)B * Hq * Sq > (int64_t)INT32_MAX || (int64_t)B * Hkv * Skv > (int64_t)INT32_MAX)
    return fail(BSA_ERR_UNSUPPORTED, "B*H*S must fit in int32");
  return BSA_OK;
}

bsa_status check_info(const bsa_mask_info* info, int32_t orientation, int64_t Sq, int64_t Skv, int32_t Hq,
                      const char* which) {
  if (!info) return fail(BSA_ERR_INVALID_ARG, std::string(which) + " MaskInfo is null");
  if (info->orientation != orientation)
    return fail(BSA_ERR_INVALID_ARG, std::string(which) + " MaskInfo has the wrong orientation");
  if (info->q_len != Sq || info->kv_len != Skv)
    return fail(BSA_ERR_INVALID_ARG, std::string(which) + " MaskInfo was compiled for other sequence lengths");
  if (info->heads != 1 && info->heads != Hq)
    return fail(BSA_ERR_INVALID_ARG, std::string(which) + " MaskInfo must have 1 or Hq mask heads");
  return BSA_OK;
}

float resolve_scale(float s, int32_t D) { return std::isnan(s) ? 1.0f / std::sqrt((float)D) : s; }

bsa_status check_transforms(float cap, const float* sinks, int32_t num_sinks) {
  if (!(cap >= 0.f) || std::isinf(cap)) return fail(BSA_ERR_INVALID_ARG, "logits_soft_cap must be finite and >= 0");
  if (num_sinks < 0 || num_sinks > 64) return fail(BSA_ERR_UNSUPPORTED, "num_sinks must be in 0..64");
  if (num_sinks > 0 && !sinks) return fail(BSA_ERR_INVALID_ARG, "sinks is null");
  if (num_sinks > 0 && (reinterpret_cast<uintptr_t>(sinks) & 3u))
    return fail(BSA_ERR_INVALID_ARG, "sinks must be 4-byte aligned");
  return BSA_OK;
}

}  // namespace

bsa_status bsa::check_bwd_args(const bsa_bwd_args* a, bool need_dsum) {
  if (!a) return fail(BSA_ERR_INVALID_ARG, "args is null");
  bsa_status s = check_shapes(a->B, a->Hq, a->Hkv, a->S_q, a->S_kv, a->D);
  if (s != BSA_OK) return s;
  const void* ptrs[] = {a->q, a->k, a->v, a->o, a->lse, a->do_, a->dq, a->dk, a->dv, need_dsum ? a->dsum : a->q};
  for (const void* p : ptrs)
    if (!p) return fail(BSA_ERR_INVALID_ARG, "a tensor pointer is null");
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(BSA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  s = check_transforms(a->logits_soft_cap, a->sinks, a->num_sinks);
  if (s != BSA_OK) return s;
  if (a->dsinks && (reinterpret_cast<uintptr_t>(a->dsinks) & 3u))
    return fail(BSA_ERR_INVALID_ARG, "dsinks must be 4-byte aligned");
  return BSA_OK;
}

namespace {
bsa_status check_bwd(const bsa_bwd_args* a) { return check_bwd_args(a, true); }
}  // namespace

extern "C" {

const char* bsa_version(void) { return "0.1.0"; }

const char* bsa_status_string(bsa_status s) {
  switch (s) {
    case BSA_OK: return "ok";
    case BSA_ERR_INVALID_ARG: return "invalid argument";
    case BSA_ERR_UNSUPPORTED: return "unsupported";
    case BSA_ERR_CUDA: return "cuda error";
    case BSA_ERR_OOM: return "out of memory";
    case BSA_ERR_TIMEOUT: return "device wait timed out";
    case BSA_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

const char* bsa_last_error(void) { return g_last_error.c_str(); }

bsa_status bsa_set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns = ns ? ns : 2000000000ull;
  return BSA_OK;
}

bsa_status bsa_debug_wait_timeout(bsa_stream stream) {
  return debug_wait_timeout_launch(static_cast<cudaStream_t>(stream));
}

bsa_status bsa_debug_selfcheck(bsa_stream stream) {
  return debug_selfcheck_launch(static_cast<cudaStream_t>(stream));
}

bsa_status bsa_debug_tile_schedule(const int32_t* row_len, const int32_t* row_order, int32_t rows, int32_t heads,
                                   int32_t n_b, int32_t n_g, int32_t group, int32_t splits, int32_t grid,
                                   int32_t* out, int32_t cap, int32_t* stride) {
  if (!row_len || !row_order || !out || !stride) return fail(BSA_ERR_INVALID_ARG, "null pointer");
  std::vector<int4> flat;
  int32_t st = 0;
  const bsa_status s = schedule_lists(row_len, row_order, rows, heads, n_b, n_g, group, splits, grid, &flat, &st);
  if (s != BSA_OK) return s;
  *stride = st;
  if (cap < st) return fail(BSA_ERR_INVALID_ARG, "cap is below the schedule's stride");
  for (int32_t c = 0; c < grid; ++c)
    for (int32_t k = 0; k < cap; ++k) {
      const int4 e = k < st ? flat[static_cast<size_t>(c) * st + k] : make_int4(0, -1, 0, 0);
      int32_t* o = out + (static_cast<size_t>(c) * cap + k) * 4;
      o[0] = e.x;
      o[1] = e.y;
      o[2] = e.z;
      o[3] = e.w;
    }
  return BSA_OK;
}

bsa_status bsa_get_device_error(bsa_stream stream, uint32_t* word) {
  if (!word) return fail(BSA_ERR_INVALID_ARG, "word is null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  // both words of the current device: the one of the ordinary launches and
  // the one of the allocation-free backward; neither is allocated here
  uint32_t h = 0;
  uint32_t* words[2] = {device_error_word_if_set(), noalloc_error_word_if_set()};
  for (uint32_t* d : words) {
    if (!d) continue;
    uint32_t x = 0;
    e = cudaMemcpy(&x, d, sizeof(x), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    e = cudaMemset(d, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    h |= x;
  }
  *word = h;
  if (h & DEV_ERR_TIMEOUT) return fail(BSA_ERR_TIMEOUT, "a device-side wait ran out");
  if (h) return fail(BSA_ERR_DEVICE, "a kernel reported a device-side error");
  return BSA_OK;
}

bsa_status bsa_mask_compile(const bsa_mask_spec* spec, const bsa_mask_opts* opts, bsa_stream stream,
                            bsa_mask_info** out) {
  if (!spec || !opts || !out) return fail(BSA_ERR_INVALID_ARG, "spec, opts and out must be non-null");
  if (opts->block_q != kBlock || opts->block_kv != kBlock)
    return fail(BSA_ERR_UNSUPPORTED, "only 128 x 128 blocks are supported");
  if (opts->orientation != BSA_ORIENT_FWD && opts->orientation != BSA_ORIENT_DKV)
    return fail(BSA_ERR_INVALID_ARG, "unknown orientation");
  if (opts->shrink != 0 && opts->shrink != 1) return fail(BSA_ERR_INVALID_ARG, "shrink must be 0 or 1");
  if (spec->q_len <= 0 || spec->kv_len <= 0 || spec->q_len % kBlock || spec->kv_len % kBlock)
    return fail(BSA_ERR_INVALID_ARG, "mask lengths must be positive multiples of 128");
  if (spec->q_len > (1 << 24) || spec->kv_len > (1 << 24))
    return fail(BSA_ERR_UNSUPPORTED, "mask lengths above 2^24 are not supported");
  if (spec->mask_heads <= 0) return fail(BSA_ERR_INVALID_ARG, "mask_heads must be positive");
  switch (spec->kind) {
    case BSA_MASK_DENSE:
      if (!spec->dense) return fail(BSA_ERR_INVALID_ARG, "dense mask pointer is null");
      if (!aligned16(spec->dense)) return fail(BSA_ERR_INVALID_ARG, "dense mask must be 16-byte aligned");
      break;
    case BSA_MASK_CAUSAL:
    case BSA_MASK_FULL:
      break;
    case BSA_MASK_LOCAL:
      if (spec->local_left < -1 || spec->local_right < -1)
        return fail(BSA_ERR_INVALID_ARG, "local windows must be >= 0 or -1 (unbounded)");
      break;
    case BSA_MASK_CHUNKED_CAUSAL:
      if (spec->chunk <= 0) return fail(BSA_ERR_INVALID_ARG, "chunk must be positive");
      break;
    default:
      return fail(BSA_ERR_INVALID_ARG, "unknown mask kind");
  }
  if (spec->kind != BSA_MASK_DENSE && spec->q_len != spec->kv_len)
    return fail(BSA_ERR_UNSUPPORTED, "computable masks need q_len == kv_len");
  return mask_compile_impl(spec, opts, static_cast<cudaStream_t>(stream), out);
}

bsa_status bsa_mask_info_view(const bsa_mask_info* info, bsa_mask_info_desc* out) {
  if (!info || !out) return fail(BSA_ERR_INVALID_ARG, "info and out must be non-null");
  std::memset(out, 0, sizeof(*out));
  out->block_mask = info->block_mask;
  out->data_next = info->data_next;
  out->data_next_bytes = info->data_next_bytes;
  out->mask_next = info->mask_next;
  out->mask_next_bytes = info->mask_next ? info->mask_next_bytes : 0;
  out->partial_mask_blocks = info->partial;
  out->q_sequence = info->q_sequence;
  out->heads = info->heads;
  out->rows = info->rows;
  out->width = info->width;
  out->cols = info->cols;
  out->num_partial = info->num_partial;
  out->n_empty = info->n_empty;
  out->n_partial = info->n_partial;
  out->n_full = info->n_full;
  out->kind = info->kind;
  out->orientation = info->orientation;
  out->shrink = info->shrink;
  out->q_len = info->q_len;
  out->kv_len = info->kv_len;
  out->row_len = info->row_len;
  out->row_order = info->row_order;
  return BSA_OK;
}

bsa_status bsa_mask_info_destroy(bsa_mask_info* info) {
  if (!info) return BSA_OK;
  // no launch may still read the arrays; they go back to the library's
  // stream-ordered pool they came from
  cudaDeviceSynchronize();
  void* ptrs[] = {info->block_mask, info->data_next, info->mask_next, info->partial,
                  info->partial_bits, info->q_sequence, info->row_len, info->row_order};
  for (void* p : ptrs)
    if (p) pool_free(p, nullptr);
  for (auto& sc : info->schedules) {
    if (sc.dev) pool_free(sc.dev, nullptr);
    if (sc.ready) cudaEventDestroy(sc.ready);
  }
  delete info;
  return BSA_OK;
}

bsa_status bsa_fwd(const bsa_fwd_args* a, const bsa_mask_info* info, bsa_stream stream) {
  if (!a) return fail(BSA_ERR_INVALID_ARG, "args is null");
  bsa_status s = check_shapes(a->B, a->Hq, a->Hkv, a->S_q, a->S_kv, a->D);
  if (s != BSA_OK) return s;
  if (!a->q || !a->k || !a->v || !a->o || !a->lse) return fail(BSA_ERR_INVALID_ARG, "a tensor pointer is null");
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o) || !aligned16(a->lse))
    return fail(BSA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  s = check_transforms(a->logits_soft_cap, a->sinks, a->num_sinks);
  if (s != BSA_OK) return s;
  s = check_info(info, BSA_ORIENT_FWD, a->S_q, a->S_kv, a->Hq, "forward");
  if (s != BSA_OK) return s;
  return fwd_launch(a, info, resolve_scale(a->softmax_scale, a->D), static_cast<cudaStream_t>(stream));
}

bsa_status bsa_fwd_partial(const bsa_fwd_partial_args* a, const bsa_mask_info* info, bsa_stream stream) {
  if (!a) return fail(BSA_ERR_INVALID_ARG, "args is null");
  bsa_status s = check_shapes(a->B, a->Hq, a->Hkv, a->S_q, a->S_kv_shard, a->D);
  if (s != BSA_OK) return s;
  if (!a->q || !a->k || !a->v || !a->o_acc || !a->m || !a->l)
    return fail(BSA_ERR_INVALID_ARG, "a tensor pointer is null");
  if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o_acc) || !aligned16(a->m) ||
      !aligned16(a->l))
    return fail(BSA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!info) return fail(BSA_ERR_INVALID_ARG, "forward MaskInfo is null");
  if (a->kv_offset < 0 || a->kv_offset % kBlock)
    return fail(BSA_ERR_INVALID_ARG, "kv_offset must be a non-negative multiple of 128");
  s = check_transforms(a->logits_soft_cap, nullptr, 0);
  if (s != BSA_OK) return s;
  if (a->kv_offset + a->S_kv_shard > info->kv_len)
    return fail(BSA_ERR_INVALID_ARG, "the shard runs past the MaskInfo's key axis");
  s = check_info(info, BSA_ORIENT_FWD, a->S_q, info->kv_len, a->Hq, "forward");
  if (s != BSA_OK) return s;
  return fwd_partial_launch(a, info, resolve_scale(a->softmax_scale, a->D), static_cast<cudaStream_t>(stream));
}

bsa_status bsa_fwd_merge(const bsa_merge_args* a, bsa_stream stream) {
  if (!a) return fail(BSA_ERR_INVALID_ARG, "args is null");
  if (a->n_shards < 1) return fail(BSA_ERR_INVALID_ARG, "n_shards must be at least 1");
  if (a->rows <= 0) return fail(BSA_ERR_INVALID_ARG, "rows must be positive");
  if (a->D != 64 && a->D != 128) return fail(BSA_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (static_cast<int64_t>(a->n_shards) * a->rows * a->D > (int64_t(1) << 40))
    return fail(BSA_ERR_UNSUPPORTED, "merge too large");
  if (!a->o_acc || !a->m || !a->l || !a->o || !a->lse) return fail(BSA_ERR_INVALID_ARG, "a tensor pointer is null");
  if (!aligned16(a->o_acc) || !aligned16(a->o))
    return fail(BSA_ERR_INVALID_ARG, "o_acc and o must be 16-byte aligned");
  return merge_launch(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_bwd_rowsum(const bsa_bwd_args* a, bsa_stream stream) {
  bsa_status s = check_bwd(a);
  if (s != BSA_OK) return s;
  return rowsum_launch(a, static_cast<cudaStream_t>(stream));
}

bsa_status bsa_bwd_dkv(const bsa_bwd_args* a, const bsa_mask_info* dkv_info, bsa_stream stream) {
  bsa_status s = check_bwd(a);
  if (s != BSA_OK) return s;
  s = check_info(dkv_info, BSA_ORIENT_DKV, a->S_q, a->S_kv, a->Hq, "dkv");
  if (s != BSA_OK) return s;
  return dkv_launch(a, dkv_info, resolve_scale(a->softmax_scale, a->D), static_cast<cudaStream_t>(stream));
}

bsa_status bsa_bwd_dq(const bsa_bwd_args* a, const bsa_mask_info* fwd_info, bsa_stream stream) {
  bsa_status s = check_bwd(a);
  if (s != BSA_OK) return s;
  s = check_info(fwd_info, BSA_ORIENT_FWD, a->S_q, a->S_kv, a->Hq, "dq");
  if (s != BSA_OK) return s;
  return dq_launch(a, fwd_info, resolve_scale(a->softmax_scale, a->D), static_cast<cudaStream_t>(stream));
}

bsa_status bsa_bwd(const bsa_bwd_args* a, const bsa_mask_info* fwd_info, const bsa_mask_info* dkv_info,
                   bsa_stream stream) {
  bsa_status s = check_bwd(a);
  if (s != BSA_OK) return s;
  s = check_info(fwd_info, BSA_ORIENT_FWD, a->S_q, a->S_kv, a->Hq, "dq");
  if (s != BSA_OK) return s;
  s = check_info(dkv_info, BSA_ORIENT_DKV, a->S_q, a->S_kv, a->Hq, "dkv");
  if (s != BSA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float scale = resolve_scale(a->softmax_scale, a->D);
  s = rowsum_launch(a, st);
  if (s != BSA_OK) return s;
  s = dkv_launch(a, dkv_info, scale, st);
  if (s != BSA_OK) return s;
  return dq_launch(a, fwd_info, scale, st);
}

}  // extern "C"
