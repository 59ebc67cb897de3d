// bsa_bwd_noalloc: the backward pass without any device allocation.
//
// The ordinary backward needs two pieces of device memory besides its
// inputs and outputs: the rowsum(dO*O) workspace (which the caller passes)
// and the library's device error word (which the library allocates on the
// first launch on each device).  Here both live in file-scope device arrays
// that exist from the moment the library is loaded on a device until the
// process exits, so a call allocates and frees nothing.  The host only
// needs their device addresses, which cudaGetSymbolAddress gives; that
// set-up runs on the first call on each device, with that device current.
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace bsa {
namespace {

// Largest B * Hq * S_q this entry point accepts (4 MiB of fp32 rowsum).
constexpr int64_t kMaxRows = int64_t(1) << 20;

// Shared by every call on a device; holds the last call's rowsum.
static __device__ __align__(256) float g_dsum_scratch[kMaxRows];
// Device-side error bits of this entry point's kernels; they stay set until
// bsa_get_device_error reads and clears them (with the library's own word).
static __device__ __align__(256) uint32_t g_err_scratch;

std::mutex g_mu;
float* g_dsum_ptr[64] = {nullptr};
uint32_t* g_err_ptr[64] = {nullptr};

// Device addresses of the two arrays for the current device.  In host code
// the arrays' names are host-side stand-ins, not device addresses, so the
// kernels are always given these resolved pointers.
bsa_status resolve(float** dsum, uint32_t** err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(BSA_ERR_UNSUPPORTED, "device index above 63");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dsum_ptr[dev]) {
    void* pd = nullptr;
    void* pe = nullptr;
    e = cudaGetSymbolAddress(&pd, g_dsum_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(rowsum scratch)");
    e = cudaGetSymbolAddress(&pe, g_err_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    g_dsum_ptr[dev] = static_cast<float*>(pd);
    g_err_ptr[dev] = static_cast<uint32_t*>(pe);
  }
  *dsum = g_dsum_ptr[dev];
  *err = g_err_ptr[dev];
  return BSA_OK;
}

bsa_status check(const bsa_bwd_args* a, const bsa_mask_info* fwd_info, const bsa_mask_info* dkv_info) {
  // the same checks as the ordinary backward, without the dsum workspace
  bsa_status s = check_bwd_args(a, false);
  if (s != BSA_OK) return s;
  const int64_t rows = static_cast<int64_t>(a->B) * a->Hq * a->S_q;
  if (rows > kMaxRows)
    return fail(BSA_ERR_UNSUPPORTED, "bsa_bwd_noalloc: B*Hq*S_q = " + std::to_string(rows) +
                                         " exceeds its fixed scratch of 1048576 rows; use bsa_bwd");
  const bsa_mask_info* infos[2] = {fwd_info, dkv_info};
  const int32_t orient[2] = {BSA_ORIENT_FWD, BSA_ORIENT_DKV};
  for (int i = 0; i < 2; ++i) {
    const bsa_mask_info* m = infos[i];
    if (!m) return fail(BSA_ERR_INVALID_ARG, "MaskInfo is null");
    if (m->orientation != orient[i]) return fail(BSA_ERR_INVALID_ARG, "MaskInfo has the wrong orientation");
    if (m->q_len != a->S_q || m->kv_len != a->S_kv)
      return fail(BSA_ERR_INVALID_ARG, "MaskInfo was compiled for other sequence lengths");
    if (m->heads != 1 && m->heads != a->Hq) return fail(BSA_ERR_INVALID_ARG, "MaskInfo must have 1 or Hq mask heads");
  }
  return BSA_OK;
}

}  // namespace

uint32_t* noalloc_error_word_if_set() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_err_ptr[dev];
}

}  // namespace bsa

using namespace bsa;

extern "C" bsa_status bsa_bwd_noalloc(const bsa_bwd_args* a, const bsa_mask_info* fwd_info,
                                      const bsa_mask_info* dkv_info, bsa_stream stream) {
  bsa_status s = check(a, fwd_info, dkv_info);
  if (s != BSA_OK) return s;
  float* dsum = nullptr;
  uint32_t* err = nullptr;
  s = resolve(&dsum, &err);
  if (s != BSA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bsa_bwd_args b;
  std::memcpy(&b, a, sizeof(b));
  b.dsum = dsum;  // every row is rewritten by the rowsum kernel before it is read
  const float scale = std::isnan(a->softmax_scale) ? 1.0f / std::sqrt(static_cast<float>(a->D)) : a->softmax_scale;
  s = rowsum_launch(&b, st);
  if (s != BSA_OK) return s;
  // round-robin tiles: a launch-time tile schedule would allocate
  s = dkv_launch(&b, dkv_info, scale, st, err, false);
  if (s != BSA_OK) return s;
  return dq_launch(&b, fwd_info, scale, st, err, false);
}
