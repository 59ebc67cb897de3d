// rowsum(dO * O): the one quantity of the backward pass that is computed
// once, outside both gradient kernels ("Flash Attention on a TPU, Line by
// Line", section "What does the TPU flash attention kernel save for the
// backward pass?").  Dsum[b,h,s] = sum_d dO[b,h,s,d] * O[b,h,s,d] in fp32.
//
// HBM-bound: it reads 4*D bytes per row and writes 4.  Each row is split
// over D/8 lanes that load 16 bytes of dO and 16 of O (coalesced, one
// 128-byte line per 8 lanes), multiply in fp32 and reduce with shuffles.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace bsa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) rowsum_kernel(const uint4* __restrict__ dout, const uint4* __restrict__ out,
                                                     float* __restrict__ dsum, int64_t n_rows) {
  constexpr int kLanesPerRow = D / 8;  // 16 bytes (8 bf16) per lane
  constexpr int kRowsPerCta = 256 / kLanesPerRow;
  griddep_launch_dependents();
  griddep_wait();  // O comes from the forward kernel
  const int sub = threadIdx.x % kLanesPerRow;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + threadIdx.x / kLanesPerRow; row < n_rows;
       row += static_cast<int64_t>(gridDim.x) * kRowsPerCta) {
    const uint4 a = __ldcs(dout + row * kLanesPerRow + sub);
    const uint4 b = __ldcs(out + row * kLanesPerRow + sub);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(a2[e]);
      const float2 fb = __bfloat1622float2(b2[e]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
#pragma unroll
    for (int o = kLanesPerRow / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, kLanesPerRow);
    if (sub == 0) dsum[row] = acc;
  }
}

// Gradient of the attention sinks (extra logits z_j of every row's
// normaliser, no value): dz_j = -sum over the rows of exp(z_j - LSE) * Dsum.
// One CTA per 128-row query block of one (b, q head): one row per thread,
// a block reduction per sink, then one atomic add per sink and CTA.
__global__ void __launch_bounds__(128) dsink_kernel(const float* __restrict__ lse, const float* __restrict__ dsum,
                                                    const float* __restrict__ sinks, float* __restrict__ dsinks,
                                                    int32_t Hq, int32_t Hkv, int64_t Sq, int32_t n_sinks,
                                                    int32_t per_kv) {
  griddep_launch_dependents();
  griddep_wait();  // Dsum comes from the rowsum kernel
  __shared__ float part[4];
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 128 + threadIdx.x;
  const int32_t hq = static_cast<int32_t>((row / Sq) % Hq);
  const int32_t srow = per_kv ? hq / (Hq / Hkv) : 0;
  const float l = lse[row], d = dsum[row];
  for (int32_t j = 0; j < n_sinks; ++j) {
    const float z = sinks[srow * n_sinks + j];
    float c = (l == -INFINITY) ? 0.f : -expf(z - l) * d;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(&dsinks[srow * n_sinks + j], (part[0] + part[1]) + (part[2] + part[3]));
    __syncthreads();
  }
}

}  // namespace

bsa_status dsink_launch(const bsa_bwd_args* a, cudaStream_t stream) {
  if (a->num_sinks <= 0 || !a->dsinks) return BSA_OK;
  const int32_t srows = a->sinks_per_kv_head ? a->Hkv : 1;
  cudaError_t e = cudaMemsetAsync(a->dsinks, 0, sizeof(float) * srows * a->num_sinks, stream);
  if (e != cudaSuccess) return cuda_fail(e, "clear dsinks");
  const int64_t blocks = static_cast<int64_t>(a->B) * a->Hq * a->S_q / 128;
  e = launch_kernel(dsink_kernel, dim3(static_cast<unsigned>(blocks)), dim3(128), 0, stream, a->lse, a->dsum,
                    a->sinks, a->dsinks, a->Hq, a->Hkv, a->S_q, a->num_sinks, a->sinks_per_kv_head ? 1 : 0);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "dsink launch");
  return BSA_OK;
}

bsa_status rowsum_launch(const bsa_bwd_args* a, cudaStream_t stream) {
  const int64_t n_rows = static_cast<int64_t>(a->B) * a->Hq * a->S_q;
  const int rows_per_cta = 256 / (a->D / 8);
  const int64_t need = (n_rows + rows_per_cta - 1) / rows_per_cta;
  const int grid = static_cast<int>(std::min<int64_t>(need, static_cast<int64_t>(num_sms()) * 16));
  const uint4* dout = static_cast<const uint4*>(a->do_);
  const uint4* out = static_cast<const uint4*>(a->o);
  cudaError_t e = a->D == 128 ? launch_kernel(rowsum_kernel<128>, dim3(grid), dim3(256), 0, stream, dout, out, a->dsum, n_rows)
                              : launch_kernel(rowsum_kernel<64>, dim3(grid), dim3(256), 0, stream, dout, out, a->dsum, n_rows);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "rowsum launch");
  return dsink_launch(a, stream);
}

}  // namespace bsa
