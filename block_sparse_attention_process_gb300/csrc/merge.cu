// Merge of key shards ("Splash Attention: When the Mask Stops Being
// Arithmetic and Becomes the Loop", section "What does ring attention add on
// top of the splash kernel?"): each shard's unnormalised accumulator is
// rescaled to the common maximum of the row and the sum divided once by the
// merged normaliser.  A shard with l = 0 for a row contributes nothing.
//
// HBM-bound: per row it reads n * (4 D + 8) bytes and writes 2 D + 4.  One
// warp per row, four columns (one float4 of each shard) per lane.
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace bsa {
namespace {

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ acc, const float* __restrict__ ms,
                                                    const float* __restrict__ ls, __nv_bfloat16* __restrict__ o,
                                                    float* __restrict__ lse, int64_t rows, int32_t n) {
  griddep_launch_dependents();
  griddep_wait();  // the shards come from the forward launches
  constexpr int kLanes = D / 4;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
       row += warps) {
    float mx = -INFINITY;
    for (int32_t i = 0; i < n; ++i) {
      const float m = ms[i * rows + row], l = ls[i * rows + row];
      if (l > 0.f) mx = fmaxf(mx, m);
    }
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float lt = 0.f;
    if (mx != -INFINITY) {
      for (int32_t i = 0; i < n; ++i) {
        const float l = ls[i * rows + row];
        if (!(l > 0.f)) continue;
        const float w = expf(ms[i * rows + row] - mx);
        lt += w * l;
        if (lane < kLanes) {
          const float4 x = __ldcs(reinterpret_cast<const float4*>(acc + (i * rows + row) * D) + lane);
          a.x += w * x.x;
          a.y += w * x.y;
          a.z += w * x.z;
          a.w += w * x.w;
        }
      }
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    if (lane < kLanes)
      reinterpret_cast<uint2*>(o + row * D)[lane] =
          make_uint2(pack_bf16x2(a.x * inv, a.y * inv), pack_bf16x2(a.z * inv, a.w * inv));
    if (lane == 0) lse[row] = lt > 0.f ? mx + logf(lt) : -INFINITY;
  }
}

}  // namespace

bsa_status merge_launch(const bsa_merge_args* a, cudaStream_t stream) {
  const int64_t need = (a->rows + 7) / 8;
  const int grid = static_cast<int>(std::min<int64_t>(need, static_cast<int64_t>(num_sms()) * 16));
  cudaError_t e;
  if (a->D == 128)
    e = launch_kernel(merge_kernel<128>, dim3(grid), dim3(256), 0, stream, a->o_acc, a->m, a->l,
                      static_cast<__nv_bfloat16*>(a->o), a->lse, a->rows, a->n_shards);
  else
    e = launch_kernel(merge_kernel<64>, dim3(grid), dim3(256), 0, stream, a->o_acc, a->m, a->l,
                      static_cast<__nv_bfloat16*>(a->o), a->lse, a->rows, a->n_shards);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return BSA_OK;
}

}  // namespace bsa
