// attention_norm of the block ("Llama 3.1 8B · Grouped-query attention",
// handoff excerpt: the attention receives attention_norm(x), an RMSNorm over
// the 4096 features with norm_eps 1e-05): y_i = g_i x_i / sqrt(mean_j x_j^2 + eps).
// One warp per token row: the 8 KB row is read once into registers (16
// 16-byte vectors per lane), its mean square reduced across the warp in fp32,
// and y written as bf16 (one rounding of x * r * g). The arithmetic is in
// norm_core.cuh, shared with the fused decode grid.
#include "kernels.h"
#include "norm_core.cuh"

namespace gqa {

namespace {

constexpr int WARPS = 8;

__global__ void __launch_bounds__(WARPS * 32) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const __nv_bfloat16* __restrict__ g, float eps, int M,
                                                             __nv_bfloat16* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  if (row >= M) return;
  uint4 v[NORM_VEC];
  norm_load_row(x + row * D_MODEL, lane, v);
  const float r = norm_inv_rms(v, eps);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4* yr = reinterpret_cast<uint4*>(y + row * D_MODEL);
#pragma unroll
  for (int i = 0; i < NORM_VEC; ++i) {
    const uint4 gv = __ldg(gr + lane + 32 * i);
    yr[lane + 32 * i] = make_uint4(norm_pair(v[i].x, r, gv.x), norm_pair(v[i].y, r, gv.y), norm_pair(v[i].z, r, gv.z),
                                   norm_pair(v[i].w, r, gv.w));
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* g, float eps, int M, __nv_bfloat16* y,
                           cudaStream_t s) {
  if (M <= 0) return cudaErrorInvalidValue;
  const int blocks = (M + WARPS - 1) / WARPS;
  rmsnorm_kernel<<<blocks, WARPS * 32, 0, s>>>(x, g, eps, M, y);
  return cudaGetLastError();
}

}  // namespace gqa
