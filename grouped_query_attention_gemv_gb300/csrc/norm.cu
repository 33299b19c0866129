// attention_norm of the block ("Llama 3.1 8B · Grouped-query attention",
// handoff excerpt: the attention receives attention_norm(x), an RMSNorm over
// the 4096 features with norm_eps 1e-05): y_i = g_i x_i / sqrt(mean_j x_j^2 + eps).
// One warp per token row: the 8 KB row is read once into registers (16
// 16-byte vectors per lane), its mean square reduced across the warp in fp32,
// and y written as bf16 (one rounding of x * r * g).
#include "kernels.h"

namespace gqa {

namespace {

constexpr int WARPS = 8;
constexpr int VEC = D_MODEL / 8 / 32;  // 16-byte vectors per lane

__global__ void __launch_bounds__(WARPS * 32) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                             const __nv_bfloat16* __restrict__ g, float eps, int M,
                                                             __nv_bfloat16* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * D_MODEL);
  uint4 v[VEC];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    v[i] = ld_stream(xr + lane + 32 * i);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
      ss = fmaf(a, a, fmaf(b, b, ss));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss * (1.f / D_MODEL) + eps);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4* yr = reinterpret_cast<uint4*>(y + row * D_MODEL);
#pragma unroll
  for (int i = 0; i < VEC; ++i) {
    const uint4 gv = __ldg(gr + lane + 32 * i);
    const uint32_t xw[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_bf16(bf16_lo(xw[e]) * r * bf16_lo(gw[e]), bf16_hi(xw[e]) * r * bf16_hi(gw[e]));
    yr[lane + 32 * i] = make_uint4(o[0], o[1], o[2], o[3]);
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
