// attention_norm arithmetic shared by the standalone norm kernel (norm.cu)
// and the fused decode grid's Q|K|V phase (proj_rows.cuh), so that both give
// bit-identical normalised rows: y_i = g_i x_i / sqrt(mean_j x_j^2 + eps)
// ("Llama 3.1 8B · Grouped-query attention", handoff excerpt: the attention
// receives attention_norm(x), RMSNorm over the 4096 features).
#pragma once

#include "common.cuh"

namespace gqa {

constexpr int NORM_VEC = D_MODEL / 8 / 32;  // 16-byte vectors of a row per lane

// One warp reads row `x` (4096 bf16) into v: lane l holds vectors l + 32 i.
__device__ __forceinline__ void norm_load_row(const __nv_bfloat16* x, int lane, uint4 (&v)[NORM_VEC]) {
  const uint4* xr = reinterpret_cast<const uint4*>(x);
#pragma unroll
  for (int i = 0; i < NORM_VEC; ++i) v[i] = ld_stream(xr + lane + 32 * i);
}

// 1 / sqrt(mean(x^2) + eps) of the row held by the warp (fp32, fixed order:
// each lane's values in sequence, then a butterfly over the lanes).
__device__ __forceinline__ float norm_inv_rms(const uint4 (&v)[NORM_VEC], float eps) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NORM_VEC; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
      ss = fmaf(a, a, fmaf(b, b, ss));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return rsqrtf(ss * (1.f / D_MODEL) + eps);
}

// Two normalised features (x * r) * g, rounded once to bf16.
__device__ __forceinline__ uint32_t norm_pair(uint32_t x2, float r, uint32_t g2) {
  return pack_bf16(bf16_lo(x2) * r * bf16_lo(g2), bf16_hi(x2) * r * bf16_hi(g2));
}

}  // namespace gqa
