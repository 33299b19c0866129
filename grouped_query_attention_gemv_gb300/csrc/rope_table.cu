// RoPE table R [rows, 64 pairs] of (cos, sin) for the decode/prefill calls.
//
// The pages rotate adjacent pairs of each head by freqs_cis ("apply_rotary_emb"
// on the "Grouped-query attention" page) and name the Llama 3.1 frequency
// rescaling (use_scaled_rope in the catalogue entry; "Prepare Q, K, V · Key
// heads" points at its source) without printing it. This kernel takes the
// plainest reading: f_i = theta^(-2i/128), rescaled band-wise by the
// wavelength 2*pi/f_i against original_context/high_freq_factor and
// original_context/low_freq_factor, linear interpolation between. Angles and
// their cos/sin are evaluated in fp64 and stored as fp32.
#include "kernels.h"

namespace gqa {

namespace {

__global__ void rope_table_kernel(float2* __restrict__ rope, int rows, double theta, int scaled, double factor,
                                  double lo, double hi, double ctx) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(rows) * ROPE_PAIRS) return;
  const int p = static_cast<int>(idx / ROPE_PAIRS);
  const int i = static_cast<int>(idx % ROPE_PAIRS);
  double f = pow(theta, -2.0 * i / HEAD_DIM);
  if (scaled) {
    const double wavelength = 2.0 * 3.14159265358979323846 / f;
    if (wavelength > ctx / lo) {
      f = f / factor;
    } else if (wavelength >= ctx / hi) {
      const double mu = (ctx / wavelength - lo) / (hi - lo);
      f = (1.0 - mu) * f / factor + mu * f;
    }
  }
  double s, c;
  sincos(static_cast<double>(p) * f, &s, &c);
  rope[idx] = make_float2(static_cast<float>(c), static_cast<float>(s));
}

}  // namespace

cudaError_t launch_rope_table(float* rope, int rows, double theta, int scaled, double factor, double lo,
                              double hi, double ctx, cudaStream_t s) {
  const size_t n = static_cast<size_t>(rows) * ROPE_PAIRS;
  const int block = 256;
  const unsigned grid = static_cast<unsigned>((n + block - 1) / block);
  rope_table_kernel<<<grid, block, 0, s>>>(reinterpret_cast<float2*>(rope), rows, theta, scaled, factor, lo, hi,
                                           ctx);
  return cudaGetLastError();
}

}  // namespace gqa
