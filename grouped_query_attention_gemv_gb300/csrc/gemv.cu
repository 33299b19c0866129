// Weight-streaming projection for few tokens (M <= 64): y = x W^T.
//
// At decode sizes the projections of the block ("Llama 3.1 8B · Query
// projection": Q = x W_Q with the weight stored [out, in]; the K, V and
// output projections of "Grouped-query attention") are bound by reading the
// 84 MB of weights once, so the kernel is organised around streaming W:
//
//   * the work is the grid of (16-row block, 64-wide k block) units of W,
//     2 KB each, cut into equal contiguous ranges, one per warp of the grid
//     (stream-K), so every SM streams the same number of bytes;
//   * a warp reads its rows straight from HBM with 128-bit loads, two k blocks
//     in flight, and multiplies on the tensor cores with mma.sync m16n8k16:
//     W rows are the A operand, the (<= 64) tokens the B operand, fp32
//     accumulators. Each thread's 16-byte load holds 8 consecutive k values;
//     the k order inside a 64-wide block is permuted identically for A and B
//     so no shuffle is needed;
//   * a warp that finishes its part of a row block adds its fp32 partial into
//     a zero-filled scratch with red.add, then takes a ticket; the warp whose
//     ticket completes the 64 k blocks of that row block applies the epilogue
//     (RoPE and KV-cache append for Q|K|V, plain bf16 store for W_O) and
//     zero-fills the scratch again. No warp ever waits for another.
#include "kernels.h"

namespace gqa {

namespace {

constexpr int KBLK = 64;                  // k values per unit
constexpr int NKB = D_MODEL / KBLK;       // 64 k blocks per row block
constexpr int GEMV_THREADS = 256;

template <int NT>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_kernel(ProjParams p, float* __restrict__ acc,
                                                            int* __restrict__ tickets) {
  constexpr int MP = NT * 8;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int warps_per_cta = GEMV_THREADS / 32;
  const long long nwarps = static_cast<long long>(gridDim.x) * warps_per_cta;
  const long long wid = static_cast<long long>(blockIdx.x) * warps_per_cta + (threadIdx.x >> 5);
  const long long units = static_cast<long long>(p.N / 16) * NKB;
  long long u = units * wid / nwarps;
  const long long u_end = units * (wid + 1) / nwarps;

  // token rows this thread feeds into the B operand
  const uint4* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = nt * 8 + g;
    xrow[nt] = m < p.M ? reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(m) * D_MODEL) : nullptr;
  }

  while (u < u_end) {
    const int rb = static_cast<int>(u / NKB);
    const int kb0 = static_cast<int>(u - static_cast<long long>(rb) * NKB);
    const int kb1 = static_cast<int>(min(static_cast<long long>(NKB), kb0 + (u_end - u)));
    const int row0 = rb * 16;
    const __nv_bfloat16* W;
    int lrow;
    if (row0 < p.r1) {
      W = p.w0;
      lrow = row0;
    } else if (row0 < p.r2) {
      W = p.w1;
      lrow = row0 - p.r1;
    } else {
      W = p.w2;
      lrow = row0 - p.r2;
    }
    const uint4* wa = reinterpret_cast<const uint4*>(W + static_cast<size_t>(lrow + g) * D_MODEL) + t;
    const uint4* wb = reinterpret_cast<const uint4*>(W + static_cast<size_t>(lrow + g + 8) * D_MODEL) + t;

    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;

    uint4 cw0 = ld_stream(wa + kb0 * 8), cw1 = ld_stream(wa + kb0 * 8 + 4);
    uint4 cw2 = ld_stream(wb + kb0 * 8), cw3 = ld_stream(wb + kb0 * 8 + 4);
    for (int kb = kb0; kb < kb1; ++kb) {
      uint4 nw0 = cw0, nw1 = cw1, nw2 = cw2, nw3 = cw3;
      if (kb + 1 < kb1) {
        nw0 = ld_stream(wa + (kb + 1) * 8);
        nw1 = ld_stream(wa + (kb + 1) * 8 + 4);
        nw2 = ld_stream(wb + (kb + 1) * 8);
        nw3 = ld_stream(wb + (kb + 1) * 8 + 4);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
        if (xrow[nt]) {
          x0 = ld_nc(xrow[nt] + kb * 8 + t);
          x1 = ld_nc(xrow[nt] + kb * 8 + t + 4);
        }
        // logical k (2t, 2t+1 | 2t+8, 2t+9) of step s <- physical 8t + 4(s&1) + {0,1 | 2,3} + 32(s>>1)
        mma16816(d[nt], cw0.x, cw2.x, cw0.y, cw2.y, x0.x, x0.y);
        mma16816(d[nt], cw0.z, cw2.z, cw0.w, cw2.w, x0.z, x0.w);
        mma16816(d[nt], cw1.x, cw3.x, cw1.y, cw3.y, x1.x, x1.y);
        mma16816(d[nt], cw1.z, cw3.z, cw1.w, cw3.w, x1.z, x1.w);
      }
      cw0 = nw0;
      cw1 = nw1;
      cw2 = nw2;
      cw3 = nw3;
    }

    // partial sums: d[nt] = (row g | g+8, tokens nt*8 + 2t, +1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = nt * 8 + 2 * t;
      if (n < p.M) {
        red_add_v2(acc + static_cast<size_t>(row0 + g) * MP + n, d[nt][0], d[nt][1]);
        red_add_v2(acc + static_cast<size_t>(row0 + g + 8) * MP + n, d[nt][2], d[nt][3]);
      }
    }
    __threadfence();
    __syncwarp();
    int prev = 0;
    if (lane == 0) prev = atomicAdd(tickets + rb, kb1 - kb0);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev + (kb1 - kb0) == NKB) {
      // this warp completed row block rb: epilogue over 8 feature pairs x M tokens
      __threadfence();
      float* a = acc + static_cast<size_t>(row0) * MP;
      for (int idx = lane; idx < 8 * p.M; idx += 32) {
        const int m = idx >> 3;
        const int pr = idx & 7;
        const float va = __ldcg(a + (2 * pr) * MP + m);
        const float vb = __ldcg(a + (2 * pr + 1) * MP + m);
        proj_store2(p, m, row0 + 2 * pr, va, vb);
      }
      __syncwarp();
      for (int idx = lane; idx < 16 * MP; idx += 32) __stcg(a + idx, 0.f);
      if (lane == 0) tickets[rb] = 0;
    }
    u += kb1 - kb0;
  }
}

}  // namespace

int gemv_padded_m(int M) {
  if (M <= 0 || M > 64) return 0;
  if (M <= 8) return 8;
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  return 64;
}

cudaError_t launch_gemv(const ProjParams& p, float* acc, int* tickets, int num_sms, cudaStream_t s) {
  const dim3 grid(2 * num_sms), block(GEMV_THREADS);
  switch (gemv_padded_m(p.M)) {
    case 8: gemv_kernel<1><<<grid, block, 0, s>>>(p, acc, tickets); break;
    case 16: gemv_kernel<2><<<grid, block, 0, s>>>(p, acc, tickets); break;
    case 32: gemv_kernel<4><<<grid, block, 0, s>>>(p, acc, tickets); break;
    case 64: gemv_kernel<8><<<grid, block, 0, s>>>(p, acc, tickets); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace gqa
