// Projection GEMM on the 5th-generation tensor cores for M > 64 tokens:
// y[M, N] = x[M, 4096] W^T with W stored [out, in] (the F.linear storage of
// the "Query projection" page), K fixed at 4096.
//
// Persistent: one CTA per SM walks the 128 x 256 output tiles t = CTA,
// CTA + grid, ... with the output features fastest within groups of at most
// 24 feature tiles (48 MB of weights): the CTAs in flight cover a few token
// tiles against one group, which L2 holds while every token tile passes over
// it, so W comes from HBM once and x once per group. Q|K|V with 8 KV heads
// (24 tiles) and W_O (16) are one group; the multi-head Q|K|V (48 tiles,
// 100 MB) is two, where one group over all of it read W ~5 times at 2048
// tokens. (Token tiles fastest made every wave sweep all of x: at 8192 tokens
// its 67 MB were read ~10 times.)
//   warp 0 (one lane)   TMA producer: 128x64 x tile and 256x64 W tile per
//                       stage, 128B-swizzled, 4-stage ring on mbarriers, one
//                       ring across the CTA's tiles
//   warp 1 (one lane)   MMA issuer: tcgen05.mma kind::f16 (bf16 in, fp32 out)
//                       into one of two 256-column TMEM accumulators;
//                       tcgen05.commit releases each stage, then the tile
//   warps 2-5           epilogue of the previous tile while the next one is
//                       multiplied: tcgen05.ld of their 32 TMEM lanes (one
//                       token each), fused RoPE + KV-cache append (Q|K|V) or a
//                       bf16 store (W_O), then the accumulator goes back.
// A 256-column tile holds two heads: the RoPE pairs of column c and c + 128
// share one (cos, sin), so each thread loads its position's 64 pairs (one
// 512-byte table row) once per tile and rotates both heads with them.
// Every barrier wait is bounded; a wait that gives up records
// DEV_WAIT_TIMEOUT, drains outstanding copies and products (bounded) and
// frees TMEM.
#include "kernels.h"

namespace gqa {

namespace {

constexpr int BM = GEMM_BM, BN = GEMM_BN, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NKB = D_MODEL / BK;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators
constexpr int EPI_WARPS = 4;
constexpr int GROUP_N = 24;  // feature tiles per group of the tile walk

// Tile t of the walk -> its first token m0 and first output feature n0.
__device__ __forceinline__ void tile_of(int t, int tiles_m, int tiles_n, int& m0, int& n0) {
  const int per_group = tiles_m * GROUP_N;
  const int g = t / per_group, r = t - g * per_group;
  const int gw = min(GROUP_N, tiles_n - g * GROUP_N);
  m0 = (r / gw) * BM;
  n0 = (g * GROUP_N + r % gw) * BN;
}

struct Bars {
  uint64_t full[STAGES], empty[STAGES];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_slot;
  int abort;
  int issued, consumed;  // k-block loads requested / consumed by the MMA issuer
};

__device__ __forceinline__ bool aborted(const Bars& bs) { return *reinterpret_cast<const volatile int*>(&bs.abort) != 0; }

// Weight map and row of output feature n0 (tiles never straddle w0/w1/w2).
__device__ __forceinline__ const CUtensorMap* weight_of(const ProjParams& p, const CUtensorMap* b0, const CUtensorMap* b1,
                                                        const CUtensorMap* b2, int n0, int& brow) {
  if (n0 < p.r1) {
    brow = n0;
    return b0;
  }
  if (n0 < p.r2) {
    brow = n0 - p.r1;
    return b1;
  }
  brow = n0 - p.r2;
  return b2;
}

__device__ __forceinline__ void store32(__nv_bfloat16* dst, const float (&v)[16]) {
  uint4 lo, hi;
  lo.x = pack_bf16(v[0], v[1]);
  lo.y = pack_bf16(v[2], v[3]);
  lo.z = pack_bf16(v[4], v[5]);
  lo.w = pack_bf16(v[6], v[7]);
  hi.x = pack_bf16(v[8], v[9]);
  hi.y = pack_bf16(v[10], v[11]);
  hi.z = pack_bf16(v[12], v[13]);
  hi.w = pack_bf16(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = lo;
  reinterpret_cast<uint4*>(dst)[1] = hi;
}

// v[e] += src[e] for 16 bf16 values (16-byte aligned).
__device__ __forceinline__ void add_bf16_16(float (&v)[16], const __nv_bfloat16* src) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 u = __ldg(s4 + h);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * h + 2 * e] += bf16_lo(w[e]);
      v[8 * h + 2 * e + 1] += bf16_hi(w[e]);
    }
  }
}

// Rotate the 8 pairs of v by (cos, sin) pairs cs[0..3] (two pairs per float4).
__device__ __forceinline__ void rotate16(float (&v)[16], const float4* cs) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 c = cs[j];
    float a = v[4 * j], b = v[4 * j + 1];
    v[4 * j] = a * c.x - b * c.y;
    v[4 * j + 1] = a * c.y + b * c.x;
    a = v[4 * j + 2];
    b = v[4 * j + 3];
    v[4 * j + 2] = a * c.z - b * c.w;
    v[4 * j + 3] = a * c.w + b * c.z;
  }
}

// Epilogue of one tile for token m (this thread's TMEM lane): columns n0 .. n0+255.
__device__ __forceinline__ void epilogue_tile(const ProjParams& p, uint32_t acc, int m, int n0) {
  __nv_bfloat16* dst = nullptr;
  int pos = 0;
  bool rope = false;
  if (m < p.M) {
    if (!p.qkv) {
      dst = p.out + static_cast<size_t>(m) * p.N + n0;
    } else {
      const int b = m / p.T;
      const int t = m - b * p.T;
      const int start = p.sp.get(b);
      if (p.sp.ok(start)) {
        pos = start + t;
        if (n0 < D_MODEL) {
          dst = p.out + static_cast<size_t>(m) * D_MODEL + n0;
          rope = true;
        } else {
          const size_t row = (static_cast<size_t>(b) * p.s_max + pos) * (p.r2 - p.r1);
          rope = n0 < p.r2;
          dst = rope ? p.cache_k + row + (n0 - D_MODEL) : p.cache_v + row + (n0 - p.r2);
        }
      } else if (t == 0 && n0 == 0) {
        report(p.status, DEV_BAD_POSITION);
      }
    }
  }
  float4 cs[32];  // (cos, sin) of the 64 pairs at this position
  if (rope) {
    const float4* row = reinterpret_cast<const float4*>(p.rope + static_cast<size_t>(pos) * ROPE_PAIRS * 2);
#pragma unroll
    for (int j = 0; j < 32; ++j) cs[j] = __ldg(row + j);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t r0[16], r1[16];
    tmem_ld16(acc + c * 16, r0);
    tmem_ld16(acc + 128 + c * 16, r1);
    tmem_ld_wait();
    float v0[16], v1[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      v0[e] = __uint_as_float(r0[e]);
      v1[e] = __uint_as_float(r1[e]);
    }
    if (rope) {
      rotate16(v0, cs + 4 * c);
      rotate16(v1, cs + 4 * c);
    }
    if (dst && p.resid) {  // the block's residual (plain store only)
      add_bf16_16(v0, p.resid + static_cast<size_t>(m) * p.N + n0 + c * 16);
      add_bf16_16(v1, p.resid + static_cast<size_t>(m) * p.N + n0 + 128 + c * 16);
    }
    if (dst) {
      store32(dst + c * 16, v0);
      store32(dst + 128 + c * 16, v1);
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                   ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bs = *reinterpret_cast<Bars*>(smem + STAGES * STAGE_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_n = p.N / BN;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles = tiles_m * tiles_n;
  const int G = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bs.full[s]), 1);
      mbar_init(smem_u32(&bs.empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bs.acc_full[i]), 1);
      mbar_init(smem_u32(&bs.acc_empty[i]), EPI_WARPS);
    }
    mbar_init(smem_u32(&bs.mma_done), 1);
    bs.abort = 0;
    bs.issued = 0;
    bs.consumed = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_b0);
    tma_prefetch_desc(&map_b1);
    tma_prefetch_desc(&map_b2);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bs.tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs.tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // every token tile is read by the CTAs of its group at about the same
      // time and never again; every weight tile by each token tile in turn:
      // L2 keeps the weights before the token rows
      const uint64_t pol_x = l2_evict_first(), pol_w = l2_evict_last();
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += G) {
        int m0, n0;
        tile_of(t, tiles_m, tiles_n, m0, n0);
        int brow;
        const CUtensorMap* mb = weight_of(p, &map_b0, &map_b1, &map_b2, n0, brow);
        for (int kb = 0; kb < NKB; ++kb, ++it) {
          const int s = it % STAGES;
          if (it >= STAGES && !mbar_wait(smem_u32(&bs.empty[s]), ((it / STAGES) & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (aborted(bs)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&bs.full[s]);
          const uint32_t sa = sbase + s * STAGE_BYTES;
          mbar_expect_tx(fb, STAGE_BYTES);
          tma_load_2d_hint(sa, &map_a, fb, kb * BK, m0, pol_x);
          tma_load_2d_hint(sa + A_BYTES, mb, fb, kb * BK, brow, pol_w);
        }
      }
      if (!ok) atomicExch(&bs.abort, 1);
      bs.issued = it;
    }
  } else if (warp == 1) {
    // the whole warp runs the loop (descriptors stay warp-uniform); one
    // elected lane issues the products and commits
    const uint32_t idesc = umma_idesc_bf16(BM, BN);
    int it = 0, j = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += G, ++j) {
      const int buf = j & 1;
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.acc_empty[buf]), ((j >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + buf * BN;
      for (int kb = 0; kb < NKB; ++kb, ++it) {
        const int s = it % STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.full[s]), (it / STAGES) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = sbase + s * STAGE_BYTES;
        const uint32_t sb = sa + A_BYTES;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d, umma_desc_sw128(sa + k * 32), umma_desc_sw128(sb + k * 32), idesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&bs.empty[s]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) umma_commit(smem_u32(&bs.acc_full[buf]));
      __syncwarp();
    }
    if (lane == 0) {
      if (!ok) atomicExch(&bs.abort, 1);
      bs.consumed = it;
    }
    if (elect_one()) umma_commit(smem_u32(&bs.mma_done));
    __syncwarp();
    mbar_wait(smem_u32(&bs.mma_done), 0);
  } else {
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    int j = 0;
    for (int t = blockIdx.x; t < tiles; t += G, ++j) {
      const int buf = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.acc_full[buf]), (j >> 1) & 1)) ||
          __any_sync(0xffffffffu, aborted(bs))) {
        if (lane == 0) atomicExch(&bs.abort, 1);
        break;
      }
      tc_fence_after();
      int m0, n0;
      tile_of(t, tiles_m, tiles_n, m0, n0);
      epilogue_tile(p, lane_addr + buf * BN, m0 + quarter * 32 + lane, n0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bs.acc_empty[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (aborted(bs)) {
    if (threadIdx.x == 0) {
      report(p.status, DEV_WAIT_TIMEOUT);
      // copies that were requested but never consumed land before exit
      for (int it = bs.consumed; it < bs.issued; ++it)
        mbar_wait(smem_u32(&bs.full[it % STAGES]), (it / STAGES) & 1);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmMaps& maps, const ProjParams& p, int ctas, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (p.M <= 0 || p.N % BN != 0 || p.r1 % BN != 0 || p.r2 % BN != 0 || ctas <= 0) return cudaErrorInvalidValue;
  const long long tiles = static_cast<long long>((p.M + BM - 1) / BM) * (p.N / BN);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = tiles < ctas ? static_cast<int>(tiles) : ctas;
  gemm_tc_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(maps.a, maps.b[0], maps.b[1], maps.b[2], p);
  return cudaGetLastError();
}

}  // namespace gqa
