// Projection GEMM on the 5th-generation tensor cores for M > 64 tokens:
// y[M, N] = x[M, 4096] W^T with W stored [out, in] (the F.linear storage of
// the "Query projection" page), K fixed at 4096.
//
// One CTA computes a 128 x 256 output tile:
//   warp 0 (one lane)   TMA producer: 128x64 x tile and 256x64 W tile per
//                       stage, 128B-swizzled, 4-stage ring on mbarriers
//   warp 1 (one lane)   MMA issuer: tcgen05.mma kind::f16 (bf16 in, fp32 out)
//                       into a 256-column TMEM accumulator, tcgen05.commit
//                       releases each stage
//   warps 2-5           epilogue: tcgen05.ld of their 32 TMEM lanes, fused
//                       RoPE + KV-cache append (Q|K|V) or bf16 store (W_O)
// Every barrier wait is bounded; a wait that gives up records
// DEV_WAIT_TIMEOUT, drains outstanding copies (bounded) and frees TMEM.
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

__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
                   const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_b2,
                   ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_bar = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_bar + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] issued, [2] consumed

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const CUtensorMap* map_b;
  int brow;
  if (n0 < p.r1) {
    map_b = &map_b0;
    brow = n0;
  } else if (n0 < p.r2) {
    map_b = &map_b1;
    brow = n0 - p.r1;
  } else {
    map_b = &map_b2;
    brow = n0 - p.r2;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_bar), 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_barrier_init();
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(map_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    int kb = 0;
    for (; kb < NKB; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (kb >= STAGES && !mbar_wait(smem_u32(&empty[s]), ph ^ 1)) {
        atomicExch(&flags[0], 1);
        break;
      }
      if (*reinterpret_cast<volatile int*>(&flags[0])) break;
      const uint32_t fb = smem_u32(&full[s]);
      const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
      mbar_expect_tx(fb, STAGE_BYTES);
      tma_load_2d(sa, &map_a, fb, kb * BK, m0);
      tma_load_2d(sa + A_BYTES, map_b, fb, kb * BK, brow);
    }
    flags[1] = kb;
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = umma_idesc_bf16(BM, BN);
    int kb = 0;
    for (; kb < NKB; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait(smem_u32(&full[s]), ph)) {
        atomicExch(&flags[0], 1);
        break;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
      const uint32_t sb = sa + A_BYTES;
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        umma_bf16(tmem, umma_desc_sw128(sa + k * 32), umma_desc_sw128(sb + k * 32), idesc,
                  (kb | k) != 0 ? 1u : 0u);
      }
      umma_commit(smem_u32(&empty[s]));
    }
    flags[2] = kb;
    umma_commit(smem_u32(acc_bar));
  } else if (warp >= 2) {
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    bool ok = mbar_wait(smem_u32(acc_bar), 0);
    tc_fence_after();
    ok = __all_sync(0xffffffffu, ok && !*reinterpret_cast<volatile int*>(&flags[0]));
    if (ok) {
      const int m = m0 + quarter * 32 + lane;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        tmem_ld16(lane_addr + c, r);
        tmem_ld_wait();
        if (m < p.M) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          proj_store16(p, m, n0 + c, v);
        }
      }
    } else if (lane == 0) {
      atomicExch(&flags[0], 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (flags[0]) {
    if (threadIdx.x == 0) {
      report(p.status, DEV_WAIT_TIMEOUT);
      // let copies that were issued but never consumed land before exit
      for (int kb = flags[2]; kb < flags[1]; ++kb) mbar_wait(smem_u32(&full[kb % STAGES]), (kb / STAGES) & 1);
      mbar_wait(smem_u32(acc_bar), 0);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmMaps& maps, const ProjParams& p, cudaStream_t s) {
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
  if (p.N % BN != 0 || p.r1 % BN != 0 || p.r2 % BN != 0) return cudaErrorInvalidValue;
  const dim3 grid(p.N / BN, (p.M + BM - 1) / BM);
  gemm_tc_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(maps.a, maps.b[0], maps.b[1], maps.b[2], p);
  return cudaGetLastError();
}

}  // namespace gqa
