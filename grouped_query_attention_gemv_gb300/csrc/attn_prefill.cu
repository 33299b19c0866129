// Causal prefill attention: T new tokens per sequence after start_pos cached
// rows. Query t (position start_pos + t) of head h attends to cache rows
// 0..start_pos+t of KV head h / 4 ("Llama 3.1 8B · Grouped-query attention":
// the mask of Transformer.forward is -inf above the diagonal, left-padded with
// start_pos visible columns; softmax in fp32; output heads merged h*128 + d).
//
// One CTA takes 32 query positions of one sequence and the 4 query heads of
// one KV group (8 warps, 16 rows each). K/V tiles of 64 keys come in by 4-D
// TMA (128B swizzle, 2-stage mbarrier ring) once for all 4 heads; QK^T and PV
// run on mma.sync m16n8k16 with an online softmax in fp32. Tiles above a
// warp's diagonal are skipped; CTAs with the longest key range launch first.
#include <math.h>

#include "kernels.h"

namespace gqa {

namespace {

constexpr int TILE = PREFILL_TILE;  // keys per stage (= TMA box height)
constexpr int QT = 32;                          // query positions per CTA
constexpr int STAGES = 2;
constexpr int HALF_BYTES = TILE * 128;
constexpr int KV_TILE_BYTES = 2 * HALF_BYTES;
constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;
constexpr int THREADS = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 128;
constexpr float SCALE_LOG2 = 0.08838834764831845f * 1.4426950408889634f;

__device__ __forceinline__ void issue_tile(uint8_t* smem, uint64_t* full, const CUtensorMap* mk,
                                           const CUtensorMap* mv, int i, int g, int b) {
  const int st = i % STAGES;
  const uint32_t fb = smem_u32(&full[st]);
  const uint32_t base = smem_u32(smem + st * STAGE_BYTES);
  const int pos = i * TILE;
  mbar_expect_tx(fb, STAGE_BYTES);
  tma_load_4d(base, mk, fb, 0, g, pos, b);
  tma_load_4d(base + HALF_BYTES, mk, fb, 64, g, pos, b);
  tma_load_4d(base + KV_TILE_BYTES, mv, fb, 0, g, pos, b);
  tma_load_4d(base + KV_TILE_BYTES + HALF_BYTES, mv, fb, 64, g, pos, b);
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                        PrefillAttnParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  int* sflag = reinterpret_cast<int*>(empty + STAGES);  // [0] abort, [2] issued

  const int nqt = (a.T + QT - 1) / QT;
  const int qtile = nqt - 1 - static_cast<int>(blockIdx.x);  // longest key ranges first
  const int g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;
  const int hh = warp >> 1;
  const int h = g * N_REP + hh;
  const int start = a.sp.get(b);
  if (!a.sp.ok(start)) {
    if (qtile == nqt - 1 && g == 0 && threadIdx.x == 0) report(a.status, DEV_BAD_POSITION);
    return;
  }
  const int q0 = qtile * QT;
  const int kv_end = start + min(q0 + QT, a.T);
  const int ntiles = (kv_end + TILE - 1) / TILE;
  const int row0 = q0 + (warp & 1) * 16 + gr;  // query index t of rows gr and gr+8
  const int row1 = row0 + 8;
  const int qp0 = row0 < a.T ? start + row0 : -1;  // absolute positions (-1: no such row)
  const int qp1 = row1 < a.T ? start + row1 : -1;
  const int wmax = start + min(q0 + (warp & 1) * 16 + 15, a.T - 1);  // last position of this warp

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), THREADS / 32);
    }
    sflag[0] = 0;
    fence_barrier_init();
    const int first = min(STAGES, ntiles);
    for (int i = 0; i < first; ++i) issue_tile(smem, full, &mk, &mv, i, g, b);
    sflag[2] = first;
  }

  // Q fragments: rows gr / gr+8 = query rows row0 / row1, cols = dims
  uint32_t qa[8][4];
  {
    const size_t tok0 = static_cast<size_t>(b) * a.T + row0;
    const uint32_t* q0p = reinterpret_cast<const uint32_t*>(a.q + tok0 * D_MODEL + static_cast<size_t>(h) * HEAD_DIM);
    const uint32_t* q1p = q0p + 8 * D_MODEL / 2;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = row0 < a.T ? q0p[ks * 8 + t] : 0u;
      qa[ks][1] = row1 < a.T ? q1p[ks * 8 + t] : 0u;
      qa[ks][2] = row0 < a.T ? q0p[ks * 8 + 4 + t] : 0u;
      qa[ks][3] = row1 < a.T ? q1p[ks * 8 + 4 + t] : 0u;
    }
  }
  __syncthreads();

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;

  bool aborted = false;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % STAGES;
    const uint32_t ph = (i / STAGES) & 1;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[st]), ph))) {
      aborted = true;
      break;
    }
    const int base_key = i * TILE;
    if (base_key <= wmax) {
      const uint32_t kt = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t vt = kt + KV_TILE_BYTES;
      float sc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
        const int r = j * 8 + (lane & 7);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int ch = 4 * c + (lane >> 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kt + (ch >> 3) * HALF_BYTES + sw128(r, ch & 7), b0, b1, b2, b3);
          mma16816(sc[j], qa[2 * c][0], qa[2 * c][1], qa[2 * c][2], qa[2 * c][3], b0, b1);
          mma16816(sc[j], qa[2 * c + 1][0], qa[2 * c + 1][1], qa[2 * c + 1][2], qa[2 * c + 1][3], b2, b3);
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = base_key + 8 * j + 2 * t + e;
          const float v0 = key <= qp0 ? sc[j][e] * SCALE_LOG2 : -INFINITY;
          const float v1 = key <= qp1 ? sc[j][2 + e] * SCALE_LOG2 : -INFINITY;
          sc[j][e] = v0;
          sc[j][2 + e] = v1;
          mx0 = fmaxf(mx0, v0);
          mx1 = fmaxf(mx1, v1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
      const float al0 = exp2f(m0 - u0), al1 = exp2f(m1 - u1);
      m0 = n0;
      m1 = n1;
      float s0 = 0.f, s1 = 0.f;
      uint32_t pa[4][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = exp2f(sc[j][0] - u0), p1 = exp2f(sc[j][1] - u0);
        const float p2 = exp2f(sc[j][2] - u1), p3 = exp2f(sc[j][3] - u1);
        s0 += p0 + p1;
        s1 += p2 + p3;
        pa[j >> 1][(j & 1) * 2] = pack_bf16(p0, p1);
        pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16(p2, p3);
      }
      l0 = l0 * al0 + s0;
      l1 = l1 * al1 + s1;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        oacc[nt][0] *= al0;
        oacc[nt][1] *= al0;
        oacc[nt][2] *= al1;
        oacc[nt][3] *= al1;
      }
      const bool ragged = base_key + TILE > kv_end;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t mask_a = 0xffffffffu, mask_b = 0xffffffffu;
        if (ragged) {
          const int ka = base_key + 16 * kk + 2 * t, kb = ka + 8;
          mask_a = (ka < kv_end ? 0x0000ffffu : 0u) | (ka + 1 < kv_end ? 0xffff0000u : 0u);
          mask_b = (kb < kv_end ? 0x0000ffffu : 0u) | (kb + 1 < kv_end ? 0xffff0000u : 0u);
        }
        const int vr = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const int ch = 2 * dp + (lane >> 4);
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vt + (ch >> 3) * HALF_BYTES + sw128(vr, ch & 7), v0, v1, v2, v3);
          mma16816(oacc[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], v0 & mask_a, v1 & mask_b);
          mma16816(oacc[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], v2 & mask_a, v3 & mask_b);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    if (threadIdx.x == 0 && i + STAGES < ntiles) {
      if (mbar_wait(smem_u32(&empty[st]), ph)) {
        issue_tile(smem, full, &mk, &mv, i + STAGES, g, b);
        sflag[2] = i + STAGES + 1;
      } else {
        aborted = true;
      }
    }
    if (__any_sync(0xffffffffu, aborted)) {
      aborted = true;
      break;
    }
  }
  if (aborted) atomicExch(&sflag[0], 1);
  __syncthreads();
  if (sflag[0]) {
    if (threadIdx.x == 0) {
      report(a.status, DEV_WAIT_TIMEOUT);
      const int issued = sflag[2];
      for (int i = max(0, issued - STAGES); i < issued; ++i)
        mbar_wait(smem_u32(&full[i % STAGES]), (i / STAGES) & 1);
    }
    return;
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  __nv_bfloat16* o0 = a.o + (static_cast<size_t>(b) * a.T + row0) * D_MODEL + static_cast<size_t>(h) * HEAD_DIM;
  __nv_bfloat16* o1 = o0 + 8 * static_cast<size_t>(D_MODEL);
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    if (row0 < a.T)
      *reinterpret_cast<uint32_t*>(o0 + nt * 8 + 2 * t) = pack_bf16(oacc[nt][0] * inv0, oacc[nt][1] * inv0);
    if (row1 < a.T)
      *reinterpret_cast<uint32_t*>(o1 + nt * 8 + 2 * t) = pack_bf16(oacc[nt][2] * inv1, oacc[nt][3] * inv1);
  }
}

}  // namespace

cudaError_t launch_attn_prefill(const CUtensorMap& mk, const CUtensorMap& mv, const PrefillAttnParams& a,
                                cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid((a.T + QT - 1) / QT, N_KV, a.B);
  attn_prefill_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace gqa
