// Decode attention (one new token per sequence) over the KV cache.
//
// "Llama 3.1 8B · Grouped-query attention" (mode decode): for every query
// head h the scores q_h . k_j / sqrt(128) over cache rows j = 0..P, a softmax
// in fp32 and the weighted sum of the value rows; KV head g = h / 4 serves
// query heads 4g..4g+3 (repeat_kv). Grouping is what makes this step cheap:
// each K/V row is loaded from HBM once for its 4 query heads.
//
// Layout of the work (flash-decoding):
//   grid (split, g, b); split s covers keys [s*chunk, min((s+1)*chunk, P+1)).
//   One producer lane streams 64-key K and V tiles with 4-D TMA loads
//   (128B-swizzled, 3-stage mbarrier ring); each of the 4 warps takes 16 keys
//   of every tile and runs QK^T and PV on mma.sync m16n8k16 with the 4 query
//   heads as the (zero-padded) M = 16 rows, an online softmax in fp32 (base-2
//   exponent, scale folded in) and fp32 accumulators. The warps merge their
//   (max, sum, o) through shared memory; a sequence split over several CTAs
//   writes fp32 partials and the last CTA to take the (b, g) ticket merges
//   them with the log-sum-exp rule and writes the bf16 head outputs.
#include <math.h>

#include "kernels.h"

namespace gqa {

namespace {

constexpr int TILE = 64;                        // keys per stage
constexpr int STAGES = 3;
constexpr int HALF_BYTES = TILE * 128;          // 64 keys x 64 dims x bf16
constexpr int KV_TILE_BYTES = 2 * HALF_BYTES;   // 128 dims
constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;  // K and V
constexpr int THREADS = 128;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 128;
// 1/sqrt(128) * log2(e): scores become base-2 exponents directly.
constexpr float SCALE_LOG2 = 0.08838834764831845f * 1.4426950408889634f;

__device__ __forceinline__ void issue_tile(uint8_t* smem, uint64_t* full, const CUtensorMap* mk,
                                           const CUtensorMap* mv, int i, int pos, int g, int b) {
  const int st = i % STAGES;
  const uint32_t fb = smem_u32(&full[st]);
  const uint32_t base = smem_u32(smem + st * STAGE_BYTES);
  mbar_expect_tx(fb, STAGE_BYTES);
  tma_load_4d(base, mk, fb, 0, g, pos, b);
  tma_load_4d(base + HALF_BYTES, mk, fb, 64, g, pos, b);
  tma_load_4d(base + KV_TILE_BYTES, mv, fb, 0, g, pos, b);
  tma_load_4d(base + KV_TILE_BYTES + HALF_BYTES, mv, fb, 64, g, pos, b);
}

__global__ void __launch_bounds__(THREADS, 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                       DecodeAttnParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  int* sflag = reinterpret_cast<int*>(empty + STAGES);  // [0] abort, [1] ticket, [2] issued

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;

  const int P = a.sp.get(b);
  if (!a.sp.ok(P)) {
    if (split == 0 && g == 0 && threadIdx.x == 0) report(a.status, DEV_BAD_POSITION);
    return;
  }
  const int L = P + 1;
  const int nsplit_b = (L + a.chunk - 1) / a.chunk;
  if (split >= nsplit_b) return;
  const int k0 = split * a.chunk;
  const int k1 = min(L, k0 + a.chunk);
  const int ntiles = (k1 - k0 + TILE - 1) / TILE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), THREADS / 32);
    }
    sflag[0] = 0;
    fence_barrier_init();
    const int first = min(STAGES, ntiles);
    for (int i = 0; i < first; ++i) issue_tile(smem, full, &mk, &mv, i, k0 + i * TILE, g, b);
    sflag[2] = first;
  }

  // A operand of QK^T: rows = the 4 query heads of group g (rows 4..15 zero),
  // cols = head dims; qa[ks] = {cols 2t,2t+1 ; cols 2t+8,2t+9} of k-step ks.
  uint32_t qa[8][2];
  {
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(a.q + static_cast<size_t>(b) * D_MODEL +
                                                            static_cast<size_t>(g * N_REP + (gr & 3)) * HEAD_DIM);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = gr < N_REP ? q32[ks * 8 + t] : 0u;
      qa[ks][1] = gr < N_REP ? q32[ks * 8 + 4 + t] : 0u;
    }
  }
  __syncthreads();

  float m_run = -INFINITY, l_run = 0.f;
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
    const uint32_t kt = smem_u32(smem + st * STAGE_BYTES);
    const uint32_t vt = kt + KV_TILE_BYTES;
    const int key_w = k0 + i * TILE + warp * 16;  // first key of this warp

    float sc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
      const int r = warp * 16 + j * 8 + (lane & 7);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int ch = 4 * c + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + (ch >> 3) * HALF_BYTES + sw128(r, ch & 7), b0, b1, b2, b3);
        mma16816(sc[j], qa[2 * c][0], 0u, qa[2 * c][1], 0u, b0, b1);
        mma16816(sc[j], qa[2 * c + 1][0], 0u, qa[2 * c + 1][1], 0u, b2, b3);
      }
    }

    // online softmax for row gr (keys key_w + 8j + 2t + e)
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key_w + 8 * j + 2 * t + e;
        const float v = key < k1 ? sc[j][e] * SCALE_LOG2 : -INFINITY;
        sc[j][e] = v;
        mx = fmaxf(mx, v);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);
    float p[2][2];
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[j][e] = exp2f(sc[j][e] - m_use);
        psum += p[j][e];
      }
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      oacc[nt][0] *= alpha;
      oacc[nt][1] *= alpha;
    }
    const bool real_row = gr < N_REP;
    const uint32_t pa0 = real_row ? pack_bf16(p[0][0], p[0][1]) : 0u;
    const uint32_t pa2 = real_row ? pack_bf16(p[1][0], p[1][1]) : 0u;

    // zero value rows past the range in a ragged tile (they may hold anything)
    uint32_t mask_a = 0xffffffffu, mask_b = 0xffffffffu;
    if (key_w + 16 > k1) {
      const int ka = key_w + 2 * t, kb = ka + 8;
      mask_a = (ka < k1 ? 0x0000ffffu : 0u) | (ka + 1 < k1 ? 0xffff0000u : 0u);
      mask_b = (kb < k1 ? 0x0000ffffu : 0u) | (kb + 1 < k1 ? 0xffff0000u : 0u);
    }
    const int vr = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      const int ch = 2 * dp + (lane >> 4);
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vt + (ch >> 3) * HALF_BYTES + sw128(vr, ch & 7), v0, v1, v2, v3);
      mma16816(oacc[2 * dp], pa0, 0u, pa2, 0u, v0 & mask_a, v1 & mask_b);
      mma16816(oacc[2 * dp + 1], pa0, 0u, pa2, 0u, v2 & mask_a, v3 & mask_b);
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    if (threadIdx.x == 0 && i + STAGES < ntiles) {
      if (mbar_wait(smem_u32(&empty[st]), ph)) {
        issue_tile(smem, full, &mk, &mv, i + STAGES, k0 + (i + STAGES) * TILE, g, b);
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

  // merge the 4 warps of this CTA (pipeline buffers are free now)
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  float* wml = reinterpret_cast<float*>(smem);  // [warp][head][2]
  float* wo = wml + 32;                         // [warp][head][128]
  if (gr < N_REP) {
    if (t == 0) {
      wml[(warp * 4 + gr) * 2] = m_run;
      wml[(warp * 4 + gr) * 2 + 1] = l_run;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      *reinterpret_cast<float2*>(&wo[(warp * 4 + gr) * 128 + nt * 8 + 2 * t]) = make_float2(oacc[nt][0], oacc[nt][1]);
    }
  }
  __syncthreads();
  const int hh = threadIdx.x >> 5;  // head within the group
  const int d0 = lane * 4;
  float mmax = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) mmax = fmaxf(mmax, wml[(w * 4 + hh) * 2]);
  float lsum = 0.f;
  float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float mw = wml[(w * 4 + hh) * 2];
    const float sc = mw == -INFINITY ? 0.f : exp2f(mw - mmax);
    lsum += wml[(w * 4 + hh) * 2 + 1] * sc;
    const float4 ov = *reinterpret_cast<const float4*>(&wo[(w * 4 + hh) * 128 + d0]);
    o4[0] += ov.x * sc;
    o4[1] += ov.y * sc;
    o4[2] += ov.z * sc;
    o4[3] += ov.w * sc;
  }
  __nv_bfloat16* out = a.o + static_cast<size_t>(b) * D_MODEL + static_cast<size_t>(g * N_REP + hh) * HEAD_DIM + d0;
  if (nsplit_b == 1) {
    const float inv = 1.f / lsum;
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(o4[0] * inv, o4[1] * inv), pack_bf16(o4[2] * inv, o4[3] * inv));
    return;
  }

  // split: publish the partial, take a ticket, the last CTA merges
  const size_t bg = static_cast<size_t>(b) * N_KV + g;
  const size_t pidx = (bg * a.nsplit + split) * N_REP + hh;
  __stcg(reinterpret_cast<float4*>(a.part_o + pidx * HEAD_DIM + d0), make_float4(o4[0], o4[1], o4[2], o4[3]));
  if (lane == 0) __stcg(reinterpret_cast<float2*>(a.part_ml + pidx * 2), make_float2(mmax, lsum));
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sflag[1] = atomicAdd(a.tickets + bg, 1);
  __syncthreads();
  if (sflag[1] != nsplit_b - 1) return;
  __threadfence();
  float gmax = -INFINITY;
  for (int s = 0; s < nsplit_b; ++s) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + ((bg * a.nsplit + s) * N_REP + hh) * 2));
    gmax = fmaxf(gmax, ml.x);
  }
  float gl = 0.f;
  float go[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < nsplit_b; ++s) {
    const size_t q = (bg * a.nsplit + s) * N_REP + hh;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + q * 2));
    const float sc = exp2f(ml.x - gmax);
    gl += ml.y * sc;
    const float4 ov = __ldcg(reinterpret_cast<const float4*>(a.part_o + q * HEAD_DIM + d0));
    go[0] += ov.x * sc;
    go[1] += ov.y * sc;
    go[2] += ov.z * sc;
    go[3] += ov.w * sc;
  }
  const float inv = 1.f / gl;
  *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(go[0] * inv, go[1] * inv), pack_bf16(go[2] * inv, go[3] * inv));
  if (threadIdx.x == 0) a.tickets[bg] = 0;
}

}  // namespace

int decode_chunk(int B, int max_keys, int num_sms) {
  // aim for about four CTAs per SM of a 152-SM part, at most 2048 keys (1 MB of K+V) each
  const long long target = 4LL * num_sms;
  const long long work = static_cast<long long>(B) * N_KV * max_keys;
  long long chunk = (work + target - 1) / target;
  chunk = ((chunk + TILE - 1) / TILE) * TILE;
  if (chunk < TILE) chunk = TILE;
  if (chunk > 2048) chunk = 2048;
  return static_cast<int>(chunk);
}

cudaError_t launch_attn_decode(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeAttnParams& a,
                               cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const dim3 grid(a.nsplit, N_KV, a.B);
  attn_decode_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(mk, mv, a);
  return cudaGetLastError();
}

}  // namespace gqa
