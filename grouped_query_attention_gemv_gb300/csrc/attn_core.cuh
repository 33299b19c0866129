// Decode attention (one new token per sequence) over the KV cache: the
// device-side phase shared by the standalone kernel (attn_decode.cu) and the
// fused decode kernel (decode_fused.cu).
//
// "Llama 3.1 8B · Grouped-query attention" (mode decode): for every query
// head h the scores q_h . k_j / sqrt(128) over cache rows j = 0..P, a softmax
// in fp32 and the weighted sum of the value rows; KV head g = h / 4 serves
// query heads 4g..4g+3 (repeat_kv). Grouping is what makes this step cheap:
// each K/V row is loaded from HBM once for its 4 query heads.
//
// Work decomposition (persistent, stream-K over position chunks):
//   * the cache rows of every sequence are cut into 16-position units; all
//     units of the batch, in (b, chunk) order, are split into equal contiguous
//     ranges, one per CTA (one CTA per SM), so every SM streams the same bytes
//     whatever the mix of sequence lengths;
//   * a producer warp fetches each unit for all 8 KV heads at once: a TMA box
//     of 16 positions x 8 heads x 64 dims over a transposed view of the cache
//     (K and V, two halves each: 64 KB per unit, 3-stage mbarrier ring), so
//     every 2 KB position row is read in one burst;
//   * compute warp g (of 8) owns KV head g: QK^T and PV on mma.sync m16n8k16
//     with its 4 query heads as the (zero-padded) M = 16 rows, online softmax
//     in fp32 (base-2, scale folded in);
//   * a sequence wholly inside one CTA's range is finished in registers; one
//     split between CTAs leaves fp32 partials (max, sum, o) in two slots per
//     CTA, and the CTA whose ticket completes the sequence merges them with
//     the log-sum-exp rule in CTA order (deterministic). Nothing waits on
//     another CTA;
//   * units are requested before `gate` (the queries and the new rows may
//     still be in the making) except a sequence's last unit, which holds the
//     row the projection writes; queries are read after it.
#pragma once

#include <math.h>

#include "kernels.h"

namespace gqa {
namespace attnk {

constexpr int UNIT = DECODE_UNIT;              // positions per unit (= TMA box height)
constexpr int STAGES = 3;
constexpr int BOX_BYTES = UNIT * N_KV * 128;   // 16 positions x 8 heads x 64 dims x bf16 = 16 KB
constexpr int UNIT_BYTES = 4 * BOX_BYTES;      // K lo | K hi | V lo | V hi
constexpr int RING = STAGES * UNIT_BYTES;
constexpr int HEAD_BYTES = UNIT * 128;         // one head's slice of a box
constexpr int COMPUTE_WARPS = N_KV;            // warps 0..7; warp 8 is the producer
constexpr float SCALE_LOG2 = 0.08838834764831845f * 1.4426950408889634f;

struct Cursor {
  int b, j;  // sequence, unit within it
};

__device__ __forceinline__ int units_of(const int* pre, int b) { return pre[b + 1] - pre[b]; }

__device__ __forceinline__ void advance(Cursor& c, const int* pre, int B) {
  if (++c.j < units_of(pre, c.b)) return;
  c.j = 0;
  do {
    ++c.b;
  } while (c.b < B && units_of(pre, c.b) == 0);
}

__device__ __forceinline__ Cursor locate(long long u, const int* pre, int B) {
  int lo = 0, hi = B - 1;  // largest b with pre[b] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= u) lo = mid; else hi = mid - 1;
  }
  while (units_of(pre, lo) == 0) ++lo;
  return Cursor{lo, static_cast<int>(u - pre[lo])};
}

__device__ __forceinline__ int cta_of(long long u, long long U, long long C) {
  return static_cast<int>(((u + 1) * C + U - 1) / U) - 1;
}
__device__ __forceinline__ long long range_start(long long c, long long U, long long C) { return U * c / C; }

// Units per sequence prefix-summed into pre[0..B]; returns (on every lane) the
// number of sequences with a valid start position. Run by one whole warp.
__device__ __forceinline__ int build_prefix(const DecodeAttnParams& a, int* pre) {
  const int lane = threadIdx.x & 31;
  int run = 0, valid = 0;
  if (lane == 0) pre[0] = 0;
  for (int base = 0; base < a.B; base += 32) {
    const int b = base + lane;
    int v = 0;
    if (b < a.B) {
      const int P = a.sp.get(b);
      if (a.sp.ok(P)) v = (P + 1 + UNIT - 1) / UNIT;
      else if (blockIdx.x == 0) report(a.status, DEV_BAD_POSITION);
    }
    valid += __popc(__ballot_sync(0xffffffffu, v > 0));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += x;
    }
    if (b < a.B) pre[b + 1] = run + v;
    run += __shfl_sync(0xffffffffu, v, 31);
  }
  return valid;
}

// AND of `v` over the 256 compute threads, with a barrier: the compute warps
// always take the same branch, so none is left alone at a later barrier.
__device__ __forceinline__ bool compute_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 3, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

struct Shared {
  uint8_t* ring;    // RING bytes, 1024-aligned
  uint64_t* full;   // [STAGES], count 1
  uint64_t* empty;  // [STAGES], count COMPUTE_WARPS
  int* flags;       // [0] abort, [1] ticket, [2] issued
  const int* pre;   // [B + 1] from build_prefix
};

// This CTA's range of units. Roles: warps 0..7 compute (KV head = warp), warp 8
// lane 0 produces. gate_lane() is called by the producer lane before the units
// that need the projection's output, gate_warp() by every lane of each compute
// warp before it reads queries; false = give up. seq_done(b) runs on thread 0
// once sequence b's attention output is written.
template <class GateLane, class GateWarp, class SeqDone>
__device__ __forceinline__ void attn_phase(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeAttnParams& a,
                                           const Shared& sh, GateLane gate_lane, GateWarp gate_warp,
                                           SeqDone seq_done) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B;
  const int* pre = sh.pre;
  int* flags = sh.flags;
  const long long U = pre[B];
  const long long C = gridDim.x;
  const long long u0 = range_start(blockIdx.x, U, C), u1 = range_start(blockIdx.x + 1, U, C);
  const int n = static_cast<int>(u1 - u0);
  if (n <= 0) return;

  if (warp == COMPUTE_WARPS) {
    if (lane != 0) return;
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    Cursor iss = locate(u0, pre, B);
    auto issue = [&](int i) {
      const int s = i % STAGES;
      const uint32_t dst = smem_u32(sh.ring + s * UNIT_BYTES);
      const uint32_t fb = smem_u32(&sh.full[s]);
      const int pos = iss.j * UNIT;
      mbar_expect_tx(fb, UNIT_BYTES);
      tma_load_4d(dst, &mk, fb, 0, pos, 0, iss.b);
      tma_load_4d(dst + BOX_BYTES, &mk, fb, 64, pos, 0, iss.b);
      tma_load_4d(dst + 2 * BOX_BYTES, &mv, fb, 0, pos, 0, iss.b);
      tma_load_4d(dst + 3 * BOX_BYTES, &mv, fb, 64, pos, 0, iss.b);
      advance(iss, pre, B);
    };
    int i = 0;
    // before the gate: units that do not hold a sequence's new row
    while (i < n && i < STAGES && iss.j + 1 < units_of(pre, iss.b)) issue(i++);
    bool ok = gate_lane();
    for (; ok && i < n; ++i) {
      if (i >= STAGES && !mbar_wait(smem_u32(&sh.empty[i % STAGES]), ((i / STAGES) & 1) ^ 1)) {
        ok = false;
        break;
      }
      issue(i);
    }
    if (!ok) atomicExch(&flags[0], 1);
    flags[2] = i;
    return;
  }
  if (warp > COMPUTE_WARPS) return;

  if (!compute_all(gate_warp())) {
    if (lane == 0) atomicExch(&flags[0], 1);
    return;
  }
  const int g = warp;               // KV head of this warp
  const int gr = lane >> 2, t = lane & 3;
  const bool real_row = gr < N_REP;
  Cursor cur = locate(u0, pre, B);
  uint32_t qa[8][2];
  float m_run = -INFINITY, l_run = 0.f;
  float oacc[16][4];
  int seg_units = 0;
  long long seg_start = u0;

  for (int i = 0; i < n; ++i) {
    const long long u = u0 + i;
    const int L = a.sp.get(cur.b) + 1;
    if (i == 0 || cur.j == 0) {
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(
          a.q + static_cast<size_t>(cur.b) * D_MODEL + static_cast<size_t>(g * N_REP + (gr & 3)) * HEAD_DIM);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = real_row ? q32[ks * 8 + t] : 0u;
        qa[ks][1] = real_row ? q32[ks * 8 + 4 + t] : 0u;
      }
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;
      seg_units = 0;
      seg_start = u;
    }
    const int s = i % STAGES;
    const bool landed = mbar_wait(smem_u32(&sh.full[s]), (i / STAGES) & 1);
    if (!compute_all(landed && !*reinterpret_cast<volatile int*>(&flags[0]))) {
      if (lane == 0) atomicExch(&flags[0], 1);
      break;
    }
    // this warp's head inside the four boxes: rows g*16 + r (r = key within the unit)
    const uint32_t kt = smem_u32(sh.ring + s * UNIT_BYTES) + g * HEAD_BYTES;
    const uint32_t vt = kt + 2 * BOX_BYTES;
    const int key0 = cur.j * UNIT;

    float sc[2][4];
#pragma unroll
    for (int jn = 0; jn < 2; ++jn) {
      sc[jn][0] = sc[jn][1] = sc[jn][2] = sc[jn][3] = 0.f;
      const int r = jn * 8 + (lane & 7);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int ch = 4 * c + (lane >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + (ch >> 3) * BOX_BYTES + sw128(r, ch & 7), b0, b1, b2, b3);
        mma16816(sc[jn], qa[2 * c][0], 0u, qa[2 * c][1], 0u, b0, b1);
        mma16816(sc[jn], qa[2 * c + 1][0], 0u, qa[2 * c + 1][1], 0u, b2, b3);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int jn = 0; jn < 2; ++jn) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + 8 * jn + 2 * t + e;
        const float v = key < L ? sc[jn][e] * SCALE_LOG2 : -INFINITY;
        sc[jn][e] = v;
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
    for (int jn = 0; jn < 2; ++jn) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        p[jn][e] = exp2f(sc[jn][e] - m_use);
        psum += p[jn][e];
      }
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      oacc[nt][0] *= alpha;
      oacc[nt][1] *= alpha;
    }
    const uint32_t pa0 = real_row ? pack_bf16(p[0][0], p[0][1]) : 0u;
    const uint32_t pa2 = real_row ? pack_bf16(p[1][0], p[1][1]) : 0u;
    uint32_t mask_a = 0xffffffffu, mask_b = 0xffffffffu;
    if (key0 + UNIT > L) {  // value rows past the sequence may hold anything
      const int ka = key0 + 2 * t, kb = ka + 8;
      mask_a = (ka < L ? 0x0000ffffu : 0u) | (ka + 1 < L ? 0xffff0000u : 0u);
      mask_b = (kb < L ? 0x0000ffffu : 0u) | (kb + 1 < L ? 0xffff0000u : 0u);
    }
    const int vr = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      const int ch = 2 * dp + (lane >> 4);
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vt + (ch >> 3) * BOX_BYTES + sw128(vr, ch & 7), v0, v1, v2, v3);
      mma16816(oacc[2 * dp], pa0, 0u, pa2, 0u, v0 & mask_a, v1 & mask_b);
      mma16816(oacc[2 * dp + 1], pa0, 0u, pa2, 0u, v2 & mask_a, v3 & mask_b);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
    ++seg_units;

    const Cursor here = cur;
    advance(cur, pre, B);
    if (i + 1 < n && cur.j != 0) continue;

    // ---- end of this CTA's part of sequence `here.b`
    float lsum = l_run;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    const int nu = units_of(pre, here.b);
    __nv_bfloat16* out = a.o + static_cast<size_t>(here.b) * D_MODEL + static_cast<size_t>(g * N_REP) * HEAD_DIM;
    if (seg_units == nu) {
      if (real_row) {
        const float inv = 1.f / lsum;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          *reinterpret_cast<uint32_t*>(out + gr * HEAD_DIM + nt * 8 + 2 * t) =
              pack_bf16(oacc[nt][0] * inv, oacc[nt][1] * inv);
      }
      fence_proxy_async_global();  // a later phase of the same grid reads o by TMA
      __threadfence();
      asm volatile("bar.sync 2, 256;" ::: "memory");   // the 8 compute warps
      if (threadIdx.x == 0) seq_done(here.b);
      continue;
    }
    const long long slot = (2LL * blockIdx.x + (seg_start == u0 ? 0 : 1)) * N_KV + g;
    if (real_row) {
      float* po = a.part_o + (slot * N_REP + gr) * HEAD_DIM;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt)
        __stcg(reinterpret_cast<float2*>(po + nt * 8 + 2 * t), make_float2(oacc[nt][0], oacc[nt][1]));
      if (t == 0) __stcg(reinterpret_cast<float2*>(a.part_ml + (slot * N_REP + gr) * 2), make_float2(m_run, lsum));
    }
    __threadfence();
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (threadIdx.x == 0) flags[1] = atomicAdd(a.tickets + here.b, seg_units);
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (flags[1] + seg_units != nu) continue;

    // last contribution to sequence here.b: warp g merges KV head g over every CTA's slot
    __threadfence();
    const long long ub = pre[here.b];
    const int cf = cta_of(ub, U, C), cl = cta_of(ub + nu - 1, U, C);
    const int hh = lane >> 3;        // query head within the group
    const int d0 = (lane & 7) * 16;  // 16 dims per lane
    float gmax = -INFINITY;
    for (int cc = cf; cc <= cl; ++cc) {
      const long long sl = (2LL * cc + (range_start(cc, U, C) >= ub ? 0 : 1)) * N_KV + g;
      gmax = fmaxf(gmax, __ldcg(a.part_ml + (sl * N_REP + hh) * 2));
    }
    float gl = 0.f;
    float go[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) go[e] = 0.f;
    for (int cc = cf; cc <= cl; ++cc) {
      const long long sl = (2LL * cc + (range_start(cc, U, C) >= ub ? 0 : 1)) * N_KV + g;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + (sl * N_REP + hh) * 2));
      const float sc2 = exp2f(ml.x - gmax);
      gl += ml.y * sc2;
      const float4* po = reinterpret_cast<const float4*>(a.part_o + (sl * N_REP + hh) * HEAD_DIM + d0);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 v = __ldcg(po + e);
        go[4 * e] += v.x * sc2;
        go[4 * e + 1] += v.y * sc2;
        go[4 * e + 2] += v.z * sc2;
        go[4 * e + 3] += v.w * sc2;
      }
    }
    const float inv = 1.f / gl;
    uint4 lo, hi2;
    lo.x = pack_bf16(go[0] * inv, go[1] * inv);
    lo.y = pack_bf16(go[2] * inv, go[3] * inv);
    lo.z = pack_bf16(go[4] * inv, go[5] * inv);
    lo.w = pack_bf16(go[6] * inv, go[7] * inv);
    hi2.x = pack_bf16(go[8] * inv, go[9] * inv);
    hi2.y = pack_bf16(go[10] * inv, go[11] * inv);
    hi2.z = pack_bf16(go[12] * inv, go[13] * inv);
    hi2.w = pack_bf16(go[14] * inv, go[15] * inv);
    reinterpret_cast<uint4*>(out + hh * HEAD_DIM + d0)[0] = lo;
    reinterpret_cast<uint4*>(out + hh * HEAD_DIM + d0)[1] = hi2;
    fence_proxy_async_global();
    __threadfence();
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (threadIdx.x == 0) {
      a.tickets[here.b] = 0;
      seq_done(here.b);
    }
  }
}

// After an aborted phase: let loads that were issued but never consumed land
// (bounded). One thread.
__device__ __forceinline__ void attn_drain(const Shared& sh) {
  const int issued = sh.flags[2];
  for (int i = max(0, issued - STAGES); i < issued; ++i) mbar_wait(smem_u32(&sh.full[i % STAGES]), (i / STAGES) & 1);
}

}  // namespace attnk
}  // namespace gqa
