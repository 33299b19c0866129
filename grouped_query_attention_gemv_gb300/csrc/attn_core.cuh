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
//     units of the batch, in (sequence, chunk) order, are split into equal
//     contiguous ranges, one per CTA (one CTA per SM), so every SM streams
//     the same bytes whatever the mix of sequence lengths;
//   * a producer lane fetches each unit for all 8 KV heads at once: TMA boxes
//     of 16 positions x 8 heads x 64 dims over a (dim, position, head,
//     sequence) view of the cache, K and V in two halves each (64 KB per
//     unit, 3 units in flight), so every 2 KB position row is read whole;
//   * compute warp g (of 8) owns KV head g. Its 16 keys go on the M side of
//     mma.sync m16n8k16 and its 4 query heads (padded to 8) on the N side:
//     S^T = K Q^T, online softmax per head in fp32 (base 2, scale folded in),
//     O^T += V^T P^T with P^T moved into B-operand layout by movmatrix: half
//     the tensor instructions of the query-rows-as-M form, whose 16 rows
//     would hold 4 heads;
//   * a sequence wholly inside one CTA's range is finished in registers; one
//     split between CTAs leaves an fp32 partial (running max, sum, o) in one
//     of the CTA's two slots;
//   * after every CTA's last unit the grid meets once (a counter), and every
//     warp of the grid merges one (sequence, query head) of the split
//     sequences over its slots by the log-sum-exp rule, in CTA order
//     (deterministic). All slot loads of a merge are issued together, so the
//     merge costs one round trip however many CTAs shared the sequence;
//   * units are requested before `gate` (the queries and the new rows may
//     still be in the making) except a sequence's last unit, which holds the
//     row the projection writes; queries are read after it.
// The multi-head variant (32 KV heads, one query head each: repeat_kv is the
// identity) runs the same units over groups of 8 KV heads: every sequence
// becomes NG = 4 "virtual sequences" (sequence b, heads 8j..8j+7), so a unit
// is still 16 positions x 8 heads and a warp still owns one KV head. NREP
// (query heads per KV head: 4, or 1 for the multi-head variant) is a
// template parameter of the phase.
#pragma once

#include <math.h>

#include "kernels.h"

namespace gqa {
namespace attnk {

constexpr int UNIT = DECODE_UNIT;             // positions per unit
constexpr int COMPUTE_WARPS = N_KV;           // warps 0..7 (KV head = warp); warp 8 lane 0 produces
constexpr int STAGES = 3;
constexpr int HEAD_BYTES = UNIT * 128;        // one head's 16 positions x 64 dims
constexpr int BOX_BYTES = N_KV * HEAD_BYTES;  // 16 positions x 8 heads x 64 dims = 16 KB
constexpr int UNIT_BYTES = 4 * BOX_BYTES;     // K lo | K hi | V lo | V hi
constexpr int RING = STAGES * UNIT_BYTES;
constexpr int STAGE_OUT_BYTES = COMPUTE_WARPS * N_REP * HEAD_DIM * 4;  // per-warp o staging
constexpr float SCALE_LOG2 = 0.08838834764831845f * 1.4426950408889634f;
constexpr int MERGE_SLOTS = 16;               // slots whose loads are in flight together in a merge
constexpr int PRE_GATE_UNITS = STAGES;        // units requested before the gate (at most STAGES)
constexpr int ITEM_POS = DECODE_ITEM_POS;      // positions per stage of the head-major phase (16 per warp)
static_assert(ITEM_POS == COMPUTE_WARPS * UNIT, "a head-major stage gives every compute warp 16 keys");

struct Cursor {
  int b, j;  // virtual sequence (sequence b / NG, head group b % NG), unit within it
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

// Units split over the grid: CTA c takes units [U c / C, U (c + 1) / C).
// With U >= C every CTA has a unit; with U < C each has at most one.
// Calls are refused unless (units + 1) x (CTAs + 1) < 2^32, so 32-bit
// unsigned arithmetic is exact here (a 64-bit division is a long software
// sequence, and a merge takes one per partial it reads).
__device__ __forceinline__ int cta_of(long long u, long long U, long long C) {
  const uint32_t uu = static_cast<uint32_t>(u), UU = static_cast<uint32_t>(U), CC = static_cast<uint32_t>(C);
  return static_cast<int>(((uu + 1) * CC + UU - 1) / UU) - 1;
}
__device__ __forceinline__ long long range_start(long long c, long long U, long long C) {
  return static_cast<uint32_t>(U) * static_cast<uint32_t>(c) / static_cast<uint32_t>(C);
}

// The CTAs that hold units of a sequence (first unit ub, nu units), in
// order: participant p is cf + p when every CTA has units, else the owner of
// the sequence's p-th unit (one unit per CTA; the CTAs between own none and
// write no partial).
__device__ __forceinline__ int participants(long long ub, int nu, long long U, long long C) {
  return U >= C ? cta_of(ub + nu - 1, U, C) - cta_of(ub, U, C) + 1 : nu;
}
// cf = cta_of(ub): the first participant
__device__ __forceinline__ int participant(long long ub, int cf, int p, long long U, long long C) {
  return U >= C ? cf + p : cta_of(ub + p, U, C);
}

// Units per virtual sequence (NG per sequence) prefix-summed into
// pre[0..B*NG]; returns (on every lane) the number of virtual sequences with a
// valid start position. Run by one whole warp.
template <int NG>
__device__ __forceinline__ int build_prefix(const DecodeAttnParams& a, int* pre) {
  const int lane = threadIdx.x & 31;
  const int VB = a.B * NG;
  int run = 0, valid = 0;
  if (lane == 0) pre[0] = 0;
  for (int base = 0; base < VB; base += 32) {
    const int b = base + lane;
    int v = 0;
    if (b < VB) {
      const int P = a.sp.get(b / NG);
      if (a.sp.ok(P)) v = (P + 1 + UNIT - 1) / UNIT;
      else if (blockIdx.x == 0 && b % NG == 0) report(a.status, DEV_BAD_POSITION);
    }
    valid += __popc(__ballot_sync(0xffffffffu, v > 0));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += x;
    }
    if (b < VB) pre[b + 1] = run + v;
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

// OR of `v` over the 256 compute threads, with a barrier.
__device__ __forceinline__ bool compute_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 3, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

struct Shared {
  uint8_t* ring;     // RING bytes, 1024-aligned
  uint64_t* full;    // [STAGES], count 1
  uint64_t* empty;   // [STAGES], count COMPUTE_WARPS
  int* flags;        // [0] abort, [2] units issued
  const int* pre;    // [B + 1] from build_prefix
  float* stage_out;  // STAGE_OUT_BYTES
};

// One warp's 16 keys of one KV head against its query heads (NREP real,
// padded to 8 on the N side of m16n8k16): S^T = K Q^T, an online-softmax
// update of the running (max, sum) per query head (base 2, scale folded in),
// and O^T += V^T P^T with P^T moved into B-operand layout by movmatrix.
// kt / vt: shared addresses of the keys' K and V rows (dims 0-63; dims 64-127
// one box further, BOX_BYTES), 128-byte swizzled rows; key0: position of the
// first key, L: keys of the sequence (keys >= L are masked). At least one of
// the 16 keys must be below L. qb: Q^T as B fragments; m_run, l_run: running
// max and sum of query heads 2t, 2t+1 (t = lane % 4); oacc: O^T tiles
// (dim 16d + lane/4 (+8), heads 2t, 2t+1).
template <int NREP>
__device__ __forceinline__ void block16(uint32_t kt, uint32_t vt, int key0, int L, const uint32_t (&qb)[8][2],
                                        float (&m_run)[2], float (&l_run)[2], float (&oacc)[8][4]) {
  const int lane = threadIdx.x & 31;
  const int gr = lane >> 2, t = lane & 3;
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(kt + (ks >> 2) * BOX_BYTES + sw128(lane & 15, 2 * (ks & 3) + (lane >> 4)), a0, a1, a2, a3);
    mma16816(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
  }
  // sc: (key gr, heads 2t, 2t+1), (key gr + 8, heads 2t, 2t+1)
  const bool v0 = key0 + gr < L, v1 = key0 + gr + 8 < L;
  sc[0] = v0 ? sc[0] * SCALE_LOG2 : -INFINITY;
  sc[1] = v0 ? sc[1] * SCALE_LOG2 : -INFINITY;
  sc[2] = v1 ? sc[2] * SCALE_LOG2 : -INFINITY;
  sc[3] = v1 ? sc[3] * SCALE_LOG2 : -INFINITY;
  float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);  // finite: key0 < L
  const float al0 = exp2f(m_run[0] - mn0), al1 = exp2f(m_run[1] - mn1);
  const float p0 = exp2f(sc[0] - mn0), p1 = exp2f(sc[1] - mn1);
  const float p2 = exp2f(sc[2] - mn0), p3 = exp2f(sc[3] - mn1);
  float ps0 = p0 + p2, ps1 = p1 + p3;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    ps0 += __shfl_xor_sync(0xffffffffu, ps0, o);
    ps1 += __shfl_xor_sync(0xffffffffu, ps1, o);
  }
  l_run[0] = l_run[0] * al0 + ps0;
  l_run[1] = l_run[1] * al1 + ps1;
  m_run[0] = mn0;
  m_run[1] = mn1;
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    oacc[d][0] *= al0;
    oacc[d][1] *= al1;
    oacc[d][2] *= al0;
    oacc[d][3] *= al1;
  }
  // P^T as the B operand: (head gr, keys 2t, 2t+1) and (head gr, keys 2t+8, 2t+9)
  const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1));
  const uint32_t pb1 = movmatrix_t(pack_bf16(p2, p3));
  uint32_t mask_a = 0xffffffffu, mask_b = 0xffffffffu;
  if (key0 + UNIT > L) {  // value rows past the sequence may hold anything
    const int ka = key0 + 2 * t, kb = ka + 8;
    mask_a = (ka < L ? 0x0000ffffu : 0u) | (ka + 1 < L ? 0xffff0000u : 0u);
    mask_b = (kb < L ? 0x0000ffffu : 0u) | (kb + 1 < L ? 0xffff0000u : 0u);
  }
  const int vr = (lane & 7) + ((lane >> 4) << 3);  // key row of this lane's ldmatrix address
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(vt + (d >> 2) * BOX_BYTES + sw128(vr, 2 * (d & 3) + ((lane >> 3) & 1)), a0, a1, a2, a3);
    mma16816(oacc[d], a0 & mask_a, a1 & mask_a, a2 & mask_b, a3 & mask_b, pb0, pb1);
  }
}

// This CTA's range of units: outputs of the sequences it holds whole,
// partials of the others. Every thread of the CTA calls this. Roles: warps
// 0..7 compute, warp 8 lane 0 produces. gate_lane() is called by the producer
// lane before the units that need the projection's output, gate_warp() by
// every lane of each compute warp before it reads queries; false = give up.
// issued() runs on the producer lane once all its loads are requested.
// Returns false (on the compute threads) when the phase gave up; on return
// every unit is consumed and the ring is free.
template <int NREP, class GateLane, class GateWarp, class Issued>
__device__ __forceinline__ bool attn_units(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeAttnParams& a,
                                           const Shared& sh, GateLane gate_lane, GateWarp gate_warp, Issued issued) {
  constexpr int NG = N_REP / NREP;  // head groups of 8 KV heads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B * NG;           // virtual sequences
  const int* pre = sh.pre;
  int* flags = sh.flags;
  const long long U = pre[B];
  const long long C = gridDim.x;
  const long long u0 = range_start(blockIdx.x, U, C), u1 = range_start(blockIdx.x + 1, U, C);
  const int n = static_cast<int>(u1 - u0);

  if (warp == COMPUTE_WARPS) {
    if (lane != 0 || n <= 0) return true;
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    Cursor iss = locate(u0, pre, B);
    auto issue = [&](int i) {
      const int s = i % STAGES;
      const uint32_t dst = smem_u32(sh.ring + s * UNIT_BYTES);
      const uint32_t fb = smem_u32(&sh.full[s]);
      const int pos = iss.j * UNIT, h0 = (iss.b % NG) * N_KV, sb = iss.b / NG;
      const uint64_t pol = l2_evict_first();
      mbar_expect_tx(fb, UNIT_BYTES);
      tma_load_4d_stream(dst, &mk, fb, 0, pos, h0, sb, pol);
      tma_load_4d_stream(dst + BOX_BYTES, &mk, fb, 64, pos, h0, sb, pol);
      tma_load_4d_stream(dst + 2 * BOX_BYTES, &mv, fb, 0, pos, h0, sb, pol);
      tma_load_4d_stream(dst + 3 * BOX_BYTES, &mv, fb, 64, pos, h0, sb, pol);
      advance(iss, pre, B);
    };
    int i = 0;
    // before the gate: units that do not hold a sequence's new row
    while (i < n && i < PRE_GATE_UNITS && iss.j + 1 < units_of(pre, iss.b)) issue(i++);
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
    if (ok) issued();
    return true;
  }
  if (warp > COMPUTE_WARPS) return true;

  const int g = warp;  // KV head of this warp within its group
  const int gr = lane >> 2, t = lane & 3;
  bool ok = true;
  if (n > 0) ok = compute_all(gate_warp());
  if (n > 0 && ok) {
    Cursor cur = locate(u0, pre, B);
    uint32_t qb[8][2];         // Q^T as B fragments: dims 16s + 2t (+1) | +8, query head gr (0-3 real)
    float m_run[2], l_run[2];  // query heads 2t, 2t+1
    float oacc[8][4];          // O^T tile d: (dim 16d + gr (+8), heads 2t, 2t+1)
    int seg_units = 0;
    long long seg_start = u0;
    float* so = sh.stage_out + g * N_REP * HEAD_DIM;  // this warp's [4][128] staging (NREP rows used)
    for (int i = 0; i < n; ++i) {
      const long long u = u0 + i;
      const int L = a.sp.get(cur.b / NG) + 1;
      if (i == 0 || cur.j == 0) {
        // query heads (8 (b % NG) + g) NREP + 0..NREP-1 of sequence b / NG
        const int qh0 = ((cur.b % NG) * N_KV + g) * NREP;
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(
            a.q + static_cast<size_t>(cur.b / NG) * D_MODEL + static_cast<size_t>(qh0 + (gr % NREP)) * HEAD_DIM);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          qb[s][0] = gr < NREP ? q32[s * 8 + t] : 0u;
          qb[s][1] = gr < NREP ? q32[s * 8 + 4 + t] : 0u;
        }
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d) oacc[d][0] = oacc[d][1] = oacc[d][2] = oacc[d][3] = 0.f;
        seg_units = 0;
        seg_start = u;
      }
      // each warp on its own: no barrier per unit (the merge step makes the
      // outcome uniform)
      const int s = i % STAGES;
      const bool landed = mbar_wait(smem_u32(&sh.full[s]), (i / STAGES) & 1);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) atomicExch(&flags[0], 1);
        ok = false;
        break;
      }
      // this warp's head inside the four boxes: rows g*16 + r (r = key within the unit)
      const uint32_t kt = smem_u32(sh.ring + s * UNIT_BYTES) + g * HEAD_BYTES;
      block16<NREP>(kt, kt + 2 * BOX_BYTES, cur.j * UNIT, L, qb, m_run, l_run, oacc);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
      ++seg_units;

      const Cursor here = cur;
      advance(cur, pre, B);
      if (i + 1 < n && cur.j != 0) continue;

      // ---- end of this CTA's part of sequence here.b: stage o (this warp's 4 heads) as [4][128]
      const bool whole = seg_units == units_of(pre, here.b);
      const float inv0 = whole ? 1.f / l_run[0] : 1.f, inv1 = whole ? 1.f / l_run[1] : 1.f;
      if (t < 2) {
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          float* o0 = so + 2 * t * HEAD_DIM + 16 * d + gr;
          o0[0] = oacc[d][0] * inv0;
          o0[HEAD_DIM] = oacc[d][1] * inv1;
          o0[8] = oacc[d][2] * inv0;
          o0[HEAD_DIM + 8] = oacc[d][3] * inv1;
        }
      }
      __syncwarp();
      // lane -> head lane / 8, dims 16 (lane % 8) .. + 15
      const int hh = lane >> 3, d0 = (lane & 7) * 16;
      const float4* src = reinterpret_cast<const float4*>(so + hh * HEAD_DIM + d0);
      const int qh = ((here.b % NG) * N_KV + g) * NREP + hh;  // query head of this lane's row
      const bool real = hh < NREP;  // rows past NREP: padding of the multi-head variant
      if (whole) {
        if (real) {
          __nv_bfloat16* out = a.o + static_cast<size_t>(here.b / NG) * D_MODEL + static_cast<size_t>(qh) * HEAD_DIM + d0;
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 v = src[e];
            w[2 * e] = pack_bf16(v.x, v.y);
            w[2 * e + 1] = pack_bf16(v.z, v.w);
          }
          reinterpret_cast<uint4*>(out)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(out)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      } else {
        const long long slot = 2LL * blockIdx.x + (seg_start == u0 ? 0 : 1);
        if (real) {
          float4* dst = reinterpret_cast<float4*>(a.part_o + (slot * N_HEADS + g * NREP + hh) * HEAD_DIM + d0);
#pragma unroll
          for (int e = 0; e < 4; ++e) __stcg(dst + e, src[e]);
        }
        // (max, sum) of the warp's query head q is held by the lanes with t = q / 2
        const int srcl = (lane >> 1) & 1;
        const float mq0 = __shfl_sync(0xffffffffu, m_run[0], srcl), mq1 = __shfl_sync(0xffffffffu, m_run[1], srcl);
        const float lq0 = __shfl_sync(0xffffffffu, l_run[0], srcl), lq1 = __shfl_sync(0xffffffffu, l_run[1], srcl);
        if (lane < NREP)
          __stcg(reinterpret_cast<float2*>(a.part_ml + (slot * N_HEADS + g * NREP + lane) * 2),
                 (lane & 1) ? make_float2(mq1, lq1) : make_float2(mq0, lq0));
      }
      __syncwarp();  // the staging area is reused by the next sequence
    }
  }
  // its outputs and partials are out
  fence_proxy_async_global();  // a later phase of the same grid reads o by TMA
  __threadfence();
  return ok;
}

// Head-major decode attention, for a batch whose (sequence, KV head) pairs
// fit the grid one per CTA: CTA c < 8B takes item (b = c / 8, g = c % 8), all
// cache rows 0..P_b of KV head g of sequence b, so no sequence is split
// between CTAs and nothing is merged across them. The producer lane streams
// stages of ITEM_POS positions (boxes of 64 dims x 1 head x 128 positions
// over a (dim, head, position, sequence) view, K and V in two halves each,
// 64 KB per stage); compute warp w takes keys 16w..16w+15 of every stage,
// all against the pair's 4 query heads (the same 16-row tile shape as a
// position-major unit, so block16 serves both). At the end the 8 warps'
// (max, sum, o) states are combined in shared memory by the log-sum-exp rule
// in warp order and o[b, heads 4g..4g+3] written as bf16. The first stages
// (up to the ring's depth) are requested before `gate_lane`, the one holding
// position P_b too, although the projection writes that row concurrently:
// after the gate, the warp whose keys include P_b loads the new K and V rows
// (plain loads, published like the queries) and writes them over the stale
// copy once the stage has landed. Roles, gates and the return value as in
// attn_units; the
// standalone kernel does not use this phase (its queries are ready at launch
// and its batches are larger).
// Stage i occupies ring slot (i + ITEM_ROT) % STAGES: the first stages then
// lie past the ring's first slot, which a preceding projection phase still
// uses for its cross-warp sums after its last weight stage is consumed, so
// attn_items_early can request them during that phase's epilogue. One stage
// (64 KB) lands within the epilogue; a second is still in flight when the
// epilogue publishes its rows, and that release waits for the SM's loads
// (B = 16 at 500-2,000 keys: 0.9 us saved with one, 0.5 us with two).
constexpr int ITEM_ROT = 1;
constexpr int EARLY_ITEMS = 1;
static_assert(EARLY_ITEMS + ITEM_ROT <= STAGES, "early stages fit past the first slot");
__device__ __forceinline__ int item_slot(int i) { return (i + ITEM_ROT) % STAGES; }

// One head-major stage: positions i*ITEM_POS .. +127 of KV head g of sequence
// b, K and V, into its ring slot (producer lane).
__device__ __forceinline__ void item_issue(const CUtensorMap& mk, const CUtensorMap& mv, const Shared& sh, int b,
                                           int g, int i) {
  const int s = item_slot(i);
  const uint32_t dst = smem_u32(sh.ring + s * UNIT_BYTES);
  const uint32_t fb = smem_u32(&sh.full[s]);
  const int pos = i * ITEM_POS;
  const uint64_t pol = l2_evict_first();
  mbar_expect_tx(fb, UNIT_BYTES);
  tma_load_4d_stream(dst, &mk, fb, 0, g, pos, b, pol);
  tma_load_4d_stream(dst + BOX_BYTES, &mk, fb, 64, g, pos, b, pol);
  tma_load_4d_stream(dst + 2 * BOX_BYTES, &mv, fb, 0, g, pos, b, pol);
  tma_load_4d_stream(dst + 3 * BOX_BYTES, &mv, fb, 64, g, pos, b, pol);
}

// Requests this CTA's first head-major stages (at most EARLY_ITEMS) before
// phase B: called by the producer lane once the
// ring's slots past the first are free (every stage of the preceding phase
// consumed, no load of it in flight). Records the count in sh.flags[2], where
// attn_items (same lane) continues and attn_drain looks. Returns the count.
__device__ __forceinline__ int attn_items_early(const CUtensorMap& mk, const CUtensorMap& mv,
                                                const DecodeAttnParams& a, const Shared& sh) {
  const int item = blockIdx.x;
  if (item >= a.B * N_KV) return 0;
  const int b = item / N_KV, g = item % N_KV;
  const int P = a.sp.get(b);
  if (!a.sp.ok(P)) return 0;
  const int n = (P + 1 + ITEM_POS - 1) / ITEM_POS;
  tma_prefetch_desc(&mk);
  tma_prefetch_desc(&mv);
  int i = 0;
  while (i < n && i < EARLY_ITEMS) item_issue(mk, mv, sh, b, g, i++);
  sh.flags[2] = i;
  return i;
}

template <class GateLane, class GateWarp>
__device__ __forceinline__ bool attn_items(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeAttnParams& a,
                                           const Shared& sh, GateLane gate_lane, GateWarp gate_warp) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  if (item >= a.B * N_KV) return true;
  const int b = item / N_KV, g = item % N_KV;
  const int P = a.sp.get(b);
  if (!a.sp.ok(P)) {
    if (g == 0 && threadIdx.x == 0) report(a.status, DEV_BAD_POSITION);
    return true;
  }
  const int L = P + 1;
  const int n = (L + ITEM_POS - 1) / ITEM_POS;
  int* flags = sh.flags;

  if (warp == COMPUTE_WARPS) {
    if (lane != 0) return true;
    tma_prefetch_desc(&mk);
    tma_prefetch_desc(&mv);
    auto issue = [&](int i) { item_issue(mk, mv, sh, b, g, i); };
    int i = flags[2];  // stages attn_items_early requested (0 if none)
    while (i < n && i < PRE_GATE_UNITS) issue(i++);  // row P is put in place after the gate
    bool ok = gate_lane();
    for (; ok && i < n; ++i) {
      if (i >= STAGES && !mbar_wait(smem_u32(&sh.empty[item_slot(i)]), ((i / STAGES) & 1) ^ 1)) {
        ok = false;
        break;
      }
      issue(i);
    }
    if (!ok) atomicExch(&flags[0], 1);
    flags[2] = i;
    return true;
  }
  if (warp > COMPUTE_WARPS) return true;

  const int gr = lane >> 2, t = lane & 3;
  bool ok = compute_all(gate_warp());
  uint32_t qb[8][2];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float oacc[8][4];
#pragma unroll
  for (int d = 0; d < 8; ++d) oacc[d][0] = oacc[d][1] = oacc[d][2] = oacc[d][3] = 0.f;
  if (ok) {
    // query heads 4g + gr (gr < 4; rows 4-7 of the N tile are padding)
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(
        a.q + static_cast<size_t>(b) * D_MODEL + static_cast<size_t>(g * N_REP + (gr % N_REP)) * HEAD_DIM);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      qb[s][0] = gr < N_REP ? q32[s * 8 + t] : 0u;
      qb[s][1] = gr < N_REP ? q32[s * 8 + 4 + t] : 0u;
    }
    // the new row P: lane l holds 16 bytes of box l / 8 (K lo, K hi, V lo,
    // V hi), chunk l % 8; the warp whose keys include P writes it into stage
    // P / ITEM_POS, which may have been read before the projection wrote it
    const int iP = P / ITEM_POS, rP = P % ITEM_POS;
    const bool ownP = rP / UNIT == warp;
    const int bx = lane >> 3, ch = lane & 7;
    uint4 rowP = make_uint4(0u, 0u, 0u, 0u);
    if (ownP) {
      const __nv_bfloat16* src = (bx < 2 ? a.cache_k : a.cache_v) +
                                 (static_cast<size_t>(b) * a.s_max + P) * (N_KV * HEAD_DIM) + g * HEAD_DIM +
                                 (bx & 1) * 64 + ch * 8;
      rowP = *reinterpret_cast<const uint4*>(src);
    }
    for (int i = 0; i < n; ++i) {
      const int s = item_slot(i);
      const bool landed = mbar_wait(smem_u32(&sh.full[s]), (i / STAGES) & 1);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) atomicExch(&flags[0], 1);
        ok = false;
        break;
      }
      if (i == iP && ownP) {  // warp-uniform
        st_shared_v4(smem_u32(sh.ring + s * UNIT_BYTES + bx * BOX_BYTES) + sw128(rP, ch), rowP);
        fence_proxy_async_smem();  // before any later TMA write into this slot
        __syncwarp();
      }
      const int key0 = i * ITEM_POS + warp * UNIT;
      if (key0 < L) {  // warp-uniform: a warp whose keys all lie past the sequence skips the stage
        const uint32_t kt = smem_u32(sh.ring + s * UNIT_BYTES) + warp * HEAD_BYTES;
        block16<N_REP>(kt, kt + 2 * BOX_BYTES, key0, L, qb, m_run, l_run, oacc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
    }
  }
  ok = compute_all(ok);
  if (ok) {
    // stage the warp's unnormalised o [4 heads][128] and (max, sum) per head;
    // every stage is consumed, so the ring's first bytes hold the (max, sum)
    float* so = sh.stage_out + warp * N_REP * HEAD_DIM;
    float* ml = reinterpret_cast<float*>(sh.ring);  // [8 warps][4 heads][2]
    if (t < 2) {
#pragma unroll
      for (int d = 0; d < 8; ++d) {
        float* o0 = so + 2 * t * HEAD_DIM + 16 * d + gr;
        o0[0] = oacc[d][0];
        o0[HEAD_DIM] = oacc[d][1];
        o0[8] = oacc[d][2];
        o0[HEAD_DIM + 8] = oacc[d][3];
      }
      if (gr == 0) {
        ml[(warp * N_REP + 2 * t) * 2] = m_run[0];
        ml[(warp * N_REP + 2 * t) * 2 + 1] = l_run[0];
        ml[(warp * N_REP + 2 * t + 1) * 2] = m_run[1];
        ml[(warp * N_REP + 2 * t + 1) * 2 + 1] = l_run[1];
      }
    }
    asm volatile("bar.sync 3, 256;" ::: "memory");
    // thread -> query head hh, dims d2, d2 + 1; warp 0 always holds key 0, so M is finite.
    // Warps past the first nw hold no key (max -inf, sum 0, o 0): their
    // terms are exact zeros and are skipped
    const int hh = threadIdx.x >> 6, d2 = (threadIdx.x & 63) * 2;
    const int nw = min(COMPUTE_WARPS, (L + UNIT - 1) / UNIT);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < COMPUTE_WARPS; ++w)
      if (w < nw) M = fmaxf(M, ml[(w * N_REP + hh) * 2]);
    float den = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < COMPUTE_WARPS; ++w) {
      if (w < nw) {
        const float f = exp2f(ml[(w * N_REP + hh) * 2] - M);
        den += f * ml[(w * N_REP + hh) * 2 + 1];
        const float2 v = *reinterpret_cast<const float2*>(sh.stage_out + (w * N_REP + hh) * HEAD_DIM + d2);
        o0 += f * v.x;
        o1 += f * v.y;
      }
    }
    const float inv = 1.f / den;
    *reinterpret_cast<uint32_t*>(a.o + static_cast<size_t>(b) * D_MODEL + static_cast<size_t>(g * N_REP + hh) * HEAD_DIM +
                                 d2) = pack_bf16(o0 * inv, o1 * inv);
  }
  // its output is out: a later phase of the same grid reads o by TMA, after
  // the caller's release on one thread behind a CTA barrier (it covers every
  // thread's stores; see the caller)
  fence_proxy_async_global();
  return ok;
}

// The merges, after every CTA's units: the grid meets once on `meet` (a
// zero-filled counter, left equal to the grid size: the caller resets it),
// then every warp merges one (sequence, query head) of the split sequences.
// Called by the 256 compute threads of every CTA with `ok` from attn_units
// (a CTA that gave up still meets, so that no other CTA waits in vain).
// When no CTA boundary falls inside a sequence (every sequence was finished
// whole by one CTA: a small batch of short sequences) there is nothing to
// merge and the grid does not meet.
// Returns false when any thread of the CTA gave up or the meeting timed out.
template <int NREP>
__device__ __forceinline__ bool attn_merge(const DecodeAttnParams& a, const Shared& sh, int* meet, bool ok) {
  constexpr int NG = N_REP / NREP;   // virtual sequences per sequence
  constexpr int HV = N_HEADS / NG;   // query heads of one virtual sequence
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B * NG;
  const int* pre = sh.pre;
  int* flags = sh.flags;
  const long long U = pre[B];
  const long long C = gridDim.x;
  const bool all_ok = compute_all(ok);
  bool cut = false;  // a CTA boundary inside a sequence: its partials need merging
  for (long long c = threadIdx.x + 1; c < C; c += COMPUTE_WARPS * 32) {
    const long long u = range_start(c, U, C);
    if (u > 0 && u < U) cut = cut || locate(u, pre, B).j != 0;
  }
  if (!compute_any(cut)) {
    if (!all_ok && lane == 0) atomicExch(&flags[0], 1);
    return all_ok;
  }
  if (threadIdx.x == 0) {
    atomicAdd(meet, 1);
    flags[3] = wait_counter(meet, static_cast<int>(C), a.wait_ns) ? 1 : 0;
  }
  asm volatile("bar.sync 2, 256;" ::: "memory");
  if (!all_ok || flags[3] == 0) {
    if (lane == 0) atomicExch(&flags[0], 1);
    return false;
  }
  // merges: one warp per (virtual sequence, query head) of every split one,
  // spread over the SMs first (warp w of CTA c takes task w * C + c)
  const int hh4 = lane * 4;  // dims of this lane
  for (long long task = static_cast<long long>(warp) * C + blockIdx.x; task < static_cast<long long>(B) * HV;
       task += C * COMPUTE_WARPS) {
    const int b = static_cast<int>(task / HV), h = static_cast<int>(task % HV);
    const int nu = units_of(pre, b);
    if (nu == 0) continue;
    const long long ub = pre[b];
    const int np = participants(ub, nu, U, C), cf = cta_of(ub, U, C);
    if (np == 1) continue;  // finished by its CTA
    float GM = -INFINITY, GL = 0.f;
    float4 go = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < np; p0 += MERGE_SLOTS) {
      float2 mlv[MERGE_SLOTS];
      float4 ov[MERGE_SLOTS];
#pragma unroll
      for (int k = 0; k < MERGE_SLOTS; ++k) {
        if (p0 + k < np) {
          const int cc = participant(ub, cf, p0 + k, U, C);
          const long long sl = 2LL * cc + (range_start(cc, U, C) >= ub ? 0 : 1);
          mlv[k] = __ldcg(reinterpret_cast<const float2*>(a.part_ml + (sl * N_HEADS + h) * 2));
          ov[k] = __ldcg(reinterpret_cast<const float4*>(a.part_o + (sl * N_HEADS + h) * HEAD_DIM + hh4));
        } else {
          mlv[k] = make_float2(-INFINITY, 0.f);
          ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < MERGE_SLOTS; ++k) {
        if (mlv[k].x == -INFINITY) continue;
        const float mn = fmaxf(GM, mlv[k].x);
        const float sa = GM == -INFINITY ? 0.f : exp2f(GM - mn), sb = exp2f(mlv[k].x - mn);
        GL = GL * sa + mlv[k].y * sb;
        go.x = go.x * sa + ov[k].x * sb;
        go.y = go.y * sa + ov[k].y * sb;
        go.z = go.z * sa + ov[k].z * sb;
        go.w = go.w * sa + ov[k].w * sb;
        GM = mn;
      }
    }
    const float inv = 1.f / GL;
    __nv_bfloat16* out = a.o + static_cast<size_t>(b / NG) * D_MODEL + static_cast<size_t>((b % NG) * HV + h) * HEAD_DIM + hh4;
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(go.x * inv, go.y * inv), pack_bf16(go.z * inv, go.w * inv));
  }
  fence_proxy_async_global();
  __threadfence();
  asm volatile("bar.sync 2, 256;" ::: "memory");
  return true;
}

// After an aborted phase: let loads that were issued but never consumed land
// (bounded). One thread. `rot`: the split's slot rotation (ITEM_ROT for the
// head-major stages, 0 for position-major units).
__device__ __forceinline__ void attn_drain(const Shared& sh, int rot = 0) {
  const int issued = sh.flags[2];
  for (int i = max(0, issued - STAGES); i < issued; ++i)
    mbar_wait(smem_u32(&sh.full[(i + rot) % STAGES]), (i / STAGES) & 1);
}

}  // namespace attnk
}  // namespace gqa
