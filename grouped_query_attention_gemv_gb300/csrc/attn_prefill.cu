// Causal prefill attention on the 5th-generation tensor cores. Query t
// (position start_pos + t) of head h attends to cache rows 0..start_pos+t of
// KV head h / 4 ("Llama 3.1 8B · Grouped-query attention": the mask of
// Transformer.forward is -inf above the diagonal, left-padded with start_pos
// visible columns; softmax in fp32; output heads merged h*128 + d).
//
// A work item is 64 query positions of one sequence and the 4 query heads of
// one KV group, as two 128-row Q tiles (32 positions x 4 heads each; row
// r = position r/4, head r%4), so every 64-key K/V tile is staged once for
// 8 x 32 query rows. In the multi-head variant (32 KV heads, one query head
// each) a Q tile is 128 positions of one head and an item 256 positions:
// the kernel is templated on the query heads per KV head, NREP.
// The grid is persistent: one CTA per SM (its shared memory and TMEM admit
// no second) walks a fixed list of items, longest key range first, so that
// the next item's Q tiles, K/V tiles and first score products overlap the
// current item's last P.V products and epilogue. One CTA per item measured
// ~4 us of set-up, first loads and epilogue per item with nothing else on
// the SM, a third of the kernel at 4 x 2048 tokens.
//   warp 8 (one lane)  TMA producer: per item its K/V stages (stage j: K_j
//                      and V_{j-1}, the tiles the issuers' iteration j
//                      reads, on one full and one empty barrier), after the
//                      first item stages 0..3 first (their slots free up
//                      during the previous item), both Q tiles once the
//                      previous item's last score products are done (128B
//                      swizzle, 4-stage rings shared by all items)
//   warps 9, 10        MMA issuers, one lane each, one per Q tile t: for key
//                      tile j, S_{t,j} = Q_t K_j^T (M=128, N=64) into TMEM
//                      slot j%2 of the tile, then O_t += P_{t,j-1} V_{j-1}
//                      (M=128, N=128) with P read from TMEM and V as an
//                      MN-major shared-memory operand. A single issuing
//                      thread measured ~100 cycles per tcgen05.mma at these
//                      sizes, so each tile has its own.
//   warps 0-3 / 4-7    one softmax warpgroup per Q tile, one thread per row:
//                      loads S from TMEM, masks keys past the row's position,
//                      keeps a running max / sum in fp32, writes
//                      P = 2^(S*scale - max) as bf16 over S, and at the end
//                      of the item reads O, divides by the sum, stores bf16
//                      and frees O for the next item's products.
// TMEM (512 columns): Q tile t owns [256t, 256t+256): S slots at +0 and +64,
// O at +128. While one warpgroup works on its scores the tensor core runs
// the other tile's products and the next key tile's scores. The K/V ring
// holds 4 stages. Cycle stamps of one CTA in steady state: a key tile every
// ~1450 cycles, set by each issuer's loop (a barrier wait, S_j, a wait on
// P_{j-1}, O_{j-1}, commits) in step with the softmax chain (~800 cycles
// from S to P); the copies land well ahead (these K tiles stream at ~70
// bytes a cycle per SM), and a fifth stage left the period as it was; two
// stages made the copy latency the period.
// O is rescaled only when a row's running max grows by more than 2^8 over the
// max its P values were taken against (the result is the same: every P and
// the sum use that reference).
// Every barrier wait is bounded; a wait that gives up records
// DEV_WAIT_TIMEOUT, lets issued copies and products finish (bounded) and frees
// TMEM before the CTA exits.
#include <math.h>

#include "kernels.h"

namespace gqa {

namespace {

constexpr int ROWS = 128;                 // rows of a Q tile = MMA M
constexpr int NQ = 2;                     // Q tiles per CTA
constexpr int KT = PREFILL_TILE;          // keys per tile (= TMA box height)
constexpr int STAGES = 4;                 // K tiles and V tiles in flight
constexpr int Q_HALF = ROWS * 128;        // 128 rows x 64 dims
constexpr int Q_TILE = 2 * Q_HALF;
constexpr int KV_HALF = KT * 128;         // 64 keys x 64 dims
constexpr int KV_TILE = 2 * KV_HALF;
constexpr int K_OFF = NQ * Q_TILE;
constexpr int V_OFF = K_OFF + STAGES * KV_TILE;
constexpr int BAR_OFF = V_OFF + STAGES * KV_TILE;
constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;
constexpr int THREADS = 352;
constexpr int PRODUCER_WARP = 8, MMA_WARP = 9;  // MMA warps 9 (Q tile 0) and 10 (Q tile 1)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TILE_COLS = 256;       // TMEM columns of one Q tile
constexpr uint32_t O_COL = 128;
constexpr float SCALE_LOG2 = 0.08838834764831845f * 1.4426950408889634f;  // log2(e) / sqrt(128)
constexpr float RESCALE_LOG2 = 8.f;

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[STAGES], kv_empty[STAGES];  // stage j of an item: K_j and V_{j-1}
  uint64_t s_full[NQ][2], p_full[NQ][2];
  uint64_t o_done[NQ], mma_done[NQ];
  uint32_t tmem_slot;
  int abort;
  int q_issued, kv_issued;
};
static_assert(sizeof(Bars) <= 512, "barrier block");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ bool aborted(const Bars& bs) { return *reinterpret_cast<const volatile int*>(&bs.abort) != 0; }

// One work item: 2 Q tiles (NQ x QP query positions) of one KV head g of
// sequence b, and the key tiles they see.
struct Item {
  int g, b, q0, start, n;  // n: key tiles of the item (the longer of its Q tiles)
  int nt[NQ];              // key tiles of each Q tile (0: the tile is past T)
  bool valid;              // start position in range
  bool report;             // the item that reports an invalid start of sequence b
};

// Items are numbered longest key range first: item idx is KV head idx % NKV of
// sequence (idx / NKV) % B, pair npairs - 1 - idx / (NKV * B).
template <int NREP>
__device__ __forceinline__ Item item_at(int idx, const PrefillAttnParams& a) {
  constexpr int QP = ROWS / NREP, NKV = N_HEADS / NREP;
  const int npairs = ((a.T + QP - 1) / QP + NQ - 1) / NQ;
  Item it;
  it.g = idx % NKV;
  const int rest = idx / NKV;
  it.b = rest % a.B;
  const int pair = npairs - 1 - rest / a.B;
  it.start = a.sp.get(it.b);
  it.valid = a.sp.ok(it.start);
  it.report = pair == npairs - 1 && it.g == 0;
  it.q0 = pair * NQ * QP;
  it.n = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int qt = it.q0 + t * QP;
    it.nt[t] = it.valid && qt < a.T ? (it.start + min(qt + QP, a.T) + KT - 1) / KT : 0;
    it.n = max(it.n, it.nt[t]);
  }
  return it;
}

// The items of this CTA in order: round k takes item k * G + c on even rounds
// and k * G + G - 1 - c on odd ones (G CTAs, c = blockIdx.x), so that the CTA
// with the longest item of one round gets the shortest of the next. Every
// role of the CTA walks the same sequence; items with an invalid start are
// skipped by all of them.
template <int NREP>
struct ItemWalk {
  int k, nitems;
  __device__ __forceinline__ explicit ItemWalk(const PrefillAttnParams& a) : k(0) {
    constexpr int QP = ROWS / NREP, NKV = N_HEADS / NREP;
    nitems = ((a.T + QP - 1) / QP + NQ - 1) / NQ * NKV * a.B;
  }
  // the next valid item, or false at the end of the list
  __device__ __forceinline__ bool next(const PrefillAttnParams& a, Item& it) {
    const int G = gridDim.x, c = blockIdx.x;
    for (; k * G < nitems; ++k) {
      const int idx = k * G + ((k & 1) ? G - 1 - c : c);
      if (idx >= nitems) continue;
      it = item_at<NREP>(idx, a);
      if (!it.valid) {
        if (it.report && threadIdx.x == 0) report(a.status, DEV_BAD_POSITION);
        continue;
      }
      ++k;
      return true;
    }
    return false;
  }
};

template <int NREP>
__global__ void __launch_bounds__(THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, PrefillAttnParams a) {
  constexpr int QP = ROWS / NREP;         // query positions per Q tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bs = *reinterpret_cast<Bars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bs.q_full), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bs.kv_full[s]), 1);
      mbar_init(smem_u32(&bs.kv_empty[s]), NQ);  // one arrival per MMA issuer
    }
    for (int t = 0; t < NQ; ++t) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(smem_u32(&bs.s_full[t][s]), 1);
        mbar_init(smem_u32(&bs.p_full[t][s]), 4);
      }
      mbar_init(smem_u32(&bs.o_done[t]), 1);
      mbar_init(smem_u32(&bs.mma_done[t]), 1);
    }
    bs.abort = 0;
    bs.q_issued = 0;
    bs.kv_issued = 0;
    fence_barrier_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(&bs.tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs.tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      tma_prefetch_desc(&mv);
      // stage j of an item holds K_j (j < n) and V_{j-1} (j >= 1), the tiles
      // its two issuers' iteration j reads: one full and one empty barrier a
      // stage. u counts stages over the CTA's items, ring slot u % STAGES.
      int u0 = 0, kvn = 0, qn = 0;
      int cs[NQ] = {};  // score tiles of each Q tile so far (as its issuer counts them)
      bool ok = true, stop = false;
      ItemWalk<NREP> walk(a);
      Item it;
      // copies of stage j; false when a wait gave up or the kernel is aborting
      auto load_stage = [&](const Item& it, int j) -> bool {
        const int u = u0 + j, s = u % STAGES;
        if (u >= STAGES) ok = mbar_wait(smem_u32(&bs.kv_empty[s]), ((u / STAGES) - 1) & 1);
        if (!ok || aborted(bs)) return false;
        const uint32_t fb = smem_u32(&bs.kv_full[s]);
        mbar_expect_tx(fb, (j < it.n ? KV_TILE : 0) + (j >= 1 ? KV_TILE : 0));
        if (j < it.n) {
          const uint32_t dst = sbase + K_OFF + s * KV_TILE;
          tma_load_4d(dst, &mk, fb, 0, it.g, j * KT, it.b);
          tma_load_4d(dst + KV_HALF, &mk, fb, 64, it.g, j * KT, it.b);
        }
        if (j >= 1) {
          const uint32_t dst = sbase + V_OFF + s * KV_TILE;
          tma_load_4d(dst, &mv, fb, 0, it.g, (j - 1) * KT, it.b);
          tma_load_4d(dst + KV_HALF, &mv, fb, 64, it.g, (j - 1) * KT, it.b);
        }
        kvn = u + 1;
        return true;
      };
      for (int ii = 0; !stop && walk.next(a, it); ++ii) {
        // after the first item, the item's first stages go out before its Q
        // tiles: their ring slots free up while the previous item's last
        // products run, the Q tiles only after its last score products have
        // completed
        const int la = ii > 0 ? min(STAGES, it.n + 1) : 0;
        for (int j = 0; j < la && !stop; ++j) stop = !load_stage(it, j);
        if (stop) break;
        // Q tile t is free once the last score product of the previous item
        // that read it has completed (its s_full phase; the next product on
        // that slot needs the new Q, so the phase cannot have moved on)
#pragma unroll
        for (int t = 0; t < NQ; ++t)
          if (ok && cs[t] > 0) ok = mbar_wait(smem_u32(&bs.s_full[t][(cs[t] - 1) & 1]), ((cs[t] - 1) >> 1) & 1);
        if (!ok || aborted(bs)) break;
        const uint32_t qb = smem_u32(&bs.q_full);
        mbar_expect_tx(qb, NQ * Q_TILE);
        // a tile past T reads as zeros (its rows are never stored)
        for (int t = 0; t < NQ; ++t) {
          tma_load_4d(sbase + t * Q_TILE, &mq, qb, 0, it.g * NREP, it.q0 + t * QP, it.b);
          tma_load_4d(sbase + t * Q_TILE + Q_HALF, &mq, qb, 64, it.g * NREP, it.q0 + t * QP, it.b);
        }
        qn = ii + 1;
        for (int j = la; j <= it.n && !stop; ++j) stop = !load_stage(it, j);
        if (stop) break;
        u0 += it.n + 1;
#pragma unroll
        for (int t = 0; t < NQ; ++t) cs[t] += it.nt[t];
      }
      if (!ok) atomicExch(&bs.abort, 1);
      bs.q_issued = qn;
      bs.kv_issued = kvn;
    }
  } else if (warp >= MMA_WARP) {
    // issuer of Q tile t (the whole warp runs the loop; one elected lane
    // issues): waits on every K/V stage so that its arrivals on the empty
    // barriers stay in step with the other issuer's; a stage past this
    // tile's causal range gets a plain arrival. cs counts this tile's score
    // tiles over the items (S slot cs % 2, one O product group each).
    const int t = warp - MMA_WARP;
    const uint32_t idesc_s = umma_idesc_bf16(ROWS, KT);
    const uint32_t idesc_o = umma_idesc_bf16(ROWS, HEAD_DIM) | (1u << 16);  // B (V) MN-major
    const uint32_t qt = sbase + t * Q_TILE;
    const uint32_t base = tmem + t * TILE_COLS;
    unsigned u0 = 0, cs = 0;
    bool ok = true;
    ItemWalk<NREP> walk(a);
    Item it;
    for (int ii = 0; ok && walk.next(a, it); ++ii) {
      const int n_t = t ? it.nt[1] : it.nt[0];
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.q_full), ii & 1));
      if (!ok) break;
      for (int j = 0; ok && j <= it.n; ++j) {
        const unsigned u = u0 + j, s = u % STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.kv_full[s]), (u / STAGES) & 1));
        if (!ok) break;
        bool used = false;
        if (j < n_t) {
          tc_fence_after();
          const uint32_t kt = sbase + K_OFF + s * KV_TILE;
          const unsigned slot = (cs + j) & 1u;
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
              const uint32_t off = (ks & 3) * 32;
              umma_bf16(base + slot * KT, umma_desc_sw128(qt + (ks >> 2) * Q_HALF + off),
                        umma_desc_sw128(kt + (ks >> 2) * KV_HALF + off), idesc_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(smem_u32(&bs.s_full[t][slot]));
          }
          __syncwarp();
          used = true;
        }
        if (j >= 1 && j - 1 < n_t) {
          const int i = j - 1;
          // P of the item's first key tile also tells that the softmax
          // warps have read the previous item's O (their epilogue comes
          // first), so that the first product may overwrite it
          const unsigned c = cs + i;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.p_full[t][c & 1]), (c >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t vt = sbase + V_OFF + s * KV_TILE;
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < KT / 16; ++ks)
              umma_bf16_ts(base + O_COL, base + (c & 1) * KT + ks * 8,
                           umma_desc_sw128_mn(vt + ks * 16 * 128, KV_HALF), idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
            umma_commit(smem_u32(&bs.o_done[t]));
          }
          __syncwarp();
          used = true;
        }
        // the stage is free once this issuer's products on it are done (a
        // commit covers every product the thread issued before it)
        if (elect_one()) {
          if (used)
            umma_commit(smem_u32(&bs.kv_empty[s]));
          else
            mbar_arrive(smem_u32(&bs.kv_empty[s]));
        }
        __syncwarp();
      }
      if (!ok) break;
      u0 += it.n + 1;
      cs += n_t;
    }
    if (!ok && lane == 0) atomicExch(&bs.abort, 1);
    if (elect_one()) umma_commit(smem_u32(&bs.mma_done[t]));
    __syncwarp();
    mbar_wait(smem_u32(&bs.mma_done[t]), 0);
  } else {
    // softmax / epilogue: warpgroup t, thread r owns row r = TMEM lane r of Q tile t
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int hh = r % NREP;
    const uint32_t lane_addr = tmem + t * TILE_COLS + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    unsigned cs = 0;  // score tiles of this Q tile over the items (as the issuer counts them)
    bool ok = true;
    ItemWalk<NREP> walk(a);
    Item it;
    while (ok && walk.next(a, it)) {
      const int n_t = t ? it.nt[1] : it.nt[0];
      const int pos = it.q0 + t * QP + r / NREP;  // query index within the sequence
      const int kv_end = it.start + min(it.q0 + t * QP + QP, a.T);
      const int lim = min(it.start + pos, kv_end - 1);  // last key this row sees
      float m_ref = -INFINITY;  // max the current P values and O are taken against (raw score units)
      float l = 0.f;
      for (int j = 0; j < n_t; ++j) {
        const unsigned c = cs + j;
        const unsigned s = c & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.s_full[t][s]), (c >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[KT];
        tmem_ld32(lane_addr + s * KT, sr);
        tmem_ld32(lane_addr + s * KT + 32, sr + 32);
        tmem_ld_wait();
        const int vis = lim - j * KT;  // columns 0..vis are visible to this row
        if (vis < KT - 1) {
#pragma unroll
          for (int cc = 0; cc < KT; ++cc)
            if (cc > vis) sr[cc] = __float_as_uint(-INFINITY);
        }
        float mx = fmaxf(__uint_as_float(sr[0]), __uint_as_float(sr[1]));
#pragma unroll
        for (int cc = 2; cc < KT; cc += 2) mx = max3(mx, __uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1]));
        float alpha = 1.f;
        const bool grow = mx > m_ref && (m_ref == -INFINITY || (mx - m_ref) * SCALE_LOG2 > RESCALE_LOG2);
        if (grow) {
          alpha = m_ref == -INFINITY ? 0.f : ex2_approx((m_ref - mx) * SCALE_LOG2);
          m_ref = mx;
        }
        const float neg = m_ref == -INFINITY ? 0.f : -m_ref * SCALE_LOG2;
        // exponent arguments and the row sum two columns per instruction
        const float2 sc2 = make_float2(SCALE_LOG2, SCALE_LOG2), ng2 = make_float2(neg, neg);
        float2 sum2 = make_float2(0.f, 0.f);
        uint32_t pk[KT / 2];
#pragma unroll
        for (int cc = 0; cc < KT; cc += 2) {
          const float2 e = fma2(make_float2(__uint_as_float(sr[cc]), __uint_as_float(sr[cc + 1])), sc2, ng2);
          const float2 p = make_float2(ex2_approx(e.x), ex2_approx(e.y));
          sum2 = add2(sum2, p);
          pk[cc >> 1] = pack_bf16(p.x, p.y);
        }
        l = l * alpha + (sum2.x + sum2.y);
        if (j > 0) {
          // O must hold P_{j-1} V_{j-1} before it is rescaled (and this keeps
          // the o_done phases in step with the score tiles)
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.o_done[t]), (c - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
            for (int cc = 0; cc < HEAD_DIM; cc += 32) {
              uint32_t o[32];
              tmem_ld32(lane_addr + O_COL + cc, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st32(lane_addr + O_COL + cc, o);
            }
          }
        }
        tmem_st32(lane_addr + s * KT, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bs.p_full[t][s]));
      }
      if (!ok) break;
      if (n_t > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.o_done[t]), (cs + n_t - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16* dst = a.o + (static_cast<size_t>(it.b) * a.T + pos) * D_MODEL +
                             static_cast<size_t>(it.g * NREP + hh) * HEAD_DIM;
#pragma unroll 1
        for (int cc = 0; cc < HEAD_DIM; cc += 32) {
          uint32_t o[32];
          tmem_ld32(lane_addr + O_COL + cc, o);
          tmem_ld_wait();
          if (pos < a.T) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
              w.y = pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
              w.z = pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
              w.w = pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
              d4[e] = w;
            }
          }
        }
      }
      cs += n_t;
    }
    if (!ok && lane == 0) atomicExch(&bs.abort, 1);
  }

  tc_fence_before();
  __syncthreads();
  if (aborted(bs)) {
    if (threadIdx.x == 0) report(a.status, DEV_WAIT_TIMEOUT);
    if (warp == PRODUCER_WARP && lane == 0) {
      // the last copy into each buffer may still be in flight
      if (bs.q_issued > 0) mbar_wait(smem_u32(&bs.q_full), (bs.q_issued - 1) & 1);
      for (int u = max(0, bs.kv_issued - STAGES); u < bs.kv_issued; ++u)
        mbar_wait(smem_u32(&bs.kv_full[u % STAGES]), (u / STAGES) & 1);
    }
    __syncthreads();
  }
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int NREP>
cudaError_t launch_nrep(const PrefillMaps& maps, const PrefillAttnParams& a, cudaStream_t s) {
  constexpr int QP = ROWS / NREP, NKV = N_HEADS / NREP;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = attn_prefill_kernel<NREP>;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (a.B <= 0 || a.T <= 0 || a.num_sms <= 0) return cudaErrorInvalidValue;
  // one CTA per SM (shared memory and TMEM admit no second), each walking its items
  const long long items = static_cast<long long>(((a.T + QP - 1) / QP + NQ - 1) / NQ) * NKV * a.B;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned ctas = static_cast<unsigned>(items < a.num_sms ? items : a.num_sms);
  kern<<<ctas, THREADS, SMEM_BYTES, s>>>(maps.q, maps.k, maps.v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_prefill(const PrefillMaps& maps, const PrefillAttnParams& a, cudaStream_t s) {
  switch (a.n_kv) {
    case N_KV: return launch_nrep<N_REP>(maps, a, s);
    case N_HEADS: return launch_nrep<1>(maps, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gqa
