// Causal prefill attention on the 5th-generation tensor cores. Query t
// (position start_pos + t) of head h attends to cache rows 0..start_pos+t of
// KV head h / 4 ("Llama 3.1 8B · Grouped-query attention": the mask of
// Transformer.forward is -inf above the diagonal, left-padded with start_pos
// visible columns; softmax in fp32; output heads merged h*128 + d).
//
// One CTA owns 64 query positions of one sequence and the 4 query heads of
// one KV group, as two 128-row Q tiles (32 positions x 4 heads each; row
// r = position r/4, head r%4), so every 64-key K/V tile is staged once for
// 8 x 32 query rows. In the multi-head variant (32 KV heads, one query head
// each) a Q tile is 128 positions of one head and a CTA owns 256 positions:
// the kernel is templated on the query heads per KV head, NREP.
//   warp 8 (one lane)  TMA producer: both Q tiles once, then K_j / V_j
//                      (128B swizzle, 4-stage rings on mbarriers)
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
//                      reads O, divides by the sum and stores bf16.
// TMEM (512 columns): Q tile t owns [256t, 256t+256): S slots at +0 and +64,
// O at +128. While one warpgroup works on its scores the tensor core runs
// the other tile's products and the next key tile's scores. The K/V rings
// hold 4 tiles each: a 16 KB K tile takes ~1.4 us from request to arrival
// under load, and two stages made that latency the period of the whole
// kernel.
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
  uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
  uint64_t s_full[NQ][2], p_full[NQ][2];
  uint64_t o_done[NQ], mma_done[NQ];
  uint32_t tmem_slot;
  int abort;
  int k_issued, v_issued;
};
static_assert(sizeof(Bars) <= 512, "barrier block");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

__device__ __forceinline__ bool aborted(const Bars& bs) { return *reinterpret_cast<const volatile int*>(&bs.abort) != 0; }

template <int NREP>
__global__ void __launch_bounds__(THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, PrefillAttnParams a) {
  constexpr int QP = ROWS / NREP;         // query positions per Q tile
  constexpr int NKV = N_HEADS / NREP;     // KV heads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars& bs = *reinterpret_cast<Bars*>(smem + BAR_OFF);

  // longest key ranges first: the pair of query tiles falls with blockIdx.x
  const int nqt = (a.T + QP - 1) / QP;
  const int npairs = (nqt + NQ - 1) / NQ;
  const int g = blockIdx.x % NKV;
  const int rest = blockIdx.x / NKV;
  const int b = rest % a.B;
  const int pair = npairs - 1 - rest / a.B;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int start = a.sp.get(b);
  if (!a.sp.ok(start)) {
    if (pair == npairs - 1 && g == 0 && threadIdx.x == 0) report(a.status, DEV_BAD_POSITION);
    return;
  }
  const int q0 = pair * NQ * QP;  // first position (index t) of Q tile 0
  int nt[NQ];                     // key tiles of each Q tile (0: the tile is past T)
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int qt = q0 + t * QP;
    nt[t] = qt < a.T ? (start + min(qt + QP, a.T) + KT - 1) / KT : 0;
  }
  const int n = nt[NQ - 1] > nt[0] ? nt[NQ - 1] : nt[0];

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bs.q_full), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bs.k_full[s]), 1);
      mbar_init(smem_u32(&bs.k_empty[s]), NQ);  // one arrival per MMA issuer
      mbar_init(smem_u32(&bs.v_full[s]), 1);
      mbar_init(smem_u32(&bs.v_empty[s]), NQ);
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
    bs.k_issued = 0;
    bs.v_issued = 0;
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
      const uint32_t qb = smem_u32(&bs.q_full);
      mbar_expect_tx(qb, NQ * Q_TILE);
      // a tile past T reads as zeros (its rows are never stored)
      for (int t = 0; t < NQ; ++t) {
        tma_load_4d(sbase + t * Q_TILE, &mq, qb, 0, g * NREP, q0 + t * QP, b);
        tma_load_4d(sbase + t * Q_TILE + Q_HALF, &mq, qb, 64, g * NREP, q0 + t * QP, b);
      }
      int kn = 0, vn = 0;
      bool ok = true;
      for (int j = 0; j <= n && ok; ++j) {
        if (j < n) {
          const int s = j % STAGES;
          if (j >= STAGES) ok = mbar_wait(smem_u32(&bs.k_empty[s]), ((j / STAGES) - 1) & 1);
          if (!ok || aborted(bs)) break;
          const uint32_t fb = smem_u32(&bs.k_full[s]);
          const uint32_t dst = sbase + K_OFF + s * KV_TILE;
          mbar_expect_tx(fb, KV_TILE);
          tma_load_4d(dst, &mk, fb, 0, g, j * KT, b);
          tma_load_4d(dst + KV_HALF, &mk, fb, 64, g, j * KT, b);
          kn = j + 1;
        }
        if (j >= 1) {
          const int i = j - 1, s = i % STAGES;
          if (i >= STAGES) ok = mbar_wait(smem_u32(&bs.v_empty[s]), ((i / STAGES) - 1) & 1);
          if (!ok || aborted(bs)) break;
          const uint32_t fb = smem_u32(&bs.v_full[s]);
          const uint32_t dst = sbase + V_OFF + s * KV_TILE;
          mbar_expect_tx(fb, KV_TILE);
          tma_load_4d(dst, &mv, fb, 0, g, i * KT, b);
          tma_load_4d(dst + KV_HALF, &mv, fb, 64, g, i * KT, b);
          vn = i + 1;
        }
      }
      if (!ok) atomicExch(&bs.abort, 1);
      bs.k_issued = kn;
      bs.v_issued = vn;
    }
  } else if (warp >= MMA_WARP) {
    // issuer of Q tile t (the whole warp runs the loop; one elected lane
    // issues): waits on every K/V stage so that its arrivals on the empty
    // barriers stay in step with the other issuer's; a stage past this
    // tile's causal range gets a plain arrival
    const int t = warp - MMA_WARP;
    const int n_t = t ? nt[1] : nt[0];
    const uint32_t idesc_s = umma_idesc_bf16(ROWS, KT);
    const uint32_t idesc_o = umma_idesc_bf16(ROWS, HEAD_DIM) | (1u << 16);  // B (V) MN-major
    const uint32_t qt = sbase + t * Q_TILE;
    const uint32_t base = tmem + t * TILE_COLS;
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.q_full), 0));
    for (int j = 0; ok && j <= n; ++j) {
      if (j < n) {
        const int s = j % STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.k_full[s]), (j / STAGES) & 1));
        if (!ok) break;
        if (j < n_t) {
          tc_fence_after();
          const uint32_t kt = sbase + K_OFF + s * KV_TILE;
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < HEAD_DIM / 16; ++ks) {
              const uint32_t off = (ks & 3) * 32;
              umma_bf16(base + (j & 1) * KT, umma_desc_sw128(qt + (ks >> 2) * Q_HALF + off),
                        umma_desc_sw128(kt + (ks >> 2) * KV_HALF + off), idesc_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(smem_u32(&bs.s_full[t][j & 1]));
            umma_commit(smem_u32(&bs.k_empty[s]));
          }
        } else if (elect_one()) {
          mbar_arrive(smem_u32(&bs.k_empty[s]));
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int i = j - 1, s = i % STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.v_full[s]), (i / STAGES) & 1));
        if (!ok) break;
        if (i < n_t) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.p_full[t][i & 1]), (i >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
          const uint32_t vt = sbase + V_OFF + s * KV_TILE;
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < KT / 16; ++ks)
              umma_bf16_ts(base + O_COL, base + (i & 1) * KT + ks * 8,
                           umma_desc_sw128_mn(vt + ks * 16 * 128, KV_HALF), idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
            umma_commit(smem_u32(&bs.o_done[t]));
            umma_commit(smem_u32(&bs.v_empty[s]));
          }
        } else if (elect_one()) {
          mbar_arrive(smem_u32(&bs.v_empty[s]));
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) atomicExch(&bs.abort, 1);
    if (elect_one()) umma_commit(smem_u32(&bs.mma_done[t]));
    __syncwarp();
    mbar_wait(smem_u32(&bs.mma_done[t]), 0);
  } else {
    // softmax / epilogue: warpgroup t, thread r owns row r = TMEM lane r of Q tile t
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int n_t = t ? nt[1] : nt[0];
    const int pos = q0 + t * QP + r / NREP;  // query index within the sequence
    const int hh = r % NREP;
    const int kv_end = start + min(q0 + t * QP + QP, a.T);
    const int lim = min(start + pos, kv_end - 1);  // last key this row sees
    const uint32_t lane_addr = tmem + t * TILE_COLS + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float m_ref = -INFINITY;  // max the current P values and O are taken against (raw score units)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_t; ++j) {
      const int s = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.s_full[t][s]), (j >> 1) & 1))) {
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
        for (int c = 0; c < KT; ++c)
          if (c > vis) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx = fmaxf(__uint_as_float(sr[0]), __uint_as_float(sr[1]));
#pragma unroll
      for (int c = 2; c < KT; c += 2) mx = max3(mx, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
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
      for (int c = 0; c < KT; c += 2) {
        const float2 e = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, ng2);
        const float2 p = make_float2(ex2_approx(e.x), ex2_approx(e.y));
        sum2 = add2(sum2, p);
        pk[c >> 1] = pack_bf16(p.x, p.y);
      }
      const float sum = sum2.x + sum2.y;
      l = l * alpha + sum;
      if (j > 0) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled (and this keeps
        // the o_done phases in step with j)
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.o_done[t]), (j - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c = 0; c < HEAD_DIM; c += 32) {
            uint32_t o[32];
            tmem_ld32(lane_addr + O_COL + c, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(lane_addr + O_COL + c, o);
          }
        }
      }
      tmem_st32(lane_addr + s * KT, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bs.p_full[t][s]));
    }
    if (ok && n_t > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bs.o_done[t]), (n_t - 1) & 1))) ok = false;
    if (ok && n_t > 0) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* dst = a.o + (static_cast<size_t>(b) * a.T + pos) * D_MODEL +
                           static_cast<size_t>(g * NREP + hh) * HEAD_DIM;
#pragma unroll 1
      for (int c = 0; c < HEAD_DIM; c += 32) {
        uint32_t o[32];
        tmem_ld32(lane_addr + O_COL + c, o);
        tmem_ld_wait();
        if (pos < a.T) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c);
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
    } else if (!ok && lane == 0) {
      atomicExch(&bs.abort, 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (aborted(bs)) {
    if (threadIdx.x == 0) report(a.status, DEV_WAIT_TIMEOUT);
    if (warp == PRODUCER_WARP && lane == 0) {
      // the last copy into each stage may still be in flight
      mbar_wait(smem_u32(&bs.q_full), 0);
      for (int u = max(0, bs.k_issued - STAGES); u < bs.k_issued; ++u)
        mbar_wait(smem_u32(&bs.k_full[u % STAGES]), (u / STAGES) & 1);
      for (int u = max(0, bs.v_issued - STAGES); u < bs.v_issued; ++u)
        mbar_wait(smem_u32(&bs.v_full[u % STAGES]), (u / STAGES) & 1);
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
  if (a.B <= 0 || a.T <= 0) return cudaErrorInvalidValue;
  const long long ctas = static_cast<long long>(((a.T + QP - 1) / QP + NQ - 1) / NQ) * NKV * a.B;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(ctas), THREADS, SMEM_BYTES, s>>>(maps.q, maps.k, maps.v, a);
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
