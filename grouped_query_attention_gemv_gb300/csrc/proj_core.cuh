// Few-token projection (M <= 64 tokens) on the 5th-generation tensor cores:
// y = x W^T with W stored [out, in] ("Llama 3.1 8B · Query projection": the
// F.linear storage; the K, V and output projections of "Grouped-query
// attention" likewise). Device-side phase shared by the standalone kernel
// (proj_stream.cu) and the fused decode kernel (decode_fused.cu).
//
// At decode sizes this step is a pure stream of the weights (50 MB for Q|K|V,
// 34 MB for W_O), so it is built to keep HBM busy:
//   * swap-AB: a 128-row tile of W is the MMA's A operand (M = 128) and the
//     token block the B operand (N = 16/32/64, zero-padded by TMA), so one
//     tcgen05.mma kind::f16 covers 128 weight rows x all tokens x 16 k;
//   * persistent stream-K: the (128-row tile, 64-wide k block) units of W are
//     cut into one contiguous range per CTA (one CTA per SM), so every SM
//     streams the same bytes; a range covers at most a few row tiles
//     ("segments");
//   * one producer lane keeps a ring of TMA loads in flight; a stage holds up
//     to 4 consecutive 64-wide k blocks of the same 128 rows, fetched as ONE
//     box of a 3-D view of W (k within block, row, block), so each weight
//     row is read 512 contiguous bytes at a time; a stretch of n k blocks
//     takes ceil(n / 4) stages (boxes of 1-4 blocks), so stage counts, which
//     set a CTA's time more than its bytes do, differ by at most one between
//     CTAs;
//   * one lane issues the MMAs into a double-buffered TMEM accumulator; four
//     epilogue warps drain a finished segment with tcgen05.ld while the next
//     one accumulates;
//   * a segment's fp32 partial goes to its own slot; the CTA whose ticket
//     completes the 64 k blocks of a row tile sums the slots in CTA order
//     (deterministic) and runs the epilogue (RoPE + KV-cache append for
//     Q|K|V, bf16 store for W_O) through a shared-memory staging tile written
//     out as 16-byte vectors. Nothing waits on another CTA;
//   * the weights of the first stages are requested before the token rows,
//     which may come from an earlier phase: `gate` is passed in by the kernel.
#pragma once

#include "kernels.h"

namespace gqa {
namespace projk {

constexpr int TILE_ROWS = 128;
constexpr int KBLK = 64;
constexpr int NKB = D_MODEL / KBLK;            // 64 k blocks per row tile
constexpr int A_BYTES = TILE_ROWS * KBLK * 2;  // 16 KB
constexpr int KC = 4;                          // k blocks per full stage

template <int NP>
struct Cfg {
  static constexpr int B_BYTES = NP * KBLK * 2;  // one k block of the token tile
  static constexpr int STAGE = KC * (A_BYTES + B_BYTES);
  static constexpr int STAGES = NP == 16 ? 3 : 2;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int TMEM_COLS = 2 * NP < 32 ? 32 : 2 * NP;
  static constexpr int OUT_BYTES = NP * TILE_ROWS * 2;  // bf16 [NP][128] staging of one row tile's outputs
};

// k blocks in the next stage when `left` remain in the segment.
__device__ __forceinline__ int stage_blocks(long long left) { return left >= KC ? KC : static_cast<int>(left); }

// CTA whose stream-K range contains unit u (ranges start at floor(c*U/C)).
__device__ __forceinline__ int cta_of(long long u, long long U, long long C) {
  return static_cast<int>(((u + 1) * C + U - 1) / U) - 1;
}
__device__ __forceinline__ long long range_start(long long c, long long U, long long C) { return U * c / C; }

// AND of `v` over the 128 epilogue threads (warps 2-5), with a barrier.
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

template <int NP>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NP]) {
#pragma unroll
  for (int j = 0; j < NP / 16; ++j) {
    uint32_t r[16];
    tmem_ld16(taddr + j * 16, r);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e) v[j * 16 + e] = __uint_as_float(r[e]);
  }
}

// Epilogue of row tile rt: every epilogue thread holds the full sums of one
// weight row f (= rt*128 + r) for all tokens; RoPE pairs (f, f^1) are
// neighbouring lanes. Results are staged in shared memory as [token][128]
// bf16 and written as 16-byte vectors, one contiguous 256-byte run per token
// (its 128 features of q, or its new K or V row in the cache). Ends with the
// writes fenced and a barrier of the epilogue warps.
template <int NP, bool QKV>
__device__ __forceinline__ void store_tile(const ProjParams& p, int rt, int r, float (&acc)[NP],
                                           __nv_bfloat16* stage) {
  const int f = rt * TILE_ROWS + r;
#pragma unroll
  for (int m = 0; m < NP; ++m) {
    float v = acc[m];
    if constexpr (QKV) {
      const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
      if (m < p.M && f < p.r2) {
        const int b = m / p.T;
        const int start = p.sp.get(b);
        if (p.sp.ok(start)) {
          const float2 cs = *reinterpret_cast<const float2*>(
              p.rope + (static_cast<size_t>(start + m - b * p.T) * ROPE_PAIRS + ((f & (HEAD_DIM - 1)) >> 1)) * 2);
          v = (f & 1) ? partner * cs.y + v * cs.x : v * cs.x - partner * cs.y;
        }
      }
    }
    if constexpr (!QKV) {
      if (p.resid && m < p.M) v += __bfloat162float(p.resid[static_cast<size_t>(m) * p.N + f]);  // the block's residual
    }
    stage[m * TILE_ROWS + r] = __float2bfloat16_rn(v);
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  const int t = threadIdx.x - 64;  // 0..127 over the epilogue warps
  for (int idx = t; idx < p.M * 16; idx += 128) {
    const int m = idx >> 4, ch = idx & 15;
    __nv_bfloat16* dst;
    if constexpr (QKV) {
      const int b = m / p.T;
      const int start = p.sp.get(b);
      if (!p.sp.ok(start)) {
        if (ch == 0 && m - b * p.T == 0 && (rt & 3) == 0) report(p.status, DEV_BAD_POSITION);
        continue;
      }
      const int pos = start + (m - b * p.T);
      const int f0 = rt * TILE_ROWS;
      if (f0 < D_MODEL) {
        dst = p.out + static_cast<size_t>(m) * D_MODEL + f0;
      } else {
        const size_t row = (static_cast<size_t>(b) * p.s_max + pos) * (p.r2 - p.r1);
        dst = f0 < p.r2 ? p.cache_k + row + (f0 - D_MODEL) : p.cache_v + row + (f0 - p.r2);
      }
    } else {
      dst = p.out + static_cast<size_t>(m) * p.N + rt * TILE_ROWS;
    }
    reinterpret_cast<uint4*>(dst)[ch] = reinterpret_cast<const uint4*>(stage + m * TILE_ROWS)[ch];
  }
  fence_proxy_async_global();  // a later phase of the same grid may read these rows by TMA
  __threadfence();
  asm volatile("bar.sync 1, 128;" ::: "memory");  // the staging tile is reused by the next merge
}

// Shared-memory objects of one projection phase. Barriers are initialised by
// the kernel: full/empty count 1, acc_full count 1, acc_empty count 4.
template <int NP>
struct Shared {
  uint8_t* ring;       // Cfg<NP>::RING bytes, 1024-aligned
  uint64_t* full;      // [STAGES]
  uint64_t* empty;     // [STAGES]
  uint64_t* acc_full;  // [2]
  uint64_t* acc_empty; // [2]
  __nv_bfloat16* stage;  // Cfg<NP>::OUT_BYTES
  int* flags;          // [0] abort, [1] ticket, [2] issued, [3] consumed
  uint32_t tmem;       // TMEM base of >= 2*NP columns
};

// One projection over this CTA's stream-K range of units. Roles: warp 0 lane 0
// producer, warp 1 lane 0 MMA issuer, warps 2-5 epilogue; other warps return
// at once. gate() runs on the producer before the first token load (false =
// give up); tile_done(rt) runs on thread 64 once row tile rt is written.
template <int NP, bool QKV, class Gate, class TileDone>
__device__ __forceinline__ void proj_phase(const ProjStreamMaps& maps, const ProjParams& p, float* __restrict__ part,
                                           int* __restrict__ tickets, int segmax, const Shared<NP>& sh, Gate gate,
                                           TileDone tile_done) {
  using C_ = Cfg<NP>;
  constexpr int S = C_::STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long C = gridDim.x, c = blockIdx.x;
  const long long U = static_cast<long long>(p.N / TILE_ROWS) * NKB;
  const long long u0 = range_start(c, U, C), u1 = range_start(c + 1, U, C);
  int* flags = sh.flags;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer: stage i holds k blocks [u, u + nch) of one row tile
    tma_prefetch_desc(&maps.x[KC - 1]);
    long long u = u0;
    int i = 0;
    long long seg_end = u0;
    auto load = [&](bool weights, bool tokens) {
      const int rt = static_cast<int>(u / NKB), kb = static_cast<int>(u % NKB);
      const int nch = stage_blocks(seg_end - u);
      const int s = i % S;
      const uint32_t base = smem_u32(sh.ring + s * C_::STAGE);
      const uint32_t fb = smem_u32(&sh.full[s]);
      if (weights) {
        const int row0 = rt * TILE_ROWS;
        const int w = row0 < p.r1 ? 0 : (row0 < p.r2 ? 1 : 2);
        const int lrow = row0 - (w == 0 ? 0 : (w == 1 ? p.r1 : p.r2));
        mbar_expect_tx(fb, nch * (A_BYTES + C_::B_BYTES));
        tma_load_3d(base, &maps.w[nch - 1][w], fb, 0, lrow, kb);
      }
      if (tokens) tma_load_3d(base + KC * A_BYTES, &maps.x[nch - 1], fb, 0, 0, kb);
      return nch;
    };
    // weights do not depend on earlier work: request the first stages' weights before the gate
    int pre = 0;
    {
      long long uu = u0, se = u0;
      while (uu < u1 && pre < S) {
        if (uu == se) se = min(u1, (uu / NKB + 1) * NKB);
        u = uu;
        seg_end = se;
        uu += load(true, false);
        ++i;
        ++pre;
      }
    }
    // even when the gate gives up, the pre-issued stages get their token
    // loads, so that every issued stage completes and can be drained
    bool ok = gate();
    u = u0;
    seg_end = u0;
    i = 0;
    for (; u < u1; ++i) {
      if (u == seg_end) seg_end = min(u1, (u / NKB + 1) * NKB);
      if (i >= pre) {
        if (!ok) break;
        if (!mbar_wait(smem_u32(&sh.empty[i % S]), ((i / S) & 1) ^ 1)) {
          ok = false;
          break;
        }
      }
      u += load(i >= pre, true);
    }
    if (!ok) atomicExch(&flags[0], 1);
    flags[2] = i;  // stages whose loads were issued
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer (same stage walk as the producer)
    constexpr uint32_t idesc = umma_idesc_bf16(TILE_ROWS, NP);
    int seg = 0, i = 0;
    long long u = u0, seg_end = u0;
    for (; u < u1; ++i) {
      const bool first = u == seg_end;
      if (first) seg_end = min(u1, (u / NKB + 1) * NKB);
      const int nch = stage_blocks(seg_end - u);
      const int s = i % S;
      if (!mbar_wait(smem_u32(&sh.full[s]), (i / S) & 1)) {
        atomicExch(&flags[0], 1);
        break;
      }
      const int buf = seg & 1;
      if (first && seg >= 2 && !mbar_wait(smem_u32(&sh.acc_empty[buf]), ((seg >> 1) & 1) ^ 1)) {
        atomicExch(&flags[0], 1);
        break;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(sh.ring + s * C_::STAGE);
      const uint32_t sb = sa + KC * A_BYTES;
      for (int cb = 0; cb < nch; ++cb) {
#pragma unroll
        for (int k = 0; k < KBLK / 16; ++k)
          umma_bf16(sh.tmem + buf * NP, umma_desc_sw128(sa + cb * A_BYTES + k * 32),
                    umma_desc_sw128(sb + cb * C_::B_BYTES + k * 32), idesc, (first && cb == 0 && k == 0) ? 0u : 1u);
      }
      umma_commit(smem_u32(&sh.empty[s]));
      u += nch;
      if (u == seg_end) {
        umma_commit(smem_u32(&sh.acc_full[buf]));
        ++seg;
      }
    }
    flags[3] = i;
  } else if (warp >= 2 && warp < 6) {
    // ---------------- epilogue warps: TMEM lanes 32*(warp%4) .. +31
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the 128-row tile
    const uint32_t lane_addr = sh.tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    long long u = u0;
    int seg = 0;
    while (u < u1) {
      const int rt = static_cast<int>(u / NKB);
      const long long seg_end = min(u1, static_cast<long long>(rt + 1) * NKB);
      const int nunits = static_cast<int>(seg_end - u);
      const int buf = seg & 1;
      bool ok = mbar_wait(smem_u32(&sh.acc_full[buf]), (seg >> 1) & 1);
      // the four epilogue warps decide together: they meet at named barrier 1 below
      ok = epilogue_all(ok && !*reinterpret_cast<volatile int*>(&flags[0]));
      if (!ok) {
        if (lane == 0) atomicExch(&flags[0], 1);
        break;
      }
      tc_fence_after();
      float v[NP];
      tmem_ld_cols<NP>(lane_addr + buf * NP, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[buf]));
      // publish the partial of this segment
      float4* dst = reinterpret_cast<float4*>(part + ((static_cast<size_t>(c) * segmax + seg) * TILE_ROWS + r) * NP);
#pragma unroll
      for (int j = 0; j < NP / 4; ++j) __stcg(dst + j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
      __threadfence();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (threadIdx.x == 64) flags[1] = atomicAdd(tickets + rt, nunits);
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (flags[1] + nunits == NKB) {
        // last contribution to row tile rt: sum every CTA's slot in CTA order
        __threadfence();
        const long long uf = static_cast<long long>(rt) * NKB;
        const int cf = cta_of(uf, U, C), cl = cta_of(uf + NKB - 1, U, C);
        float acc[NP];
#pragma unroll
        for (int m = 0; m < NP; ++m) acc[m] = 0.f;
        for (int cc = cf; cc <= cl; ++cc) {
          const int ordinal = rt - static_cast<int>(range_start(cc, U, C) / NKB);
          const float4* src =
              reinterpret_cast<const float4*>(part + ((static_cast<size_t>(cc) * segmax + ordinal) * TILE_ROWS + r) * NP);
#pragma unroll
          for (int j = 0; j < NP / 4; ++j) {
            const float4 q = __ldcg(src + j);
            acc[4 * j] += q.x;
            acc[4 * j + 1] += q.y;
            acc[4 * j + 2] += q.z;
            acc[4 * j + 3] += q.w;
          }
        }
        store_tile<NP, QKV>(p, rt, r, acc, sh.stage);
        if (threadIdx.x == 64) {
          tickets[rt] = 0;
          tile_done(rt);
        }
      }
      u = seg_end;
      ++seg;
    }
  }
}

// After an aborted phase: let loads that were issued but never consumed land
// (bounded) before the shared memory is reused or the CTA exits. One thread.
template <int NP>
__device__ __forceinline__ void proj_drain(const Shared<NP>& sh) {
  constexpr int S = Cfg<NP>::STAGES;
  for (int i = max(sh.flags[3], sh.flags[2] - S); i < sh.flags[2]; ++i)
    mbar_wait(smem_u32(&sh.full[i % S]), (i / S) & 1);
}

}  // namespace projk
}  // namespace gqa
