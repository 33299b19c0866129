// Few-token projection y = x W^T (W stored [out, in]) in which every CTA owns
// whole output rows: the projection phases of the fused decode grid
// (decode_fused.cu). "Llama 3.1 8B · Query projection" and the K, V and
// output projections of "Grouped-query attention".
//
// At decode sizes a projection is a stream of its weights (50 MB for Q|K|V,
// 34 MB for W_O at bf16) against a handful of token rows, and in a grid that
// runs several phases back to back its end matters as much as its rate:
//   * the rows of each weight matrix are split over a share of the grid
//     proportional to its size (Q|K|V: 102 + 25 + 25 CTAs of 40 or 42 rows on
//     152 SMs; W_O: 152 CTAs of 26 or 28 rows), in pairs so that RoPE partners
//     stay together. Every CTA reads all 64 k blocks of its rows, so every CTA
//     streams the same bytes to within one row pair, and no CTA waits on
//     another: there is no cross-CTA reduction (the stream-K projection of
//     proj_core.cuh pays a chain of global round trips per row tile for it);
//   * a weight stage holds 4 k blocks of the CTA's h rows, fetched as ONE TMA
//     box of (64 k x h rows x 4 blocks) over a (k, row, k block) view of W: a
//     TMA request has a fixed cost, and four smaller boxes per stage measured
//     a lower rate per SM than the weight stream needs. The box lands dense,
//     row R = block * h + r at R * 128 bytes with the 128-byte swizzle of R,
//     which ldmatrix addresses directly (the MMAs here need no tensor-core
//     descriptor layout). The token rows of the same 4 k blocks (one box of 64
//     k x NP tokens x 4 blocks over the same view of x) go to a separate
//     ring: they come from L2, and every CTA reads all of them. One TMA
//     request a stage: 512 16-byte cp.async a stage through one warp issued
//     at ~0.27 us a stage and bounded the W_O phase, whose tokens only
//     become ready at its gate;
//   * CTAs walk the 16 stages from different starting points: were they in
//     step, every request in flight would fall in the same 512-byte window of
//     the 8 KB weight rows;
//   * the arithmetic is mma.sync m16n8k16 (bf16 in, fp32 accumulate) on the 8
//     compute warps: warp w takes k block w % 4 of every stage, up to 3 row
//     tiles of 16, and either half of that block's 64 k and every token (up
//     to 32 tokens: each weight fragment is read from shared memory once) or
//     all of its k and half of the tokens (64 tokens: the accumulators of all
//     tokens would not fit in registers). The step is bound by HBM, and with
//     so few tokens the cost per tensor instruction, not FLOPs, decides
//     whether the arithmetic keeps up: with 40-42 rows per CTA a tcgen05.mma
//     covers 16 k of a 64-row tile, and the 256 of them a CTA needs measured
//     slower than the weight stream itself, while 8 warps of mma.sync keep up;
//   * at the end the 8 warps' partials of every (row, token) are added in
//     shared memory, the pair (f, f+1) is rotated (Q|K|V), written as bf16
//     and published with one counter increment.
#pragma once

#include "kernels.h"
#include "norm_core.cuh"

namespace gqa {
namespace rowsk {

constexpr int KBLK = 64;
constexpr int NKB = D_MODEL / KBLK;      // 64 k blocks
constexpr int MT_MAX = ROWS_MAX_H / 16;  // row tiles of 16
constexpr int WARPS = 8;                 // compute warps 0-7; warp 8 lane 0 loads W, warp 9 lane 0 loads x
constexpr int MAX_STAGES = 12;           // weight stages (barrier pairs)
constexpr int RING_BYTES = 224 * 1024;   // weight ring + token ring
constexpr int OVERREAD = 1024;           // the last row tile may read up to 15 rows past a stage

constexpr int XS_MAX = 16;               // token stages at most (all of a phase's tokens)

// NP padded tokens; KC k blocks per stage (rows_kc: 8, or 4 at 64 tokens,
// whose warps split the tokens); XS token stages in flight (0: the default,
// 2). A phase whose weights come from HBM wants most of shared memory for
// them (few token stages); one whose weights are already in L2 but whose
// tokens only become ready when it starts wants the tokens in flight
// instead. INFL: weight stages requested but not yet landed, at most (the
// ring may hold more landed ones): with every SM streaming, ~85 KB a SM keep
// HBM busy, and each SM's reads and counter polls queue behind what it has
// in flight, so more only adds latency. Stages of 8 k blocks halve the
// per-stage cost every warp pays (a barrier wait and an arrive for the
// weights and for the tokens, ~0.25 us a stage).
// ONE: a single token (M = 1): its whole row is the one token slot, loaded
// once after the gate, and each warp builds the n8 tile's token fragments
// from it in registers (lanes 0-3 hold the token's column, the others the
// zero padding) instead of streaming 8-row token stages: the weight ring
// keeps the rest of shared memory.
template <int NP_, int XS_ = 0, int INFL_ = 0, bool ONE_ = false>
struct Cfg {
  static constexpr int NP = NP_;
  static constexpr bool ONE = ONE_;
  static constexpr int KC = rows_kc(NP_);
  static constexpr int NST = NKB / KC;              // stages per CTA
  static constexpr int INFL = INFL_ ? INFL_ : 4 * KBLK * 4 / (KC * KBLK);  // ~4 stages of 4 k blocks
  static constexpr int B_BYTES = NP * KBLK * 2;      // one k block of the token tile
  static constexpr int X_STAGE = KC * B_BYTES;       // the token rows of one weight stage
  static constexpr int XS = XS_ ? XS_ : 2;           // token stages
  static_assert(XS >= 1 && XS <= XS_MAX && XS <= NST, "token stages");
  static_assert(KC * (WARPS / KC) == WARPS || KC == WARPS, "warps per k block");
  static constexpr int X_RING = XS * X_STAGE;
  static constexpr int W_RING = RING_BYTES - X_RING;
  static constexpr bool TOKEN_SPLIT = NP > 32;      // warps split the tokens (else the k of a block)
  static constexpr int NT = TOKEN_SPLIT ? NP / 16 : NP / 8;  // n8 token tiles per warp
  static constexpr int RED_BYTES = WARPS * ROWS_MAX_H * NP * 4;  // per-warp partials, reuse the weight ring
  static_assert(RED_BYTES <= W_RING, "the reduction fits in the weight ring");
  static_assert(!ONE || (NT == 1 && XS == 1 && X_STAGE == D_MODEL * 2), "one token row fills the one token slot");
};

// Weight stage: kc k blocks of the phase's largest row count, rounded up to
// whole 1 KB swizzle atoms (so that every stage starts 1024-byte aligned).
__device__ __forceinline__ int wstage_bytes(const RowPlan& plan, int kc) {
  int hmax = 0;
  for (int i = 0; i < plan.nmat; ++i) hmax = max(hmax, plan.h_lo[i] + 2);
  return ((kc * hmax * 128 + 1023) / 1024) * 1024;
}

// This CTA's rows: matrix `mat`, rows [row0, row0 + h), map index hi (0: h_lo, 1: h_lo + 2).
// CTA c >= plan.cta0 (the others own no rows and run no phase of the plan).
struct MyRows {
  int mat, row0, h, hi;
};
__device__ __forceinline__ MyRows my_rows(const RowPlan& plan, int c) {
  c -= plan.cta0;
  int mat = 0;
  while (mat + 1 < plan.nmat && c >= plan.ctas[mat]) c -= plan.ctas[mat++];
  const int pairs = plan.rows[mat] / 2, n = plan.ctas[mat];
  const int p0 = static_cast<int>(static_cast<long long>(pairs) * c / n);
  const int p1 = static_cast<int>(static_cast<long long>(pairs) * (c + 1) / n);
  MyRows r;
  r.mat = plan.mat0 + mat;  // the RowMaps (and feature range) index
  r.row0 = 2 * p0;
  r.h = 2 * (p1 - p0);
  r.hi = r.h == plan.h_lo[mat] ? 0 : 1;
  return r;
}

// AND of `v` over the 256 compute threads (warps 0-7), with a barrier.
__device__ __forceinline__ bool compute_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 4, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

struct Shared {
  uint8_t* ring;    // RING_BYTES, 1024-aligned: weight ring, then token ring
  uint64_t* full;   // [MAX_STAGES], count 1
  uint64_t* empty;  // [MAX_STAGES], count WARPS
  uint64_t* xfull;  // [XS_MAX], count 1 (expect-tx)
  uint64_t* xempty; // [XS_MAX], count WARPS
  int* flags;       // [0] abort, [2] weight stages issued, [3] token stages issued
  float* rs;        // [NP] attention_norm scale of each token (Q|K|V phase of a layer call), or null
};

// One weight stage (i-th of this CTA's walk) into ring slot i % S.
template <class C_>
__device__ __forceinline__ void issue_w_stage(const CUtensorMap* wmap, const Shared& sh, int i, int S, int wstage,
                                              const MyRows& mr, int rot) {
  const int s = i % S, ks = (i + rot) % C_::NST;
  const uint32_t fb = smem_u32(&sh.full[s]);
  mbar_expect_tx(fb, C_::KC * mr.h * 128);
  tma_load_3d_stream(smem_u32(sh.ring + s * wstage), wmap, fb, 0, mr.row0, ks * C_::KC, l2_evict_first());
}
// The token rows of stage i into token slot i % XS.
template <class C_>
__device__ __forceinline__ void issue_x_stage(const CUtensorMap* xmap, const Shared& sh, int i, int rot) {
  const int s = i % C_::XS, ks = (i + rot) % C_::NST;
  const uint32_t fb = smem_u32(&sh.xfull[s]);
  mbar_expect_tx(fb, C_::X_STAGE);
  tma_load_3d(smem_u32(sh.ring + C_::W_RING + s * C_::X_STAGE), xmap, fb, 0, 0, ks * C_::KC);
}
template <class C_>
__device__ __forceinline__ int ring_stages(const RowPlan& plan) {
  return min(MAX_STAGES, (C_::W_RING - OVERREAD) / wstage_bytes(plan, C_::KC));
}

// Starts a phase's streams before the rest of the CTA is ready, for a phase
// that needs nothing from earlier phases: run by the weight producer (warp
// 8 lane 0) or the token producer (warp 9 lane 0) right after it has
// initialised its own barriers; it fills its ring and returns the stages
// requested, which rows_phase then skips.
template <class C_>
__device__ __forceinline__ int rows_start(const RowMaps& maps, const RowPlan& plan, const Shared& sh) {
  const MyRows mr = my_rows(plan, blockIdx.x);
  const int rot = (blockIdx.x * 7) % C_::NST;
  if ((threadIdx.x >> 5) == WARPS) {
    const int S = ring_stages<C_>(plan);
    const int D = min(S, C_::INFL);
    for (int i = 0; i < D; ++i)
      issue_w_stage<C_>(&maps.w[mr.mat][mr.hi], sh, i, S, wstage_bytes(plan, C_::KC), mr, rot);
    return D;
  }
  for (int i = 0; i < C_::XS; ++i) issue_x_stage<C_>(&maps.x, sh, i, rot);
  return C_::XS;
}

// One projection phase. Roles: warps 0-7 compute, warp 8 lane 0 loads the
// weights, warp 9 lane 0 the token rows; other lanes return at once. gate()
// runs on the token producer before its first load (false = give up; it
// orders the earlier phases' plain stores of the token rows before the
// token producer's TMA reads);
// prologue() runs on the 256 compute threads before they consume anything
// (other work of the grid that may overlap the first weight loads; false =
// give up); w_issued(drained) runs on the weight producer once all its loads
// are requested, `drained` a callable that waits until the phase no longer
// uses the ring past the cross-warp sums (the first RED_BYTES, which the
// epilogue reads); rows_done() runs on thread 0 once this CTA's rows are
// written and fenced. `started`: the stages the calling producer thread already
// requested in rows_start (0 if none).
template <class C_, bool QKV, class Gate, class Prologue, class WIssued, class RowsDone>
__device__ __forceinline__ void rows_phase(const RowMaps& maps, const ProjParams& p, const RowPlan& plan,
                                           const Shared& sh, Gate gate, Prologue prologue, WIssued w_issued,
                                           RowsDone rows_done, int started) {
  constexpr int NP = C_::NP;
  constexpr int XS = C_::XS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NST = C_::NST, KC = C_::KC;
  const MyRows mr = my_rows(plan, blockIdx.x);
  const int rot = (blockIdx.x * 7) % NST;  // this CTA's first k stage
  const int wstage = wstage_bytes(plan, KC);
  const int S = ring_stages<C_>(plan);
  uint8_t* const xring = sh.ring + C_::W_RING;
  int* flags = sh.flags;

  if (warp == WARPS) {
    if (lane != 0) return;
    // ---------------- weight producer: needs nothing from earlier phases
    const CUtensorMap* wmap = &maps.w[mr.mat][mr.hi];
    if (started == 0) tma_prefetch_desc(wmap);
    int i = started;
    for (; i < NST; ++i) {
      if (i >= S && !mbar_wait_or_abort(smem_u32(&sh.empty[i % S]), ((i / S) & 1) ^ 1, &flags[0])) {
        atomicExch(&flags[0], 1);
        break;
      }
      // at most INFL stages in flight: stage i - INFL must have landed
      if (i >= C_::INFL && C_::INFL < S &&
          !mbar_wait_or_abort(smem_u32(&sh.full[(i - C_::INFL) % S]), ((i - C_::INFL) / S) & 1, &flags[0])) {
        atomicExch(&flags[0], 1);
        break;
      }
      issue_w_stage<C_>(wmap, sh, i, S, wstage, mr, rot);
    }
    flags[2] = i;
    if (i == NST) {
      // drained(): waits (bounded) until the compute warps have released the
      // last stage's weights and tokens; every stage is then consumed and no
      // load of the phase is in flight. False if the phase gave up.
      const int l = NST - 1;
      w_issued([&]() {
        return mbar_wait_or_abort(smem_u32(&sh.empty[l % S]), (l / S) & 1, &flags[0]) &&
               (C_::ONE || mbar_wait_or_abort(smem_u32(&sh.xempty[l % XS]), (l / XS) & 1, &flags[0]));
      });
    }
    return;
  }
  if (warp == WARPS + 1) {
    if (lane != 0) return;
    // ---------------- token producer: the token rows may come from an earlier
    // phase (gate() waits for them). Rows past M read as zero (the map's rows
    // end at M).
    if constexpr (C_::ONE) {
      // the token's row, once
      const bool ok = gate();
      if (ok) {
        const uint32_t fb = smem_u32(&sh.xfull[0]);
        mbar_expect_tx(fb, C_::X_STAGE);
        bulk_load(smem_u32(xring), p.x, C_::X_STAGE, fb);
      } else {
        atomicExch(&flags[0], 1);
      }
      flags[3] = ok ? 1 : 0;
      return;
    }
    if (started == 0) tma_prefetch_desc(&maps.x);
    bool ok = gate();
    int i = started;
    for (; ok && i < NST; ++i) {
      if (i >= XS && !mbar_wait_or_abort(smem_u32(&sh.xempty[i % XS]), ((i / XS) & 1) ^ 1, &flags[0])) {
        ok = false;
        break;
      }
      issue_x_stage<C_>(&maps.x, sh, i, rot);
    }
    if (!ok) atomicExch(&flags[0], 1);
    flags[3] = i;
    return;
  }
  if (warp > WARPS + 1) return;

  // ---------------- compute warps: k block kb of every stage; k16 steps [ks0, ks0 + KS) of it and
  // tokens [tok0, tok0 + 8 NT)
  const int kb = warp & (KC - 1);
  constexpr int KS = C_::TOKEN_SPLIT ? 4 : 4 * KC / WARPS;
  const int ks0 = C_::TOKEN_SPLIT ? 0 : KS * (warp / KC);
  const int tok0 = C_::TOKEN_SPLIT ? (warp / KC) * (NP / 2) : 0;
  const int mtc = (mr.h + 15) >> 4;  // row tiles holding this CTA's rows
  // With few tokens the two k16 halves of a stage accumulate separately
  // (summed after the stream): an mma.sync result feeds the next product on
  // the same accumulator only after a long fixed latency, and one chain per
  // accumulator instead of two halves the stall each stage pays for it.
  constexpr int KH = C_::NT <= 2 ? 2 : 1;
  float acc[KH][MT_MAX][C_::NT][4];
#pragma unroll
  for (int h = 0; h < KH; ++h)
#pragma unroll
    for (int mt = 0; mt < MT_MAX; ++mt)
#pragma unroll
      for (int nt = 0; nt < C_::NT; ++nt)
        acc[h][mt][nt][0] = acc[h][mt][nt][1] = acc[h][mt][nt][2] = acc[h][mt][nt][3] = 0.f;

  // Each warp runs through the stages on its own (no per-stage barrier, so
  // that warps drift and cover each other's latencies); a warp whose bounded
  // wait gives up records it and leaves the loop. Every warp then meets the
  // others at the barrier after the loop, where the outcome is read.
  bool ok = prologue();
  // attention_norm folded in (a layer call): each token's 1/rms from its raw
  // row, while the first weight stages are in flight; the token fragments are
  // then normalised feature by feature (x * r * g, one bf16 rounding, as the
  // standalone norm kernel) just before the products
  const bool norm = QKV && p.norm_w != nullptr;
  float rn[C_::NT];
  if (norm) {
    for (int tok = warp; tok < NP; tok += WARPS) {
      float r = 0.f;
      if (tok < p.M) {
        uint4 v[NORM_VEC];
        norm_load_row(p.x + static_cast<size_t>(tok) * D_MODEL, lane, v);
        r = norm_inv_rms(v, p.eps);
      }
      if (lane == 0) sh.rs[tok] = r;
    }
    asm volatile("bar.sync 4, 256;" ::: "memory");
#pragma unroll
    for (int nt = 0; nt < C_::NT; ++nt) rn[nt] = sh.rs[tok0 + nt * 8 + (lane >> 2)];
  }
  // norm weights of this warp's features, one stage ahead of their use
  constexpr int NG = KS * 2;  // (KS / 2) k16 pairs x 4 chunks
  uint32_t gnext[NG];
  auto load_g = [&](int stage, uint32_t(&g)[NG]) {
    const int kbase = (((stage + rot) % NST) * KC + kb) * KBLK + 2 * (lane & 3);
#pragma unroll
    for (int j = 0; j < NG; ++j)
      g[j] = __ldg(reinterpret_cast<const uint32_t*>(p.norm_w + kbase + (2 * (ks0 + 2 * (j >> 2)) + (j & 3)) * 8));
  };
  if (norm) load_g(0, gnext);
  // the epilogue's first EPF items of this thread (item = (row pair, token)):
  // their start positions and RoPE factors are loaded during the stream, in
  // two steps (the start positions after stage EPF_SP, the factors, whose
  // address depends on them, after stage EPF_ROPE), so that no compute warp
  // waits on a load before its first stage: at the start of the grid every
  // load that misses L2 queues behind the whole grid's first weight stages
  const int fbase = (mr.mat == 0 ? 0 : (mr.mat == 1 ? p.r1 : p.r2)) + mr.row0;  // feature of row 0
  const int items = (mr.h / 2) * p.M;
  constexpr int EPF = 2, EPF_SP = 1, EPF_ROPE = NST / 2;
  int pos_pf[EPF], sp_pf[EPF];
  float2 cs_pf[EPF];
#pragma unroll
  for (int k = 0; k < EPF; ++k) {
    pos_pf[k] = -1;
    sp_pf[k] = -1;
    cs_pf[k] = make_float2(1.f, 0.f);
  }
  auto epf_start_positions = [&]() {
#pragma unroll
    for (int k = 0; k < EPF; ++k) {
      const int idx = threadIdx.x + k * WARPS * 32;
      if (idx < items) sp_pf[k] = p.sp.get((idx % p.M) / p.T);
    }
  };
  auto epf_rope = [&]() {
#pragma unroll
    for (int k = 0; k < EPF; ++k) {
      const int idx = threadIdx.x + k * WARPS * 32;
      if (idx < items && p.sp.ok(sp_pf[k])) {
        const int m = idx % p.M, f = fbase + 2 * (idx / p.M);
        pos_pf[k] = sp_pf[k] + (m - (m / p.T) * p.T);
        if (f < p.r2)
          cs_pf[k] = *reinterpret_cast<const float2*>(
              p.rope + (static_cast<size_t>(pos_pf[k]) * ROPE_PAIRS + ((f & (HEAD_DIM - 1)) >> 1)) * 2);
      }
    }
  };
  // stage i's slots in the two rings and their barrier phases, advanced by
  // one each stage: the ring size S is only known at run time, and a
  // division by it costs the consumer ~150 cycles a stage
  int s = 0, xs = 0;
  uint32_t ph = 0, xph = 0;
  if constexpr (C_::ONE) {
    // the token's row first
    if (ok && !__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&sh.xfull[0]), 0, &flags[0]))) {
      if (lane == 0) atomicExch(&flags[0], 1);
      ok = false;
    }
    // One token, every stage but the last already in the ring: the stages
    // are walked two deep, the fragments of stage i + 1 loaded while stage
    // i's products issue (one stage at a time measured ~0.33 us a stage, the
    // loads' and products' latencies in series). At most two row tiles
    // (the grid checks rows <= 32 before it picks this path).
    constexpr int NKS = KS / 2;
    constexpr int MT1 = 2;
    uint32_t af[2][NKS][2][MT1][4];
    uint32_t bf[2][NKS][4];
    auto load = [&](int i, int slot, uint32_t(&a)[NKS][2][MT1][4], uint32_t(&b)[NKS][4]) {
      const uint32_t wa = smem_u32(sh.ring + slot * wstage);
      const int rb = kb * mr.h;
      // fragment q of lane l < 4: features 16 ks + 8 q + 2 l, +1 of the token's row
      const uint32_t* xr = reinterpret_cast<const uint32_t*>(xring) + ((((i + rot) % NST) * KC + kb) * KBLK + 2 * lane) / 2;
#pragma unroll
      for (int j = 0; j < NKS; ++j) {
        const int ks = ks0 + 2 * j;
#pragma unroll
        for (int q = 0; q < 4; ++q) b[j][q] = lane < 4 ? xr[8 * ks + 4 * q] : 0u;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
          for (int mt = 0; mt < MT1; ++mt)
            if (mt < mtc) {
              const int r = rb + mt * 16 + (lane & 15);
              ldsm_x4(wa + sw128(r, 2 * (ks + kk) + (lane >> 4)), a[j][kk][mt][0], a[j][kk][mt][1], a[j][kk][mt][2],
                      a[j][kk][mt][3]);
            }
      }
    };
    auto products = [&](const uint32_t(&a)[NKS][2][MT1][4], const uint32_t(&b)[NKS][4]) {
#pragma unroll
      for (int j = 0; j < NKS; ++j)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
          for (int mt = 0; mt < MT1; ++mt)
            if (mt < mtc) mma16816(acc[kk % KH][mt][0], a[j][kk][mt][0], a[j][kk][mt][1], a[j][kk][mt][2], a[j][kk][mt][3],
                                   b[j][2 * kk], b[j][2 * kk + 1]);
    };
    // stage i: wait for its weights, load its fragments, release its slot
    auto take = [&](int i, int slot, uint32_t phase, uint32_t(&a)[NKS][2][MT1][4], uint32_t(&b)[NKS][4]) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&sh.full[slot]), phase, &flags[0]))) {
        if (lane == 0) atomicExch(&flags[0], 1);
        return false;
      }
      load(i, slot, a, b);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
      return true;
    };
    if (ok) ok = take(0, 0, 0u, af[0], bf[0]);
#pragma unroll
    for (int i = 0; i < NST; ++i) {
      if (!ok) break;
      if (i + 1 < NST) {
        if (++s == S) { s = 0; ph ^= 1u; }
        ok = take(i + 1, s, ph, af[(i + 1) & 1], bf[(i + 1) & 1]);
      }
      products(af[i & 1], bf[i & 1]);
    }
  }
  for (int i = 0; !C_::ONE && ok && i < NST; ++i) {
    uint32_t gcur[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) gcur[j] = gnext[j];
    if (norm && i + 1 < NST) load_g(i + 1, gnext);
    if (i > 0) {
      if (++s == S) { s = 0; ph ^= 1u; }
      if (++xs == XS) { xs = 0; xph ^= 1u; }
    }
    bool landed = mbar_wait_or_abort(smem_u32(&sh.full[s]), ph, &flags[0]);
    landed = landed && mbar_wait_or_abort(smem_u32(&sh.xfull[xs]), xph, &flags[0]);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) atomicExch(&flags[0], 1);
      ok = false;
      break;
    }
    const uint32_t wa = smem_u32(sh.ring + s * wstage);
    const int rb = kb * mr.h;  // this warp's k block starts at row rb of the stage
    const uint32_t xb = smem_u32(xring + xs * C_::X_STAGE + kb * C_::B_BYTES);
    if constexpr (C_::NT <= 2) {
      // with few tokens, every fragment of the stage first, then the
      // products: the loads are in flight together instead of one load's
      // latency before each product (more tokens: the registers are not there)
      constexpr int NKS = KS / 2;  // k16 pairs of this warp in the stage
      uint32_t bf[NKS][C_::NT][4];
      uint32_t af[NKS][2][MT_MAX][4];
#pragma unroll
      for (int j = 0; j < NKS; ++j) {
        const int ks = ks0 + 2 * j;
        // token fragments of two k16 steps: matrices (tokens, 16-byte chunks 2ks .. 2ks+3)
#pragma unroll
        for (int nt = 0; nt < C_::NT; ++nt) {
          const int tr = tok0 + nt * 8 + (lane & 7);
          ldsm_x4(xb + sw128(tr, 2 * ks + (lane >> 3)), bf[j][nt][0], bf[j][nt][1], bf[j][nt][2], bf[j][nt][3]);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
          for (int mt = 0; mt < MT_MAX; ++mt)
            if (mt < mtc) {
              const int r = rb + mt * 16 + (lane & 15);
              ldsm_x4(wa + sw128(r, 2 * (ks + kk) + (lane >> 4)), af[j][kk][mt][0], af[j][kk][mt][1], af[j][kk][mt][2],
                      af[j][kk][mt][3]);
            }
      }
      // the stage's slots are no longer read: release them before the
      // products (the arrive orders the warp's loads, which __syncwarp
      // orders before lane 0's arrive)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.empty[s]));
        mbar_arrive(smem_u32(&sh.xempty[xs]));
      }
      if (norm) {
        // fragment q holds token tok0 + nt*8 + lane/4, features k, k+1 of chunk 2ks + q
#pragma unroll
        for (int j = 0; j < NKS; ++j)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t g2 = gcur[j * 4 + q];
#pragma unroll
            for (int nt = 0; nt < C_::NT; ++nt) bf[j][nt][q] = norm_pair(bf[j][nt][q], rn[nt], g2);
          }
      }
#pragma unroll
      for (int j = 0; j < NKS; ++j)
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
          for (int mt = 0; mt < MT_MAX; ++mt)
            if (mt < mtc)
#pragma unroll
              for (int nt = 0; nt < C_::NT; ++nt)
                mma16816(acc[kk % KH][mt][nt], af[j][kk][mt][0], af[j][kk][mt][1], af[j][kk][mt][2], af[j][kk][mt][3],
                         bf[j][nt][2 * kk], bf[j][nt][2 * kk + 1]);
    } else {
#pragma unroll
      for (int ks = ks0; ks < ks0 + KS; ks += 2) {
        // token fragments of two k16 steps: matrices (tokens, 16-byte chunks 2ks .. 2ks+3)
        uint32_t b[C_::NT][4];
#pragma unroll
        for (int nt = 0; nt < C_::NT; ++nt) {
          const int tr = tok0 + nt * 8 + (lane & 7);
          ldsm_x4(xb + sw128(tr, 2 * ks + (lane >> 3)), b[nt][0], b[nt][1], b[nt][2], b[nt][3]);
        }
        if (norm) {
          // fragment q holds token tok0 + nt*8 + lane/4, features k, k+1 of chunk 2ks + q
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t g2 = gcur[((ks - ks0) >> 1) * 4 + q];
#pragma unroll
            for (int nt = 0; nt < C_::NT; ++nt) b[nt][q] = norm_pair(b[nt][q], rn[nt], g2);
          }
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
          for (int mt = 0; mt < MT_MAX; ++mt) {
            if (mt < mtc) {
              uint32_t a0, a1, a2, a3;
              const int r = rb + mt * 16 + (lane & 15);
              ldsm_x4(wa + sw128(r, 2 * (ks + kk) + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < C_::NT; ++nt)
                mma16816(acc[kk % KH][mt][nt], a0, a1, a2, a3, b[nt][2 * kk], b[nt][2 * kk + 1]);
            }
          }
        }
      }
    }
    if constexpr (C_::NT > 2) {  // the interleaved form reads the ring up to its last product
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sh.empty[s]));
        mbar_arrive(smem_u32(&sh.xempty[xs]));
      }
    }
    if constexpr (QKV) {
      if (i == EPF_SP) epf_start_positions();
      if (i == EPF_ROPE) epf_rope();
    }
  }
  if (!ok && lane == 0) atomicExch(&flags[0], 1);
  // every warp is past its stages (a producer may still give up at any time:
  // the vote gives every compute thread the same answer)
  if (!compute_all(ok && !*reinterpret_cast<volatile int*>(&flags[0]))) {
    if (lane == 0) atomicExch(&flags[0], 1);
    return;
  }
  // the weight ring now holds the warps' partials [WARPS][ROWS_MAX_H][NP]
  float* red = reinterpret_cast<float*>(sh.ring);
  {
    const int gr = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mt = 0; mt < MT_MAX; ++mt) {
      if (mt < mtc) {
#pragma unroll
        for (int nt = 0; nt < C_::NT; ++nt) {
          const int row = mt * 16 + gr, tok = tok0 + nt * 8 + 2 * t;
          float* d = red + (warp * ROWS_MAX_H + row) * NP + tok;
          float v[4] = {acc[0][mt][nt][0], acc[0][mt][nt][1], acc[0][mt][nt][2], acc[0][mt][nt][3]};
#pragma unroll
          for (int h = 1; h < KH; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] += acc[h][mt][nt][e];
          *reinterpret_cast<float2*>(d) = make_float2(v[0], v[1]);
          *reinterpret_cast<float2*>(d + 8 * NP) = make_float2(v[2], v[3]);
        }
      }
    }
  }
  asm volatile("bar.sync 4, 256;" ::: "memory");
  // epilogue: thread -> (row pair, token)
  auto item = [&](int idx, int pos, float2 cs) {
    const int m = idx % p.M, pr = idx / p.M;
    const int r = 2 * pr, f = fbase + r;
    float x0 = 0.f, x1 = 0.f;
    // the warps that hold token m: all 8, or the 4 of its half
    const int w0 = C_::TOKEN_SPLIT ? (m / (NP / 2)) * KC : 0;
#pragma unroll
    for (int w = 0; w < (C_::TOKEN_SPLIT ? KC : WARPS); ++w) {
      x0 += red[((w0 + w) * ROWS_MAX_H + r) * NP + m];
      x1 += red[((w0 + w) * ROWS_MAX_H + r + 1) * NP + m];
    }
    __nv_bfloat16* dst;
    if constexpr (QKV) {
      if (pos < 0) return;  // a start position out of range (reported by the attention)
      const int b = m / p.T;
      if (f < p.r2) {
        const float y0 = x0 * cs.x - x1 * cs.y;
        const float y1 = x0 * cs.y + x1 * cs.x;
        x0 = y0;
        x1 = y1;
      }
      if (f < D_MODEL) {
        dst = p.out + static_cast<size_t>(m) * D_MODEL + f;
      } else {
        const size_t row = (static_cast<size_t>(b) * p.s_max + pos) * (p.r2 - p.r1);
        dst = f < p.r2 ? p.cache_k + row + (f - D_MODEL) : p.cache_v + row + (f - p.r2);
      }
    } else {
      dst = p.out + static_cast<size_t>(m) * p.N + f;
      if (p.resid) {  // the block's residual
        const uint32_t rv = *reinterpret_cast<const uint32_t*>(p.resid + static_cast<size_t>(m) * p.N + f);
        x0 += bf16_lo(rv);
        x1 += bf16_hi(rv);
      }
    }
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(x0, x1);
  };
#pragma unroll
  for (int k = 0; k < EPF; ++k) {
    const int idx = threadIdx.x + k * WARPS * 32;
    if (idx < items) item(idx, pos_pf[k], cs_pf[k]);
  }
  for (int idx = threadIdx.x + EPF * WARPS * 32; idx < items; idx += WARPS * 32) {
    float2 cs = make_float2(1.f, 0.f);
    int pos = -1;
    if constexpr (QKV) {
      const int m = idx % p.M, f = fbase + 2 * (idx / p.M);
      const int b = m / p.T;
      const int start = p.sp.get(b);
      if (p.sp.ok(start)) {
        pos = start + (m - b * p.T);
        if (f < p.r2)
          cs = *reinterpret_cast<const float2*>(
              p.rope + (static_cast<size_t>(pos) * ROPE_PAIRS + ((f & (HEAD_DIM - 1)) >> 1)) * 2);
      }
    }
    item(idx, pos, cs);
  }
  // later phases of the grid read the Q|K|V rows by TMA (the W_O phase is
  // the grid's last: its rows are only read after the kernel boundary). The
  // rows reach other CTAs through rows_done's release on thread 0 after the
  // barrier, which covers every thread's stores before it; a full fence per
  // thread would wait for each thread's own stores (~0.5 us) for nothing
  if constexpr (QKV) fence_proxy_async_global();
  asm volatile("bar.sync 4, 256;" ::: "memory");
  if (threadIdx.x == 0) rows_done();
}

// After an aborted phase: let loads that were issued but never consumed land
// (bounded) before the shared memory is reused or the CTA exits. One thread.
template <class C_>
__device__ __forceinline__ void rows_drain(const Shared& sh, const RowPlan& plan) {
  constexpr int XS = C_::XS;
  const int S = ring_stages<C_>(plan);
  for (int i = max(0, sh.flags[2] - S); i < sh.flags[2]; ++i) mbar_wait(smem_u32(&sh.full[i % S]), (i / S) & 1);
  for (int i = max(0, sh.flags[3] - XS); i < sh.flags[3]; ++i) mbar_wait(smem_u32(&sh.xfull[i % XS]), (i / XS) & 1);
}

}  // namespace rowsk
}  // namespace gqa
