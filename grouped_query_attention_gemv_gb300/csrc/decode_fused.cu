// One decode step of the attention block in a single persistent grid: the
// Q|K|V projection with RoPE and cache append (phase A), the decode attention
// (phase B) and the W_O projection (phase C) of "Llama 3.1 8B · Grouped-query
// attention", run back to back by one CTA per SM (cooperative launch, so
// every CTA is resident).
//
// Why one grid: each phase alone is a short, HBM-bound stream (50, 66 and
// 34 MB at B = 16, P = 1000). Run as separate kernels, every boundary costs
// the slowest CTA's tail plus the teardown and launch of the next grid, all
// with HBM idle. Here phases are ordered by grid-wide counters instead:
//   * both projections are row-owner phases (proj_rows.cuh): a CTA finishes
//     its rows without waiting on any other CTA;
//   * phase B needs the rotated queries and the new K/V rows: a CTA leaving
//     phase A at once requests its first KV stages (all but the one holding a
//     sequence's new row) and waits until every CTA has published its phase
//     A rows;
//   * phase B runs one of two work splits (attn_core.cuh): position-major
//     units spread evenly over the grid, whose CTAs meet once and merge the
//     partials of sequences split between them; or, for a small batch of
//     short contexts, one (sequence, KV head) pair per CTA, with nothing to
//     merge across CTAs (the host picks; see the launch arguments);
//   * phase C needs every sequence's attention output: a CTA leaving phase B
//     at once requests its first W_O stages and waits until every CTA has
//     published its outputs.
// Each phase keeps at most a few weight stages in flight per SM: deeper
// queues do not raise the stream's rate, and every counter poll and grid
// hand-over waits behind the bytes an SM has in flight.
// The grid is launched with programmatic stream serialization: a step that
// follows another kernel of the stream is set up by the hardware while that
// kernel finishes (~0.4 us per step), and every thread executes
// griddepcontrol.wait before its first global access, so the step sees all
// that the previous kernel wrote and overwrites nothing it still reads, as
// in plain stream order. (Its CTAs, one per SM, start only when the previous
// grid has left the SMs: a request of weights before the wait gained nothing
// measurable and is not made.)
// Waits are bounded (DEV_WAIT_TIMEOUT in the status word, then a clean exit).
// The last CTA out resets the counters, so the workspace is ready for the
// next call.
#include "attn_core.cuh"
#include "proj_rows.cuh"

namespace gqa {

bool make_row_plan(int nmat, const int* rows, int ctas, RowPlan* plan) {
  if (nmat < 1 || nmat > 3 || ctas < nmat) return false;
  long long total = 0;
  for (int i = 0; i < nmat; ++i) {
    if (rows[i] <= 0 || (rows[i] & 1)) return false;
    total += rows[i];
  }
  *plan = RowPlan{};
  plan->nmat = nmat;
  int given = 0;
  for (int i = nmat - 1; i >= 1; --i) {  // the smaller matrices first, the rest to matrix 0
    plan->ctas[i] = static_cast<int>((static_cast<long long>(ctas) * rows[i] + total / 2) / total);
    if (plan->ctas[i] < 1) plan->ctas[i] = 1;
    given += plan->ctas[i];
  }
  plan->ctas[0] = ctas - given;
  for (int i = 0; i < nmat; ++i) {
    if (plan->ctas[i] < 1) return false;
    const int pairs = rows[i] / 2;
    plan->rows[i] = rows[i];
    plan->h_lo[i] = 2 * (pairs / plan->ctas[i]);
    const int h_hi = 2 * ((pairs + plan->ctas[i] - 1) / plan->ctas[i]);
    if (plan->h_lo[i] < 2 || h_hi > ROWS_MAX_H) return false;
  }
  return true;
}

namespace {

// warps 0-7 compute; 8 loads (weights in the projections, the cache in the
// attention); 9 loads the projections' token rows
constexpr int THREADS = (rowsk::WARPS + 2) * 32;
static_assert(attnk::COMPUTE_WARPS == rowsk::WARPS, "phases share the compute warps");
struct FusedMaps {
  RowMaps qkv, o;
  DecodeCacheMaps cache;     // position-major view (units of 16 positions x 8 heads)
  DecodeCacheMaps cache_hm;  // head-major view (stages of 128 positions of one head)
};

struct FusedParams {
  ProjParams pq, po;
  RowPlan qkv_plan, o_plan;
  DecodeAttnParams at;
  int* counters;   // [0] CTAs whose Q|K|V rows are published, [1] CTAs whose attention outputs are published,
                   // [2] CTAs done, [3] the attention's meeting before its merges
  int head_major;  // phase B: one (sequence, KV head) pair per CTA (1) or position-major units (0)
};

// Phase A streams its weights from HBM as soon as the grid starts: the
// default (short) token ring, about 85 KB of weight stages in flight per SM
// (13 MB over the grid, 2 us of HBM time). Phase C requests its first weight
// stages while the grid finishes the attention; its tokens, the attention
// output, only become ready at the gate. Once past the gate its consumer
// waits on weight stages that take ~1.2 us to land, so the period per stage
// is that latency over the stages in flight: up to 16 tokens, 4 token stages
// (half the output) leave 5-6 weight slots, 3 of them in flight (B = 16:
// -0.3 us per step, B = 1: -0.6 us against 8 token stages and 2 in flight).
// (Asking L2 for the rest of W_O at the same time measured 1.5 us slower per
// step at B = 16: the requests queue ahead of the merge and the gate.)
template <int NP>
using CfgA = rowsk::Cfg<NP>;
template <int NP>
using CfgC = rowsk::Cfg<NP, NP <= 16 ? 4 : (NP == 32 ? 4 : 3), NP <= 16 ? 3 : 0>;
// One sequence (one token): its attention output row is loaded once after
// the gate and the W_O ring keeps the four token stages' 24 KB, 7 of a CTA's
// 8 weight stages instead of 6, all requested before the gate.
using CfgC1 = rowsk::Cfg<8, 1, 3, true>;

template <int NP>
struct Layout {
  static constexpr int RING = rowsk::RING_BYTES > attnk::RING ? rowsk::RING_BYTES : attnk::RING;
  static constexpr int PSET = 2 * rowsk::MAX_STAGES + 2 * rowsk::XS_MAX;   // barriers of one projection
  static constexpr int BARS = 2 * PSET + 2 * attnk::STAGES;                // two projections + attention
  static constexpr int FIXED = RING + BARS * 8 + 16 * 4 + FUSED_MAX_B * 4 + 1024;  // ..., flags, norm scales
  // the attention's output staging lies past its ring, inside the projections' ring
  static_assert(attnk::RING + attnk::STAGE_OUT_BYTES <= RING, "attention staging fits");
  static_assert(FIXED + (FUSED_MAX_B + 1) * 4 <= 227 * 1024, "shared memory of one CTA");
};

// NREP: query heads per KV head, 4 (8 KV heads) or 1 (the multi-head variant:
// 32 KV heads, Wk and Wv of 4,096 rows each; phase A walks Wq, Wk and Wv in
// three passes over the grid, the attention runs each sequence as 4 groups
// of 8 KV heads, position-major).
template <int NP, int NREP>
__global__ void __launch_bounds__(THREADS, 1) decode_fused_kernel(const __grid_constant__ FusedMaps m, FusedParams fp) {
  using L = Layout<NP>;
  constexpr int NG = N_REP / NREP;  // head groups of 8 KV heads per sequence
  constexpr int MS = rowsk::MAX_STAGES, XS = rowsk::XS_MAX;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::RING);
  uint64_t* a_bars = bars;                // phase A: full[MS] empty[MS] xfull[XS] xempty[XS]
  uint64_t* c_bars = bars + L::PSET;      // phase C: same
  uint64_t* b_bars = bars + 2 * L::PSET;  // phase B: full[3] empty[3]
  int* ints = reinterpret_cast<int*>(bars + L::BARS);
  int* flags_a = ints + 4;
  int* flags_b = ints + 8;
  int* flags_c = ints + 12;
  float* rs = reinterpret_cast<float*>(ints + 16);  // [FUSED_MAX_B] attention_norm scales (layer calls)
  int* pre = ints + 16 + FUSED_MAX_B;

  // everything below may touch what the previous kernel of the stream wrote;
  // a dependent step may be set up as soon as every CTA of this one runs
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5;
  const rowsk::Shared sha{smem, a_bars, a_bars + MS, a_bars + 2 * MS, a_bars + 2 * MS + XS, flags_a, rs};
  // phase A needs nothing from the grid: its two producers set up their own
  // barriers and request their first stages at once, before the CTA's setup
  // (the prefix of attention units reads the start positions) is done
  int a_started = 0;
  if (threadIdx.x == rowsk::WARPS * 32 || threadIdx.x == (rowsk::WARPS + 1) * 32) {
    const bool wprod = threadIdx.x == rowsk::WARPS * 32;
    const int n = wprod ? MS : XS;
    uint64_t* fullb = wprod ? sha.full : sha.xfull;
    uint64_t* emptyb = wprod ? sha.empty : sha.xempty;
    for (int s = 0; s < n; ++s) {
      mbar_init(smem_u32(&fullb[s]), 1);
      mbar_init(smem_u32(&emptyb[s]), rowsk::WARPS);
    }
    fence_barrier_init();
    a_started = rowsk::rows_start<CfgA<NP>>(m.qkv, fp.qkv_plan, sha);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < MS; ++s) {
      mbar_init(smem_u32(&c_bars[s]), 1);
      mbar_init(smem_u32(&c_bars[MS + s]), rowsk::WARPS);
    }
    for (int s = 0; s < XS; ++s) {
      mbar_init(smem_u32(&c_bars[2 * MS + s]), 1);
      mbar_init(smem_u32(&c_bars[2 * MS + XS + s]), rowsk::WARPS);
    }
    for (int s = 0; s < attnk::STAGES; ++s) {
      mbar_init(smem_u32(&b_bars[s]), 1);
      mbar_init(smem_u32(&b_bars[attnk::STAGES + s]), attnk::COMPUTE_WARPS);
    }
    for (int i = 0; i < 4; ++i) flags_a[i] = flags_b[i] = flags_c[i] = 0;
    fence_barrier_init();
  }
  // (nothing here may wait on a global load: at the start of the grid a load
  // that misses L2 queues behind every CTA's first weight stages, ~3 us)
  __syncthreads();
  const int grid = static_cast<int>(gridDim.x);
  int* const cnt = fp.counters;

  const attnk::Shared shb{smem, b_bars, b_bars + attnk::STAGES, flags_b, pre,
                          reinterpret_cast<float*>(smem + attnk::RING)};

  // ---------------- phase A: Q|K|V projection, RoPE, cache append. With the
  // head-major split, its weight producer requests the first KV stage (into
  // a ring slot past the first, which holds the epilogue's sums) once the
  // phase's last stage is consumed: HBM keeps streaming through the
  // epilogue, and the stage has landed before the gate's poll.
  if constexpr (NREP == N_REP) {
    rowsk::rows_phase<CfgA<NP>, true>(
        m.qkv, fp.pq, fp.qkv_plan, sha, []() { return true; }, []() { return true; },
        [&fp, &m, &shb](auto drained) {
          if constexpr (CfgA<NP>::RED_BYTES <= attnk::UNIT_BYTES) {
            if (fp.head_major && drained()) attnk::attn_items_early(m.cache_hm.k, m.cache_hm.v, fp.at, shb);
          }
        },
        [cnt]() { signal_counter(&cnt[0], 1); }, a_started);
  } else {
    // 32 KV heads: Wq, Wk and Wv in turn, each of its 4,096 rows split over
    // the grid as W_O's are; the CTA publishes its rows once, after the last
    // pass (thread 0's release after the epilogue's barrier covers all three)
    for (int pass = 0; pass < 3; ++pass) {
      if (pass > 0) {
        // the ring's generic reads and writes precede the next pass's TMA
        // writes; every load of the pass has landed and been consumed, so
        // its barriers start again from phase 0
        fence_proxy_async_smem();
        __syncthreads();
        if (flags_a[0]) break;
        if (threadIdx.x == 0) {
          for (int s = 0; s < MS; ++s) {
            mbar_inval(smem_u32(&sha.full[s]));
            mbar_inval(smem_u32(&sha.empty[s]));
            mbar_init(smem_u32(&sha.full[s]), 1);
            mbar_init(smem_u32(&sha.empty[s]), rowsk::WARPS);
          }
          for (int s = 0; s < XS; ++s) {
            mbar_inval(smem_u32(&sha.xfull[s]));
            mbar_inval(smem_u32(&sha.xempty[s]));
            mbar_init(smem_u32(&sha.xfull[s]), 1);
            mbar_init(smem_u32(&sha.xempty[s]), rowsk::WARPS);
          }
          flags_a[2] = 0;
          fence_barrier_init();
        }
        __syncthreads();
      }
      RowPlan pp = fp.qkv_plan;
      pp.mat0 = pass;
      rowsk::rows_phase<CfgA<NP>, true>(
          m.qkv, fp.pq, pp, sha, []() { return true; }, []() { return true; }, [](auto) {},
          [cnt, pass]() {
            if (pass == 2) signal_counter(&cnt[0], 1);
          },
          pass == 0 ? a_started : 0);
    }
  }
  fence_proxy_async_smem();  // the ring's generic reads and writes precede phase B's TMA writes into it
  __syncthreads();
  bool aborted = flags_a[0] != 0;
  if (!fp.head_major) {
    // the position-major split's unit prefix (the start positions are in L2 by now)
    if (warp == rowsk::WARPS - 1) attnk::build_prefix<NG>(fp.at, pre);
    __syncthreads();
  }

  // ---------------- phase B: attention units (waits for every CTA's Q|K|V rows)
  bool units_ok = true;
  if (!aborted) {
    // one poller per CTA: the producer lane waits on the grid counter and
    // hands the outcome to the compute warps through shared memory (lane 0
    // of every compute warp polling the counter as well measured 0.4 us
    // slower at B = 16)
    auto gate_lane = [cnt, grid, flags_b, &fp]() {
      const bool ok = wait_counter(&cnt[0], grid, fp.at.wait_ns);
      fence_proxy_async_global();  // the new K/V rows were written by plain stores
      st_release_cta(&flags_b[1], ok ? 1 : 2);
      return ok;
    };
    auto gate_warp = [flags_b]() {
      int v = 0;
      if ((threadIdx.x & 31) == 0) v = wait_flag_cta(&flags_b[1]);
      return __shfl_sync(0xffffffffu, v, 0) == 1;
    };
    if constexpr (NREP == N_REP) {
      if (fp.head_major)
        units_ok = attnk::attn_items(m.cache_hm.k, m.cache_hm.v, fp.at, shb, gate_lane, gate_warp);
      else
        units_ok = attnk::attn_units<NREP>(m.cache.k, m.cache.v, fp.at, shb, gate_lane, gate_warp, []() {});
    } else {
      units_ok = attnk::attn_units<NREP>(m.cache.k, m.cache.v, fp.at, shb, gate_lane, gate_warp, []() {});
    }
    fence_proxy_async_smem();  // ldmatrix reads of the ring precede phase C's TMA writes into it
  }
  __syncthreads();
  // Head-major outputs are complete: publish them (thread 0's release after
  // the barrier covers every thread's stores) before phase C's weight loads
  // are in flight, because a release on an SM waits for the bulk loads that
  // SM has in flight (~1.5 us more when W_O's stages are out).
  const bool early_signal = fp.head_major && !aborted;
  if (early_signal) {
    if (threadIdx.x == 0) signal_counter(&cnt[1], 1);
    __syncthreads();
  }

  // ---------------- phase C: W_O projection. Its weight loads start at once;
  // meanwhile the compute warps meet the grid and merge the attention
  // outputs of split sequences; its token loads wait for every CTA's outputs.
  const rowsk::Shared shc{smem, c_bars, c_bars + MS, c_bars + 2 * MS, c_bars + 2 * MS + XS, flags_c, nullptr};
  // one sequence, and W_O rows of at most two row tiles per CTA
  const bool one_token_c = NP == 8 && fp.po.M == 1 && fp.o_plan.h_lo[0] + 2 <= 32;
  if (!aborted && flags_b[0]) {
    // this CTA's units gave up: it still meets the grid (no other CTA waits in vain)
    if (warp < attnk::COMPUTE_WARPS) {
      if (!fp.head_major) attnk::attn_merge<NREP>(fp.at, shb, &cnt[3], false);
      if (threadIdx.x == 0 && !early_signal) signal_counter(&cnt[1], 1);
    }
  } else if (!aborted && static_cast<int>(blockIdx.x) < fp.o_plan.cta0) {
    // no W_O rows here (a head-major attention CTA of a small batch: its
    // outputs are published already, it has nothing to merge)
  } else if (!aborted) {
    auto phase_c = [&](auto cfg) {
      rowsk::rows_phase<decltype(cfg), false>(m.o, fp.po, fp.o_plan, shc,
                                              [cnt, grid, &fp]() {
                                                const bool ok = wait_counter(&cnt[1], grid, fp.at.wait_ns);
                                                fence_proxy_async_global();  // o was written by plain stores
                                                return ok;
                                              },
                                              [&fp, &shb, cnt, units_ok, early_signal]() {
                                                // head-major outputs need no merge (attn_items fenced them
                                                // and they are published already)
                                                if (early_signal) return units_ok;
                                                const bool ok = attnk::attn_merge<NREP>(fp.at, shb, &cnt[3], units_ok);
                                                // this CTA's attention outputs (whole sequences, merges)
                                                // are fenced
                                                if (threadIdx.x == 0) signal_counter(&cnt[1], 1);
                                                return ok;
                                              },
                                              [](auto) {}, []() {}, 0);
    };
    if (one_token_c)
      phase_c(CfgC1{});
    else
      phase_c(CfgC<NP>{});
  }
  aborted = aborted || flags_b[0] != 0;
  __syncthreads();
  if (threadIdx.x == 0 && (aborted || flags_c[0])) {
    report(fp.pq.status, DEV_WAIT_TIMEOUT);
    if (flags_a[0]) rowsk::rows_drain<CfgA<NP>>(sha, fp.qkv_plan);
    // (phase A's producer may have requested head-major stages before phase A gave up)
    if (flags_a[0] || flags_b[0]) attnk::attn_drain(shb, fp.head_major ? attnk::ITEM_ROT : 0);
    if (flags_c[0]) {
      if (one_token_c)
        rowsk::rows_drain<CfgC1>(shc, fp.o_plan);
      else
        rowsk::rows_drain<CfgC<NP>>(shc, fp.o_plan);
    }
  }
  if (threadIdx.x == 0) {
    // the last CTA out resets the grid counters for the next call (every
    // CTA has passed its last wait when it arrives here; the next call sees
    // the reset through the kernel boundary, so no fence is needed)
    if (atomicAdd(&cnt[2], 1) == grid - 1) {
      cnt[0] = 0;
      cnt[1] = 0;
      cnt[2] = 0;
      cnt[3] = 0;
    }
  }
}

template <int NP, int NREP>
cudaError_t launch_fused_np(const DecodeFusedArgs& a, cudaStream_t s) {
  static bool attr_set[64] = {};
  constexpr int NG = N_REP / NREP;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = decode_fused_kernel<NP, NREP>;
  const int max_smem = Layout<NP>::FIXED + (FUSED_MAX_B + 1) * 4;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // the unit prefix over B * NG virtual sequences lives in shared memory
  if (a.at.B <= 0 || a.at.B * NG > FUSED_MAX_B) return cudaErrorInvalidValue;
  if (a.qkv_passes != (NREP == N_REP ? 1 : 3) || (NREP != N_REP && a.qkv_plan.nmat != 1)) return cudaErrorInvalidValue;
  int planned = 0;
  for (int i = 0; i < a.qkv_plan.nmat; ++i) planned += a.qkv_plan.ctas[i];
  if (planned != a.ctas || a.qkv_plan.cta0 != 0 || a.o_plan.nmat != 1 || a.o_plan.cta0 < 0 ||
      a.o_plan.cta0 + a.o_plan.ctas[0] != a.ctas || (a.o_plan.cta0 > 0 && !a.head_major))
    return cudaErrorInvalidValue;
  FusedMaps m;
  m.qkv = a.qkv_maps;
  m.o = a.o_maps;
  m.cache = a.cache;
  m.cache_hm = a.cache_hm;
  FusedParams fp;
  fp.pq = a.pq;
  fp.po = a.po;
  fp.qkv_plan = a.qkv_plan;
  fp.o_plan = a.o_plan;
  fp.at = a.at;
  fp.counters = a.counters;
  fp.head_major = a.head_major;
  if (a.head_major && (NREP != N_REP || a.at.B * N_KV > a.ctas)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Layout<NP>::FIXED + (a.at.B * NG + 1) * 4;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, m, fp);
}

}  // namespace

int decode_fused_np(int M) {
  return M <= 8 ? 8 : proj_stream_np(M);  // 8: half the tensor work of 16 padded tokens
}

cudaError_t launch_decode_fused(const DecodeFusedArgs& a, cudaStream_t s) {
  if (a.at.n_kv == N_KV) {
    switch (decode_fused_np(a.pq.M)) {
      case 8: return launch_fused_np<8, N_REP>(a, s);
      case 16: return launch_fused_np<16, N_REP>(a, s);
      case 32: return launch_fused_np<32, N_REP>(a, s);
      case 64: return launch_fused_np<64, N_REP>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (a.at.n_kv == N_HEADS) {  // the multi-head variant, up to 16 sequences
    switch (decode_fused_np(a.pq.M)) {
      case 8: return launch_fused_np<8, 1>(a, s);
      case 16: return launch_fused_np<16, 1>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace gqa
