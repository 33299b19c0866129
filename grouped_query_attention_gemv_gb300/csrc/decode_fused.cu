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
//   * phase B needs the rotated queries and the new K/V rows: a CTA leaving
//     phase A at once requests its first KV units (all but a sequence's last
//     one) and waits until all 48 row tiles of phase A are published;
//   * phase C needs every sequence's attention output: a CTA leaving phase B
//     at once requests its first W_O tiles and waits until all valid
//     sequences are published.
// Waits are bounded (DEV_WAIT_TIMEOUT in the status word, then a clean exit).
// The last CTA out resets the counters, so the workspace is ready for the
// next call.
#include "attn_core.cuh"
#include "proj_core.cuh"

namespace gqa {

namespace {

constexpr int THREADS = (attnk::COMPUTE_WARPS + 1) * 32;  // 9 warps: attention needs them all
constexpr int QKV_TILES = QKV_ROWS / projk::TILE_ROWS;

struct FusedMaps {
  ProjStreamMaps qkv, o;
  CUtensorMap mk, mv;
};

struct FusedParams {
  ProjParams pq, po;
  float* part;     // projection partial slots
  int* tickets;    // projection row-tile tickets
  int segmax_q, segmax_o;
  DecodeAttnParams at;
  int* counters;   // [0] Q|K|V row tiles published, [1] sequences published, [2] CTAs done
};

template <int NP>
struct Layout {
  static constexpr int RING = projk::Cfg<NP>::RING > attnk::RING ? projk::Cfg<NP>::RING : attnk::RING;
  static constexpr int S = projk::Cfg<NP>::STAGES;
  static constexpr int BARS = 2 * (2 * S + 4) + 2 * attnk::STAGES;  // two projection sets + attention
  static constexpr int FIXED = RING + projk::Cfg<NP>::OUT_BYTES + BARS * 8 + 16 * 4 + 1024;
};

template <int NP>
__global__ void __launch_bounds__(THREADS, 1) decode_fused_kernel(const __grid_constant__ FusedMaps m, FusedParams fp) {
  using L = Layout<NP>;
  constexpr int S = L::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + L::RING);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::RING + projk::Cfg<NP>::OUT_BYTES);
  uint64_t* a_bars = bars;                       // phase A: full[S] empty[S] acc_full[2] acc_empty[2]
  uint64_t* c_bars = bars + (2 * S + 4);         // phase C: same
  uint64_t* b_bars = bars + 2 * (2 * S + 4);     // phase B: full[3] empty[3]
  int* ints = reinterpret_cast<int*>(bars + L::BARS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ints);
  int* flags_a = ints + 4;
  int* flags_b = ints + 8;
  int* flags_c = ints + 12;
  int* n_valid_s = ints + 1;
  int* pre = ints + 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (uint64_t* set : {a_bars, c_bars}) {
      for (int s = 0; s < S; ++s) {
        mbar_init(smem_u32(&set[s]), 1);
        mbar_init(smem_u32(&set[S + s]), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(smem_u32(&set[2 * S + b]), 1);
        mbar_init(smem_u32(&set[2 * S + 2 + b]), 4);
      }
    }
    for (int s = 0; s < attnk::STAGES; ++s) {
      mbar_init(smem_u32(&b_bars[s]), 1);
      mbar_init(smem_u32(&b_bars[attnk::STAGES + s]), attnk::COMPUTE_WARPS);
    }
    for (int i = 0; i < 4; ++i) flags_a[i] = flags_b[i] = flags_c[i] = 0;
    fence_barrier_init();
  }
  if (warp == attnk::COMPUTE_WARPS) {
    const int valid = attnk::build_prefix(fp.at, pre);
    if (lane == 0) *n_valid_s = valid;
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), projk::Cfg<NP>::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_valid = *n_valid_s;
  int* const cnt = fp.counters;

  // ---------------- phase A: Q|K|V projection, RoPE, cache append
  const projk::Shared<NP> sha{smem, a_bars, a_bars + S, a_bars + 2 * S, a_bars + 2 * S + 2, stage, flags_a, tmem};
  projk::proj_phase<NP, true>(
      m.qkv, fp.pq, fp.part, fp.tickets, fp.segmax_q, sha, []() { return true; },
      [cnt](int) { signal_counter(&cnt[0], 1); });
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool aborted = flags_a[0] != 0;

  // ---------------- phase B: attention (waits for every Q|K|V row tile)
  const attnk::Shared shb{smem, b_bars, b_bars + attnk::STAGES, flags_b, pre};
  if (!aborted) {
    attnk::attn_phase(
        m.mk, m.mv, fp.at, shb,
        [cnt]() {
          const bool ok = wait_counter(&cnt[0], QKV_TILES);
          fence_proxy_async_global();  // the new K/V rows were written by plain stores
          return ok;
        },
        [cnt]() {
          int ok = 0;
          if ((threadIdx.x & 31) == 0) ok = wait_counter(&cnt[0], QKV_TILES);
          return __shfl_sync(0xffffffffu, ok, 0) != 0;
        },
        [cnt](int) { signal_counter(&cnt[1], 1); });
    fence_proxy_async_smem();  // ldmatrix reads of the ring precede phase C's TMA writes into it
  }
  __syncthreads();
  aborted = aborted || flags_b[0] != 0;

  // ---------------- phase C: W_O projection (waits for every valid sequence)
  const projk::Shared<NP> shc{smem, c_bars, c_bars + S, c_bars + 2 * S, c_bars + 2 * S + 2, stage, flags_c, tmem};
  if (!aborted) {
    tc_fence_after();
    // The partial slots and tickets are phase A's as well. The producer's gate
    // below orders this phase's loads after every phase A merge; the epilogue
    // warps, which write the slots and take tickets, acquire the same counter
    // themselves (their first barrier passes it on to all four warps).
    if (threadIdx.x == 64) wait_counter(&cnt[0], QKV_TILES);
    projk::proj_phase<NP, false>(
        m.o, fp.po, fp.part, fp.tickets, fp.segmax_o, shc,
        [cnt, n_valid]() {
          // every Q|K|V tile as well: with no valid sequence phase B waits on
          // nothing, and the partial slots and tickets are shared with phase A
          const bool ok = wait_counter(&cnt[0], QKV_TILES) && wait_counter(&cnt[1], n_valid);
          fence_proxy_async_global();  // o was written by plain stores
          return ok;
        },
        [](int) {});
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && (aborted || flags_c[0])) {
    report(fp.pq.status, DEV_WAIT_TIMEOUT);
    if (flags_a[0]) projk::proj_drain(sha);
    if (flags_b[0]) attnk::attn_drain(shb);
    if (flags_c[0]) projk::proj_drain(shc);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, projk::Cfg<NP>::TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    // the last CTA out resets the grid counters for the next call
    __threadfence();
    if (atomicAdd(&cnt[2], 1) == static_cast<int>(gridDim.x) - 1) {
      cnt[0] = 0;
      cnt[1] = 0;
      cnt[2] = 0;
      __threadfence();
    }
  }
}

template <int NP>
cudaError_t launch_fused_np(const DecodeFusedArgs& a, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = decode_fused_kernel<NP>;
  const int max_smem = Layout<NP>::FIXED + (FUSED_MAX_B + 1) * 4;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (a.at.B <= 0 || a.at.B > FUSED_MAX_B) return cudaErrorInvalidValue;
  FusedMaps m;
  m.qkv = a.qkv_maps;
  m.o = a.o_maps;
  m.mk = a.mk;
  m.mv = a.mv;
  FusedParams fp;
  fp.pq = a.pq;
  fp.po = a.po;
  fp.part = a.part;
  fp.tickets = a.tickets;
  fp.segmax_q = a.segmax_q;
  fp.segmax_o = a.segmax_o;
  fp.at = a.at;
  fp.counters = a.counters;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = Layout<NP>::FIXED + (a.at.B + 1) * 4;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m, fp);
}

}  // namespace

cudaError_t launch_decode_fused(const DecodeFusedArgs& a, cudaStream_t s) {
  switch (proj_stream_np(a.pq.M)) {
    case 16: return launch_fused_np<16>(a, s);
    case 32: return launch_fused_np<32>(a, s);
    case 64: return launch_fused_np<64>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gqa
