// Standalone decode attention kernel (the decode path for batches above the
// few-token projection size): the attention phase of attn_core.cuh in its own
// persistent grid, launched cooperatively because its CTAs meet before the
// merges.
#include "attn_core.cuh"

namespace gqa {

namespace {

constexpr int THREADS = (attnk::COMPUTE_WARPS + 1) * 32;
constexpr int FIXED_SMEM = attnk::RING + attnk::STAGE_OUT_BYTES + 1024 + 2 * attnk::STAGES * 8 + 4 * 4;

// NREP: query heads per KV head (4; 1 for the multi-head variant)
template <int NREP>
__global__ void __launch_bounds__(THREADS, 1) attn_decode_kernel(const __grid_constant__ DecodeCacheMaps maps,
                                                                 DecodeAttnParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stage_out = reinterpret_cast<float*>(smem + attnk::RING);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + attnk::RING + attnk::STAGE_OUT_BYTES);
  uint64_t* empty = full + attnk::STAGES;
  int* flags = reinterpret_cast<int*>(empty + attnk::STAGES);
  int* pre = flags + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == attnk::COMPUTE_WARPS) {
    attnk::build_prefix<N_REP / NREP>(a, pre);
    if (lane == 0) {
      for (int s = 0; s < attnk::STAGES; ++s) {
        mbar_init(smem_u32(&full[s]), 1);
        mbar_init(smem_u32(&empty[s]), attnk::COMPUTE_WARPS);
      }
      flags[0] = flags[1] = flags[2] = flags[3] = 0;
      fence_barrier_init();
    }
  }
  __syncthreads();
  const attnk::Shared sh{smem, full, empty, flags, pre, stage_out};
  // the projection that wrote the queries and the new rows ran before this grid
  auto pass = []() { return true; };
  const bool ok = attnk::attn_units<NREP>(maps.k, maps.v, a, sh, pass, pass, []() {});
  if (warp < attnk::COMPUTE_WARPS) attnk::attn_merge<NREP>(a, sh, &a.counters[0], ok);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (flags[0]) {
      report(a.status, DEV_WAIT_TIMEOUT);
      attnk::attn_drain(sh);
    }
    // the last CTA out resets the grid counters for the next call
    __threadfence();
    if (atomicAdd(&a.counters[1], 1) == static_cast<int>(gridDim.x) - 1) {
      a.counters[0] = 0;
      a.counters[1] = 0;
      __threadfence();
    }
  }
}

template <int NREP>
cudaError_t launch_nrep(const DecodeCacheMaps& maps, const DecodeAttnParams& a, cudaStream_t s) {
  static bool attr_set[64] = {};
  constexpr int NG = N_REP / NREP;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = attn_decode_kernel<NREP>;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FIXED_SMEM + (DECODE_MAX_B + 1) * 4);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // the prefix over B * NG virtual sequences lives in shared memory
  if (a.B <= 0 || a.B * NG > DECODE_MAX_B) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = FIXED_SMEM + (a.B * NG + 1) * 4;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps, a);
}

}  // namespace

int attn_decode_ctas(int num_sms) { return num_sms; }
int attn_decode_slots(int ctas) { return 2 * ctas * N_KV; }

cudaError_t launch_attn_decode(const DecodeCacheMaps& maps, const DecodeAttnParams& a, cudaStream_t s) {
  switch (a.n_kv) {
    case N_KV: return launch_nrep<N_REP>(maps, a, s);
    case N_HEADS: return launch_nrep<1>(maps, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gqa
