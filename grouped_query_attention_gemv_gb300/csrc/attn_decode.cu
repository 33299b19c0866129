// Standalone decode attention kernel (the decode path for batches above the
// few-token projection size): the attention phase of attn_core.cuh in its own
// grid, ordered after the projection by programmatic dependent launch.
#include "attn_core.cuh"

namespace gqa {

namespace {

constexpr int THREADS = (attnk::COMPUTE_WARPS + 1) * 32;
constexpr int FIXED_SMEM = attnk::RING + 1024 + 2 * attnk::STAGES * 8 + 4 * 4;

__global__ void __launch_bounds__(THREADS, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                       DecodeAttnParams a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + attnk::RING);
  uint64_t* empty = full + attnk::STAGES;
  int* flags = reinterpret_cast<int*>(empty + attnk::STAGES);
  int* pre = flags + 4;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == attnk::COMPUTE_WARPS) {
    attnk::build_prefix(a, pre);
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
  const attnk::Shared sh{smem, full, empty, flags, pre};
  auto gate = []() {
    pdl_wait();
    return true;
  };
  attnk::attn_phase(mk, mv, a, sh, gate, gate, [](int) {});
  pdl_wait();  // never complete before the predecessor grid: the next kernel relies on it
  __syncthreads();
  if (flags[0] && threadIdx.x == attnk::COMPUTE_WARPS * 32) {
    report(a.status, DEV_WAIT_TIMEOUT);
    attnk::attn_drain(sh);
  }
}

}  // namespace

int attn_decode_ctas(int num_sms) { return num_sms; }
int attn_decode_slots(int ctas) { return 2 * ctas * N_KV; }

cudaError_t launch_attn_decode(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeAttnParams& a,
                               cudaStream_t s, bool pdl) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             FIXED_SMEM + (DECODE_MAX_B + 1) * 4);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (a.B <= 0 || a.B > DECODE_MAX_B) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = FIXED_SMEM + (a.B + 1) * 4;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel, mk, mv, a);
}

}  // namespace gqa
