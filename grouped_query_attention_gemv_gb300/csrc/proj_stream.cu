// Standalone few-token projection kernel (small prefills, and the decode path
// when it is not fused): the projection phase of proj_core.cuh in its own
// grid, token loads ordered after the predecessor by griddepcontrol.wait.
#include "proj_core.cuh"

namespace gqa {

namespace {

using namespace projk;
constexpr int THREADS = 192;

template <int NP>
constexpr int smem_bytes() {
  return Cfg<NP>::RING + Cfg<NP>::OUT_BYTES + 1024 + 256;
}

template <int NP, bool QKV>
__global__ void __launch_bounds__(THREADS, 1)
    proj_stream_kernel(const __grid_constant__ ProjStreamMaps maps, ProjParams p, float* __restrict__ part,
                       int* __restrict__ tickets, int segmax) {
  using C_ = Cfg<NP>;
  constexpr int S = C_::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C_::RING);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);
  __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + C_::RING + 256);

  pdl_trigger();
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), 4);
    }
    flags[0] = flags[1] = flags[2] = flags[3] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C_::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const Shared<NP> sh{smem, full, empty, acc_full, acc_empty, stage, flags, *tmem_slot};
  proj_phase<NP, QKV>(
      maps, p, part, tickets, segmax, sh,
      []() {
        pdl_wait();
        return true;
      },
      [](int) {});
  tc_fence_before();
  __syncthreads();
  if (flags[0]) {
    if (threadIdx.x == 0) {
      report(p.status, DEV_WAIT_TIMEOUT);
      proj_drain(sh);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(sh.tmem, C_::TMEM_COLS);
  }
}

template <int NP, bool QKV>
cudaError_t launch_np(const ProjStreamArgs& a, cudaStream_t s, bool pdl) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = proj_stream_kernel<NP, QKV>;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes<NP>());
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ctas);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem_bytes<NP>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a.maps, a.p, a.part, a.tickets, a.segmax);
}

}  // namespace

int proj_stream_np(int M) {
  if (M <= 0 || M > 64) return 0;
  return M <= 16 ? 16 : (M <= 32 ? 32 : 64);
}

int proj_stream_segmax(int N, int ctas) {
  const long long U = static_cast<long long>(N / TILE_ROWS) * NKB;
  const long long per = (U + ctas - 1) / ctas;
  return static_cast<int>((per + NKB - 1) / NKB) + 1;
}

cudaError_t launch_proj_stream(const ProjStreamArgs& a, cudaStream_t s, bool pdl) {
  const bool qkv = a.p.qkv != 0;
  switch (proj_stream_np(a.p.M)) {
    case 16: return qkv ? launch_np<16, true>(a, s, pdl) : launch_np<16, false>(a, s, pdl);
    case 32: return qkv ? launch_np<32, true>(a, s, pdl) : launch_np<32, false>(a, s, pdl);
    case 64: return qkv ? launch_np<64, true>(a, s, pdl) : launch_np<64, false>(a, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gqa
