// C ABI of libgqa (declared in include/gqa.h): argument validation on the
// host, workspace layout, TMA descriptor encoding and the launch sequence of
// one block call on the caller's stream. Nothing here allocates or waits.
#include <stdio.h>
#include <string.h>

#include "gqa.h"
#include "kernels.h"

using namespace gqa;

namespace {

thread_local cudaError_t t_last_cuda = cudaSuccess;
thread_local int t_launches = 0;
thread_local char t_msg[256];
thread_local void* const* t_prof_events = nullptr;
thread_local int t_prof_count = 0;
thread_local int t_fused = 1;
thread_local int t_attn_split = 0;  // fused decode attention: 0 chosen per call, 1 position-major, 2 head-major
thread_local unsigned long long t_wait_ns = WAIT_LIMIT_NS;  // grid-wide waits of the decode kernels

thread_local int t_prof_base = 0;  // 1 while a layer call's norm kernel occupies events[0..1]
void prof_mark(int i, cudaStream_t s) {
  i += t_prof_base;
  if (t_prof_events && i < t_prof_count && t_prof_events[i])
    cudaEventRecord(static_cast<cudaEvent_t>(t_prof_events[i]), s);
}

// Workspace regions, each 256-byte aligned. The status region is always
// first: the status word at offset 0, the fused decode grid's progress
// counters at COUNTERS_OFFSET.
constexpr size_t COUNTERS_OFFSET = 16;
struct Layout {
  size_t status = 0, q = 0, o = 0, proj_part = 0, proj_tickets = 0, part_o = 0, part_ml = 0;
  size_t total = 0;
  int np = 0;            // padded tokens of the few-token projection (0: tensor-core GEMM path)
  int proj_slots = 0;    // partial slots of the few-token projection
  int att_slots = 0;     // partial slots of the decode attention
};

// SM count the workspace sizing assumes (GB300); launches use at most this many.
constexpr int REF_SMS = 152;

bool make_layout(int B, int T, int max_keys, Layout* L) {
  if (B <= 0 || T <= 0 || max_keys < T) return false;
  const long long M = static_cast<long long>(B) * T;
  if (M > (1LL << 24)) return false;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t r = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return r;
  };
  L->status = take(256);
  L->q = take(static_cast<size_t>(M) * D_MODEL * 2);
  L->o = take(static_cast<size_t>(M) * D_MODEL * 2);
  L->np = proj_stream_np(static_cast<int>(M));
  if (L->np) {
    const int segmax = proj_stream_segmax(QKV_ROWS_MAX, REF_SMS) > proj_stream_segmax(D_MODEL, REF_SMS)
                           ? proj_stream_segmax(QKV_ROWS_MAX, REF_SMS) : proj_stream_segmax(D_MODEL, REF_SMS);
    L->proj_slots = REF_SMS * segmax;
    L->proj_part = take(static_cast<size_t>(L->proj_slots) * 128 * L->np * 4);
    L->proj_tickets = take(static_cast<size_t>(QKV_ROWS_MAX / 128) * 4);
  }
  if (T == 1) {
    if (B > DECODE_MAX_B) return false;
    L->att_slots = attn_decode_slots(attn_decode_ctas(REF_SMS));
    const size_t slots = static_cast<size_t>(L->att_slots) * N_REP;
    L->part_o = take(slots * HEAD_DIM * 4);
    L->part_ml = take(slots * 2 * 4);
  }
  L->total = off;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail_cuda(cudaError_t e) {
  t_last_cuda = e;
  return GQA_ECUDA;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Every tensor map of this library: bf16, 128-byte swizzle, no interleave,
// 256-byte L2 promotion, zero fill. Encoding one costs the host about a
// microsecond and a decode call needs ~16, so each thread keeps the last
// ones it encoded (a map depends only on these arguments; the buffers behind
// the pointers are the caller's and are not read).
struct MapKey {
  const void* ptr;
  cuuint32_t rank;
  cuuint64_t dims[4];
  cuuint64_t strides[3];
  cuuint32_t box[4];
  bool operator==(const MapKey& o) const {
    if (ptr != o.ptr || rank != o.rank) return false;
    for (cuuint32_t i = 0; i < rank; ++i)
      if (dims[i] != o.dims[i] || box[i] != o.box[i] || (i + 1 < rank && strides[i] != o.strides[i])) return false;
    return true;
  }
};
constexpr int MAP_CACHE = 256;
struct MapCacheEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};

bool encode_bf16(CUtensorMap* m, cuuint32_t rank, const void* ptr, const cuuint64_t* dims, const cuuint64_t* strides,
                 const cuuint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 1 || rank > 4) return false;
  MapKey k{};
  k.ptr = ptr;
  k.rank = rank;
  uint64_t h = reinterpret_cast<uintptr_t>(ptr) * 0x9E3779B97F4A7C15ull ^ rank;
  for (cuuint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    h = (h ^ dims[i]) * 0x100000001B3ull;
    h = (h ^ box[i]) * 0x100000001B3ull;
    if (i + 1 < rank) {
      k.strides[i] = strides[i];
      h = (h ^ strides[i]) * 0x100000001B3ull;
    }
  }
  thread_local MapCacheEntry cache[MAP_CACHE];
  MapCacheEntry& e = cache[(h >> 32) % MAP_CACHE];
  if (e.used && e.key == k) {
    *m = e.map;
    return true;
  }
  const cuuint32_t es[4] = {1, 1, 1, 1};
  if (enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  e.key = k;
  e.map = *m;
  e.used = true;
  return true;
}

// bf16 [outer, 4096] row-major, boxes of box_rows x 64 (128B swizzle).
bool map_rows(CUtensorMap* m, const void* ptr, long long rows, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D_MODEL), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D_MODEL) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  return encode_bf16(m, 2, ptr, dims, strides, box);
}

// bf16 [rows, 4096] row-major viewed as (64 values, row, 64 k blocks), boxes
// of 64 x box_rows x kblocks: one box reads kblocks*128 contiguous bytes of
// each of box_rows rows.
bool map_rows_kblocks(CUtensorMap* m, const void* ptr, long long rows, int box_rows, int kblocks) {
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), D_MODEL / 64};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D_MODEL) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(kblocks)};
  return encode_bf16(m, 3, ptr, dims, strides, box);
}

// Decode view of the KV cache [B, s_max, n_kv, 128] bf16: dims (d, pos, g, b)
// so that one box of 64 dims x box_pos positions x 8 heads covers whole
// position rows of 8 KV heads (all of them, or one group of the multi-head
// variant). Positions past s_max read as zero.
bool map_cache_by_position(CUtensorMap* m, const void* ptr, int B, int s_max, int n_kv, int box_pos) {
  const cuuint64_t row = static_cast<cuuint64_t>(n_kv) * HEAD_DIM * 2;  // bytes of one cache position
  const cuuint64_t dims[4] = {HEAD_DIM, static_cast<cuuint64_t>(s_max), static_cast<cuuint64_t>(n_kv),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {row, HEAD_DIM * 2, static_cast<cuuint64_t>(s_max) * row};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_pos), N_KV, 1};
  return encode_bf16(m, 4, ptr, dims, strides, box);
}

// KV cache [B, s_max, n_kv, 128] bf16 as a 4-D tensor (d, g, pos, b); boxes
// of 64 dims x 1 head x box_pos positions. Positions at or past `rows`
// (<= s_max) read as zero.
bool map_cache(CUtensorMap* m, const void* ptr, int B, int s_max, int n_kv, int rows, int box_pos) {
  if (rows <= 0 || rows > s_max) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(n_kv) * HEAD_DIM * 2;
  const cuuint64_t dims[4] = {HEAD_DIM, static_cast<cuuint64_t>(n_kv), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {HEAD_DIM * 2, row, static_cast<cuuint64_t>(s_max) * row};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(box_pos), 1};
  return encode_bf16(m, 4, ptr, dims, strides, box);
}

// Rotated queries [B*T, 4096] bf16 as a 4-D tensor (d, head, t, b); boxes of
// 64 dims x n_rep heads (one KV group) x 128 / n_rep tokens (128 rows). Tokens
// past T read as zero.
bool map_q_prefill(CUtensorMap* m, const void* ptr, int B, int T, int n_rep) {
  const cuuint64_t dims[4] = {HEAD_DIM, N_HEADS, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {HEAD_DIM * 2, D_MODEL * 2, static_cast<cuuint64_t>(T) * D_MODEL * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(n_rep), static_cast<cuuint32_t>(128 / n_rep), 1};
  return encode_bf16(m, 4, ptr, dims, strides, box);
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return REF_SMS;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = REF_SMS;
    cached[dev] = n;
  }
  return cached[dev];
}

struct Call {
  const gqa_bf16* x;
  const gqa_bf16* norm_w;  // layer entries: attention_norm weight (x is normalised first, then added back)
  float eps;
  int B, T;
  StartPos sp;
  int max_keys;
  const gqa_bf16 *wq, *wk, *wv, *wo;
  const float* rope;
  gqa_bf16 *cache_k, *cache_v;
  int s_max;
  int n_kv;  // KV heads: 8 (Llama 3.1 8B), or 32 (the multi-head variant)
  gqa_bf16* out;
  uint8_t* ws;
  cudaStream_t stream;
  Layout L;
  int kv_row() const { return n_kv * HEAD_DIM; }
};

int check_common(const gqa_bf16* x, int B, int T, const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                 const gqa_bf16* wo, const float* rope, int rope_rows, const gqa_bf16* ck, const gqa_bf16* cv,
                 int s_max, const gqa_bf16* out, const void* ws, int max_keys, size_t ws_bytes, Layout* L) {
  if (!x || !wq || !wk || !wv || !wo || !rope || !ck || !cv || !out || !ws) return GQA_EINVAL;
  if (B <= 0 || T <= 0 || s_max <= 0 || rope_rows <= 0) return GQA_EINVAL;
  if (max_keys > s_max || max_keys > rope_rows) return GQA_EINVAL;
  if (!aligned16(x) || !aligned16(wq) || !aligned16(wk) || !aligned16(wv) || !aligned16(wo) ||
      !aligned16(rope) || !aligned16(ck) || !aligned16(cv) || !aligned16(out) || !aligned16(ws))
    return GQA_EALIGN;
  if (!make_layout(B, T, max_keys, L)) return GQA_EINVAL;
  if (ws_bytes < L->total) return GQA_EWORKSPACE;
  return GQA_OK;
}

// fold_norm: the kernel applies attention_norm to x itself (the fused decode
// grid); otherwise a layer call's projection reads the norm kernel's rows.
ProjParams proj_params(const Call& c, bool qkv, bool fold_norm = false) {
  ProjParams p{};
  p.M = c.B * c.T;
  p.T = c.T;
  if (qkv) {
    // the layer entries project the normalised rows, which the norm kernel
    // left in the attention-output buffer (the attention overwrites them
    // only after this projection)
    p.x = reinterpret_cast<const __nv_bfloat16*>(c.norm_w && !fold_norm ? reinterpret_cast<const gqa_bf16*>(c.ws + c.L.o)
                                                                         : c.x);
    p.norm_w = fold_norm ? reinterpret_cast<const __nv_bfloat16*>(c.norm_w) : nullptr;
    p.eps = c.eps;
    p.w0 = reinterpret_cast<const __nv_bfloat16*>(c.wq);
    p.w1 = reinterpret_cast<const __nv_bfloat16*>(c.wk);
    p.w2 = reinterpret_cast<const __nv_bfloat16*>(c.wv);
    p.r1 = D_MODEL;
    p.r2 = D_MODEL + c.kv_row();
    p.N = D_MODEL + 2 * c.kv_row();
    p.qkv = 1;
    p.out = reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.q);
  } else {
    p.x = reinterpret_cast<const __nv_bfloat16*>(c.ws + c.L.o);
    p.w0 = p.w1 = p.w2 = reinterpret_cast<const __nv_bfloat16*>(c.wo);
    p.r1 = p.r2 = p.N = D_MODEL;
    p.qkv = 0;
    p.out = reinterpret_cast<__nv_bfloat16*>(c.out);
    p.resid = c.norm_w ? reinterpret_cast<const __nv_bfloat16*>(c.x) : nullptr;  // h = x + delta
  }
  p.cache_k = reinterpret_cast<__nv_bfloat16*>(c.cache_k);
  p.cache_v = reinterpret_cast<__nv_bfloat16*>(c.cache_v);
  p.s_max = c.s_max;
  p.rope = c.rope;
  p.sp = c.sp;
  p.status = reinterpret_cast<int*>(c.ws + c.L.status);
  return p;
}

int launch_sms() {
  const int n = sm_count();
  return n < REF_SMS ? n : REF_SMS;
}

// Tensor maps of the few-token projection: boxes of 1..4 k blocks of the
// weights (128 rows) and of the tokens (np rows).
bool stream_maps(const Call& c, bool qkv, const ProjParams& p, ProjStreamMaps* m) {
  const gqa_bf16* w[3] = {qkv ? c.wq : c.wo, qkv ? c.wk : c.wo, qkv ? c.wv : c.wo};
  const long long rows[3] = {D_MODEL, qkv ? c.kv_row() : D_MODEL, qkv ? c.kv_row() : D_MODEL};
  for (int kc = 1; kc <= 4; ++kc) {
    for (int i = 0; i < 3; ++i)
      if (!map_rows_kblocks(&m->w[kc - 1][i], w[i], rows[i], 128, kc)) return false;
    if (!map_rows_kblocks(&m->x[kc - 1], p.x, p.M, c.L.np, kc)) return false;
  }
  return true;
}

DecodeAttnParams decode_attn_params(const Call& c) {
  DecodeAttnParams a{};
  a.q = reinterpret_cast<const __nv_bfloat16*>(c.ws + c.L.q);
  a.B = c.B;
  a.n_kv = c.n_kv;
  a.sp = c.sp;
  a.ctas = attn_decode_ctas(launch_sms());
  a.part_o = reinterpret_cast<float*>(c.ws + c.L.part_o);
  a.part_ml = reinterpret_cast<float*>(c.ws + c.L.part_ml);
  a.counters = reinterpret_cast<int*>(c.ws + c.L.status + COUNTERS_OFFSET);
  a.o = reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.o);
  a.status = reinterpret_cast<int*>(c.ws + c.L.status);
  a.cache_k = reinterpret_cast<const __nv_bfloat16*>(c.cache_k);
  a.cache_v = reinterpret_cast<const __nv_bfloat16*>(c.cache_v);
  a.s_max = c.s_max;
  a.wait_ns = t_wait_ns;
  return a;
}

bool decode_cache_maps(const Call& c, DecodeCacheMaps* m) {
  return map_cache_by_position(&m->k, c.cache_k, c.B, c.s_max, c.n_kv, DECODE_UNIT) &&
         map_cache_by_position(&m->v, c.cache_v, c.B, c.s_max, c.n_kv, DECODE_UNIT);
}

// PDL (programmatic dependent launch) is only requested for kernels that
// execute griddepcontrol.wait before reading what earlier kernels wrote.
int run_projection(const Call& c, bool qkv, bool pdl) {
  const ProjParams p = proj_params(c, qkv);
  cudaError_t e;
  GemmMaps maps;
  if (c.L.np) {
    ProjStreamArgs a;
    if (!stream_maps(c, qkv, p, &a.maps)) return fail_cuda(cudaErrorInvalidValue);
    a.p = p;
    a.ctas = launch_sms();
    a.segmax = proj_stream_segmax(p.N, a.ctas);
    if (a.ctas * a.segmax > c.L.proj_slots) return fail_cuda(cudaErrorInvalidConfiguration);
    a.part = reinterpret_cast<float*>(c.ws + c.L.proj_part);
    a.tickets = reinterpret_cast<int*>(c.ws + c.L.proj_tickets);
    e = launch_proj_stream(a, c.stream, pdl);
  } else {
    if (!map_rows(&maps.a, p.x, p.M, GEMM_BM)) return fail_cuda(cudaErrorInvalidValue);
    if (qkv) {
      if (!map_rows(&maps.b[0], c.wq, D_MODEL, GEMM_BN) || !map_rows(&maps.b[1], c.wk, c.kv_row(), GEMM_BN) ||
          !map_rows(&maps.b[2], c.wv, c.kv_row(), GEMM_BN))
        return fail_cuda(cudaErrorInvalidValue);
    } else {
      if (!map_rows(&maps.b[0], c.wo, D_MODEL, GEMM_BN)) return fail_cuda(cudaErrorInvalidValue);
      maps.b[1] = maps.b[0];
      maps.b[2] = maps.b[0];
    }
    e = launch_gemm_tc(maps, p, launch_sms(), c.stream);
  }
  if (e != cudaSuccess) return fail_cuda(e);
  ++t_launches;
  return GQA_OK;
}

int run_attention(const Call& c) {
  cudaError_t e;
  if (c.T == 1) {
    DecodeCacheMaps maps;
    if (!decode_cache_maps(c, &maps)) return fail_cuda(cudaErrorInvalidValue);
    const DecodeAttnParams a = decode_attn_params(c);
    if (attn_decode_slots(a.ctas) > c.L.att_slots) return fail_cuda(cudaErrorInvalidConfiguration);
    e = launch_attn_decode(maps, a, c.stream);
  } else {
    PrefillMaps maps;
    const void* q = c.ws + c.L.q;
    if (!map_q_prefill(&maps.q, q, c.B, c.T, N_HEADS / c.n_kv) ||
        !map_cache(&maps.k, c.cache_k, c.B, c.s_max, c.n_kv, c.max_keys, PREFILL_TILE) ||
        !map_cache(&maps.v, c.cache_v, c.B, c.s_max, c.n_kv, c.max_keys, PREFILL_TILE))
      return fail_cuda(cudaErrorInvalidValue);
    PrefillAttnParams a{};
    a.q = reinterpret_cast<const __nv_bfloat16*>(q);
    a.B = c.B;
    a.T = c.T;
    a.n_kv = c.n_kv;
    a.sp = c.sp;
    a.o = reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.o);
    a.status = reinterpret_cast<int*>(c.ws + c.L.status);
    a.num_sms = sm_count();
    e = launch_attn_prefill(maps, a, c.stream);
  }
  if (e != cudaSuccess) return fail_cuda(e);
  ++t_launches;
  return GQA_OK;
}

// Tensor maps of a row-owner projection: per matrix, boxes of its two row
// counts; the token rows x (M of them), boxes of np rows.
bool row_maps(const gqa_bf16* const* w, const RowPlan& plan, const void* x, int M, int np, RowMaps* m) {
  const int kc = rows_kc(np);
  for (int i = 0; i < 3; ++i) {
    const int mi = i < plan.nmat ? i : 0;
    for (int hi = 0; hi < 2; ++hi)
      if (!map_rows_kblocks(&m->w[i][hi], w[mi], plan.rows[mi], plan.h_lo[mi] + 2 * hi, kc)) return false;
  }
  return np > 0 && map_rows_kblocks(&m->x, x, M, np, kc);
}

// Tensor maps of the multi-head Q|K|V phase: Wq, Wk and Wv (4,096 rows
// each) walked in three passes of one plan, so every matrix gets that plan's
// boxes.
bool row_maps_passes(const gqa_bf16* const* w, const RowPlan& plan, const void* x, int M, int np, RowMaps* m) {
  const int kc = rows_kc(np);
  for (int i = 0; i < 3; ++i)
    for (int hi = 0; hi < 2; ++hi)
      if (!map_rows_kblocks(&m->w[i][hi], w[i], plan.rows[0], plan.h_lo[0] + 2 * hi, kc)) return false;
  return np > 0 && map_rows_kblocks(&m->x, x, M, np, kc);
}

// Work split of the fused grid's attention for one call. Head-major (one
// (sequence, KV head) pair per CTA) streams each head of a sequence on one
// SM, at about 50 GB/s per SM (measured with 128 SMs streaming at B = 16,
// P = 1000); position-major units spread the batch over every SM (about
// 6.8 TB/s) but pay a grid meeting and a merge round, about 5 us at B = 16,
// when sequences are split between CTAs. Head-major wins while one head's
// stream is shorter than the whole batch's stream plus that overhead: small
// batches of short contexts.
bool head_major_pays(int B, int max_keys, int ctas) {
  if (B * N_KV > ctas) return false;
  const double item_us = max_keys * 512.0 / 5.0e4;                 // 512 B of K and V per position and head
  const double split_us = static_cast<double>(B) * max_keys * 4096.0 / 6.8e6 + 5.0;
  return item_us < split_us;
}

// The whole decode step as one persistent grid (B <= FUSED_MAX_B). Returns
// GQA_EINVAL without launching anything when this GPU cannot run it (too few
// SMs for the row split); the caller then takes the three-kernel path.
int run_decode_fused(const Call& c) {
  // 8 KV heads: one Q|K|V pass over 6,144 rows. 32 KV heads (12,288 rows):
  // three passes of 4,096, up to 16 sequences (the attention's unit prefix
  // covers 4 head groups per sequence), block entries only.
  const bool mha = c.n_kv == N_HEADS;
  if (c.n_kv != N_KV && !(mha && c.B * N_REP <= FUSED_MAX_B && !c.norm_w)) return GQA_EINVAL;
  DecodeFusedArgs a;
  a.ctas = launch_sms();
  const int qkv_rows[3] = {D_MODEL, KV_ROW, KV_ROW};
  const int o_rows[1] = {D_MODEL};
  a.qkv_passes = mha ? 3 : 1;
  a.head_major = mha                 ? 0
                 : t_attn_split == 2 ? (c.B * N_KV <= a.ctas)
                 : t_attn_split == 1 ? 0
                                     : head_major_pays(c.B, c.max_keys, a.ctas);
  // One sequence with head-major attention: its 8 attention CTAs finish
  // phase B last and would only then request their W_O stages (their ring
  // held the attention's), so W_O's rows go to the other CTAs, whose stages
  // are in shared memory before the W_O gate opens.
  const int o_cta0 = a.head_major && c.B == 1 ? N_KV : 0;
  if (!(mha ? make_row_plan(1, o_rows, a.ctas, &a.qkv_plan) : make_row_plan(3, qkv_rows, a.ctas, &a.qkv_plan)) ||
      !make_row_plan(1, o_rows, a.ctas - o_cta0, &a.o_plan))
    return GQA_EINVAL;
  a.o_plan.cta0 = o_cta0;
  a.pq = proj_params(c, true, /*fold_norm=*/true);
  a.po = proj_params(c, false);
  const gqa_bf16* wqkv[3] = {c.wq, c.wk, c.wv};
  const gqa_bf16* wo[1] = {c.wo};
  const int np = decode_fused_np(a.pq.M);
  if (!(mha ? row_maps_passes(wqkv, a.qkv_plan, a.pq.x, a.pq.M, np, &a.qkv_maps)
            : row_maps(wqkv, a.qkv_plan, a.pq.x, a.pq.M, np, &a.qkv_maps)) ||
      !row_maps(wo, a.o_plan, a.po.x, a.po.M, np, &a.o_maps) ||
      !decode_cache_maps(c, &a.cache))
    return fail_cuda(cudaErrorInvalidValue);
  if (a.head_major) {
    if (!map_cache(&a.cache_hm.k, c.cache_k, c.B, c.s_max, c.n_kv, c.s_max, DECODE_ITEM_POS) ||
        !map_cache(&a.cache_hm.v, c.cache_v, c.B, c.s_max, c.n_kv, c.s_max, DECODE_ITEM_POS))
      return fail_cuda(cudaErrorInvalidValue);
  } else {
    a.cache_hm = a.cache;  // unused
  }
  a.at = decode_attn_params(c);
  if (a.at.ctas != a.ctas || attn_decode_slots(a.ctas) > c.L.att_slots) return fail_cuda(cudaErrorInvalidConfiguration);
  a.counters = reinterpret_cast<int*>(c.ws + c.L.status + COUNTERS_OFFSET);
  prof_mark(0, c.stream);
  const cudaError_t e = launch_decode_fused(a, c.stream);
  prof_mark(1, c.stream);
  if (e != cudaSuccess) return fail_cuda(e);
  ++t_launches;
  return GQA_OK;
}

// attention_norm of the layer entries: the normalised rows go to the
// attention-output buffer of the workspace.
int run_norm(const Call& c) {
  const cudaError_t e = launch_rmsnorm(reinterpret_cast<const __nv_bfloat16*>(c.x),
                                       reinterpret_cast<const __nv_bfloat16*>(c.norm_w), c.eps, c.B * c.T,
                                       reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.o), c.stream);
  if (e != cudaSuccess) return fail_cuda(e);
  ++t_launches;
  return GQA_OK;
}

int run_block(Call& c) {
  t_launches = 0;
  t_prof_base = 0;
  // the fused decode grid applies a layer call's norm itself
  if (c.T == 1 && c.L.np && c.B <= FUSED_MAX_B && t_fused) {
    const int r = run_decode_fused(c);
    if (r != GQA_EINVAL) return r;
  }
  if (c.norm_w) {
    prof_mark(0, c.stream);
    const int r = run_norm(c);
    prof_mark(1, c.stream);
    if (r != GQA_OK) return r;
    t_prof_base = 1;  // the block's kernels follow in the event list
  }
  prof_mark(0, c.stream);
  int r = run_projection(c, true, false);
  prof_mark(1, c.stream);
  if (r == GQA_OK) r = run_attention(c);
  prof_mark(2, c.stream);
  // W_O: the few-token kernel overlaps its weight stream with attention's tail
  if (r == GQA_OK) r = run_projection(c, false, c.L.np != 0 && t_prof_events == nullptr);
  prof_mark(3, c.stream);
  return r;
}

}  // namespace

extern "C" {

size_t gqa_workspace_bytes(int B, int T, int max_keys) {
  Layout L;
  return make_layout(B, T, max_keys, &L) ? L.total : 0;
}

int gqa_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes == 0) return GQA_EINVAL;
  if (!aligned16(workspace)) return GQA_EALIGN;
  cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GQA_OK : fail_cuda(e);
}

int gqa_device_status(void* workspace, int* status, int clear) {
  if (!workspace || !status) return GQA_EINVAL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(status, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(workspace, 0, sizeof(int));
  if (e != cudaSuccess) return fail_cuda(e);
  return *status ? GQA_EDEVICE : GQA_OK;
}

int gqa_rope_table(float* rope, int rows, double theta, int scaled, double factor, double low_freq_factor,
                   double high_freq_factor, double original_context, void* stream) {
  if (!rope || rows <= 0 || !(theta > 1.0)) return GQA_EINVAL;
  if (scaled && !(factor > 0.0 && high_freq_factor > low_freq_factor && low_freq_factor > 0.0 &&
                  original_context > 0.0))
    return GQA_EINVAL;
  if (!aligned16(rope)) return GQA_EALIGN;
  t_launches = 0;
  cudaError_t e = launch_rope_table(rope, rows, theta, scaled, factor, low_freq_factor, high_freq_factor,
                                    original_context, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  t_launches = 1;
  return GQA_OK;
}

static bool valid_n_kv(int n_kv) { return n_kv == N_KV || n_kv == N_HEADS; }

// dry: validate only (GQA_OK when the call would be launched)
static int block_call(const gqa_bf16* x, int B, int T, int start_pos, int n_kv, const gqa_bf16* norm_w, float eps,
                      const gqa_bf16* wq, const gqa_bf16* wk,
                      const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                      gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace, size_t workspace_bytes,
                      void* stream, bool dry = false) {
  if (start_pos < 0 || T <= 0 || start_pos > (1 << 30) || !valid_n_kv(n_kv)) return GQA_EINVAL;
  Call c{};
  const int max_keys = start_pos + T;
  int r = check_common(x, B, T, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max, out, workspace, max_keys,
                       workspace_bytes, &c.L);
  if (r != GQA_OK) return r;
  c.norm_w = norm_w;
  c.eps = eps;
  c.x = x;
  c.B = B;
  c.T = T;
  c.sp = StartPos{nullptr, start_pos, start_pos};
  c.n_kv = n_kv;
  c.max_keys = max_keys;
  c.wq = wq;
  c.wk = wk;
  c.wv = wv;
  c.wo = wo;
  c.rope = rope;
  c.cache_k = cache_k;
  c.cache_v = cache_v;
  c.s_max = s_max;
  c.out = out;
  c.ws = static_cast<uint8_t*>(workspace);
  c.stream = static_cast<cudaStream_t>(stream);
  return dry ? GQA_OK : run_block(c);
}

// Arguments of the layer entries beyond the block's.
static int check_layer(const gqa_bf16* x, const gqa_bf16* norm_w, float eps, const gqa_bf16* h) {
  if (!norm_w || !(eps > 0.f) || !(eps < 1e30f)) return GQA_EINVAL;
  if (!aligned16(norm_w)) return GQA_EALIGN;
  if (h == x) return GQA_EINVAL;
  return GQA_OK;
}

int gqa_rms_norm(const gqa_bf16* x, int M, const gqa_bf16* norm_w, float eps, gqa_bf16* y, void* stream) {
  if (!x || !norm_w || !y || M <= 0 || !(eps > 0.f) || !(eps < 1e30f)) return GQA_EINVAL;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(y)) return GQA_EALIGN;
  t_launches = 0;
  const cudaError_t e = launch_rmsnorm(reinterpret_cast<const __nv_bfloat16*>(x),
                                       reinterpret_cast<const __nv_bfloat16*>(norm_w), eps, M,
                                       reinterpret_cast<__nv_bfloat16*>(y), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  t_launches = 1;
  return GQA_OK;
}

int gqa_block_forward(const gqa_bf16* x, int B, int T, int start_pos, const gqa_bf16* wq, const gqa_bf16* wk,
                      const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                      gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return block_call(x, B, T, start_pos, N_KV, nullptr, 0.f, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max,
                    out, workspace, workspace_bytes, stream);
}

int gqa_block_forward_nkv(const gqa_bf16* x, int B, int T, int start_pos, int n_kv_heads, const gqa_bf16* wq,
                          const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows,
                          gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return block_call(x, B, T, start_pos, n_kv_heads, nullptr, 0.f, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v,
                    s_max, out, workspace, workspace_bytes, stream);
}

int gqa_layer_forward(const gqa_bf16* x, int B, int T, int start_pos, const gqa_bf16* norm_w, float eps,
                      const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
                      const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max,
                      gqa_bf16* h, void* workspace, size_t workspace_bytes, void* stream) {
  const int r = check_layer(x, norm_w, eps, h);
  if (r != GQA_OK) return r;
  return block_call(x, B, T, start_pos, N_KV, norm_w, eps, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max,
                    h, workspace, workspace_bytes, stream);
}

int gqa_prefill(const gqa_bf16* x, int B, int T, int start_pos, const gqa_bf16* wq, const gqa_bf16* wk,
                const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace, size_t workspace_bytes, void* stream) {
  return gqa_block_forward(x, B, T, start_pos, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max, out,
                           workspace, workspace_bytes, stream);
}

static int decode_call(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos, int n_kv,
                       const gqa_bf16* norm_w, float eps, const gqa_bf16* wq, const gqa_bf16* wk,
                       const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                       gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace, size_t workspace_bytes,
                       void* stream, bool dry = false) {
  if (!start_pos || max_start_pos < 0 || max_start_pos > (1 << 30) || !valid_n_kv(n_kv)) return GQA_EINVAL;
  // the attention runs n_kv / 8 head groups of every sequence as units of their own
  const int groups = n_kv / N_KV;
  if (B > DECODE_MAX_B / groups) return GQA_EINVAL;
  Call c{};
  const int max_keys = max_start_pos + 1;
  int r = check_common(x, B, 1, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max, out, workspace, max_keys,
                       workspace_bytes, &c.L);
  if (r != GQA_OK) return r;
  if ((reinterpret_cast<uintptr_t>(start_pos) & 3u) != 0) return GQA_EALIGN;
  // the attention splits its units over the grid in 32-bit arithmetic
  const unsigned long long units =
      static_cast<unsigned long long>(B) * groups * ((max_keys + DECODE_UNIT - 1) / DECODE_UNIT);
  if ((units + 1) * (static_cast<unsigned long long>(attn_decode_ctas(launch_sms())) + 1) >= (1ull << 32))
    return GQA_EINVAL;
  c.norm_w = norm_w;
  c.eps = eps;
  c.x = x;
  c.B = B;
  c.T = 1;
  c.sp = StartPos{start_pos, 0, max_start_pos};
  c.n_kv = n_kv;
  c.max_keys = max_keys;
  c.wq = wq;
  c.wk = wk;
  c.wv = wv;
  c.wo = wo;
  c.rope = rope;
  c.cache_k = cache_k;
  c.cache_v = cache_v;
  c.s_max = s_max;
  c.out = out;
  c.ws = static_cast<uint8_t*>(workspace);
  c.stream = static_cast<cudaStream_t>(stream);
  return dry ? GQA_OK : run_block(c);
}

int gqa_decode(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos, const gqa_bf16* wq,
               const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows,
               gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace,
               size_t workspace_bytes, void* stream) {
  return decode_call(x, B, start_pos, max_start_pos, N_KV, nullptr, 0.f, wq, wk, wv, wo, rope, rope_rows, cache_k,
                     cache_v, s_max, out, workspace, workspace_bytes, stream);
}

int gqa_decode_nkv(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos, int n_kv_heads,
                   const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo, const float* rope,
                   int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace,
                   size_t workspace_bytes, void* stream) {
  return decode_call(x, B, start_pos, max_start_pos, n_kv_heads, nullptr, 0.f, wq, wk, wv, wo, rope, rope_rows,
                     cache_k, cache_v, s_max, out, workspace, workspace_bytes, stream);
}

int gqa_layer_decode(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos, const gqa_bf16* norm_w,
                     float eps, const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
                     const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max,
                     gqa_bf16* h, void* workspace, size_t workspace_bytes, void* stream) {
  const int r = check_layer(x, norm_w, eps, h);
  if (r != GQA_OK) return r;
  return decode_call(x, B, start_pos, max_start_pos, N_KV, norm_w, eps, wq, wk, wv, wo, rope, rope_rows, cache_k,
                     cache_v, s_max, h, workspace, workspace_bytes, stream);
}

const char* gqa_strerror(int status) {
  switch (status) {
    case GQA_OK: return "success";
    case GQA_EINVAL: return "invalid argument (null pointer, non-positive size, or position beyond cache/table)";
    case GQA_EALIGN: return "pointer not 16-byte aligned";
    case GQA_EWORKSPACE: return "workspace smaller than gqa_workspace_bytes()";
    case GQA_EDEVICE: return "a kernel recorded an error in the workspace status word";
    case GQA_ESCRATCH:
      return "call needs more scratch than gqa_decode_static's static array (GQA_STATIC_SCRATCH_BYTES = 16 MiB); "
             "use gqa_decode with a workspace";
    case GQA_ECUDA:
      snprintf(t_msg, sizeof(t_msg), "CUDA error: %s", cudaGetErrorName(t_last_cuda));
      return t_msg;
    default: return "unknown status";
  }
}

int gqa_last_launch_count(void) { return t_launches; }

int gqa_set_decode_fusion(int enable) {
  const int prev = t_fused;
  t_fused = enable ? 1 : 0;
  return prev;
}

unsigned long long gqa_set_wait_limit_ns(unsigned long long ns) {
  const unsigned long long prev = t_wait_ns;
  t_wait_ns = ns ? ns : WAIT_LIMIT_NS;
  return prev;
}

int gqa_set_decode_attention_split(int mode) {
  if (mode < 0 || mode > 2) return -1;
  const int prev = t_attn_split;
  t_attn_split = mode;
  return prev;
}

int gqa_set_profile_events(void* const* events, int count) {
  if (count < 0) return GQA_EINVAL;
  t_prof_events = count > 0 ? events : nullptr;
  t_prof_count = events ? count : 0;
  return GQA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gqa_decode_static: the decode step with its scratch in a static device array
// instead of a caller-provided workspace, for callers that cannot allocate.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GQA_STATIC_SCRATCH_BYTES];

std::mutex g_static_mu;
void* g_static_ptr[64] = {};

// Device address of g_static_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current.
int static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= 64) return fail_cuda(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return fail_cuda(e);
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return GQA_OK;
}

}  // namespace

extern "C" int gqa_decode_static(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos,
                                 const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
                                 const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max,
                                 gqa_bf16* out, void* stream) {
  if (!start_pos || max_start_pos < 0 || max_start_pos > (1 << 30) || B <= 0) return GQA_EINVAL;
  Layout need;
  if (!make_layout(B, 1, max_start_pos + 1, &need)) return GQA_EINVAL;
  if (need.total > GQA_STATIC_SCRATCH_BYTES) return GQA_ESCRATCH;
  if (!x || !wq || !wk || !wv || !wo || !rope || !cache_k || !cache_v || !out) return GQA_EINVAL;
  void* scratch = nullptr;
  int r = static_scratch(&scratch);
  if (r != GQA_OK) return r;
  // everything gqa_decode checks, checked before the clear is enqueued
  Layout L;
  r = check_common(x, B, 1, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max, out, scratch,
                   max_start_pos + 1, GQA_STATIC_SCRATCH_BYTES, &L);
  if (r != GQA_OK) return r;
  if ((reinterpret_cast<uintptr_t>(start_pos) & 3u) != 0) return GQA_EALIGN;
  cudaError_t e = cudaMemsetAsync(scratch, 0, L.total, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e);
  return gqa_decode(x, B, start_pos, max_start_pos, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v, s_max, out,
                    scratch, GQA_STATIC_SCRATCH_BYTES, stream);
}

extern "C" int gqa_static_device_status(int* status, int clear) {
  if (!status) return GQA_EINVAL;
  void* scratch = nullptr;
  int r = static_scratch(&scratch);
  if (r != GQA_OK) return r;
  return gqa_device_status(scratch, status, clear);
}

// ---------------------------------------------------------------------------
// Host-buffer entries: x and the result in host memory. A caller-provided
// device stage holds two input and two output buffers; call k uses pair
// k % 2. Per stage the library keeps an upload and a read-back stream: call
// k's input is uploaded while call k-1 computes, its block runs on the
// caller's stream, and its result is read back while call k+1 computes.
// gqa_host_stage_wait joins the read-backs into the caller's stream.
// ---------------------------------------------------------------------------
#include <map>

namespace {

struct HostPipe {
  int dev = -1;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t uploaded[2] = {nullptr, nullptr};   // on `up`, after pair k's input is in
  cudaEvent_t computed[2] = {nullptr, nullptr};   // on the caller's stream, after pair k's block
  cudaEvent_t read_back[2] = {nullptr, nullptr};  // on `down`, after pair k's result is out
  bool used[2] = {false, false};
  int next = 0;
};

std::mutex g_pipe_mu;
std::map<const void*, HostPipe> g_pipes;

size_t stage_bytes_for(int B, int T) {
  if (B <= 0 || T <= 0) return 0;
  const size_t m = static_cast<size_t>(B) * T * D_MODEL * 2;
  const size_t slot = (m + 255) & ~static_cast<size_t>(255);
  return 4 * slot;
}

void release_pipe(HostPipe& p) {
  for (int i = 0; i < 2; ++i) {
    for (cudaEvent_t ev : {p.uploaded[i], p.computed[i], p.read_back[i]})
      if (ev) cudaEventDestroy(ev);
  }
  if (p.up) cudaStreamDestroy(p.up);
  if (p.down) cudaStreamDestroy(p.down);
}

// The stage's pipe on the current device (created on first use).
int get_pipe(const void* stage, HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  auto it = g_pipes.find(stage);
  if (it != g_pipes.end()) {
    if (it->second.dev != dev) return GQA_EINVAL;  // a stage belongs to one device
    *out = &it->second;
    return GQA_OK;
  }
  HostPipe p;
  p.dev = dev;
  e = cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&p.uploaded[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.computed[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.read_back[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    release_pipe(p);
    return fail_cuda(e);
  }
  *out = &g_pipes.emplace(stage, p).first->second;
  return GQA_OK;
}

// Upload x_host into pair k's input buffer, run(x_dev, out_dev) on `stream`,
// read out_dev back into out_host.
template <class Run>
int host_call(const gqa_bf16* x_host, gqa_bf16* out_host, int B, int T, void* stage, size_t stage_bytes,
              void* stream, Run run) {
  // run(x_dev, out_dev, dry): dry validates the block's arguments only
  if (!x_host || !out_host || !stage) return GQA_EINVAL;
  const size_t need = stage_bytes_for(B, T);
  if (need == 0) return GQA_EINVAL;
  if (!aligned16(stage)) return GQA_EALIGN;
  if (stage_bytes < need) return GQA_EWORKSPACE;
  const size_t bytes = static_cast<size_t>(B) * T * D_MODEL * 2;
  const size_t slot = need / 4;
  uint8_t* base = static_cast<uint8_t*>(stage);
  // every argument checked before anything is created or enqueued
  int r = run(reinterpret_cast<gqa_bf16*>(base), reinterpret_cast<gqa_bf16*>(base + 2 * slot), true);
  if (r != GQA_OK) return r;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* p = nullptr;
  r = get_pipe(stage, &p);
  if (r != GQA_OK) return r;
  const int k = p->next;
  gqa_bf16* x_dev = reinterpret_cast<gqa_bf16*>(base + k * slot);
  gqa_bf16* out_dev = reinterpret_cast<gqa_bf16*>(base + (2 + k) * slot);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // pair k was last used two calls ago: its block must be done before the
  // upload overwrites its input, its read-back before this block writes
  if (p->used[k]) e = cudaStreamWaitEvent(p->up, p->computed[k], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, p->up);
  if (e == cudaSuccess) e = cudaEventRecord(p->uploaded[k], p->up);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p->uploaded[k], 0);
  if (e == cudaSuccess && p->used[k]) e = cudaStreamWaitEvent(s, p->read_back[k], 0);
  if (e != cudaSuccess) return fail_cuda(e);
  r = run(x_dev, out_dev, false);
  const int launches = t_launches;
  if (r != GQA_OK) return r;
  e = cudaEventRecord(p->computed[k], s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->down, p->computed[k], 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, p->down);
  if (e == cudaSuccess) e = cudaEventRecord(p->read_back[k], p->down);
  if (e != cudaSuccess) return fail_cuda(e);
  p->used[k] = true;
  p->next = k ^ 1;
  t_launches = launches;
  return GQA_OK;
}

}  // namespace

extern "C" size_t gqa_host_stage_bytes(int B, int T) { return stage_bytes_for(B, T); }

extern "C" int gqa_block_forward_host(const gqa_bf16* x_host, int B, int T, int start_pos, int n_kv_heads,
                                      const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
                                      const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v,
                                      int s_max, gqa_bf16* out_host, void* stage, size_t stage_bytes,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return host_call(x_host, out_host, B, T, stage, stage_bytes, stream, [&](gqa_bf16* x, gqa_bf16* out, bool dry) {
    return block_call(x, B, T, start_pos, n_kv_heads, nullptr, 0.f, wq, wk, wv, wo, rope, rope_rows, cache_k, cache_v,
                      s_max, out, workspace, workspace_bytes, stream, dry);
  });
}

extern "C" int gqa_decode_host(const gqa_bf16* x_host, int B, const int32_t* start_pos, int max_start_pos,
                               int n_kv_heads, const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                               const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                               gqa_bf16* cache_v, int s_max, gqa_bf16* out_host, void* stage, size_t stage_bytes,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return host_call(x_host, out_host, B, 1, stage, stage_bytes, stream, [&](gqa_bf16* x, gqa_bf16* out, bool dry) {
    return decode_call(x, B, start_pos, max_start_pos, n_kv_heads, nullptr, 0.f, wq, wk, wv, wo, rope, rope_rows,
                       cache_k, cache_v, s_max, out, workspace, workspace_bytes, stream, dry);
  });
}

extern "C" int gqa_host_stage_wait(void* stage, void* stream) {
  if (!stage) return GQA_EINVAL;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  auto it = g_pipes.find(stage);
  if (it == g_pipes.end()) return GQA_OK;  // no call made on it: nothing to wait for
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != it->second.dev) return GQA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int k = 0; k < 2; ++k) {
    if (!it->second.used[k]) continue;
    const cudaError_t e = cudaStreamWaitEvent(s, it->second.read_back[k], 0);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  return GQA_OK;
}

extern "C" int gqa_host_stage_release(void* stage) {
  if (!stage) return GQA_EINVAL;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  auto it = g_pipes.find(stage);
  if (it == g_pipes.end()) return GQA_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != it->second.dev) return GQA_EINVAL;
  cudaError_t e = cudaStreamSynchronize(it->second.up);
  if (e == cudaSuccess) e = cudaStreamSynchronize(it->second.down);
  release_pipe(it->second);
  g_pipes.erase(it);
  return e == cudaSuccess ? GQA_OK : fail_cuda(e);
}
