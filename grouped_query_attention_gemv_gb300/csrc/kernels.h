// Internal interface between the C ABI (api.cu) and the kernel translation
// units. Not installed; the public contract is include/gqa.h.
#pragma once

#include "common.cuh"

namespace gqa {

// One projection y = x W^T over M tokens (rows of x, stride 4096) and N
// output features. The weight is up to three [rows, 4096] matrices stacked
// along the output axis: rows [0, r1) from w0, [r1, r2) from w1, [r2, N) from
// w2 (the fused Q|K|V projection uses wq, wk, wv with r1 = 4096 and
// r2 - r1 = N - r2 = the cache row: 1024 for 8 KV heads, 4096 for 32).
struct ProjParams {
  const __nv_bfloat16* x;
  int M;   // tokens
  int T;   // tokens per sequence: token m is (b = m / T, t = m % T)
  const __nv_bfloat16* w0;
  const __nv_bfloat16* w1;
  const __nv_bfloat16* w2;
  int r1, r2, N;
  int qkv;  // 0: plain store out[m][n]; 1: Q|K|V epilogue (RoPE, cache append)
  __nv_bfloat16* out;  // plain: [M][N]; Q|K|V: rotated queries [M][4096]
  __nv_bfloat16* cache_k;
  __nv_bfloat16* cache_v;
  int s_max;
  const float* rope;  // [rope_rows][64][2] (cos, sin)
  StartPos sp;
  int* status;
  const __nv_bfloat16* resid;  // plain store only: [M][N] added to the output (the block's residual), or null
  const __nv_bfloat16* norm_w; // fused decode Q|K|V phase only: attention_norm weight applied to x, or null
  float eps;
};

// Rotate pair (a, b) of feature f (even) by the table row `pos`.
__device__ __forceinline__ void rope_pair(const float* rope, int pos, int f, float& a, float& b) {
  const float2 cs = *reinterpret_cast<const float2*>(rope + (static_cast<size_t>(pos) * ROPE_PAIRS +
                                                             ((f & (HEAD_DIM - 1)) >> 1)) * 2);
  const float ra = a * cs.x - b * cs.y;
  const float rb = a * cs.y + b * cs.x;
  a = ra;
  b = rb;
}

// Destination of features [f, f+n) of token m, n <= 16 and inside one head.
// Returns null (and records the error) when the token's position is invalid.
__device__ __forceinline__ __nv_bfloat16* proj_dst(const ProjParams& p, int m, int f, int& pos) {
  if (!p.qkv) {
    pos = 0;
    return p.out + static_cast<size_t>(m) * p.N + f;
  }
  const int b = m / p.T;
  const int t = m - b * p.T;
  const int start = p.sp.get(b);
  if (!p.sp.ok(start)) {
    if (t == 0 && (f & 127) == 0) report(p.status, DEV_BAD_POSITION);
    return nullptr;
  }
  pos = start + t;
  if (f < D_MODEL) return p.out + static_cast<size_t>(m) * D_MODEL + f;
  const size_t row = (static_cast<size_t>(b) * p.s_max + pos) * (p.r2 - p.r1);
  if (f < p.r2) return p.cache_k + row + (f - D_MODEL);
  return p.cache_v + row + (f - p.r2);
}

// Epilogue for 16 consecutive features f..f+15 (f multiple of 16) of token m.
__device__ __forceinline__ void proj_store16(const ProjParams& p, int m, int f, float (&v)[16]) {
  int pos;
  __nv_bfloat16* dst = proj_dst(p, m, f, pos);
  if (!dst) return;
  if (p.qkv && f < p.r2) {
    const float4* cs = reinterpret_cast<const float4*>(
        p.rope + (static_cast<size_t>(pos) * ROPE_PAIRS + ((f & (HEAD_DIM - 1)) >> 1)) * 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 c = cs[j];  // pairs 2j, 2j+1: (cos, sin, cos, sin)
      float a = v[4 * j], b = v[4 * j + 1];
      v[4 * j] = a * c.x - b * c.y;
      v[4 * j + 1] = a * c.y + b * c.x;
      a = v[4 * j + 2];
      b = v[4 * j + 3];
      v[4 * j + 2] = a * c.z - b * c.w;
      v[4 * j + 3] = a * c.w + b * c.z;
    }
  }
  uint4 lo, hi;
  lo.x = pack_bf16(v[0], v[1]);
  lo.y = pack_bf16(v[2], v[3]);
  lo.z = pack_bf16(v[4], v[5]);
  lo.w = pack_bf16(v[6], v[7]);
  hi.x = pack_bf16(v[8], v[9]);
  hi.y = pack_bf16(v[10], v[11]);
  hi.z = pack_bf16(v[12], v[13]);
  hi.w = pack_bf16(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = lo;
  reinterpret_cast<uint4*>(dst)[1] = hi;
}

// Epilogue for the feature pair (f, f+1), f even.
__device__ __forceinline__ void proj_store2(const ProjParams& p, int m, int f, float a, float b) {
  int pos;
  __nv_bfloat16* dst = proj_dst(p, m, f, pos);
  if (!dst) return;
  if (p.qkv && f < p.r2) rope_pair(p.rope, pos, f, a, b);
  *reinterpret_cast<uint32_t*>(dst) = pack_bf16(a, b);
}

// ----------------------------------------------------------------- launches
// tcgen05 GEMM for M > 64 tokens, persistent over at most `ctas` CTAs (one
// per SM). Maps are created by the caller.
struct GemmMaps {
  CUtensorMap a;      // activations [M][4096]
  CUtensorMap b[3];   // w0, w1, w2
};
cudaError_t launch_gemm_tc(const GemmMaps& maps, const ProjParams& p, int ctas, cudaStream_t s);
constexpr int GEMM_BN = 256;
constexpr int GEMM_BM = 128;

// Few-token projection on tcgen05 (swap-AB, persistent stream-K), M <= 64.
// Tensor maps view a [rows][4096] matrix in 3-D as (64 values, row, k block)
// so that one box carries several consecutive k blocks of the same rows:
// w[kc-1][i] / x[kc-1] boxes hold kc = 1..4 k blocks, so every stretch of k
// blocks is fetched in ceil(len / 4) boxes.
struct ProjStreamMaps {
  CUtensorMap w[4][3];  // weights: box 64 x 128 rows x kc, matrices w0, w1, w2
  CUtensorMap x[4];     // tokens: box 64 x NP x kc
};
// part: fp32 [ctas * segmax][128][NP] slots; tickets: int [N/128], zero-filled,
// left zero-filled.
struct ProjStreamArgs {
  ProjStreamMaps maps;
  ProjParams p;
  float* part;
  int* tickets;
  int segmax;
  int ctas;
};
int proj_stream_np(int M);                 // padded token count (0 if M > 64)
int proj_stream_segmax(int N, int ctas);   // partial slots per CTA
cudaError_t launch_proj_stream(const ProjStreamArgs& a, cudaStream_t s, bool pdl);

// Decode attention (one new token per sequence), persistent stream-K over
// 16-position units of the batch, all 8 KV heads per unit.
constexpr int DECODE_MAX_B = 2048;  // sequences per launch (prefix sums live in shared memory)
constexpr int DECODE_UNIT = 16;     // cache positions per unit (TMA box) of the decode attention
constexpr int PREFILL_TILE = 64;    // cache positions per TMA box of the prefill kernel
constexpr int DECODE_ITEM_POS = 128; // cache positions per TMA box of the head-major decode attention
struct DecodeAttnParams {
  const __nv_bfloat16* q;  // [B][4096] rotated queries
  int B;
  int n_kv;                // KV heads: 8, or 32 (the multi-head variant)
  StartPos sp;             // keys 0..sp(b) are read
  int ctas;                // grid size (one CTA per SM)
  float* part_o;           // [attn_decode_slots(ctas) / 8][32 query heads][128]
  float* part_ml;          // [attn_decode_slots(ctas) / 8][32][2] (running max in log2 units, sum)
  int* counters;           // [2] grid counters (meeting, exit), zero-filled, left zero-filled
  __nv_bfloat16* o;        // [B][4096]
  int* status;
  const __nv_bfloat16* cache_k;  // [B][s_max][n_kv][128]: L2 prefetches; the head-major split's new row
  const __nv_bfloat16* cache_v;
  int s_max;
  unsigned long long wait_ns;    // limit of the grid-wide waits (the meeting; the fused grid's gates)
};
int attn_decode_ctas(int num_sms);
int attn_decode_slots(int ctas);   // (CTA, first or last stretch, KV head) partial slots
// Cache tensor maps of the decode attention: (dim, position, KV head,
// sequence) with boxes of 64 dims x 16 positions x 8 heads.
struct DecodeCacheMaps {
  CUtensorMap k, v;
};
// Cooperative launch: the CTAs meet once before the merges.
cudaError_t launch_attn_decode(const DecodeCacheMaps& maps, const DecodeAttnParams& a, cudaStream_t s);

// Causal prefill attention.
struct PrefillAttnParams {
  const __nv_bfloat16* q;  // [B*T][4096] rotated queries
  int B, T;
  int n_kv;                // KV heads: 8, or 32 (the multi-head variant)
  StartPos sp;             // common start position (chunked prefill when > 0)
  __nv_bfloat16* o;        // [B*T][4096]
  int* status;
  int num_sms;             // CTAs of the persistent grid at most
};
// Tensor maps of the prefill attention: q over (dim, head, token, sequence)
// with boxes of 64 dims x n_rep heads x 128 / n_rep tokens; k / v over (dim, KV head,
// position, sequence) with boxes of 64 dims x 1 head x PREFILL_TILE positions
// and a position extent of start_pos + T, so later positions read as zero.
struct PrefillMaps {
  CUtensorMap q, k, v;
};
cudaError_t launch_attn_prefill(const PrefillMaps& maps, const PrefillAttnParams& a, cudaStream_t s);

// Row-owner projection of the fused decode grid: the rows of matrix i are
// split over ctas[i] CTAs in row pairs; a CTA owns h_lo[i] or h_lo[i] + 2
// rows. CTAs of matrix 0 come first, then 1, then 2.
struct RowPlan {
  int nmat;
  int rows[3];
  int ctas[3];
  int h_lo[3];
  int mat0;  // RowMaps index of matrix 0 (0; a pass over one matrix of three sets it to that matrix)
  int cta0;  // first CTA of the split: CTAs [0, cta0) own no rows (0 unless set after make_row_plan)
};
constexpr int ROWS_MAX_H = 48;   // rows one CTA can own (3 row tiles of 16)
// k blocks of 64 per stage of the row-owner projections for np padded tokens
// (8; 4 at 64 tokens, where the warps split the tokens): the weight and token
// boxes of the fused grid's tensor maps hold this many k blocks.
__host__ __device__ constexpr int rows_kc(int np) { return np <= 32 ? 8 : 4; }
// Tensor maps over (64 k, row, k block) views of the weight matrices:
// w[i][0] / w[i][1] are matrix i with boxes of 64 x h_lo[i] (or h_lo[i] + 2)
// rows x rows_kc(NP) k blocks; x is the same view of the M token rows with
// boxes of 64 x NP tokens x rows_kc(NP) k blocks (NP = decode_fused_np(M)).
struct RowMaps {
  CUtensorMap w[3][2];
  CUtensorMap x;
};
// Splits nmat matrices of the given row counts over `ctas` CTAs; false if a
// CTA would own more than ROWS_MAX_H rows or a matrix gets no CTA.
bool make_row_plan(int nmat, const int* rows, int ctas, RowPlan* plan);

// The whole decode step (Q|K|V projection, attention, W_O projection) in one
// persistent cooperative grid, for batches of up to FUSED_MAX_B sequences.
constexpr int FUSED_MAX_B = 64;
struct DecodeFusedArgs {
  RowMaps qkv_maps, o_maps;
  RowPlan qkv_plan, o_plan;
  DecodeCacheMaps cache;     // position-major view (DecodeCacheMaps above)
  DecodeCacheMaps cache_hm;  // head-major view: (dim, KV head, position, sequence), boxes of 64 dims x 1 head x
                             // 128 positions (used when head_major)
  int head_major;            // attention split: one (sequence, KV head) pair per CTA (B * 8 <= ctas) or
                             // position-major units with merges
  ProjParams pq, po;       // Q|K|V (qkv = 1) and W_O (qkv = 0) projections
  DecodeAttnParams at;
  int* counters;           // [3] grid progress counters, zero-filled, left zero-filled
  int ctas;                // one CTA per SM
  int qkv_passes;          // 1 (8 KV heads: qkv_plan splits all 6,144 rows) or 3 (32 KV heads: qkv_plan
                           // splits one 4,096-row matrix, walked for Wq, Wk, Wv in turn)
};
cudaError_t launch_decode_fused(const DecodeFusedArgs& a, cudaStream_t s);
int decode_fused_np(int M);   // padded tokens of the fused grid's projections (0 if M > 64)

// attention_norm: y[m] = g * x[m] / sqrt(mean(x[m]^2) + eps) for M rows of 4096.
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* g, float eps, int M, __nv_bfloat16* y,
                           cudaStream_t s);

cudaError_t launch_rope_table(float* rope, int rows, double theta, int scaled, double factor, double lo,
                              double hi, double ctx, cudaStream_t s);

}  // namespace gqa
