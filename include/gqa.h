/*
 * gqa.h — C ABI of the GB300 grouped-query attention block library (libgqa.so).
 *
 * One call runs the attention half of a Llama-3.1-8B transformer block on one
 * GPU: x [B,T,4096] -> delta_attn [B,T,4096], updating the KV cache in place.
 * The operation is the one the page "Llama 3.1 8B · Grouped-query attention"
 * states in its header ("in: x [B batch, T positions, 4096 d], R [positions,
 * 64 pairs]; out: delta_attn; state: KV cache, writes the new rows, reads rows
 * 0..start_pos+T-1") and spells out in its Attention.forward excerpts:
 *
 *   q = x Wq^T, k = x Wk^T, v = x Wv^T                    (bias-free linears,
 *                                                         weights stored [out,in])
 *   q, k rotated by RoPE at position start_pos + t        (apply_rotary_emb)
 *   cache_k/v[b, start_pos + t] = k, v   (bf16)           (the KV-cache state)
 *   o_h = softmax(q_h K_g^T / sqrt(128) + causal mask) V_g, g = h / 4  (repeat_kv)
 *   delta = o Wo^T, o features ordered h*128 + d          (head merge + wo)
 *
 * Fixed dimensions (the Llama 3.1 8B catalogue entry): d_model 4096, 32 query
 * heads, 8 KV heads, head_dim 128. The *_nkv and *_host entries also take 32
 * KV heads (the multi-head variant).
 *
 * Conventions shared by every entry point
 *   - bf16 tensors are raw 16-bit bfloat16 storage (gqa_bf16); all tensors are
 *     dense row-major with the shapes given; device pointers unless stated.
 *   - Every device pointer must be 16-byte aligned (128-bit loads and TMA).
 *   - The caller owns all memory. The library never allocates device memory,
 *     frees it or synchronises: it validates the arguments on the host, then
 *     enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns. Results are ready when the stream reaches that
 *     point. The exceptions are named where they occur: gqa_device_status and
 *     gqa_host_stage_release synchronise; the host-buffer entries create an
 *     upload and a read-back stream with their events per stage on first use.
 *   - Validation happens before any launch; on a non-zero return nothing was
 *     enqueued (except GQA_ECUDA, which reports a failed launch).
 *   - Conditions only the device can see (a per-sequence start position out of
 *     range, a bounded wait that gave up) are recorded in the workspace status
 *     word; read it with gqa_device_status().
 *   - One workspace may serve one call at a time: calls that overlap on the
 *     GPU must use different workspaces.
 */
#ifndef GQA_H
#define GQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gqa_bf16;

#define GQA_D_MODEL 4096
#define GQA_N_HEADS 32
#define GQA_N_KV_HEADS 8
#define GQA_HEAD_DIM 128
#define GQA_ROPE_PAIRS 64

/* Return codes (0 = success). */
#define GQA_OK 0
#define GQA_EINVAL (-1)      /* null pointer, non-positive size, position beyond cache/table */
#define GQA_EALIGN (-2)      /* a pointer is not 16-byte aligned */
#define GQA_EWORKSPACE (-3)  /* workspace smaller than gqa_workspace_bytes() */
#define GQA_ECUDA (-4)       /* a CUDA runtime call or launch failed (see gqa_strerror) */
#define GQA_EDEVICE (-5)     /* gqa_device_status(): a kernel recorded an error */
#define GQA_ESCRATCH (-6)    /* gqa_decode_static: call needs more than GQA_STATIC_SCRATCH_BYTES */

/* Device status codes stored in the workspace status word. */
#define GQA_DEV_OK 0
#define GQA_DEV_BAD_POSITION 1  /* a start position < 0 or >= S_max / rope rows */
#define GQA_DEV_WAIT_TIMEOUT 2  /* a bounded barrier wait gave up */

/* Bytes of workspace a call with batch B, T new tokens per sequence and at
 * most max_keys = start_pos + T cache rows read per sequence needs. The
 * workspace holds the rotated queries, the attention output, split-K
 * partials and tickets. It must be zero-filled before its first use (for
 * example with gqa_workspace_init); every successful call leaves it ready
 * for the next one. Returns 0 for invalid sizes. */
size_t gqa_workspace_bytes(int B, int T, int max_keys);

/* Zero-fill a workspace on `stream` (cudaMemsetAsync). */
int gqa_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Synchronously read the workspace status word into *status (GQA_DEV_*).
 * Returns GQA_EDEVICE when it is non-zero, GQA_OK otherwise. Resets it to 0
 * when `clear` is non-zero. Blocks until all prior work on the device is done. */
int gqa_device_status(void* workspace, int* status, int clear);

/* RoPE table R for positions 0..rows-1: rope[p][i] = (cos, sin) of p * f_i,
 * fp32, shape [rows, 64, 2]. f_i = theta^(-2i/128); with `scaled` non-zero
 * the Llama 3.1 frequency rescaling is applied (pairs whose wavelength
 * 2*pi/f_i exceeds original_context/low_freq_factor are divided by
 * `factor`, those shorter than original_context/high_freq_factor are kept,
 * the band between is interpolated linearly in
 * mu = (original_context/wavelength - low_freq_factor) /
 *      (high_freq_factor - low_freq_factor)).
 * The page "Prepare Q, K, V · Key heads" names the rule; the pages do not
 * print it, and this reading is stated in the design notes. Angles are
 * formed and evaluated in fp64 on the device, then stored as fp32. */
int gqa_rope_table(float* rope, int rows, double theta, int scaled, double factor,
                   double low_freq_factor, double high_freq_factor,
                   double original_context, void* stream);

/* The block for one batch with a common start position (the pages'
 * forward(x, start_pos, freqs_cis, mask)).
 *   x        [B, T, 4096] bf16, the (normalised) block input
 *   wq       [4096, 4096], wk [1024, 4096], wv [1024, 4096], wo [4096, 4096] bf16
 *   rope     [rope_rows, 64, 2] fp32 table from gqa_rope_table (row = position)
 *   cache_k, cache_v  [B, s_max, 8, 128] bf16; rows start_pos..start_pos+T-1
 *            are overwritten with the new rotated keys / values, rows
 *            0..start_pos+T-1 are read, every other row is left untouched
 *   out      [B, T, 4096] bf16, delta_attn
 * Requires start_pos >= 0, start_pos + T <= s_max and <= rope_rows.
 * T == 1 runs the decode path, T > 1 the causal prefill path (the mask of
 * Transformer.forward: query t sees keys 0..start_pos+t). */
int gqa_block_forward(const gqa_bf16* x, int B, int T, int start_pos,
                      const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                      const gqa_bf16* wo, const float* rope, int rope_rows,
                      gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* One decode step (T = 1) with a start position per sequence.
 *   start_pos  device int32 [B]: sequence b has start_pos[b] cached rows,
 *              writes row start_pos[b] and attends over rows 0..start_pos[b]
 *   max_start_pos  a host-side bound with start_pos[b] <= max_start_pos for
 *              every b; it sizes the split-K work and must satisfy
 *              max_start_pos + 1 <= s_max and <= rope_rows.
 * A start_pos[b] outside [0, max_start_pos] is reported as
 * GQA_DEV_BAD_POSITION in the status word and sequence b is skipped: its
 * cache rows are not written and its output row is unspecified. Other
 * arguments as in
 * gqa_block_forward with x [B, 1, 4096] and out [B, 1, 4096]. The split
 * work is counted in 32 bits: B x ceil((max_start_pos + 1) / 16) x (SMs + 1)
 * must stay below 2^32 (about 28 million cache positions over the batch on
 * 152 SMs, far past what one GPU's memory holds), else GQA_EINVAL. */
int gqa_decode(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos,
               const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
               const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v,
               int s_max, gqa_bf16* out, void* workspace, size_t workspace_bytes,
               void* stream);

/* The multi-head variant next to the grouped one: "Llama 3.1 8B ·
 * Grouped-query attention" sets the model's 8 KV heads against MHA with 32
 * K/V heads (its table of KV cache per token: 512 KiB over all layers
 * against 128 KiB), and its repeat_kv excerpt returns the keys and values
 * unchanged when n_rep = 1. n_kv_heads selects the KV heads:
 *   8   the Llama 3.1 8B block (the same operation as gqa_block_forward /
 *       gqa_decode)
 *   32  one KV head per query head: wk, wv [4096, 4096]; cache_k, cache_v
 *       [B, s_max, 32, 128] bf16 (8 KB of K and 8 KB of V per position);
 *       query head h attends with KV head h
 * Any other value is GQA_EINVAL. Every other argument, the workspace size
 * (gqa_workspace_bytes covers both), the cache update and the error
 * behaviour as in gqa_block_forward / gqa_decode; gqa_decode_nkv with 32 KV
 * heads also requires B <= 512. The multi-head decode step of up to 16
 * sequences runs as one grid like the grouped one (its Q|K|V projection in
 * three passes over Wq, Wk and Wv; see gqa_set_decode_fusion), larger batches
 * as three kernels. */
int gqa_block_forward_nkv(const gqa_bf16* x, int B, int T, int start_pos, int n_kv_heads,
                          const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                          const gqa_bf16* wo, const float* rope, int rope_rows,
                          gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out,
                          void* workspace, size_t workspace_bytes, void* stream);
int gqa_decode_nkv(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos,
                   int n_kv_heads, const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                   const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                   gqa_bf16* cache_v, int s_max, gqa_bf16* out, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Causal prefill of T >= 1 new tokens per sequence after start_pos cached
 * rows (start_pos > 0 is a chunked prefill over an existing prefix).
 * Arguments as in gqa_block_forward. */
int gqa_prefill(const gqa_bf16* x, int B, int T, int start_pos, const gqa_bf16* wq,
                const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
                const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v,
                int s_max, gqa_bf16* out, void* workspace, size_t workspace_bytes,
                void* stream);

/* The attention half of a transformer block with its norm and residual: the
 * TransformerBlock.forward excerpt of "Llama 3.1 8B · Grouped-query
 * attention" (handoff) and "Llama 3 8B · Attention update"
 * (block-residuals):
 *     h = x + attention(attention_norm(x))
 * attention_norm is RMSNorm over the 4096 features,
 *     g_i x_i / sqrt(mean_j x_j^2 + eps)
 * (norm_eps 1e-05 in the catalogue entries; the pages name the module but
 * do not print its body), and attention() is gqa_block_forward's operation
 * on the normalised rows.
 *   x       [B, T, 4096] bf16, the block input (the residual stream)
 *   norm_w  [4096] bf16, the RMSNorm weight g (16-byte aligned)
 *   eps     finite, > 0
 *   h       [B, T, 4096] bf16, x + delta_attn; must not be x itself
 * Every other argument, the cache update and the error behaviour as in
 * gqa_block_forward. One more kernel than gqa_block_forward (the norm). */
int gqa_layer_forward(const gqa_bf16* x, int B, int T, int start_pos, const gqa_bf16* norm_w, float eps,
                      const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv, const gqa_bf16* wo,
                      const float* rope, int rope_rows, gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max,
                      gqa_bf16* h, void* workspace, size_t workspace_bytes, void* stream);

/* attention_norm alone: y[m] = g * x[m] / sqrt(mean(x[m]^2) + eps) for M rows
 * of 4096 features (x, y [M, 4096] bf16, norm_w [4096] bf16, all 16-byte
 * aligned; y may be x). The same kernel gqa_layer_forward runs first;
 * computed in fp32, rounded once to bf16. */
int gqa_rms_norm(const gqa_bf16* x, int M, const gqa_bf16* norm_w, float eps, gqa_bf16* y, void* stream);

/* gqa_layer_forward for one decode step with a start position per sequence
 * (start_pos, max_start_pos as in gqa_decode). */
int gqa_layer_decode(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos,
                     const gqa_bf16* norm_w, float eps, const gqa_bf16* wq, const gqa_bf16* wk,
                     const gqa_bf16* wv, const gqa_bf16* wo, const float* rope, int rope_rows,
                     gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* h, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Static description of a return code (GQA_ECUDA appends the last CUDA
 * error name seen by this library on the calling thread). */
const char* gqa_strerror(int status);

/* Number of kernels the most recent successful call on this thread enqueued. */
int gqa_last_launch_count(void);

/* Selects, for the calling thread, how a decode step (T = 1) of at most 64
 * sequences (16 with 32 KV heads) is launched: enable != 0 (the default) runs it as one persistent
 * cooperative kernel (projection, attention and output projection ordered by
 * counters in the workspace's status region; launched with programmatic
 * stream serialization, it touches no memory before the previous kernel of
 * the stream has completed, so stream order holds as usual); enable = 0 as
 * three kernels.
 * Both compute the same function. Returns the previous setting. */
int gqa_set_decode_fusion(int enable);

/* Selects, for the calling thread, how the one-kernel decode step (see
 * gqa_set_decode_fusion) splits its attention over the grid:
 *   0  (the default) chosen per call: head-major when the batch has at most
 *      SMs / 8 sequences and one head's cache rows stream faster on one SM
 *      than the whole batch's rows over every SM plus a merge round (small
 *      batches of short contexts: B = 16 at 1,001 keys is head-major, B = 8
 *      at 131,072 keys and every batch above 19 position-major);
 *   1  position-major: the cache rows of the batch in 16-position units
 *      spread evenly over the grid; sequences split between CTAs are merged
 *      by the log-sum-exp rule after a grid-wide meeting;
 *   2  head-major where the batch fits (B * 8 <= SMs; else position-major):
 *      one CTA per (sequence, KV head) pair reads all of that head's rows,
 *      nothing is merged across CTAs.
 * Every mode computes the same function (reassociated fp32 sums). Returns
 * the previous setting, or -1 (nothing changed) for another value. */
int gqa_set_decode_attention_split(int mode);

/* Limit, for calls made on the calling thread, of the grid-wide waits of the
 * decode kernels: the one-kernel step's two gates (every CTA's Q|K|V rows
 * published; every attention output published) and the attention's meeting
 * before its merges. A wait that runs out records GQA_DEV_WAIT_TIMEOUT in the
 * workspace status word; the kernel then skips the work that needed the
 * wait, lets its own loads land, leaves the grid counters reset and exits
 * (the call's output is unspecified). ns = 0 restores the default of 2 s
 * (2,000,000,000 ns). Returns the previous limit. Meant for tests and for
 * callers that prefer a fast error over a long stall; the waits on the
 * kernels' own data loads keep their 2 s limit. */
unsigned long long gqa_set_wait_limit_ns(unsigned long long ns);

/* Measurement hook; it changes nothing the block computes. While set, every
 * block call on the calling thread records events[0] on its stream before its
 * first kernel and events[i] right after its i-th kernel (for i < count), so
 * a profiler can time each kernel with cudaEventElapsedTime. `events` holds
 * caller-created cudaEvent_t handles and must stay valid while set;
 * count = 0 (or events = NULL) stops the recording. */
int gqa_set_profile_events(void* const* events, int count);

/* Size of the scratch array gqa_decode_static works in (16 MiB). */
#define GQA_STATIC_SCRATCH_BYTES (16u << 20)

/* gqa_decode without a workspace argument, for callers that cannot allocate
 * device memory when they run a step: for instance an engine plugin whose
 * enqueue hook must not call cudaMalloc, or a real-time serving loop where a
 * synchronous allocation would stall the device. The pages have no
 * counterpart to this; it only changes where the scratch memory lives.
 *
 * The scratch (rotated queries, attention output, split-K partials, tickets,
 * status word) is a file-scope __device__ array of GQA_STATIC_SCRATCH_BYTES
 * inside libgqa, so every GPU that loads the library holds it until the
 * process exits. Arguments and results are exactly those of gqa_decode; the
 * caller still passes every input and output buffer.
 *   - A call whose workspace (gqa_workspace_bytes(B, 1, max_start_pos + 1))
 *     exceeds GQA_STATIC_SCRATCH_BYTES returns GQA_ESCRATCH and enqueues
 *     nothing; every batch of up to 64 sequences fits, at any length.
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress); make that first call before any stream
 *     capture.
 *   - Each call clears the part of the array it uses (cudaMemsetAsync on
 *     `stream`) before its kernels; it allocates and frees nothing.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents: calls that overlap on the GPU (different streams, or several
 *     host threads) race and must be serialised by the caller.
 *   - Device-side errors go to the array's status word; read them with
 *     gqa_static_device_status. */
int gqa_decode_static(const gqa_bf16* x, int B, const int32_t* start_pos, int max_start_pos,
                      const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                      const gqa_bf16* wo, const float* rope, int rope_rows,
                      gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out,
                      void* stream);

/* Status word of the gqa_decode_static scratch on the current device (as
 * gqa_device_status: synchronises, returns GQA_EDEVICE when non-zero). */
int gqa_static_device_status(int* status, int clear);

/* Host-buffer entries: the block input in host memory and the result
 * written back to host memory, for a caller whose tokens live on the host
 * (a serving loop reading requests, a test harness).
 *   x_host    [B, T, 4096] bf16 in host memory; pinned (page-locked) memory
 *             lets the copies run asynchronously (pageable memory works, the
 *             driver then stages the copy). It must stay unchanged until
 *             `stream` has reached the call.
 *   out_host  [B, T, 4096] bf16 in host memory: delta_attn
 *   stage     device buffer of gqa_host_stage_bytes(B, T) bytes, 16-byte
 *             aligned, owned by the caller and used on one device: two input
 *             and two output buffers. Call k on a stage uses pair k % 2.
 * Per stage the library keeps an upload stream and a read-back stream: call
 * k's input is uploaded while call k-1's block runs, the block runs on
 * `stream` (after the upload, and after call k-2's read-back released the
 * pair), and the result is read back while call k+1's block runs. The
 * results of every call made so far on a stage are in host memory once
 * `stream` has reached a later gqa_host_stage_wait(stage, stream).
 * Every other argument, the cache update and the error behaviour as in
 * gqa_block_forward_nkv / gqa_decode_nkv (all arguments are checked before
 * anything is enqueued; GQA_EWORKSPACE also when stage_bytes is too small).
 * Not for stream capture (the copy streams are outside any capture).
 * gqa_host_stage_release(stage) waits for the stage's copy streams and
 * frees them and their events; GQA_EINVAL for a stage it does not know. */
size_t gqa_host_stage_bytes(int B, int T);
int gqa_block_forward_host(const gqa_bf16* x_host, int B, int T, int start_pos, int n_kv_heads,
                           const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                           const gqa_bf16* wo, const float* rope, int rope_rows,
                           gqa_bf16* cache_k, gqa_bf16* cache_v, int s_max, gqa_bf16* out_host,
                           void* stage, size_t stage_bytes, void* workspace,
                           size_t workspace_bytes, void* stream);
int gqa_decode_host(const gqa_bf16* x_host, int B, const int32_t* start_pos, int max_start_pos,
                    int n_kv_heads, const gqa_bf16* wq, const gqa_bf16* wk, const gqa_bf16* wv,
                    const gqa_bf16* wo, const float* rope, int rope_rows, gqa_bf16* cache_k,
                    gqa_bf16* cache_v, int s_max, gqa_bf16* out_host, void* stage,
                    size_t stage_bytes, void* workspace, size_t workspace_bytes, void* stream);
int gqa_host_stage_wait(void* stage, void* stream);
int gqa_host_stage_release(void* stage);

#ifdef __cplusplus
}
#endif

#endif /* GQA_H */
