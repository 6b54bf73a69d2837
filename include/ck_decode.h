/*
 * ck_decode.h -- C ABI of the GB300 (sm_103a) single-token attention decode
 * step of an LLM layer with Q5_0 / Q8_0 quantized weights.
 *
 * The operation is the serial kernel of the page
 * "mega_fused_attention_decode_q5_0.c" (C-Kernel-Engine): RMSNorm, Q8_0
 * quantization of the normed activation, Q and K projections with Q5_0
 * weights and the V projection with Q8_0 weights (each plus a bias), RoPE,
 * the KV-cache store, GQA decode attention over the cache, Q8_0
 * quantization of the attention output, the Q5_0 O projection with bias,
 * and the residual add.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer (memory of the current CUDA
 *    device) unless stated otherwise, owned by the caller, and must be
 *    16-byte aligned.  The library allocates nothing and keeps no pointer
 *    after a call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously; no call synchronizes the stream or the device,
 *    so every call may be recorded into a CUDA graph by stream capture.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    call that returns an error has enqueued nothing.  CK_ECUDA reports a
 *    failed launch (cudaGetLastError after the launch).
 *  - Weights are row-major arrays of blocks exactly as the page lays them
 *    out: a matrix [M, K] is M rows of K/32 consecutive blocks.
 *  - fp32 vectors are dense; KV caches are head-major fp32
 *    [num_kv_heads, cache_capacity, head_dim]; RoPE tables are fp32
 *    [cache_capacity, head_dim/2] (row p holds cos / sin of position p).
 */
#ifndef CK_DECODE_H
#define CK_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define CK_OK 0
#define CK_EINVAL (-1)   /* null pointer, non-positive or inconsistent size   */
#define CK_ERANGE (-2)   /* pos / kv_tokens outside the cache                 */
#define CK_ESCRATCH (-3) /* scratch missing or smaller than the size query    */
#define CK_EALIGN (-4)   /* a pointer is not 16-byte aligned                  */
#define CK_ECUDA (-5)    /* a CUDA runtime call or a kernel launch failed     */
#define CK_ETIMEOUT (-6) /* (device status only) a bounded device wait expired */

/* Human-readable name of a status code (static storage, never NULL). */
const char *ck_status_string(int status);

/* ---- block formats (32 weights per block) ------------------------------ */
#define CK_QK 32

/* Q5_0, 22 bytes: d = fp16 scale (little-endian bits), qh = bit 4 of each of
 * the 32 codes (bit j <-> element j), qs[j] = low nibble of element j (bits
 * 0-3) and of element j+16 (bits 4-7).  Weight j = (code_j - 16) * d. */
typedef struct {
    uint16_t d;
    uint8_t qh[4];
    uint8_t qs[16];
} ck_block_q5_0;

/* Q8_0, 34 bytes: d = fp16 scale, qs = 32 signed codes.  Weight j = qs[j]*d.
 * Activations are quantized to this format with d = amax/127 (fp32) stored
 * as fp16, and code = round-half-away-from-zero(x * (1/d)). */
typedef struct {
    uint16_t d;
    int8_t qs[32];
} ck_block_q8_0;

/* ---- single steps ------------------------------------------------------ */

/* quantize_row_q8_0 (page: declared, used for the normed activation and the
 * attention output).  x: fp32 [n]; y_q8: n/32 Q8_0 blocks.  n > 0, n % 32 == 0.
 * Bit-exact: the codes and the fp16 scale follow the rule above in IEEE
 * fp32 (correctly rounded divide and reciprocal). */
int ck_quantize_q8_0(const float *x, void *y_q8, int n, void *stream);

/* gemv_q5_0_from_fp32 after its quantize step (page: Q5_0 GEMV with inline
 * processing): y[r] = sum_b d_w(r,b) * d_x(b) * isum(r,b) + bias[r] for
 * r < M, with isum the exact int32 dot of the 32 codes of block b.
 * W: [M, K] Q5_0; x_q8: K/32 Q8_0 blocks; bias: fp32 [M] or NULL; y: fp32 [M].
 * K % 32 == 0, M > 0. */
int ck_gemv_q5_0_q8_0(float *y, const void *W, const void *x_q8, const float *bias, int M, int K, void *stream);

/* gemv_q8_0_from_fp32 after its quantize step (page: Q8_0 GEMV, used for the
 * V projection).  Same arguments with W: [M, K] Q8_0. */
int ck_gemv_q8_0_q8_0(float *y, const void *W, const void *x_q8, const float *bias, int M, int K, void *stream);

/* apply_rope_inline (page: RoPE application).  Rotate-half RoPE in place:
 * with half = head_dim/2 and row `pos` of the tables, element d of every
 * head pairs with d + half: (a, b) -> (a*cos - b*sin, a*sin + b*cos).
 * q: fp32 [num_heads * head_dim] (may be NULL when num_heads == 0);
 * k: fp32 [num_kv_heads * head_dim] (may be NULL when num_kv_heads == 0);
 * rope_cos / rope_sin: fp32 [cache_capacity, head_dim/2].
 * 0 <= pos < cache_capacity (else CK_ERANGE); head_dim even. */
int ck_rope_inplace(float *q, float *k, const float *rope_cos, const float *rope_sin, int pos, int num_heads,
                    int num_kv_heads, int head_dim, int cache_capacity, void *stream);

/* KV-cache store (page: STEP 6).  k_cache[h][pos][:] = k[h*head_dim ...],
 * v_cache[h][pos][:] = v[...] for every KV head h.  0 <= pos < cache_capacity. */
int ck_kv_store(float *k_cache, float *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                int cache_capacity, int head_dim, void *stream);

/* attention_forward_decode_head_major_gqa_flash (page: declared, STEP 7).
 * For query head h, KV head g = h*num_kv_heads/num_heads and the first
 * kv_tokens rows t of that head's cache: out_h = sum_t softmax_t(q_h.k_t /
 * sqrt(head_dim)) v_t.  q, out: fp32 [num_heads * head_dim].
 * Requirements: num_heads % num_kv_heads == 0, num_heads/num_kv_heads <= 8,
 * head_dim in {32, 64, 96, 128, 256},
 * 1 <= kv_tokens <= cache_capacity (else CK_ERANGE).
 * `scratch` (device, >= ck_attn_scratch_size(...) bytes for a max_kv_tokens
 * >= kv_tokens) holds the split-KV partial results; its contents need no
 * initialization and are dead after the stream reaches the end of the call. */
size_t ck_attn_scratch_size(int num_heads, int num_kv_heads, int max_kv_tokens, int head_dim);
int ck_attn_decode_gqa(const float *q, const float *k_cache, const float *v_cache, float *out, int num_heads,
                       int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, void *scratch,
                       size_t scratch_bytes, void *stream);

/* The same attention for callers that cannot allocate device memory -- code
 * whose device memory belongs to another allocator or a fixed budget, and
 * decode loops that must not pay for a cudaMalloc, which can synchronize the
 * device.  The pages have no counterpart: this is a library convenience.
 * Arguments, requirements and result are those of ck_attn_decode_gqa minus
 * the scratch: the split-KV partials live in one buffer compiled into the
 * library, CK_ATTN_NOALLOC_MAX_BYTES of device memory that every GPU which
 * loads the library keeps until the process exits.  A shape whose partials
 * need more is rejected with CK_ESCRATCH before anything is enqueued; every supported
 * shape fits on a 152-SM GB300.  The call allocates nothing.  The first call
 * on a device looks up the buffer's device address (cudaGetSymbolAddress,
 * with that device current) and caches it; make that first call before any
 * stream capture.  All calls share the buffer and it keeps the last call's
 * contents (nothing in it needs to start at zero); calls whose work overlaps
 * on the GPU (other streams or host threads on the same device) race on it. */
#define CK_ATTN_NOALLOC_MAX_BYTES (2u * 1024u * 1024u)
int ck_attn_decode_gqa_noalloc(const float *q, const float *k_cache, const float *v_cache, float *out,
                               int num_heads, int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim,
                               void *stream);

/* ---- reduced-precision KV caches ---------------------------------------- */

/* The same decode attention over a bf16 or an fp8 cache (page
 * "prefill_attn_a.rs", layers/ops: the launchers paged_decode_attn_bf16 / paged_decode_attn_fp8:
 * bf16 and fp8 KV caches, the fp8 one with per-tensor k_scale and v_scale;
 * here on the head-major layout of ck_attn_decode_gqa, not paged).
 * k_cache / v_cache: [num_kv_heads, cache_capacity, head_dim] elements of
 *   - bf16 (ck_attn_decode_gqa_bf16): the value is the bf16 number;
 *   - fp8 E4M3 (ck_attn_decode_gqa_fp8; 1 sign, 4 exponent bits with bias 7,
 *     3 mantissa bits, subnormals, largest finite 448, 0x7F / 0xFF are NaN,
 *     no infinities): the value is code * k_scale (keys), code * v_scale
 *     (values); k_scale, v_scale finite and > 0 (else CK_EINVAL).
 * head_dim in {64, 128} (else CK_EINVAL); otherwise the arguments,
 * requirements, scratch and result of ck_attn_decode_gqa.  Arithmetic: at
 * head_dim 128 both products run on the tensor cores with fp32
 * accumulation.  The cache values are exact there, q is taken as three
 * bf16 parts (scores to fp32 quality), and the probabilities as two parts
 * (bf16 for bf16 caches, fp16 for fp8), about 2^-17 / 2^-22 relative.  At
 * head_dim 64 the arithmetic is fp32 on the CUDA cores. */
int ck_attn_decode_gqa_bf16(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                            int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, void *scratch,
                            size_t scratch_bytes, void *stream);
int ck_attn_decode_gqa_fp8(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                           int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, float k_scale,
                           float v_scale, void *scratch, size_t scratch_bytes, void *stream);

/* Split tuning.  The page "attn_v41/decode.rs" (spark_model layers) splits
 * the output dimension of each head over several blocks when one block a
 * head leaves SMs idle.  Here the same end is reached by splitting the
 * attended rows (each split a partial softmax record, merged by a combine),
 * which reads every row once; ck_attn_decode_gqa picks the split count from
 * the SM count.  This entry point takes it explicitly, for tuning: the same
 * attention as ck_attn_decode_gqa (kv_dtype 0), _bf16 (1) or _fp8 (2, with
 * k_scale / v_scale; ignored otherwise) with `splits` splits of the rows per
 * KV head, 1 <= splits <= 1024, or 0 for the built-in choice (otherwise
 * CK_EINVAL).  Splits past the last row are empty and contribute nothing.
 * `scratch`: >= ck_attn_split_scratch_size(num_heads, num_kv_heads,
 * head_dim, splits) bytes (0 for invalid arguments); with splits = 0,
 * ck_attn_scratch_size(...). */
size_t ck_attn_split_scratch_size(int num_heads, int num_kv_heads, int head_dim, int splits);
int ck_attn_decode_gqa_split(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                             int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, int kv_dtype,
                             float k_scale, float v_scale, int splits, void *scratch, size_t scratch_bytes,
                             void *stream);

/* KV-cache store (page: STEP 6) into those caches: k_cache[h][pos][:] and
 * v_cache[h][pos][:] from the fp32 rows k, v [num_kv_heads * head_dim].
 * bf16: round to nearest, ties to even.  fp8: code = E4M3(x / scale) with x /
 * scale the IEEE fp32 quotient, rounded to nearest (ties to even) and
 * saturated to +-448 (NaN stays NaN).  0 <= pos < cache_capacity (else
 * CK_ERANGE); fp8 scales finite and > 0 (else CK_EINVAL). */
int ck_kv_store_bf16(void *k_cache, void *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                     int cache_capacity, int head_dim, void *stream);
int ck_kv_store_fp8(void *k_cache, void *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                    int cache_capacity, int head_dim, float k_scale, float v_scale, void *stream);

/* Paged decode attention with an optional sliding window (page
 * "prefill_attn_a.rs", layers/ops: paged_decode_attn_bf16 / paged_decode_attn_fp8 and their GQA
 * forms, arguments block_tables, seq_lens, max_blocks_per_seq, block_size,
 * sliding_window, k_scale, v_scale), for a batch of sequences.
 *   k_pool / v_pool: [num_blocks, num_kv_heads, block_size, head_dim]
 *     elements of kv_dtype: 0 fp32, 1 bf16, 2 fp8 E4M3 (values as for
 *     ck_attn_decode_gqa_bf16 / _fp8; k_scale / v_scale used for fp8 only);
 *   block_tables: device int32 [batch, max_blocks_per_seq]: logical block i
 *     of sequence b (its rows i*block_size ..) is physical block
 *     block_tables[b][i];
 *   seq_lens: device int32 [batch]: rows of sequence b, T_b;
 *   q, out: fp32 [batch, num_heads * head_dim].
 * Sequence b attends rows [T0, T_b) with T0 = max(0, T_b - sliding_window)
 * when sliding_window > 0, else 0; out_b = the attention of
 * ck_attn_decode_gqa over those rows.  On the device, T_b outside
 * [0, max_blocks_per_seq * block_size] or a table entry outside
 * [0, num_blocks) raises CK_ERANGE in the status word (the rows concerned are
 * not read; a sequence with no rows attended gets zeros).
 * Requirements: those of ck_attn_decode_gqa (bf16 / fp8: head_dim 64 or
 * 128), 1 <= batch <= 1024, block_size >= 1, max_blocks_per_seq >= 1,
 * num_blocks >= 1, sliding_window >= 0, every pointer 16-byte aligned.
 * `scratch` >= ck_attn_paged_scratch_size(...) bytes with the same batch,
 * heads, head_dim, block_size, max_blocks_per_seq and sliding_window. */
size_t ck_attn_paged_scratch_size(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int sliding_window);
int ck_attn_decode_gqa_paged(const float *q, const void *k_pool, const void *v_pool, float *out,
                             const int32_t *block_tables, const int32_t *seq_lens, int batch, int num_heads,
                             int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                             int sliding_window, int kv_dtype, float k_scale, float v_scale, void *scratch,
                             size_t scratch_bytes, void *stream);

/* ---- the whole layer step ---------------------------------------------- */

/* mega_fused_attention_decode_q5_0 (page: MAIN KERNEL).  One token at
 * position `pos`:
 *   out = residual + bo + Wo . q8(attention(rope(Wq.q8(rms(x))+bq),
 *                                          cache with k, v stored at pos))
 * x, residual, out: fp32 [embed_dim] (residual may alias x; out may not
 * alias x, residual, weights, caches or scratch);
 * wq: Q5_0 [num_heads*head_dim, embed_dim]; wk: Q5_0 [num_kv_heads*head_dim,
 * embed_dim]; wv: Q8_0 [num_kv_heads*head_dim, embed_dim]; wo: Q5_0
 * [embed_dim, num_heads*head_dim]; gamma: fp32 [embed_dim]; bq, bk, bv, bo:
 * fp32 biases of the matching lengths, each may be NULL (= zero);
 * k_cache, v_cache: the head-major caches, row `pos` is overwritten and rows
 * 0..pos are attended; rope_cos / rope_sin: tables as above; eps: RMSNorm
 * epsilon.  Requirements: embed_dim % 32 == 0, the attention requirements
 * above, 0 <= pos < cache_capacity.
 * `scratch`: >= ck_decode_layer_scratch_size(...) bytes of device memory
 * (contents need no initialization).  The size depends on the current
 * device (its SM count). */
size_t ck_decode_layer_scratch_size(int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                    int cache_capacity);
int ck_decode_layer(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                    const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                    const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                    const float *rope_sin, int pos, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                    int cache_capacity, float eps, void *scratch, size_t scratch_bytes, void *stream);

/* The same step with the position read on the device from *d_pos (int32,
 * device memory), so that a captured CUDA graph can be replayed for
 * successive tokens by updating *d_pos alone.  The host cannot see the
 * position: the kernels check 0 <= *d_pos < cache_capacity themselves and,
 * when it fails, skip all work (nothing is written) and raise CK_ERANGE in
 * the device status word (see ck_device_status). */
int ck_decode_layer_devpos(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                           const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                           const float *bv, const float *bo, float *k_cache, float *v_cache,
                           const float *rope_cos, const float *rope_sin, const int32_t *d_pos, int embed_dim,
                           int num_heads, int num_kv_heads, int head_dim, int cache_capacity, float eps,
                           void *scratch, size_t scratch_bytes, void *stream);

/* Errors that only the device can see -- a device-side position out of
 * range (CK_ERANGE) or a bounded wait inside a kernel that expired
 * (CK_ETIMEOUT) -- are OR-ed into one status word per device.  This call
 * stores the most severe of them since the last call (CK_OK if none) in
 * *status (host pointer) and clears the word.  It synchronizes `stream`:
 * call it outside stream capture. */
int ck_device_status(int *status, void *stream);

/* Byte offset, inside a layer scratch buffer laid out for these shapes, of
 * one intermediate that the last ck_decode_layer* call left there (valid
 * until the next call on the same scratch):
 *   CK_TAP_Q    fp32 [num_heads*head_dim]   q after bias and RoPE
 *   CK_TAP_XQ8  Q8_0 [embed_dim/32]         the quantized normed input
 *   CK_TAP_ATTN fp32 [num_heads*head_dim]   the attention output
 *   CK_TAP_AQ8  Q8_0 [num_heads*head_dim/32] its quantization (O-proj input)
 * Returns (size_t)-1 for an unknown tap or invalid shapes. */
#define CK_TAP_Q 0
#define CK_TAP_XQ8 1
#define CK_TAP_ATTN 2
#define CK_TAP_AQ8 3
size_t ck_decode_layer_scratch_offset(int tap, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                      int cache_capacity);

/* ---- a batch of sequences sharing the layer ----------------------------- */

/* The decode step of the MAIN KERNEL for `batch` sequences that share the
 * layer's weights, each with its own KV cache and position (the same result,
 * sequence by sequence, as ck_decode_layer_devpos on that sequence; the
 * weights are read once for the whole batch).
 * out, x, residual: fp32 [batch, embed_dim] (device; out must not alias x or
 * residual).  Weights, biases, gamma, rope tables and eps as for
 * ck_decode_layer.  k_caches, v_caches: device arrays of `batch` pointers,
 * each to a head-major fp32 cache [num_kv_heads, cache_capacity, head_dim]
 * (16-byte aligned; the arrays and the caches are read on the device and not
 * validated by the host).  d_pos: int32 [batch] (device): sequence s writes
 * row d_pos[s] of its caches and attends rows 0..d_pos[s]; a sequence whose
 * position is outside 0..cache_capacity-1 writes nothing and raises CK_ERANGE
 * in the device status word.  Requirements: 1 <= batch <= 1024, embed_dim and
 * num_heads*head_dim multiples of 256 up to 4096, and the attention
 * requirements; otherwise CK_EINVAL.
 * `scratch`: >= ck_decode_layer_batched_scratch_size(...) bytes of device
 * memory (contents need no initialization; the size depends on the device). */
size_t ck_decode_layer_batched_scratch_size(int batch, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                            int cache_capacity);
int ck_decode_layer_batched(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                            const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                            const float *bv, const float *bo, float *const *k_caches, float *const *v_caches,
                            const float *rope_cos, const float *rope_sin, const int32_t *d_pos, int batch,
                            int embed_dim, int num_heads, int num_kv_heads, int head_dim, int cache_capacity,
                            float eps, void *scratch, size_t scratch_bytes, void *stream);
/* Byte offset of a tap (CK_TAP_*) in a batched scratch buffer: the taps hold
 * `batch` rows of the single-sequence layout, row s after row s-1. */
size_t ck_decode_layer_batched_scratch_offset(int tap, int batch, int embed_dim, int num_heads, int num_kv_heads,
                                              int head_dim, int cache_capacity);

/* ---- the multi-token (prefill) form of the layer ------------------------ */

/* Page "prefill_attn_a.rs" (layers/ops): the prefill attention launcher,
 * one query per (head, token) with a causal switch.  Read here as the same
 * layer applied to `n_tokens` consecutive tokens of ONE sequence: token i sits
 * at position pos + i, its K / V rows are stored at row pos + i, and it
 * attends cache rows 0 .. pos + i (the rows already in the cache and the
 * chunk's own rows up to and including its own).  The result equals
 * n_tokens calls of ck_decode_layer at positions pos, pos + 1, ... in order
 * (head_dim 128: the attention as ck_attn_prefill_gqa, on the tensor cores;
 * otherwise one decode attention per token).
 * out, x, residual: fp32 [n_tokens, embed_dim] (device; out must not alias x
 * or residual; residual may alias x).  k_cache, v_cache: head-major fp32
 * [num_kv_heads, cache_capacity, head_dim] (device, 16-byte aligned, else
 * CK_EALIGN); rows pos .. pos + n_tokens - 1 are written.  Weights, biases,
 * gamma, rope tables and eps as for ck_decode_layer.  Requirements: 1 <=
 * n_tokens <= 1024 and the shape requirements of ck_decode_layer_batched,
 * otherwise CK_EINVAL; pos >= 0 and pos + n_tokens <= cache_capacity,
 * otherwise CK_ERANGE (checked on the host, nothing launched).
 * `scratch`: >= ck_prefill_layer_scratch_size(...) bytes of device memory
 * (no initialization needed); the taps (CK_TAP_*) sit at
 * ck_prefill_layer_scratch_offset(...), row i for token i. */
/* The chunk's attention alone (the prefill attention launcher of the same
 * page: queries of every (token, head), causal), on the tensor cores.
 * q, out: fp32 [n_tokens, num_heads * head_dim] (device, 16-byte aligned);
 * token i (position pos + i) attends rows 0 .. pos + i of the head-major fp32
 * caches [num_kv_heads, cache_capacity, head_dim], whose rows pos ..
 * pos + n_tokens - 1 must already hold the chunk's K / V.  The result equals
 * ck_attn_decode_gqa over pos + i + 1 rows for every token.  Operands are
 * taken as bf16 pairs (hi + lo, about 17 significant bits) with fp32
 * accumulation: a relative error near 1e-5 where the fp32 kernels reach 1e-7.
 * Requirements: head_dim 128, num_heads a multiple of num_kv_heads with
 * num_heads / num_kv_heads <= 16, 1 <= n_tokens
 * <= 2^20 (else CK_EINVAL), 0 <= pos <= cache_capacity - n_tokens (else
 * CK_ERANGE).  `scratch`: >= ck_attn_prefill_scratch_size(...) bytes (0 for
 * unsupported shapes). */
size_t ck_attn_prefill_scratch_size(int num_heads, int num_kv_heads, int head_dim, int cache_capacity);
int ck_attn_prefill_gqa(const float *q, const float *k_cache, const float *v_cache, float *out, int pos,
                        int n_tokens, int num_heads, int num_kv_heads, int head_dim, int cache_capacity,
                        void *scratch, size_t scratch_bytes, void *stream);
size_t ck_prefill_layer_scratch_size(int n_tokens, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                     int cache_capacity);
size_t ck_prefill_layer_scratch_offset(int tap, int n_tokens, int embed_dim, int num_heads, int num_kv_heads,
                                       int head_dim, int cache_capacity);
int ck_prefill_layer(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                     const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                     const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                     const float *rope_sin, int pos, int n_tokens, int embed_dim, int num_heads, int num_kv_heads,
                     int head_dim, int cache_capacity, float eps, void *scratch, size_t scratch_bytes, void *stream);
/* The same with the chunk's first position read on the device from d_pos
 * (int32, device memory set before the call's first kernel), for replaying a
 * captured graph as the chunk moves.  A chunk that does not fit the cache
 * (*d_pos < 0 or *d_pos + n_tokens > cache_capacity) writes nothing (no
 * cache row, no output) and raises CK_ERANGE in the device status word
 * (ck_device_status).  d_pos null: CK_EINVAL. */
int ck_prefill_layer_devpos(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                            const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                            const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                            const float *rope_sin, const int32_t *d_pos, int n_tokens, int embed_dim, int num_heads,
                            int num_kv_heads, int head_dim, int cache_capacity, float eps, void *scratch,
                            size_t scratch_bytes, void *stream);

/* ---- test access to the integer block dots ----------------------------- */

/* The per-block int32 dots that the GEMVs above compute, with the same
 * device code: isum[r*(K/32) + b] = sum_j code_w(r,b,j) * code_x(b,j)
 * (Q5_0 codes offset by -16).  isum: int32 [M, K/32] (device). */
int ck_block_dots_q5_0_q8_0(int32_t *isum, const void *W, const void *x_q8, int M, int K, void *stream);
int ck_block_dots_q8_0_q8_0(int32_t *isum, const void *W, const void *x_q8, int M, int K, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CK_DECODE_H */
