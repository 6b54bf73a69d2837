// Host-side interfaces between the translation units of libck_decode.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ck {

// Per-device facts the launch planner needs (cached per device ordinal).
struct DeviceInfo {
    int device;
    int num_sms;
    size_t smem_optin;  // max dynamic shared memory per block (opt-in)
};
const DeviceInfo &device_info();

// Address of the library's device status word on the current device.
unsigned *status_word();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device (a runtime call only the first time a larger value is needed).
void ensure_smem(const void *fn, size_t bytes);

// Launch helper: optional programmatic-dependent-launch attribute.
cudaError_t launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void **args);

// ---- gemv / quantize (ck_gemv.cu) ----
int launch_quantize_q8_0(const float *x, void *y, int n, cudaStream_t s);
int launch_gemv(bool q8, float *y, const void *W, const void *xq8, const float *bias, int M, int K, cudaStream_t s);
int launch_block_dots(bool q8, int32_t *isum, const void *W, const void *xq8, int M, int K, cudaStream_t s);

// The layer's projection kernels.
struct QkvArgs {
    const float *x, *gamma;
    const uint8_t *wq, *wk, *wv;
    const float *bq, *bk, *bv;
    float *k_cache, *v_cache;
    const float *rope_cos, *rope_sin;
    float *q_out;        // [H*hd] rotated q
    uint8_t *xq8;        // [D/32] Q8_0 blocks of the normed input (written by K0, read by K1)
    const int32_t *d_pos;  // device position (or null: use pos)
    int pos;
    int D, H, KV, hd, C;
    float eps;
    int n_q_tiles, n_k_tiles, rv;  // Q / K tiles of 16 RoPE pairs, V tiles of rv rows
    int fused_norm;  // 1: the projection CTAs normalize and quantize x themselves (no K0)
    unsigned *status;
};
struct OprojArgs {
    float *out;
    const float *residual;
    const uint8_t *wo;
    const float *bo;
    const uint8_t *aq8;    // [H*hd/32] Q8_0 blocks of the attention output
    const uint8_t *apack;  // the same row packed (xpack_bytes), or null: unpack aq8
    const int32_t *d_pos;
    int D, QD, rows_per_cta, C;
    unsigned *status;
};
int launch_norm_q8(const QkvArgs &a, cudaStream_t s, bool pdl);
int launch_qkv(const QkvArgs &a, cudaStream_t s, bool pdl);
// Whether launch_qkv's CTAs can normalize and quantize x themselves.
bool qkv_fused_norm_ok(const QkvArgs &a);
int launch_oproj(const OprojArgs &a, cudaStream_t s, bool pdl);

// The batched step (ck_batched.cu).
struct BatchArgs {
    int B;
    const float *x, *residual, *gamma;
    const uint8_t *wq, *wk, *wv, *wo;
    const float *bq, *bk, *bv, *bo;
    float *const *k_caches, *const *v_caches;  // device arrays [B]
    const float *rope_cos, *rope_sin;
    const int32_t *d_pos;  // device [B]
    int D, H, KV, hd, C;
    float eps;
    float *out;      // [B][D]
    float *q;        // [B][H*hd]
    uint8_t *xq8;    // [B][D/32] Q8_0 blocks of the normed inputs
    uint8_t *xpack;  // [B] packed rows of the normed inputs
    uint8_t *apack;  // [B] packed rows of the attention outputs
    uint8_t *aq8;    // [B][H*hd/32] Q8_0 blocks of the attention outputs
    uint8_t *ximg;   // tensor-core operand image of the normed inputs (img_bytes(D/32, B)), or null
    uint8_t *aimg;   // the same for the attention outputs (img_bytes(H*hd/32, B))
    float *proj_part;  // tensor-core projections: partial tiles of the K splits
    int *tickets;      // per tile: K splits finished (QKV tiles, then O tiles from tickets_o)
    int tickets_o, n_tickets;
    unsigned *status;
};
bool batched_shape_ok(int D, int H, int hd);
// Tensor-core projections (ck_batched_tc.cu): shapes they take, their plan
// (K splits of the QKV and O launches, scratch of the partial tiles, tile
// tickets) and launch.  Without the device the splits are 1 and only the
// sizes, which do not depend on it, are meaningful.
bool batched_tc_ok(int D, int H, int KV, int hd);
struct TpPlan {
    int splits[2];
    size_t part_bytes;
    int tickets_o, tickets;
};
TpPlan tp_plan(int B, int D, int H, int KV, int hd, bool with_device);
int launch_rows_tc(const BatchArgs &a, bool oproj, cudaStream_t s, bool pdl);
int launch_norm_pack(const BatchArgs &a, cudaStream_t s, bool pdl);
// Per-token cache pointers and positions of a prefill chunk (token i at
// pos + i, pos read from d_pos when it is not null); a chunk that does not
// fit the cache gets every position at C (each kernel then skips the token)
// and raises CK_ERANGE in the status word.
int launch_prefill_setup(float **kcs, float **vcs, int32_t *pos_of, float *k_cache, float *v_cache, int pos,
                         const int32_t *d_pos, int n, int C, unsigned *status, cudaStream_t s);
int launch_rows_batched(const BatchArgs &a, bool oproj, cudaStream_t s, bool pdl);
void plan_qkv(QkvArgs &a);

// ---- attention (ck_attn.cu) ----
// Cache element types: fp32 (the layer's cache), bf16, fp8 E4M3 (with
// per-tensor scales).
constexpr int KV_F32 = 0, KV_BF16 = 1, KV_FP8 = 2;
struct AttnArgs {
    const float *q;           // [B][H*hd]
    const float *k_cache;     // single sequence: the cache; batched: unused
    const float *v_cache;
    const float *const *k_caches;  // batched: device array of B cache pointers
    const float *const *v_caches;
    const int32_t *d_pos;     // device positions [B] (T = pos + 1) or null
    int kv_tokens;            // used when d_pos is null (B == 1)
    int H, KV, hd, C;
    int splits;               // S
    int chunk;                // rows per split (0: ceil(T / S))
    float *part;              // scratch: partial results
    float *out;               // [B][H*hd] fp32 attention output
    uint8_t *out_q8;          // [B][H*hd/32] Q8_0 blocks, or null
    uint8_t *out_pack;        // [B] packed rows of those blocks (xpack_bytes each), or null
    uint8_t *out_img;         // tensor-core operand image of those blocks (img_* layout), or null
    int img_groups;           // its sequence groups: img_groups(B)
    const void *l2_prefetch;  // optional: bytes the next kernel reads, pulled into L2
    size_t l2_prefetch_bytes;
    int kv_type;              // cache elements: 0 fp32, 1 bf16, 2 fp8 E4M3 (k_cache / v_cache hold them)
    float k_scale, v_scale;   // fp8: k = code * k_scale, v = code * v_scale
    // paged caches (block_tables non-null): k_cache / v_cache are pools
    // [num_blocks][KV][block_size][hd]; sequence b attends rows [T0, T) with
    // T = seq_lens[b], T0 = max(0, T - window) when window > 0; its logical
    // block i is physical block block_tables[b * max_blocks + i]
    const int32_t *block_tables, *seq_lens;
    int block_size, max_blocks, num_blocks, window;
    // cache rows the preceding grid may have written: row T - 1 alone when
    // fresh_chunk is 0; rows fresh_from .. T - 1 otherwise (a prefill chunk)
    int fresh_chunk, fresh_from;
    unsigned *status;
};
size_t attn_part_bytes(int B, int H, int KV, int hd, int splits);
int attn_splits(int B, int KV, int max_tokens);
int attn_splits_batched(int B, int KV, int max_tokens);
int launch_attention(const AttnArgs &a, int B, cudaStream_t s, bool pdl_first, bool pdl_combine);
// bf16 / fp8 caches at head_dim 128, query groups up to 8: the split kernel
// with its scores on the tensor cores (same records, same combine).
bool attention_tc_ok(int kv_type, int H, int KV, int hd);
int launch_attention_tc(const AttnArgs &a, int B, cudaStream_t s, bool pdl_first, bool pdl_combine);
// Prefill attention on the tensor cores (head_dim 128, query groups up to 16):
// the chunk's rows of KV head g against cache rows 0 .. pos + n - 1, causal;
// outputs through the decode attention's store (o.out, o.out_q8, o.out_img,
// o.out_pack).  img: prefill_img_bytes(KV, C) bytes of scratch.
bool prefill_tc_ok(int H, int KV, int hd);
size_t prefill_img_bytes(int KV, int C);
int launch_prefill_attn(const AttnArgs &o, const float *q, const float *k_cache, const float *v_cache, uint8_t *img,
                        int n, int pos, const int32_t *d_pos, int H, int KV, int C, cudaStream_t s);
int launch_rope(float *q, float *k, const float *c, const float *sn, int pos, int H, int KV, int hd, cudaStream_t s);
int launch_kv_store(float *kc, float *vc, const float *k, const float *v, int pos, int KV, int C, int hd,
                    cudaStream_t s);
// The same into a bf16 cache (round to nearest even) or an fp8 E4M3 cache
// (code = E4M3(x / scale), round to nearest even, saturated to +-448).
int launch_kv_store_q(void *kc, void *vc, const float *k, const float *v, int pos, int KV, int C, int hd,
                      int kv_type, float k_scale, float v_scale, cudaStream_t s);

}  // namespace ck
