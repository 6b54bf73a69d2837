// C ABI of libck_decode (declared in include/ck_decode.h): argument
// validation on the host, launch planning, and the composition of the
// decode step of the page "mega_fused_attention_decode_q5_0.c" as five
// kernels on one stream:
//
//   k_norm_q8      RMSNorm + Q8_0 quantization of the input (one CTA) STEP 1-2
//   k_qkv_w        Q|K|V GEMV, bias, RoPE, KV-cache store, q         STEP 2-6
//   k_attn_split   split-KV GQA-packed flash decoding                STEP 7
//   k_attn_combine LSE merge + Q8_0 quant of the attention output    STEP 7-8
//   k_oproj        O GEMV + bias + residual                          STEP 8
//
// Each kernel after the first is launched with programmatic dependent
// launch: it starts while its predecessor drains, streams the operands that
// do not depend on it (weights, cache rows before `pos`), then waits.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>

#include "../../include/ck_decode.h"
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

__device__ unsigned g_status_word;

static std::mutex g_mu;

const DeviceInfo &device_info() {
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!have[dev]) {
        DeviceInfo d{};
        d.device = dev;
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        d.smem_optin = static_cast<size_t>(optin);
        if (d.num_sms <= 0) d.num_sms = 1;
        cache[dev] = d;
        have[dev] = true;
    }
    return cache[dev];
}

unsigned *status_word() {
    static unsigned *cache[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned *>(p);
    }
    return cache[dev];
}

void ensure_smem(const void *fn, size_t bytes) {
    static std::map<std::pair<const void *, int>, size_t> done;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(g_mu);
    size_t &have = done[{fn, dev}];
    if (have >= bytes && have != 0) return;
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    have = bytes;
}

cudaError_t launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void **args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ck

using namespace ck;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_ptrs(std::initializer_list<const void *> required, std::initializer_list<const void *> optional) {
    for (const void *p : required) {
        if (!p) return CK_EINVAL;
        if (!aligned16(p)) return CK_EALIGN;
    }
    for (const void *p : optional)
        if (p && !aligned16(p)) return CK_EALIGN;
    return CK_OK;
}

int attn_shape_ok(int H, int KV, int hd) {
    if (H <= 0 || KV <= 0 || H % KV != 0) return CK_EINVAL;
    if (H / KV > 8) return CK_EINVAL;
    if (hd % 32 != 0 || hd < 32 || hd > 256) return CK_EINVAL;
    const int dpl = hd / 32;
    if (dpl != 1 && dpl != 2 && dpl != 3 && dpl != 4 && dpl != 8) return CK_EINVAL;
    return CK_OK;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Layout of the layer scratch (all offsets 256-byte aligned).
struct LayerScratch {
    size_t off_q, off_xq8, off_attn, off_aq8, off_apack, off_part, total;
    int splits;
};

size_t a256(size_t v) { return (v + 255) / 256 * 256; }

LayerScratch layer_scratch(int D, int H, int KV, int hd, int C) {
    LayerScratch L{};
    L.splits = attn_splits(1, KV, C);
    size_t o = 0;
    L.off_q = o;
    o = a256(o + static_cast<size_t>(H) * hd * 4);
    L.off_xq8 = o;
    o = a256(o + static_cast<size_t>(D / 32) * 34);
    L.off_attn = o;
    o = a256(o + static_cast<size_t>(H) * hd * 4);
    L.off_aq8 = o;
    o = a256(o + static_cast<size_t>(H * hd / 32) * 34);
    L.off_apack = o;
    o = a256(o + xpack_bytes(H * hd / 32));
    L.off_part = o;
    o = a256(o + attn_part_bytes(1, H, KV, hd, L.splits));
    L.total = o;
    return L;
}

struct BatchScratch {
    size_t off_q, off_xq8, off_attn, off_aq8, off_xpack, off_apack, off_part, off_ximg, off_aimg, off_ppart,
        off_tickets, total;
    int splits;
    TpPlan tp;
};

BatchScratch batch_scratch(int B, int D, int H, int KV, int hd, int C) {
    BatchScratch L{};
    L.splits = attn_splits_batched(B, KV, C);
    const size_t nb = static_cast<size_t>(D / 32), nbo = static_cast<size_t>(H * hd / 32);
    size_t o = 0;
    L.off_q = o;
    o = a256(o + static_cast<size_t>(B) * H * hd * 4);
    L.off_xq8 = o;
    o = a256(o + static_cast<size_t>(B) * nb * 34);
    L.off_attn = o;
    o = a256(o + static_cast<size_t>(B) * H * hd * 4);
    L.off_aq8 = o;
    o = a256(o + static_cast<size_t>(B) * nbo * 34);
    L.off_xpack = o;
    o = a256(o + static_cast<size_t>(B) * xpack_bytes(static_cast<int>(nb)));
    L.off_apack = o;
    o = a256(o + static_cast<size_t>(B) * xpack_bytes(static_cast<int>(nbo)));
    L.off_part = o;
    o = a256(o + attn_part_bytes(B, H, KV, hd, L.splits));
    // tensor-core projections: operand images, partial tiles, tile tickets
    L.tp = tp_plan(B, D, H, KV, hd, false);
    L.off_ximg = o;
    o = a256(o + img_bytes(static_cast<int>(nb), B));
    L.off_aimg = o;
    o = a256(o + img_bytes(static_cast<int>(nbo), B));
    L.off_ppart = o;
    o = a256(o + L.tp.part_bytes);
    L.off_tickets = o;
    o = a256(o + static_cast<size_t>(L.tp.tickets) * 4);
    L.total = o;
    return L;
}

int batch_shape_check(int B, int D, int H, int KV, int hd, int C) {
    if (B < 1 || B > 1024 || D <= 0 || C <= 0) return CK_EINVAL;
    int rc = attn_shape_ok(H, KV, hd);
    if (rc) return rc;
    return batched_shape_ok(D, H, hd) ? CK_OK : CK_EINVAL;
}

int layer_common(float *out, const float *x, const float *residual, const void *wq, const void *wk, const void *wv,
                 const void *wo, const float *gamma, const float *bq, const float *bk, const float *bv,
                 const float *bo, float *k_cache, float *v_cache, const float *rope_cos, const float *rope_sin,
                 int pos, const int32_t *d_pos, int D, int H, int KV, int hd, int C, float eps, void *scratch,
                 size_t scratch_bytes, void *stream) {
    int rc = check_ptrs({out, x, residual, wq, wk, wv, wo, gamma, k_cache, v_cache, rope_cos, rope_sin},
                        {bq, bk, bv, bo, d_pos});
    if (rc) return rc;
    if (D <= 0 || D % 32 != 0 || C <= 0) return CK_EINVAL;
    if ((rc = attn_shape_ok(H, KV, hd))) return rc;
    if (!d_pos && (pos < 0 || pos >= C)) return CK_ERANGE;
    if (!scratch) return CK_ESCRATCH;
    if (!aligned16(scratch)) return CK_EALIGN;
    const LayerScratch L = layer_scratch(D, H, KV, hd, C);
    if (scratch_bytes < L.total) return CK_ESCRATCH;
    if (out == x || out == residual) return CK_EINVAL;
    uint8_t *sc = static_cast<uint8_t *>(scratch);
    cudaStream_t s = as_stream(stream);
    unsigned *st = status_word();
    if (!st) return CK_ECUDA;

    QkvArgs qa{};
    qa.x = x;
    qa.gamma = gamma;
    qa.wq = static_cast<const uint8_t *>(wq);
    qa.wk = static_cast<const uint8_t *>(wk);
    qa.wv = static_cast<const uint8_t *>(wv);
    qa.bq = bq;
    qa.bk = bk;
    qa.bv = bv;
    qa.k_cache = k_cache;
    qa.v_cache = v_cache;
    qa.rope_cos = rope_cos;
    qa.rope_sin = rope_sin;
    qa.q_out = reinterpret_cast<float *>(sc + L.off_q);
    qa.xq8 = sc + L.off_xq8;
    qa.d_pos = d_pos;
    qa.pos = pos;
    qa.D = D;
    qa.H = H;
    qa.KV = KV;
    qa.hd = hd;
    qa.C = C;
    qa.eps = eps;
    qa.status = st;
    qa.fused_norm = qkv_fused_norm_ok(qa) ? 1 : 0;
    if (!qa.fused_norm && (rc = launch_norm_q8(qa, s, true))) return rc == -1 ? CK_EINVAL : CK_ECUDA;
    if ((rc = launch_qkv(qa, s, true))) return rc == -1 ? CK_EINVAL : CK_ECUDA;

    AttnArgs aa{};
    aa.q = qa.q_out;
    aa.k_cache = k_cache;
    aa.v_cache = v_cache;
    aa.d_pos = d_pos;
    aa.kv_tokens = pos + 1;
    aa.H = H;
    aa.KV = KV;
    aa.hd = hd;
    aa.C = C;
    aa.splits = L.splits;
    aa.part = reinterpret_cast<float *>(sc + L.off_part);
    aa.out = reinterpret_cast<float *>(sc + L.off_attn);
    aa.out_q8 = sc + L.off_aq8;
    aa.out_pack = sc + L.off_apack;
    aa.l2_prefetch = wo;
    aa.l2_prefetch_bytes = static_cast<size_t>(D) * (H * hd / 32) * 22;
    aa.status = st;
    if (launch_attention(aa, 1, s, true, true)) return CK_ECUDA;

    OprojArgs oa{};
    oa.out = out;
    oa.residual = residual;
    oa.wo = static_cast<const uint8_t *>(wo);
    oa.bo = bo;
    oa.aq8 = sc + L.off_aq8;
    oa.apack = sc + L.off_apack;
    oa.d_pos = d_pos;
    oa.D = D;
    oa.QD = H * hd;
    oa.C = C;
    oa.status = st;
    if (launch_oproj(oa, s, true)) return CK_ECUDA;
    return CK_OK;
}

}  // namespace

extern "C" {

const char *ck_status_string(int status) {
    switch (status) {
        case CK_OK: return "CK_OK";
        case CK_EINVAL: return "CK_EINVAL: null pointer or invalid size";
        case CK_ERANGE: return "CK_ERANGE: position or token count outside the cache";
        case CK_ESCRATCH: return "CK_ESCRATCH: scratch missing or too small";
        case CK_EALIGN: return "CK_EALIGN: pointer not 16-byte aligned";
        case CK_ECUDA: return "CK_ECUDA: CUDA launch or runtime error";
        case CK_ETIMEOUT: return "CK_ETIMEOUT: a bounded device wait expired";
        default: return "unknown status";
    }
}

int ck_quantize_q8_0(const float *x, void *y_q8, int n, void *stream) {
    int rc = check_ptrs({x, y_q8}, {});
    if (rc) return rc;
    if (n <= 0 || n % 32 != 0) return CK_EINVAL;
    return launch_quantize_q8_0(x, y_q8, n, as_stream(stream)) ? CK_ECUDA : CK_OK;
}

static int gemv_common(bool q8, float *y, const void *W, const void *x_q8, const float *bias, int M, int K,
                       void *stream) {
    int rc = check_ptrs({y, W, x_q8}, {bias});
    if (rc) return rc;
    if (M <= 0 || K <= 0 || K % 32 != 0) return CK_EINVAL;
    if (!status_word()) return CK_ECUDA;
    return launch_gemv(q8, y, W, x_q8, bias, M, K, as_stream(stream)) ? CK_ECUDA : CK_OK;
}

int ck_gemv_q5_0_q8_0(float *y, const void *W, const void *x_q8, const float *bias, int M, int K, void *stream) {
    return gemv_common(false, y, W, x_q8, bias, M, K, stream);
}

int ck_gemv_q8_0_q8_0(float *y, const void *W, const void *x_q8, const float *bias, int M, int K, void *stream) {
    return gemv_common(true, y, W, x_q8, bias, M, K, stream);
}

int ck_rope_inplace(float *q, float *k, const float *rope_cos, const float *rope_sin, int pos, int num_heads,
                    int num_kv_heads, int head_dim, int cache_capacity, void *stream) {
    if (num_heads < 0 || num_kv_heads < 0 || head_dim <= 0 || head_dim % 2 != 0 || cache_capacity <= 0)
        return CK_EINVAL;
    if ((num_heads > 0 && !q) || (num_kv_heads > 0 && !k)) return CK_EINVAL;
    int rc = check_ptrs({rope_cos, rope_sin}, {q, k});
    if (rc) return rc;
    if (pos < 0 || pos >= cache_capacity) return CK_ERANGE;
    return launch_rope(q, k, rope_cos, rope_sin, pos, num_heads, num_kv_heads, head_dim, as_stream(stream))
               ? CK_ECUDA
               : CK_OK;
}

int ck_kv_store(float *k_cache, float *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                int cache_capacity, int head_dim, void *stream) {
    int rc = check_ptrs({k_cache, v_cache, k, v}, {});
    if (rc) return rc;
    if (num_kv_heads <= 0 || head_dim <= 0 || cache_capacity <= 0) return CK_EINVAL;
    if (pos < 0 || pos >= cache_capacity) return CK_ERANGE;
    return launch_kv_store(k_cache, v_cache, k, v, pos, num_kv_heads, cache_capacity, head_dim, as_stream(stream))
               ? CK_ECUDA
               : CK_OK;
}

size_t ck_attn_scratch_size(int num_heads, int num_kv_heads, int max_kv_tokens, int head_dim) {
    if (attn_shape_ok(num_heads, num_kv_heads, head_dim) || max_kv_tokens <= 0) return 0;
    const int S = attn_splits(1, num_kv_heads, max_kv_tokens);
    return attn_part_bytes(1, num_heads, num_kv_heads, head_dim, S) + 256;
}

static int attn_call(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                     int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, int kv_type, float k_scale,
                     float v_scale, void *scratch, size_t scratch_bytes, void *stream, int splits = 0);

int ck_attn_decode_gqa(const float *q, const float *k_cache, const float *v_cache, float *out, int num_heads,
                       int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, void *scratch,
                       size_t scratch_bytes, void *stream) {
    return attn_call(q, k_cache, v_cache, out, num_heads, num_kv_heads, kv_tokens, cache_capacity, head_dim, 0,
                     1.0f, 1.0f, scratch, scratch_bytes, stream);
}

static bool scale_ok(float s) { return std::isfinite(s) && s > 0.0f; }

int ck_attn_decode_gqa_bf16(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                            int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, void *scratch,
                            size_t scratch_bytes, void *stream) {
    return attn_call(q, k_cache, v_cache, out, num_heads, num_kv_heads, kv_tokens, cache_capacity, head_dim,
                     KV_BF16, 1.0f, 1.0f, scratch, scratch_bytes, stream);
}

int ck_attn_decode_gqa_fp8(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                           int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, float k_scale,
                           float v_scale, void *scratch, size_t scratch_bytes, void *stream) {
    if (!scale_ok(k_scale) || !scale_ok(v_scale)) return CK_EINVAL;
    return attn_call(q, k_cache, v_cache, out, num_heads, num_kv_heads, kv_tokens, cache_capacity, head_dim, KV_FP8,
                     k_scale, v_scale, scratch, scratch_bytes, stream);
}

size_t ck_attn_split_scratch_size(int num_heads, int num_kv_heads, int head_dim, int splits) {
    if (attn_shape_ok(num_heads, num_kv_heads, head_dim) || splits < 1 || splits > 1024) return 0;
    return attn_part_bytes(1, num_heads, num_kv_heads, head_dim, splits) + 256;
}

int ck_attn_decode_gqa_split(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                             int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, int kv_dtype,
                             float k_scale, float v_scale, int splits, void *scratch, size_t scratch_bytes,
                             void *stream) {
    if (splits < 0 || splits > 1024 || kv_dtype < 0 || kv_dtype > 2) return CK_EINVAL;
    if (kv_dtype == KV_FP8 && (!scale_ok(k_scale) || !scale_ok(v_scale))) return CK_EINVAL;
    if (kv_dtype != KV_FP8) k_scale = v_scale = 1.0f;
    return attn_call(q, k_cache, v_cache, out, num_heads, num_kv_heads, kv_tokens, cache_capacity, head_dim, kv_dtype,
                     k_scale, v_scale, scratch, scratch_bytes, stream, splits);
}

static int kv_store_q(void *k_cache, void *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                      int cache_capacity, int head_dim, int kv_type, float k_scale, float v_scale, void *stream) {
    int rc = check_ptrs({k_cache, v_cache, k, v}, {});
    if (rc) return rc;
    if (num_kv_heads <= 0 || head_dim <= 0 || cache_capacity <= 0) return CK_EINVAL;
    if (pos < 0 || pos >= cache_capacity) return CK_ERANGE;
    return launch_kv_store_q(k_cache, v_cache, k, v, pos, num_kv_heads, cache_capacity, head_dim, kv_type, k_scale,
                             v_scale, as_stream(stream))
               ? CK_ECUDA
               : CK_OK;
}

int ck_kv_store_bf16(void *k_cache, void *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                     int cache_capacity, int head_dim, void *stream) {
    return kv_store_q(k_cache, v_cache, k, v, pos, num_kv_heads, cache_capacity, head_dim, KV_BF16, 1.0f, 1.0f,
                      stream);
}

int ck_kv_store_fp8(void *k_cache, void *v_cache, const float *k, const float *v, int pos, int num_kv_heads,
                    int cache_capacity, int head_dim, float k_scale, float v_scale, void *stream) {
    if (!scale_ok(k_scale) || !scale_ok(v_scale)) return CK_EINVAL;
    return kv_store_q(k_cache, v_cache, k, v, pos, num_kv_heads, cache_capacity, head_dim, KV_FP8, k_scale, v_scale,
                      stream);
}

// Paged attention: the rows a split plans for (the longest sequence the
// tables can hold, or the window).
static int paged_rows(int block_size, int max_blocks, int window) {
    const long long cap = static_cast<long long>(block_size) * max_blocks;
    const long long r = window > 0 && window < cap ? window : cap;
    return r > (1 << 30) ? (1 << 30) : static_cast<int>(r);
}

size_t ck_attn_paged_scratch_size(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int sliding_window) {
    if (batch < 1 || batch > 1024 || block_size < 1 || max_blocks_per_seq < 1 || sliding_window < 0) return 0;
    if (attn_shape_ok(num_heads, num_kv_heads, head_dim)) return 0;
    const int S = attn_splits_batched(batch, num_kv_heads, paged_rows(block_size, max_blocks_per_seq, sliding_window));
    return attn_part_bytes(batch, num_heads, num_kv_heads, head_dim, S) + 256;
}

int ck_attn_decode_gqa_paged(const float *q, const void *k_pool, const void *v_pool, float *out,
                             const int32_t *block_tables, const int32_t *seq_lens, int batch, int num_heads,
                             int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                             int sliding_window, int kv_dtype, float k_scale, float v_scale, void *scratch,
                             size_t scratch_bytes, void *stream) {
    int rc = check_ptrs({q, k_pool, v_pool, out, block_tables, seq_lens}, {});
    if (rc) return rc;
    if ((rc = attn_shape_ok(num_heads, num_kv_heads, head_dim))) return rc;
    if (batch < 1 || batch > 1024 || block_size < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        sliding_window < 0)
        return CK_EINVAL;
    if (kv_dtype < 0 || kv_dtype > 2) return CK_EINVAL;
    if (kv_dtype != 0 && head_dim != 64 && head_dim != 128) return CK_EINVAL;
    if (kv_dtype == 2 && (!scale_ok(k_scale) || !scale_ok(v_scale))) return CK_EINVAL;
    if (!scratch) return CK_ESCRATCH;
    if (!aligned16(scratch)) return CK_EALIGN;
    const int rows = paged_rows(block_size, max_blocks_per_seq, sliding_window);
    int S = attn_splits_batched(batch, num_kv_heads, rows);
    // the tensor-core kernel pays more per CTA (TMEM, q image, the first
    // tiles) and overlaps two tiles per CTA: about 4 CTAs per SM instead of 8
    // (fewer splits fit the scratch sized for more)
    const int nsm = device_info().num_sms;
    if (attention_tc_ok(kv_dtype, num_heads, num_kv_heads, head_dim) && 2 * batch * num_kv_heads > nsm) {
        const int s4 = (4 * nsm + batch * num_kv_heads - 1) / (batch * num_kv_heads);
        if (s4 < S) S = s4 < 1 ? 1 : s4;
    }
    if (scratch_bytes < attn_part_bytes(batch, num_heads, num_kv_heads, head_dim, S)) return CK_ESCRATCH;
    unsigned *st = status_word();
    if (!st) return CK_ECUDA;
    AttnArgs a{};
    a.q = q;
    a.k_cache = static_cast<const float *>(k_pool);  // pools of kv_dtype elements
    a.v_cache = static_cast<const float *>(v_pool);
    a.kv_tokens = rows;  // the stage plan follows the longest split
    a.H = num_heads;
    a.KV = num_kv_heads;
    a.hd = head_dim;
    a.C = rows;
    a.splits = S;
    a.part = static_cast<float *>(scratch);
    a.out = out;
    a.kv_type = kv_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_tables = block_tables;
    a.seq_lens = seq_lens;
    a.block_size = block_size;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.window = sliding_window;
    a.status = st;
    return launch_attention(a, batch, as_stream(stream), false, false) ? CK_ECUDA : CK_OK;
}

static int attn_call(const float *q, const void *k_cache, const void *v_cache, float *out, int num_heads,
                     int num_kv_heads, int kv_tokens, int cache_capacity, int head_dim, int kv_type, float k_scale,
                     float v_scale, void *scratch, size_t scratch_bytes, void *stream, int splits) {
    int rc = check_ptrs({q, k_cache, v_cache, out}, {});
    if (rc) return rc;
    if (kv_type != 0 && head_dim != 64 && head_dim != 128) return CK_EINVAL;
    if ((rc = attn_shape_ok(num_heads, num_kv_heads, head_dim))) return rc;
    if (cache_capacity <= 0) return CK_EINVAL;
    if (kv_tokens < 1 || kv_tokens > cache_capacity) return CK_ERANGE;
    if (!scratch) return CK_ESCRATCH;
    if (!aligned16(scratch)) return CK_EALIGN;
    // the split count follows the token count actually attended (or is given)
    const int S = splits > 0 ? splits : attn_splits(1, num_kv_heads, kv_tokens);
    if (scratch_bytes < attn_part_bytes(1, num_heads, num_kv_heads, head_dim, S)) return CK_ESCRATCH;
    unsigned *st = status_word();
    if (!st) return CK_ECUDA;
    AttnArgs a{};
    a.q = q;
    a.k_cache = static_cast<const float *>(k_cache);  // elements of kv_type
    a.v_cache = static_cast<const float *>(v_cache);
    a.kv_tokens = kv_tokens;
    a.H = num_heads;
    a.KV = num_kv_heads;
    a.hd = head_dim;
    a.C = cache_capacity;
    a.splits = S;
    a.part = static_cast<float *>(scratch);
    a.out = out;
    a.kv_type = kv_type;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.status = st;
    return launch_attention(a, 1, as_stream(stream), false, false) ? CK_ECUDA : CK_OK;
}

size_t ck_decode_layer_scratch_size(int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                    int cache_capacity) {
    if (embed_dim <= 0 || embed_dim % 32 || cache_capacity <= 0) return 0;
    if (attn_shape_ok(num_heads, num_kv_heads, head_dim)) return 0;
    return layer_scratch(embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity).total;
}

int ck_decode_layer(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                    const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                    const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                    const float *rope_sin, int pos, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                    int cache_capacity, float eps, void *scratch, size_t scratch_bytes, void *stream) {
    return layer_common(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos,
                        rope_sin, pos, nullptr, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity, eps,
                        scratch, scratch_bytes, stream);
}

int ck_decode_layer_devpos(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                           const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                           const float *bv, const float *bo, float *k_cache, float *v_cache,
                           const float *rope_cos, const float *rope_sin, const int32_t *d_pos, int embed_dim,
                           int num_heads, int num_kv_heads, int head_dim, int cache_capacity, float eps,
                           void *scratch, size_t scratch_bytes, void *stream) {
    if (!d_pos) return CK_EINVAL;
    return layer_common(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos,
                        rope_sin, 0, d_pos, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity, eps,
                        scratch, scratch_bytes, stream);
}

size_t ck_decode_layer_batched_scratch_size(int batch, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                            int cache_capacity) {
    if (batch_shape_check(batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity)) return 0;
    return batch_scratch(batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity).total;
}

size_t ck_decode_layer_batched_scratch_offset(int tap, int batch, int embed_dim, int num_heads, int num_kv_heads,
                                              int head_dim, int cache_capacity) {
    if (batch_shape_check(batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity))
        return static_cast<size_t>(-1);
    const BatchScratch L = batch_scratch(batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity);
    switch (tap) {
        case CK_TAP_Q: return L.off_q;
        case CK_TAP_XQ8: return L.off_xq8;
        case CK_TAP_ATTN: return L.off_attn;
        case CK_TAP_AQ8: return L.off_aq8;
        default: return static_cast<size_t>(-1);
    }
}

// The launches of a batched step on validated arguments: norm + pack, the Q/K/V
// projections (with RoPE and the KV stores), attention, the O projection.
// pdl_first: whether the first launch may overlap the stream's preceding work.
static int batched_body(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                        const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                        const float *bv, const float *bo, float *const *k_caches, float *const *v_caches,
                        const float *rope_cos, const float *rope_sin, const int32_t *d_pos, int batch, int embed_dim,
                        int num_heads, int num_kv_heads, int head_dim, int cache_capacity, float eps, uint8_t *sc,
                        const BatchScratch &L, cudaStream_t s, bool pdl_first, int chunk_pos,
                        uint8_t *pf_img = nullptr, float *pf_k = nullptr, float *pf_v = nullptr,
                        const int32_t *pf_dpos = nullptr) {
    unsigned *st = status_word();
    if (!st) return CK_ECUDA;

    BatchArgs ba{};
    ba.B = batch;
    ba.x = x;
    ba.residual = residual;
    ba.gamma = gamma;
    ba.wq = static_cast<const uint8_t *>(wq);
    ba.wk = static_cast<const uint8_t *>(wk);
    ba.wv = static_cast<const uint8_t *>(wv);
    ba.wo = static_cast<const uint8_t *>(wo);
    ba.bq = bq;
    ba.bk = bk;
    ba.bv = bv;
    ba.bo = bo;
    ba.k_caches = k_caches;
    ba.v_caches = v_caches;
    ba.rope_cos = rope_cos;
    ba.rope_sin = rope_sin;
    ba.d_pos = d_pos;
    ba.D = embed_dim;
    ba.H = num_heads;
    ba.KV = num_kv_heads;
    ba.hd = head_dim;
    ba.C = cache_capacity;
    ba.eps = eps;
    ba.out = out;
    ba.q = reinterpret_cast<float *>(sc + L.off_q);
    ba.xq8 = sc + L.off_xq8;
    ba.xpack = sc + L.off_xpack;
    ba.apack = sc + L.off_apack;
    ba.aq8 = sc + L.off_aq8;
    ba.status = st;
    // projections on the tensor cores where the shapes allow, else dp4a
    const bool tc = batched_tc_ok(embed_dim, num_heads, num_kv_heads, head_dim);
    if (tc) {
        ba.ximg = sc + L.off_ximg;
        ba.aimg = sc + L.off_aimg;
        ba.proj_part = reinterpret_cast<float *>(sc + L.off_ppart);
        ba.tickets = reinterpret_cast<int *>(sc + L.off_tickets);
        ba.tickets_o = L.tp.tickets_o;
        ba.n_tickets = L.tp.tickets;
    }
    if (launch_norm_pack(ba, s, pdl_first)) return CK_ECUDA;
    if ((tc ? launch_rows_tc(ba, false, s, true) : launch_rows_batched(ba, false, s, true))) return CK_ECUDA;

    AttnArgs aa{};
    aa.q = ba.q;
    aa.k_caches = k_caches;
    aa.v_caches = v_caches;
    aa.d_pos = d_pos;
    aa.H = num_heads;
    aa.KV = num_kv_heads;
    aa.hd = head_dim;
    aa.C = cache_capacity;
    aa.splits = L.splits;
    aa.part = reinterpret_cast<float *>(sc + L.off_part);
    aa.out = reinterpret_cast<float *>(sc + L.off_attn);
    aa.out_q8 = sc + L.off_aq8;
    aa.out_pack = ba.apack;
    aa.out_img = ba.aimg;
    aa.img_groups = img_groups(batch);
    if (chunk_pos >= 0) {  // prefill: every row from the chunk's start is new
        aa.fresh_chunk = 1;
        aa.fresh_from = chunk_pos;
    }
    aa.l2_prefetch = wo;
    aa.l2_prefetch_bytes = static_cast<size_t>(embed_dim) * (num_heads * head_dim / 32) * 22;
    aa.status = st;
    if (pf_img) {  // a prefill chunk on the tensor cores
        if (launch_prefill_attn(aa, ba.q, pf_k, pf_v, pf_img, batch, chunk_pos, pf_dpos, num_heads, num_kv_heads,
                                cache_capacity, s))
            return CK_ECUDA;
    } else if (launch_attention(aa, batch, s, true, true)) {
        return CK_ECUDA;
    }
    if ((tc ? launch_rows_tc(ba, true, s, true) : launch_rows_batched(ba, true, s, true))) return CK_ECUDA;
    return CK_OK;
}

int ck_decode_layer_batched(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                            const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                            const float *bv, const float *bo, float *const *k_caches, float *const *v_caches,
                            const float *rope_cos, const float *rope_sin, const int32_t *d_pos, int batch,
                            int embed_dim, int num_heads, int num_kv_heads, int head_dim, int cache_capacity,
                            float eps, void *scratch, size_t scratch_bytes, void *stream) {
    int rc = check_ptrs({out, x, residual, wq, wk, wv, wo, gamma, k_caches, v_caches, rope_cos, rope_sin, d_pos},
                        {bq, bk, bv, bo});
    if (rc) return rc;
    if ((rc = batch_shape_check(batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity))) return rc;
    if (!scratch) return CK_ESCRATCH;
    if (!aligned16(scratch)) return CK_EALIGN;
    const BatchScratch L = batch_scratch(batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity);
    if (scratch_bytes < L.total) return CK_ESCRATCH;
    if (out == x || out == residual) return CK_EINVAL;
    return batched_body(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_caches, v_caches, rope_cos,
                        rope_sin, d_pos, batch, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity, eps,
                        static_cast<uint8_t *>(scratch), L, as_stream(stream), true, -1);
}

// ---- the multi-token (prefill) form ----------------------------------------
// The chunk's n tokens run as a batch of n entries over the one cache; the
// per-entry cache pointers and positions live after the batched scratch.
struct PrefillScratch {
    BatchScratch b;
    size_t off_kcs, off_vcs, off_pos, off_img, total;
    bool tc_attn;  // the chunk's attention on the tensor cores (else one decode attention per token)
};

static PrefillScratch prefill_scratch(int n, int D, int H, int KV, int hd, int C) {
    PrefillScratch P{};
    P.b = batch_scratch(n, D, H, KV, hd, C);
    size_t o = P.b.total;
    P.off_kcs = o;
    o = a256(o + static_cast<size_t>(n) * sizeof(float *));
    P.off_vcs = o;
    o = a256(o + static_cast<size_t>(n) * sizeof(float *));
    P.off_pos = o;
    o = a256(o + static_cast<size_t>(n) * 4);
    P.tc_attn = prefill_tc_ok(H, KV, hd) && batched_tc_ok(D, H, KV, hd);
    P.off_img = o;
    if (P.tc_attn) o = a256(o + prefill_img_bytes(KV, C));
    P.total = o;
    return P;
}

size_t ck_prefill_layer_scratch_size(int n_tokens, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                     int cache_capacity) {
    if (batch_shape_check(n_tokens, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity)) return 0;
    return prefill_scratch(n_tokens, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity).total;
}

size_t ck_prefill_layer_scratch_offset(int tap, int n_tokens, int embed_dim, int num_heads, int num_kv_heads,
                                       int head_dim, int cache_capacity) {
    return ck_decode_layer_batched_scratch_offset(tap, n_tokens, embed_dim, num_heads, num_kv_heads, head_dim,
                                                  cache_capacity);
}

size_t ck_attn_prefill_scratch_size(int num_heads, int num_kv_heads, int head_dim, int cache_capacity) {
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || cache_capacity <= 0) return 0;
    if (!prefill_tc_ok(num_heads, num_kv_heads, head_dim)) return 0;
    return prefill_img_bytes(num_kv_heads, cache_capacity) + 256;
}

int ck_attn_prefill_gqa(const float *q, const float *k_cache, const float *v_cache, float *out, int pos,
                        int n_tokens, int num_heads, int num_kv_heads, int head_dim, int cache_capacity,
                        void *scratch, size_t scratch_bytes, void *stream) {
    int rc = check_ptrs({q, k_cache, v_cache, out}, {});
    if (rc) return rc;
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return CK_EINVAL;
    if (!prefill_tc_ok(num_heads, num_kv_heads, head_dim) || cache_capacity <= 0 || n_tokens < 1 ||
        n_tokens > (1 << 20))
        return CK_EINVAL;
    if (pos < 0 || pos > cache_capacity - n_tokens) return CK_ERANGE;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return CK_EALIGN;
    if (!scratch) return CK_ESCRATCH;
    if (!aligned16(scratch)) return CK_EALIGN;
    if (scratch_bytes < prefill_img_bytes(num_kv_heads, cache_capacity)) return CK_ESCRATCH;
    unsigned *st = status_word();
    if (!st) return CK_ECUDA;
    AttnArgs o{};
    o.H = num_heads;
    o.KV = num_kv_heads;
    o.hd = head_dim;
    o.out = out;
    o.status = st;
    return launch_prefill_attn(o, q, k_cache, v_cache, static_cast<uint8_t *>(scratch), n_tokens, pos, nullptr,
                               num_heads, num_kv_heads, cache_capacity, as_stream(stream))
               ? CK_ECUDA
               : CK_OK;
}

static int prefill_common(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                          const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                          const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                          const float *rope_sin, int pos, const int32_t *d_pos, int n_tokens, int embed_dim,
                          int num_heads, int num_kv_heads, int head_dim, int cache_capacity, float eps, void *scratch,
                          size_t scratch_bytes, void *stream) {
    int rc = check_ptrs({out, x, residual, wq, wk, wv, wo, gamma, k_cache, v_cache, rope_cos, rope_sin},
                        {bq, bk, bv, bo, d_pos});
    if (rc) return rc;
    if ((rc = batch_shape_check(n_tokens, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity))) return rc;
    if (!d_pos && (pos < 0 || pos > cache_capacity - n_tokens)) return CK_ERANGE;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return CK_EALIGN;
    if (!scratch) return CK_ESCRATCH;
    if (!aligned16(scratch)) return CK_EALIGN;
    const PrefillScratch P = prefill_scratch(n_tokens, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity);
    if (scratch_bytes < P.total) return CK_ESCRATCH;
    if (out == x || out == residual) return CK_EINVAL;
    uint8_t *sc = static_cast<uint8_t *>(scratch);
    cudaStream_t s = as_stream(stream);
    unsigned *st = status_word();
    if (!st) return CK_ECUDA;
    float **kcs = reinterpret_cast<float **>(sc + P.off_kcs);
    float **vcs = reinterpret_cast<float **>(sc + P.off_vcs);
    int32_t *pos_of = reinterpret_cast<int32_t *>(sc + P.off_pos);
    if (launch_prefill_setup(kcs, vcs, pos_of, k_cache, v_cache, pos, d_pos, n_tokens, cache_capacity, st, s))
        return CK_ECUDA;
    // The first batched launch waits for the whole setup grid (no overlap).
    // With the position on the device the decode-path attention treats every
    // row as possibly new (chunk start 0).
    return batched_body(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, kcs, vcs, rope_cos, rope_sin,
                        pos_of, n_tokens, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity, eps, sc,
                        P.b, s, false, d_pos ? 0 : pos, P.tc_attn ? sc + P.off_img : nullptr, k_cache, v_cache,
                        d_pos);
}

int ck_prefill_layer(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                     const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                     const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                     const float *rope_sin, int pos, int n_tokens, int embed_dim, int num_heads, int num_kv_heads,
                     int head_dim, int cache_capacity, float eps, void *scratch, size_t scratch_bytes, void *stream) {
    return prefill_common(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos,
                          rope_sin, pos, nullptr, n_tokens, embed_dim, num_heads, num_kv_heads, head_dim,
                          cache_capacity, eps, scratch, scratch_bytes, stream);
}

int ck_prefill_layer_devpos(float *out, const float *x, const float *residual, const void *wq, const void *wk,
                            const void *wv, const void *wo, const float *gamma, const float *bq, const float *bk,
                            const float *bv, const float *bo, float *k_cache, float *v_cache, const float *rope_cos,
                            const float *rope_sin, const int32_t *d_pos, int n_tokens, int embed_dim, int num_heads,
                            int num_kv_heads, int head_dim, int cache_capacity, float eps, void *scratch,
                            size_t scratch_bytes, void *stream) {
    if (!d_pos) return CK_EINVAL;
    return prefill_common(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos,
                          rope_sin, 0, d_pos, n_tokens, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity,
                          eps, scratch, scratch_bytes, stream);
}

size_t ck_decode_layer_scratch_offset(int tap, int embed_dim, int num_heads, int num_kv_heads, int head_dim,
                                      int cache_capacity) {
    if (ck_decode_layer_scratch_size(embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity) == 0)
        return static_cast<size_t>(-1);
    const LayerScratch L = layer_scratch(embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity);
    switch (tap) {
        case CK_TAP_Q: return L.off_q;
        case CK_TAP_XQ8: return L.off_xq8;
        case CK_TAP_ATTN: return L.off_attn;
        case CK_TAP_AQ8: return L.off_aq8;
        default: return static_cast<size_t>(-1);
    }
}

int ck_device_status(int *status, void *stream) {
    if (!status) return CK_EINVAL;
    unsigned *w = status_word();
    if (!w) return CK_ECUDA;
    cudaStream_t s = as_stream(stream);
    unsigned flags = 0;
    if (cudaMemcpyAsync(&flags, w, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess) return CK_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CK_ECUDA;
    if (cudaMemsetAsync(w, 0, sizeof(unsigned), s) != cudaSuccess) return CK_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CK_ECUDA;
    *status = (flags & FLAG_TIMEOUT) ? CK_ETIMEOUT : ((flags & FLAG_RANGE) ? CK_ERANGE : CK_OK);
    return CK_OK;
}

int ck_block_dots_q5_0_q8_0(int32_t *isum, const void *W, const void *x_q8, int M, int K, void *stream) {
    int rc = check_ptrs({isum, W, x_q8}, {});
    if (rc) return rc;
    if (M <= 0 || K <= 0 || K % 32 != 0) return CK_EINVAL;
    return launch_block_dots(false, isum, W, x_q8, M, K, as_stream(stream)) ? CK_ECUDA : CK_OK;
}

int ck_block_dots_q8_0_q8_0(int32_t *isum, const void *W, const void *x_q8, int M, int K, void *stream) {
    int rc = check_ptrs({isum, W, x_q8}, {});
    if (rc) return rc;
    if (M <= 0 || K <= 0 || K % 32 != 0) return CK_EINVAL;
    return launch_block_dots(true, isum, W, x_q8, M, K, as_stream(stream)) ? CK_ECUDA : CK_OK;
}

}  // extern "C"
