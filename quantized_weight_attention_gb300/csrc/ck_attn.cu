// Host side of the decode attention (STEP 7 of the page
// "mega_fused_attention_decode_q5_0.c"): split planning and dispatch to the
// kernels of ck_attn_kernels.cuh, which are instantiated one head_dim per
// translation unit (ck_attn_d*.cu).  Also here: the standalone RoPE and
// KV-store kernels (STEP 5, STEP 6).
#include <cuda_bf16.h>

#include "ck_attn_kernels.cuh"

namespace ck {

// ---------------------------------------------------------------------------
// STEP 5 / STEP 6 as standalone kernels
// ---------------------------------------------------------------------------
__global__ void k_rope(float *q, float *k, const float *__restrict__ c, const float *__restrict__ sn, int pos, int H,
                       int KV, int hd) {
    const int half = hd >> 1;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (H + KV) * half) return;
    const int head = idx / half, d = idx - head * half;
    float *p = head < H ? q + static_cast<size_t>(head) * hd : k + static_cast<size_t>(head - H) * hd;
    const float A = p[d], B = p[d + half];
    const float cc = c[static_cast<size_t>(pos) * half + d], ss = sn[static_cast<size_t>(pos) * half + d];
    p[d] = __fsub_rn(__fmul_rn(A, cc), __fmul_rn(B, ss));
    p[d + half] = __fadd_rn(__fmul_rn(A, ss), __fmul_rn(B, cc));
}

__global__ void k_kv_store(float *kc, float *vc, const float *__restrict__ k, const float *__restrict__ v, int pos,
                           int KV, int C, int hd) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= KV * hd) return;
    const int h = idx / hd, d = idx - h * hd;
    const size_t o = (static_cast<size_t>(h) * C + pos) * hd + d;
    kc[o] = k[idx];
    vc[o] = v[idx];
}

// KV store into a bf16 cache (round to nearest even) or an fp8 E4M3 cache
// (the IEEE quotient x / scale, then round to nearest even onto E4M3 with
// saturation to +-448; the value is converted into both halves of the packed
// pair, so the byte taken does not depend on the pair's order).
__global__ void k_kv_store_q(uint8_t *kc, uint8_t *vc, const float *__restrict__ k, const float *__restrict__ v,
                             int pos, int KV, int C, int hd, int kv_type, float k_scale, float v_scale) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= KV * hd) return;
    const int h = idx / hd, d = idx - h * hd;
    const size_t o = (static_cast<size_t>(h) * C + pos) * hd + d;
    if (kv_type == KV_BF16) {
        reinterpret_cast<__nv_bfloat16 *>(kc)[o] = __float2bfloat16_rn(k[idx]);
        reinterpret_cast<__nv_bfloat16 *>(vc)[o] = __float2bfloat16_rn(v[idx]);
    } else {
        const float xk = __fdiv_rn(k[idx], k_scale), xv = __fdiv_rn(v[idx], v_scale);
        unsigned short pk, pv;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pk) : "f"(xk), "f"(xk));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pv) : "f"(xv), "f"(xv));
        kc[o] = static_cast<uint8_t>(pk & 0xFF);
        vc[o] = static_cast<uint8_t>(pv & 0xFF);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t attn_part_bytes(int B, int H, int KV, int hd, int splits) {
    const int G = H / KV;
    return static_cast<size_t>(B) * KV * splits * part_stride(G, hd) * 4;
}

int attn_splits(int B, int KV, int max_tokens) {
    const int ctas = device_info().num_sms;  // one CTA per SM
    int S = (ctas + B * KV - 1) / (B * KV);
    const int tiles = (max_tokens + AT_TILE - 1) / AT_TILE;
    if (S > tiles) S = tiles;
    if (S < 1) S = 1;
    if (S > 1024) S = 1024;
    return S;
}

// Batches of many sequences: about 8 CTAs per SM so that the ragged lengths
// balance across the grid; few sequences: one CTA per SM, as attn_splits.
int attn_splits_batched(int B, int KV, int max_tokens) {
    const int nsm = device_info().num_sms;
    if (2 * B * KV <= nsm) return attn_splits(B, KV, max_tokens);
    int S = (8 * nsm + B * KV - 1) / (B * KV);
    const int tiles = (max_tokens + AT_TILE - 1) / AT_TILE;
    if (S > tiles) S = tiles;
    if (S < 1) S = 1;
    if (S > 64) S = 64;
    return S;
}

extern template int launch_attention_dpl<1, KV_F32>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<2, KV_F32>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<3, KV_F32>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<4, KV_F32>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<8, KV_F32>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<2, KV_BF16>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<4, KV_BF16>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<2, KV_FP8>(const AttnArgs &, int, cudaStream_t, bool, bool);
extern template int launch_attention_dpl<4, KV_FP8>(const AttnArgs &, int, cudaStream_t, bool, bool);

int launch_attention(const AttnArgs &a, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    if (attention_tc_ok(a.kv_type, a.H, a.KV, a.hd)) return launch_attention_tc(a, B, s, pdl_first, pdl_combine);
    if (a.kv_type == KV_BF16 || a.kv_type == KV_FP8) {  // head_dim 64 and 128
        const bool f8 = a.kv_type == KV_FP8;
        switch (a.hd) {
            case 64:
                return f8 ? launch_attention_dpl<2, KV_FP8>(a, B, s, pdl_first, pdl_combine)
                          : launch_attention_dpl<2, KV_BF16>(a, B, s, pdl_first, pdl_combine);
            case 128:
                return f8 ? launch_attention_dpl<4, KV_FP8>(a, B, s, pdl_first, pdl_combine)
                          : launch_attention_dpl<4, KV_BF16>(a, B, s, pdl_first, pdl_combine);
            default: return -1;
        }
    }
    switch (a.hd / 32) {
        case 1: return launch_attention_dpl<1, KV_F32>(a, B, s, pdl_first, pdl_combine);
        case 2: return launch_attention_dpl<2, KV_F32>(a, B, s, pdl_first, pdl_combine);
        case 3: return launch_attention_dpl<3, KV_F32>(a, B, s, pdl_first, pdl_combine);
        case 4: return launch_attention_dpl<4, KV_F32>(a, B, s, pdl_first, pdl_combine);
        case 8: return launch_attention_dpl<8, KV_F32>(a, B, s, pdl_first, pdl_combine);
        default: return -1;
    }
}

int launch_rope(float *q, float *k, const float *c, const float *sn, int pos, int H, int KV, int hd, cudaStream_t s) {
    const int n = (H + KV) * (hd / 2);
    if (n == 0) return 0;
    k_rope<<<(n + 255) / 256, 256, 0, s>>>(q, k, c, sn, pos, H, KV, hd);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

int launch_kv_store_q(void *kc, void *vc, const float *k, const float *v, int pos, int KV, int C, int hd,
                      int kv_type, float k_scale, float v_scale, cudaStream_t s) {
    const int n = KV * hd;
    k_kv_store_q<<<(n + 255) / 256, 256, 0, s>>>(static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), k, v, pos,
                                                 KV, C, hd, kv_type, k_scale, v_scale);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

int launch_kv_store(float *kc, float *vc, const float *k, const float *v, int pos, int KV, int C, int hd,
                    cudaStream_t s) {
    const int n = KV * hd;
    k_kv_store<<<(n + 255) / 256, 256, 0, s>>>(kc, vc, k, v, pos, KV, C, hd);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace ck
