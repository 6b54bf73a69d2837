// Decode attention of the step (sm_103a): attention_forward_decode_head_
// major_gqa_flash of the page "mega_fused_attention_decode_q5_0.c" (STEP 7),
// as split-KV flash decoding:
//
//   k_attn_split    grid (S splits, KV heads, B sequences).  One CTA owns
//                   rows [t0, t1) of one KV head and all G = H/KV query heads
//                   that read it ("GQA-packed": each cache row is read once
//                   per KV head).  K and V tiles of 32 rows stream into a
//                   3-stage shared-memory ring through the bulk-copy engine;
//                   online softmax over the tiles; writes (m, l, acc) per
//                   query head.
//   k_attn_combine  grid (H, B).  Log-sum-exp merge of the S partials of one
//                   query head, the fp32 output, and its Q8_0 quantization
//                   (the O projection's input) in the epilogue.
//
// Scores are kept in log2 units: s2 = (q.k) * log2(e)/sqrt(hd), weights
// exp2(s2 - m2), which equals exp(s - m) of the definition.
//
// Also here: the standalone RoPE and KV-store kernels (STEP 5, STEP 6).
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

constexpr int ATT_TILE = 32;
constexpr int ATT_WARPS = 4;
constexpr int ATT_THREADS = 32 * ATT_WARPS;
constexpr int GMAX = 8;  // query heads per KV head handled by one CTA

__host__ __device__ constexpr int att_stages(int hd) { return hd > 128 ? 2 : 3; }

struct AttnSmem {
    size_t off_bar, off_stage, off_q, off_s, off_p, off_ml, total;
};

__host__ __device__ inline AttnSmem attn_smem(int hd) {
    AttnSmem L;
    size_t o = 0;
    L.off_bar = o;
    o += 64;
    L.off_stage = o;
    o += static_cast<size_t>(att_stages(hd)) * 2 * ATT_TILE * hd * 4;
    L.off_q = o;
    o += static_cast<size_t>(GMAX) * hd * 4;
    L.off_s = o;
    o += GMAX * ATT_TILE * 4;
    L.off_p = o;
    o += ATT_TILE * GMAX * 4;
    L.off_ml = o;
    o += 4 * GMAX * 4;  // m, l, alpha, spare
    L.total = (o + 127) / 128 * 128;
    return L;
}

// Partial results: for (b, g, s) a record of G m's, G l's, G*hd acc's.
__host__ __device__ inline size_t part_stride(int G, int hd) { return static_cast<size_t>(G) * (hd + 2); }

size_t attn_part_bytes(int B, int H, int KV, int hd, int splits) {
    const int G = H / KV;
    return static_cast<size_t>(B) * KV * splits * part_stride(G, hd) * 4;
}

template <int DPL>
__global__ void __launch_bounds__(ATT_THREADS, 2) k_attn_split(const AttnArgs a) {
    constexpr int HD = 32 * DPL;
    constexpr int HD4 = HD / 4;
    constexpr int NST = att_stages(HD);
    constexpr int VEC = (DPL % 4 == 0) ? 4 : ((DPL % 2 == 0) ? 2 : 1);
    constexpr int NV = DPL / VEC;
    extern __shared__ __align__(128) uint8_t smem[];
    const AttnSmem L = attn_smem(HD);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.off_bar);
    float *stage = reinterpret_cast<float *>(smem + L.off_stage);
    float *qs = reinterpret_cast<float *>(smem + L.off_q);
    float *Ss = reinterpret_cast<float *>(smem + L.off_s);   // [GMAX][TILE]
    float *Ps = reinterpret_cast<float *>(smem + L.off_p);   // [TILE][GMAX]
    float *ml = reinterpret_cast<float *>(smem + L.off_ml);  // m[GMAX], l[GMAX], alpha[GMAX]

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int S = gridDim.x;
    const int G = a.H / a.KV;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Spread an L2 prefetch of the next kernel's operand over the grid.
    const uint8_t *l2_pf = static_cast<const uint8_t *>(a.l2_prefetch);
    const size_t l2_pf_bytes = a.l2_prefetch_bytes & ~static_cast<size_t>(15);
    if (l2_pf && threadIdx.x == 0) {
        const size_t nct = static_cast<size_t>(gridDim.x) * gridDim.y * gridDim.z;
        const size_t cid = (static_cast<size_t>(b) * gridDim.y + g) * gridDim.x + s;
        const size_t per = ((l2_pf_bytes + nct - 1) / nct + 15) & ~static_cast<size_t>(15);
        const size_t beg = cid * per;
        if (beg < l2_pf_bytes) {
            size_t n = l2_pf_bytes - beg < per ? l2_pf_bytes - beg : per;
            n &= ~static_cast<size_t>(15);
            if (n) prefetch_l2(l2_pf + beg, static_cast<uint32_t>(n));
        }
    }

    int T;
    if (a.d_pos) {
        const int pos = a.d_pos[b];
        if (pos < 0 || pos >= a.C) {
            if (s == 0 && g == 0 && threadIdx.x == 0) flag_error(a.status, FLAG_RANGE);
            pdl_wait();
            return;
        }
        T = pos + 1;
    } else {
        T = a.kv_tokens;
    }
    const int chunk = (T + S - 1) / S;
    const int t0 = s * chunk;
    const int t1 = min(T, t0 + chunk);
    float *rec = a.part + ((static_cast<size_t>(b) * a.KV + g) * S + s) * part_stride(G, HD);
    if (t0 >= t1) {  // empty split: marked by m = -inf, skipped by the combine
        pdl_trigger();
        pdl_wait();  // the record may still be read by an earlier combine
        if (threadIdx.x < G) {
            rec[threadIdx.x] = -INFINITY;
            rec[G + threadIdx.x] = 0.0f;
        }
        return;
    }
    const float *kc = (a.k_caches ? a.k_caches[b] : a.k_cache) + static_cast<size_t>(g) * a.C * HD;
    const float *vc = (a.v_caches ? a.v_caches[b] : a.v_cache) + static_cast<size_t>(g) * a.C * HD;
    const int ntiles = (t1 - t0 + ATT_TILE - 1) / ATT_TILE;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Tile i of this split -> stage i % NST.  Rows before T-1 are never
    // written by the preceding grid, so they are fetched before waiting on
    // it; the tile holding row T-1 (the row just stored) waits first.
    auto issue = [&](int i) {
        const int r = t0 + i * ATT_TILE;
        const int n = min(ATT_TILE, t1 - r);
        if (r + n >= T) pdl_wait();
        float *dst = stage + static_cast<size_t>(i % NST) * 2 * ATT_TILE * HD;
        const uint32_t bytes = static_cast<uint32_t>(n) * HD * 4;
        mbar_arrive_expect_tx(&bars[i % NST], 2 * bytes);
        bulk_g2s(dst, kc + static_cast<size_t>(r) * HD, bytes, &bars[i % NST]);
        bulk_g2s(dst + ATT_TILE * HD, vc + static_cast<size_t>(r) * HD, bytes, &bars[i % NST]);
    };
    if (threadIdx.x == 0)
        for (int i = 0; i < NST && i < ntiles; ++i) issue(i);

    pdl_trigger();
    pdl_wait();  // q is the preceding grid's output
    for (int idx = threadIdx.x; idx < G * HD; idx += ATT_THREADS)
        qs[idx] = a.q[(static_cast<size_t>(b) * a.H + static_cast<size_t>(g) * G) * HD + idx];
    if (threadIdx.x < GMAX) {
        ml[threadIdx.x] = -INFINITY;
        ml[GMAX + threadIdx.x] = 0.0f;
    }
    __syncthreads();

    const float scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
    const float4 *q4 = reinterpret_cast<const float4 *>(qs);
    float acc[GMAX][DPL];
#pragma unroll
    for (int j = 0; j < GMAX; ++j)
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[j][e] = 0.0f;

    const int slice = lane & 7, rl = lane >> 3;
    const int rA = 8 * warp + rl, rB = rA + 4;
    for (int i = 0; i < ntiles; ++i) {
        const int st = i % NST;
        if (!mbar_wait(&bars[st], (i / NST) & 1)) flag_error(a.status, FLAG_TIMEOUT);
        const float *Kt = stage + static_cast<size_t>(st) * 2 * ATT_TILE * HD;
        const float *Vt = Kt + ATT_TILE * HD;
        const int n = min(ATT_TILE, t1 - (t0 + i * ATT_TILE));

        // ---- scores: lane = (row pair, 1/8 of the dims, float4-interleaved)
        {
            const float4 *K4 = reinterpret_cast<const float4 *>(Kt);
            float sa[GMAX], sb[GMAX];
#pragma unroll
            for (int j = 0; j < GMAX; ++j) sa[j] = sb[j] = 0.0f;
#pragma unroll
            for (int c = 0; c < DPL; ++c) {
                const float4 ka = K4[rA * HD4 + slice + 8 * c];
                const float4 kb = K4[rB * HD4 + slice + 8 * c];
#pragma unroll
                for (int j = 0; j < GMAX; ++j) {
                    if (j < G) {
                        const float4 qv = q4[j * HD4 + slice + 8 * c];
                        sa[j] = fmaf(qv.x, ka.x, fmaf(qv.y, ka.y, fmaf(qv.z, ka.z, fmaf(qv.w, ka.w, sa[j]))));
                        sb[j] = fmaf(qv.x, kb.x, fmaf(qv.y, kb.y, fmaf(qv.z, kb.z, fmaf(qv.w, kb.w, sb[j]))));
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < GMAX; ++j) {
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    sa[j] += __shfl_xor_sync(0xffffffffu, sa[j], o);
                    sb[j] += __shfl_xor_sync(0xffffffffu, sb[j], o);
                }
            }
            float va = 0.0f, vb = 0.0f;
#pragma unroll
            for (int j = 0; j < GMAX; ++j)
                if (j == slice) {
                    va = sa[j];
                    vb = sb[j];
                }
            if (slice < G) {
                Ss[slice * ATT_TILE + rA] = rA < n ? va * scale2 : -INFINITY;
                Ss[slice * ATT_TILE + rB] = rB < n ? vb * scale2 : -INFINITY;
            }
        }
        __syncthreads();
        // ---- online softmax update, one warp per query head
        for (int j = warp; j < G; j += ATT_WARPS) {
            const float x = Ss[j * ATT_TILE + lane];
            const float mo = ml[j];
            const float mn = fmaxf(mo, warp_max(x));
            const float alpha = (mo == -INFINITY) ? 0.0f : exp2f(mo - mn);
            const float p = (x == -INFINITY) ? 0.0f : exp2f(x - mn);
            Ps[lane * GMAX + j] = p;
            const float ps = warp_sum(p);
            if (lane == 0) {
                ml[GMAX + j] = ml[GMAX + j] * alpha + ps;
                ml[j] = mn;
                ml[2 * GMAX + j] = alpha;
            }
        }
        __syncthreads();
        // ---- acc = alpha * acc + P V over this warp's 8 rows
        {
#pragma unroll
            for (int j = 0; j < GMAX; ++j) {
                const float al = (j < G) ? ml[2 * GMAX + j] : 0.0f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[j][e] *= al;
            }
            const int rend = min(8 * warp + 8, n);
            for (int r = 8 * warp; r < rend; ++r) {
                const float4 p0 = reinterpret_cast<const float4 *>(Ps + r * GMAX)[0];
                const float4 p1 = reinterpret_cast<const float4 *>(Ps + r * GMAX)[1];
                const float pj[GMAX] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                float v[DPL];
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    const float *src = Vt + r * HD + VEC * (lane + 32 * u);
                    if constexpr (VEC == 4) {
                        const float4 t = *reinterpret_cast<const float4 *>(src);
                        v[4 * u] = t.x; v[4 * u + 1] = t.y; v[4 * u + 2] = t.z; v[4 * u + 3] = t.w;
                    } else if constexpr (VEC == 2) {
                        const float2 t = *reinterpret_cast<const float2 *>(src);
                        v[2 * u] = t.x; v[2 * u + 1] = t.y;
                    } else {
                        v[u] = *src;
                    }
                }
#pragma unroll
                for (int j = 0; j < GMAX; ++j)
                    if (j < G)
#pragma unroll
                        for (int e = 0; e < DPL; ++e) acc[j][e] = fmaf(pj[j], v[e], acc[j][e]);
            }
        }
        __syncthreads();  // stage st, Ss and Ps are free again
        if (threadIdx.x == 0 && i + NST < ntiles) issue(i + NST);
    }

    // ---- merge the 4 warps' accumulators (stage memory is idle now)
    float *red = stage;  // [ATT_WARPS][G][HD]
#pragma unroll
    for (int j = 0; j < GMAX; ++j)
        if (j < G)
#pragma unroll
            for (int u = 0; u < NV; ++u)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    red[(warp * G + j) * HD + VEC * (lane + 32 * u) + e] = acc[j][VEC * u + e];
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * HD; idx += ATT_THREADS) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < ATT_WARPS; ++w) t += red[w * G * HD + idx];
        rec[2 * G + idx] = t;
    }
    if (threadIdx.x < G) {
        rec[threadIdx.x] = ml[threadIdx.x];
        rec[G + threadIdx.x] = ml[GMAX + threadIdx.x];
    }
}

// Merge of the S partial records of one query head; fp32 output and its
// Q8_0 blocks.
template <int DPL>
__global__ void __launch_bounds__(256) k_attn_combine(const AttnArgs a) {
    constexpr int HD = 32 * DPL;
    constexpr int NW = 8;
    __shared__ float red[NW][HD];
    __shared__ float lred[NW];
    __shared__ float o_s[HD];
    const int h = blockIdx.x, b = blockIdx.y;
    const int G = a.H / a.KV;
    const int g = h / G, j = h - g * G;
    const int S = a.splits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.d_pos) {
        const int pos = a.d_pos[b];
        if (pos < 0 || pos >= a.C) {
            pdl_wait();
            return;
        }
    }
    pdl_trigger();
    pdl_wait();
    const size_t ps = part_stride(G, HD);
    const float *base = a.part + (static_cast<size_t>(b) * a.KV + g) * S * ps;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, base[s * ps + j]);
    M = warp_max(M);
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.0f;
    float Ls = 0.0f;
    for (int s = warp; s < S; s += NW) {
        const float *r = base + s * ps;
        const float ms = r[j];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        Ls = fmaf(w, r[G + j], Ls);
        const float *ac = r + 2 * G + static_cast<size_t>(j) * HD;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = fmaf(w, ac[lane + 32 * e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < DPL; ++e) red[warp][lane + 32 * e] = acc[e];
    if (lane == 0) lred[warp] = Ls;
    __syncthreads();
    float L = 0.0f;
#pragma unroll
    for (int w = 0; w < NW; ++w) L += lred[w];
    for (int d = threadIdx.x; d < HD; d += blockDim.x) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) t += red[w][d];
        const float o = __fdiv_rn(t, L);
        o_s[d] = o;
        a.out[(static_cast<size_t>(b) * a.H + h) * HD + d] = o;
    }
    __syncthreads();
    if (a.out_q8 && warp < HD / 32) {
        uint32_t dbits;
        float dq;
        const int q = q8_code(o_s[32 * warp + lane], dbits, dq);
        uint8_t *blk = a.out_q8 + ((static_cast<size_t>(b) * a.H + h) * (HD / 32) + warp) * Q8B;
        blk[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
        if (lane == 0) {
            blk[0] = static_cast<uint8_t>(dbits & 0xFF);
            blk[1] = static_cast<uint8_t>(dbits >> 8);
        }
    }
}

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

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int attn_splits(int B, int KV, int max_tokens) {
    const int nsm = device_info().num_sms;
    const int ctas = 2 * nsm;  // two CTAs fit per SM
    int S = (ctas + B * KV - 1) / (B * KV);
    const int tiles = (max_tokens + ATT_TILE - 1) / ATT_TILE;
    if (S > tiles) S = tiles;
    if (S < 1) S = 1;
    if (S > 1024) S = 1024;
    return S;
}

template <int DPL>
static int launch_attn_t(const AttnArgs &a0, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    AttnArgs a = a0;
    const AttnSmem L = attn_smem(32 * DPL);
    const void *fs = reinterpret_cast<const void *>(k_attn_split<DPL>);
    ensure_smem(fs, L.total);
    void *args1[] = {&a};
    cudaError_t e = launch(fs, dim3(a.splits, a.KV, B), dim3(ATT_THREADS), L.total, s, pdl_first, args1);
    if (e != cudaSuccess) return -5;
    void *args2[] = {&a};
    e = launch(reinterpret_cast<const void *>(k_attn_combine<DPL>), dim3(a.H, B), dim3(256), 0, s, pdl_combine,
               args2);
    return e == cudaSuccess ? 0 : -5;
}

int launch_attention(const AttnArgs &a, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    switch (a.hd / 32) {
        case 1: return launch_attn_t<1>(a, B, s, pdl_first, pdl_combine);
        case 2: return launch_attn_t<2>(a, B, s, pdl_first, pdl_combine);
        case 3: return launch_attn_t<3>(a, B, s, pdl_first, pdl_combine);
        case 4: return launch_attn_t<4>(a, B, s, pdl_first, pdl_combine);
        case 8: return launch_attn_t<8>(a, B, s, pdl_first, pdl_combine);
        default: return -1;
    }
}

int launch_rope(float *q, float *k, const float *c, const float *sn, int pos, int H, int KV, int hd, cudaStream_t s) {
    const int n = (H + KV) * (hd / 2);
    if (n == 0) return 0;
    k_rope<<<(n + 255) / 256, 256, 0, s>>>(q, k, c, sn, pos, H, KV, hd);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

int launch_kv_store(float *kc, float *vc, const float *k, const float *v, int pos, int KV, int C, int hd,
                    cudaStream_t s) {
    const int n = KV * hd;
    k_kv_store<<<(n + 255) / 256, 256, 0, s>>>(kc, vc, k, v, pos, KV, C, hd);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace ck
