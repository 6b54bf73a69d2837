// Decode attention of the step (sm_103a): attention_forward_decode_head_
// major_gqa_flash of the page "mega_fused_attention_decode_q5_0.c" (STEP 7),
// as split-KV flash decoding:
//
//   k_attn_split    grid (S splits, KV heads, B sequences), one CTA per SM.
//                   One CTA owns rows [t0, t1) of one KV head and all G =
//                   H/KV query heads that read it ("GQA-packed": each cache
//                   row is read once per KV head).  A producer warp streams
//                   16-row K and V tiles into a deep shared-memory ring
//                   through the bulk-copy engine; eight consumer warps take
//                   tiles round-robin, each with its own online softmax;
//                   writes (m, l, acc) per query head.
//   k_attn_combine  grid (H, hd/32, B).  Log-sum-exp merge of the S partials
//                   of one query head over one 32-wide slice of its dims,
//                   the fp32 output, and its Q8_0 block (the O projection's
//                   input) in the epilogue.
//
// Scores are kept in log2 units: s2 = (q.k) * log2(e)/sqrt(hd), weights
// exp2(s2 - m2), which equals exp(s - m) of the definition.
//
// Also here: the standalone RoPE and KV-store kernels (STEP 5, STEP 6).
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

constexpr int AT_TILE = 16;                          // cache rows per stage
constexpr int AT_CONSUMERS = 8;                      // consumer warps per CTA
constexpr int AT_THREADS = 32 * (AT_CONSUMERS + 1);  // + one producer warp
constexpr int GMAX = 8;                              // query heads per KV head

__host__ __device__ constexpr int at_stage_bytes(int hd) { return 2 * AT_TILE * hd * 4; }
__host__ __device__ constexpr int at_stages(int hd) {
    return (192 * 1024) / at_stage_bytes(hd) > 16 ? 16 : (192 * 1024) / at_stage_bytes(hd);
}

struct AttnSmem {
    size_t off_full, off_empty, off_stage, off_q, off_p, off_alpha, off_ml, total;
};

__host__ __device__ inline AttnSmem attn_smem(int hd) {
    AttnSmem L;
    size_t o = 0;
    L.off_full = o;
    o += 16 * 8;
    L.off_empty = o;
    o += 16 * 8;
    L.off_stage = o;
    o += static_cast<size_t>(at_stages(hd)) * at_stage_bytes(hd);
    L.off_q = o;
    o += static_cast<size_t>(GMAX) * hd * 4;
    L.off_p = o;
    o += static_cast<size_t>(AT_CONSUMERS) * AT_TILE * GMAX * 4;
    L.off_alpha = o;
    o += static_cast<size_t>(AT_CONSUMERS) * GMAX * 4;
    L.off_ml = o;
    o += static_cast<size_t>(2) * AT_CONSUMERS * GMAX * 4;
    L.total = (o + 127) / 128 * 128;
    return L;
}

// Partial results: for (b, g, s) a record of G m's, G l's, G*hd acc's.
__host__ __device__ inline size_t part_stride(int G, int hd) { return static_cast<size_t>(G) * (hd + 2); }

size_t attn_part_bytes(int B, int H, int KV, int hd, int splits) {
    const int G = H / KV;
    return static_cast<size_t>(B) * KV * splits * part_stride(G, hd) * 4;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sptr(bar)) : "memory");
}
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * AT_CONSUMERS) : "memory");
}

// One CTA per (split s, KV head g, sequence b); one CTA per SM.  Warp 0 is
// the producer: its lane 0 streams 16-row K and V tiles of rows [t0, t1)
// into an NST-stage ring (full / empty mbarrier per stage).  Warps 1..8
// consume tiles round-robin, each keeping its own online-softmax state for
// the G query heads; no CTA-wide barrier inside the loop.  At the end the
// eight states are merged (log-sum-exp) into the split's record.
//
// Scores: lane = (slice = lane & 7, row-lane rl = lane >> 3).  A slice is
// the float4 chunks {slice + 8c} of a row (interleaved so that the 8 slices
// hit 8 different bank groups); a lane accumulates 4 rows (rl + 4k) x G
// heads over its slice, then the 8 slices are summed with xor shuffles.
// Lane (slice = j, rl) then owns query head j's softmax state.
template <int DPL>
__global__ void __launch_bounds__(AT_THREADS, 1) k_attn_split(const AttnArgs a) {
    constexpr int HD = 32 * DPL;
    constexpr int HD4 = HD / 4;
    constexpr int NST = at_stages(HD);
    constexpr int VEC = (DPL % 4 == 0) ? 4 : ((DPL % 2 == 0) ? 2 : 1);
    constexpr int NV = DPL / VEC;
    extern __shared__ __align__(128) uint8_t smem[];
    const AttnSmem L = attn_smem(HD);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.off_full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.off_empty);
    float *stage = reinterpret_cast<float *>(smem + L.off_stage);
    float *qs = reinterpret_cast<float *>(smem + L.off_q);

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int S = gridDim.x;
    const int G = a.H / a.KV;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Spread an L2 prefetch of the next kernel's operand over the grid.
    if (a.l2_prefetch && threadIdx.x == 0) {
        const uint8_t *pf = static_cast<const uint8_t *>(a.l2_prefetch);
        const size_t total = a.l2_prefetch_bytes & ~static_cast<size_t>(15);
        const size_t nct = static_cast<size_t>(gridDim.x) * gridDim.y * gridDim.z;
        const size_t cid = (static_cast<size_t>(b) * gridDim.y + g) * gridDim.x + s;
        const size_t per = ((total + nct - 1) / nct + 15) & ~static_cast<size_t>(15);
        const size_t beg = cid * per;
        if (beg < total) {
            const size_t n = (total - beg < per ? total - beg : per) & ~static_cast<size_t>(15);
            if (n) prefetch_l2(pf + beg, static_cast<uint32_t>(n));
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
    const int chunk = a.chunk > 0 ? a.chunk : (T + S - 1) / S;
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
    const int ntiles = (t1 - t0 + AT_TILE - 1) / AT_TILE;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();

    if (warp == 0) {
        // ---- producer.  Rows before T-1 are never written by the preceding
        // grid, so they stream before waiting on it; the tile holding row
        // T-1 (the row just stored) waits first.
        if (lane == 0) {
            for (int t = 0; t < ntiles; ++t) {
                const int st = t % NST;
                if (t >= NST && !mbar_wait(&empty[st], ((t / NST) - 1) & 1)) {
                    flag_error(a.status, FLAG_TIMEOUT);
                    break;
                }
                const int r = t0 + t * AT_TILE;
                const int n = min(AT_TILE, t1 - r);
                if (r + n >= T) pdl_wait();
                float *dst = stage + static_cast<size_t>(st) * 2 * AT_TILE * HD;
                const uint32_t bytes = static_cast<uint32_t>(n) * HD * 4;
                mbar_arrive_expect_tx(&full[st], 2 * bytes);
                bulk_g2s(dst, kc + static_cast<size_t>(r) * HD, bytes, &full[st]);
                bulk_g2s(dst + AT_TILE * HD, vc + static_cast<size_t>(r) * HD, bytes, &full[st]);
            }
        }
        return;
    }

    // ---- consumers
    const int cw = warp - 1;
    const int ct = threadIdx.x - 32;
    float *Pw = reinterpret_cast<float *>(smem + L.off_p) + cw * AT_TILE * GMAX;  // [TILE][GMAX]
    float *alw = reinterpret_cast<float *>(smem + L.off_alpha) + cw * GMAX;
    float *mlw = reinterpret_cast<float *>(smem + L.off_ml);  // m[NC][GMAX], l[NC][GMAX]
    pdl_wait();  // q is the preceding grid's output
    for (int idx = ct; idx < G * HD; idx += 32 * AT_CONSUMERS)
        qs[idx] = a.q[(static_cast<size_t>(b) * a.H + static_cast<size_t>(g) * G) * HD + idx];
    consumers_sync();

    const float scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
    const float4 *q4 = reinterpret_cast<const float4 *>(qs);
    const int slice = lane & 7, rl = lane >> 3;
    float mrun = -INFINITY, lrun = 0.0f;  // head `slice`
    float acc[GMAX][DPL];
#pragma unroll
    for (int j = 0; j < GMAX; ++j)
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[j][e] = 0.0f;

    for (int t = cw; t < ntiles; t += AT_CONSUMERS) {
        const int st = t % NST;
        if (!mbar_wait(&full[st], (t / NST) & 1)) flag_error(a.status, FLAG_TIMEOUT);
        const float *Kt = stage + static_cast<size_t>(st) * 2 * AT_TILE * HD;
        const float *Vt = Kt + AT_TILE * HD;
        const int n = min(AT_TILE, t1 - (t0 + t * AT_TILE));

        float sc[GMAX][4];
#pragma unroll
        for (int j = 0; j < GMAX; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) sc[j][k] = 0.0f;
        const float4 *K4 = reinterpret_cast<const float4 *>(Kt);
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            float4 kk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) kk[k] = K4[(rl + 4 * k) * HD4 + slice + 8 * c];
#pragma unroll
            for (int j = 0; j < GMAX; ++j) {
                if (j < G) {
                    const float4 qv = q4[j * HD4 + slice + 8 * c];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        sc[j][k] = fmaf(qv.x, kk[k].x,
                                        fmaf(qv.y, kk[k].y, fmaf(qv.z, kk[k].z, fmaf(qv.w, kk[k].w, sc[j][k]))));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < GMAX; ++j) {
            if (j < G) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    sc[j][k] += __shfl_xor_sync(0xffffffffu, sc[j][k], 1);
                    sc[j][k] += __shfl_xor_sync(0xffffffffu, sc[j][k], 2);
                    sc[j][k] += __shfl_xor_sync(0xffffffffu, sc[j][k], 4);
                }
            }
        }
        // this lane's head j = slice, rows rl + 4k
        float my[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float v = 0.0f;
#pragma unroll
            for (int j = 0; j < GMAX; ++j)
                if (j == slice) v = sc[j][k];
            my[k] = (rl + 4 * k < n) ? v * scale2 : -INFINITY;
        }
        float tmax = fmaxf(fmaxf(my[0], my[1]), fmaxf(my[2], my[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float mnew = fmaxf(mrun, tmax);
        const float alpha = (mrun == -INFINITY) ? 0.0f : exp2f(mrun - mnew);
        float psum = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float p = (my[k] == -INFINITY || slice >= G) ? 0.0f : exp2f(my[k] - mnew);
            Pw[(rl + 4 * k) * GMAX + slice] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 8);
        psum += __shfl_xor_sync(0xffffffffu, psum, 16);
        lrun = lrun * alpha + psum;
        mrun = mnew;
        if (rl == 0) alw[slice] = alpha;
        __syncwarp();
        // ---- acc = alpha * acc + P V
#pragma unroll
        for (int j = 0; j < GMAX; ++j) {
            if (j < G) {
                const float al = alw[j];
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[j][e] *= al;
            }
        }
        for (int r = 0; r < n; ++r) {
            const float4 p0 = reinterpret_cast<const float4 *>(Pw + r * GMAX)[0];
            const float4 p1 = reinterpret_cast<const float4 *>(Pw + r * GMAX)[1];
            const float pj[GMAX] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            float v[DPL];
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const float *src = Vt + r * HD + VEC * (lane + 32 * u);
                if constexpr (VEC == 4) {
                    const float4 tv = *reinterpret_cast<const float4 *>(src);
                    v[4 * u] = tv.x; v[4 * u + 1] = tv.y; v[4 * u + 2] = tv.z; v[4 * u + 3] = tv.w;
                } else if constexpr (VEC == 2) {
                    const float2 tv = *reinterpret_cast<const float2 *>(src);
                    v[2 * u] = tv.x; v[2 * u + 1] = tv.y;
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---- merge the consumer warps' states
    if (rl == 0 && slice < G) {
        mlw[cw * GMAX + slice] = mrun;
        mlw[(AT_CONSUMERS + cw) * GMAX + slice] = lrun;
    }
    consumers_sync();  // every tile consumed: the ring is idle
    float *accw = stage;  // [NC][G][HD]
#pragma unroll
    for (int j = 0; j < GMAX; ++j)
        if (j < G)
#pragma unroll
            for (int u = 0; u < NV; ++u)
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    accw[(cw * G + j) * HD + VEC * (lane + 32 * u) + e] = acc[j][VEC * u + e];
    consumers_sync();
    for (int idx = ct; idx < G * HD; idx += 32 * AT_CONSUMERS) {
        const int j = idx / HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < AT_CONSUMERS; ++w) M = fmaxf(M, mlw[w * GMAX + j]);
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < AT_CONSUMERS; ++w) {
            const float mw = mlw[w * GMAX + j];
            if (mw != -INFINITY) t = fmaf(exp2f(mw - M), accw[(w * G + j) * HD + (idx - j * HD)], t);
        }
        rec[2 * G + idx] = t;
        if (idx - j * HD == 0) {
            float Ls = 0.0f;
#pragma unroll
            for (int w = 0; w < AT_CONSUMERS; ++w) {
                const float mw = mlw[w * GMAX + j];
                if (mw != -INFINITY) Ls = fmaf(exp2f(mw - M), mlw[(AT_CONSUMERS + w) * GMAX + j], Ls);
            }
            rec[j] = M;
            rec[G + j] = Ls;
        }
    }
}

// Merge of the S partial records of one query head, for one 32-wide slice of
// its dims (= one Q8_0 block of the output): fp32 output and the block.
template <int DPL>
__global__ void __launch_bounds__(256) k_attn_combine(const AttnArgs a) {
    constexpr int HD = 32 * DPL;
    constexpr int NW = 8;
    constexpr int U = 4;
    __shared__ float ared[NW][32];
    __shared__ float lred[NW];
    const int h = blockIdx.x, blk = blockIdx.y, b = blockIdx.z;
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
    float acc = 0.0f, Ls = 0.0f;
    for (int s0 = warp; s0 < S; s0 += NW * U) {
        float mv[U], lv[U], av[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int s = s0 + NW * u;
            const bool ok = s < S;
            const float *r = base + static_cast<size_t>(ok ? s : 0) * ps;
            mv[u] = ok ? r[j] : -INFINITY;
            lv[u] = ok ? r[G + j] : 0.0f;
            av[u] = ok ? r[2 * G + j * HD + blk * 32 + lane] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool live = mv[u] != -INFINITY;
            const float w = live ? exp2f(mv[u] - M) : 0.0f;
            Ls = fmaf(w, live ? lv[u] : 0.0f, Ls);
            acc = fmaf(w, live ? av[u] : 0.0f, acc);
        }
    }
    ared[warp][lane] = acc;
    if (lane == 0) lred[warp] = Ls;
    __syncthreads();
    if (warp == 0) {
        float t = 0.0f, L = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            t += ared[w][lane];
            L += lred[w];
        }
        const float o = __fdiv_rn(t, L);
        a.out[(static_cast<size_t>(b) * a.H + h) * HD + blk * 32 + lane] = o;
        if (a.out_q8) {
            uint32_t dbits;
            float dq;
            const int q = q8_code(o, dbits, dq);
            uint8_t *qb = a.out_q8 + ((static_cast<size_t>(b) * a.H + h) * (HD / 32) + blk) * Q8B;
            qb[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
            if (lane == 0) {
                qb[0] = static_cast<uint8_t>(dbits & 0xFF);
                qb[1] = static_cast<uint8_t>(dbits >> 8);
            }
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
    const int nsm = device_info().num_sms;  // one CTA per SM
    int S = (nsm + B * KV - 1) / (B * KV);
    const int tiles = (max_tokens + AT_TILE - 1) / AT_TILE;
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
    cudaError_t e = launch(fs, dim3(a.splits, a.KV, B), dim3(AT_THREADS), L.total, s, pdl_first, args1);
    if (e != cudaSuccess) return -5;
    void *args2[] = {&a};
    e = launch(reinterpret_cast<const void *>(k_attn_combine<DPL>), dim3(a.H, DPL, B), dim3(256), 0, s, pdl_combine,
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
