// Split-KV GQA decode attention kernels (attention_forward_decode_head_major_
// gqa_flash of the page "mega_fused_attention_decode_q5_0.c", STEP 7) and
// their host launcher, templated on head_dim / 32 (DPL) and on the query
// group size G.  Included by one translation unit per DPL.
//
//   k_attn_split    grid (S splits, KV heads, B sequences), one CTA per SM.
//                   One CTA owns rows [t0, t1) of one KV head and all G =
//                   H/KV query heads that read it ("GQA-packed": each cache
//                   row is read once per KV head).  A producer warp streams
//                   8-row K and V tiles into a shared-memory ring through
//                   the bulk-copy engine in stages of up to ~16 KB per
//                   operand (at_la stages in flight); six
//                   consumer warps take 8-row tiles round-robin, each with
//                   its own online softmax, and merge their states at the
//                   end.
//   k_attn_combine  grid (H, hd/32, B).  Log-sum-exp merge of the S partial
//                   records of one query head over one 32-wide slice of its
//                   dims (= one Q8_0 block): the fp32 output and the block.
//   k_attn_combine_w  the same merge for S <= 8, one warp per output block.
//
// Scores are kept in log2 units: s2 = (q.k) * log2(e)/sqrt(hd), weights
// exp2(s2 - m2), which equals exp(s - m) of the definition.
#pragma once

#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

constexpr int AT_TILE = 8;                           // cache rows per stage
constexpr int AT_RPL = AT_TILE / 4;                  // score rows per lane
constexpr int AT_CONSUMERS = 6;                      // consumer warps per CTA
constexpr int AT_THREADS = 32 * (AT_CONSUMERS + 1);  // + one producer warp
constexpr int GMAX = 8;                              // query heads per KV head

// The ring (192 KB) holds stages of RS rows of K and of V.  Long splits use
// the largest power-of-two RS with at most 16 KB per operand (one bulk copy
// of 16 KB for head_dim 32, 64, 128 and 256, 12 KB for 96).
// An SM's copy engine takes one bulk copy per few hundred cycles whatever its
// size, so 4 KB copies capped the stream near 3 TB/s while 16 KB copies
// reach the HBM peak.  Short splits (fewer than 8 such stages) keep 8-row
// stages, whose first tile arrives sooner.  Consumers always take 8-row
// tiles: stage k holds tiles TPS*k .. TPS*k + TPS - 1.  The slot count NSS
// makes TPS * NSS a multiple of AT_CONSUMERS: tile t goes to warp
// t % AT_CONSUMERS, so the warp that waits for a slot's phase p also consumed
// the slot's phase p - 1 and the parity wait can never pass on a stale phase.
constexpr int AT_RING_BYTES = 192 * 1024;
constexpr int AT_MAX_SLOTS = 48;
// Cache element types (KV_F32, KV_BF16, KV_FP8 of ck_internal.h); es =
// bytes per element.
__host__ __device__ constexpr int kv_es(int kt) { return kt == KV_F32 ? 4 : kt == KV_BF16 ? 2 : 1; }
// Stage heights: the largest power-of-two multiple of 8 rows (at most 128)
// with at most `bytes` per operand (tiles per stage a power of two: shifts,
// not divisions, in the consumer loop).  Large stages: 16 KB per operand;
// short splits: 8 rows of fp32, ~4 KB of bf16 or fp8 (16 or 32 rows at hd 128).
__host__ __device__ constexpr int at_rows_for(int hd, int es, int bytes) {
    return hd * es * 128 <= bytes ? 128 : hd * es * 64 <= bytes ? 64 : hd * es * 32 <= bytes ? 32
           : hd * es * 16 <= bytes ? 16 : 8;
}
__host__ __device__ constexpr int at_rs_big(int hd, int es = 4) { return at_rows_for(hd, es, 16384); }
// Ring geometry of the two stage heights (compile-time constants in each
// kernel instantiation: the consumer loop stays as lean as with fixed tiles).
__host__ __device__ constexpr int at_rs(int hd, bool big, int es = 4) {
    return big ? at_rs_big(hd, es) : es == 4 ? AT_TILE : at_rows_for(hd, es, 4096);
}
__host__ __device__ constexpr int at_ss_bytes(int hd, bool big, int es = 4) { return 2 * at_rs(hd, big, es) * hd * es; }
__host__ __device__ constexpr int at_nss_from(int hd, bool big, int n, int es = 4) {
    return n <= 1 ? 1
                  : ((at_rs(hd, big, es) / AT_TILE * n) % AT_CONSUMERS == 0 ? n : at_nss_from(hd, big, n - 1, es));
}
__host__ __device__ constexpr int at_nss(int hd, bool big, int es = 4) {
    return at_nss_from(hd, big,
                       AT_RING_BYTES / at_ss_bytes(hd, big, es) > AT_MAX_SLOTS ? AT_MAX_SLOTS
                                                                              : AT_RING_BYTES / at_ss_bytes(hd, big, es),
                       es);
}
// stages in flight: ~96 KB of large stages, ~80 KB of short-split stages
__host__ __device__ constexpr int at_la(int hd, bool big, int es = 4) {
    return ((big ? 96 : 80) * 1024) / at_ss_bytes(hd, big, es) < 1 ? 1
           : ((big ? 96 : 80) * 1024) / at_ss_bytes(hd, big, es) > at_nss(hd, big, es) - 1
               ? at_nss(hd, big, es) - 1
               : ((big ? 96 : 80) * 1024) / at_ss_bytes(hd, big, es);
}
// Large stages for splits of at least 8 of them.
__host__ __device__ inline bool at_big(int hd, int chunk_rows, int es = 4) { return chunk_rows >= 8 * at_rs_big(hd, es); }
static_assert(at_nss(32, true) >= 2 && at_nss(96, true) >= 2 && at_nss(128, true) >= 2 && at_nss(256, true) >= 2 &&
                  at_nss(32, false) >= 2 && at_nss(256, false) >= 2,
              "stage ring");
static_assert(at_rs(128, false) == AT_TILE && at_rs_big(128) == 32, "fp32 stage heights");
static_assert(at_nss(64, true, 2) >= 2 && at_nss(128, true, 2) >= 2 && at_nss(64, false, 2) >= 2 &&
                  at_nss(128, false, 2) >= 2 && at_nss(64, true, 1) >= 2 && at_nss(128, true, 1) >= 2 &&
                  at_nss(64, false, 1) >= 2 && at_nss(128, false, 1) >= 2,
              "stage ring (bf16, fp8)");

// Four (two) consecutive cache elements as fp32, exactly: bf16 by moving its
// bits into the high half of an fp32 word, E4M3 through the hardware
// conversion to fp16 pairs.
template <int KT>
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(two & 0xFFFFu)));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}
template <int KT>
__device__ __forceinline__ float4 kv_load4(const uint8_t *p) {
    if constexpr (KT == KV_F32) {
        return *reinterpret_cast<const float4 *>(p);
    } else if constexpr (KT == KV_BF16) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                           __uint_as_float(u.y & 0xFFFF0000u));
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        const float2 lo = e4m3x2_to_float2<KT>(u), hi = e4m3x2_to_float2<KT>(u >> 16);
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
}
template <int KT>
__device__ __forceinline__ float2 kv_load2(const uint8_t *p) {
    if constexpr (KT == KV_F32) {
        return *reinterpret_cast<const float2 *>(p);
    } else if constexpr (KT == KV_BF16) {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    } else {
        return e4m3x2_to_float2<KT>(*reinterpret_cast<const uint16_t *>(p));
    }
}

// P row stride (floats): G heads, each duplicated into a pair, padded so
// rows stay 16-byte aligned.
__host__ __device__ constexpr int at_prow(int G) { return 2 * ((G + 1) & ~1); }

struct AttnSmem {
    size_t off_full, off_empty, off_qbar, off_stage, off_q, off_p, off_alpha, off_ml, off_bt, total;
};
constexpr int AT_BT_CACHE = 1024;  // block-table entries of a split held in shared memory (paged caches)

__host__ __device__ inline AttnSmem attn_smem(int hd) {
    AttnSmem L;
    size_t o = 0;
    L.off_full = o;
    o += AT_MAX_SLOTS * 8;
    L.off_empty = o;
    o += AT_MAX_SLOTS * 8;
    L.off_qbar = o;
    o += 16;
    L.off_stage = o;
    o += AT_RING_BYTES;
    L.off_q = o;
    o += static_cast<size_t>(GMAX) * hd * 4;
    L.off_p = o;
    o += static_cast<size_t>(AT_CONSUMERS) * AT_TILE * at_prow(GMAX) * 4;
    L.off_alpha = o;
    o += static_cast<size_t>(AT_CONSUMERS) * GMAX * 4;
    L.off_ml = o;
    o += static_cast<size_t>(2) * AT_CONSUMERS * GMAX * 4;
    L.off_bt = o;
    o += static_cast<size_t>(AT_BT_CACHE) * 4;
    L.total = (o + 127) / 128 * 128;
    return L;
}

// Partial results: for (b, g, s) a record of G m's, G l's, G*hd acc's.
__host__ __device__ inline size_t part_stride(int G, int hd) { return static_cast<size_t>(G) * (hd + 2); }

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * AT_CONSUMERS) : "memory");
}

// Reduce-scatter of v[8][R] (8 head slots x R rows) over the 8 lanes that
// share a row-lane (xor 4, 2, 1): afterwards lane `slice` holds, in r[R],
// the full sums of head `slice` for its R rows.
template <int R>
__device__ __forceinline__ void reduce_scatter_heads(float (&v)[8][R], int slice, float (&r)[R]) {
    float w[4][R];
    const bool b2 = slice & 4, b1 = slice & 2, b0 = slice & 1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const float send = b2 ? v[j][k] : v[j + 4][k];
            const float keep = b2 ? v[j + 4][k] : v[j][k];
            w[j][k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    float x[2][R];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const float send = b1 ? w[j][k] : w[j + 2][k];
            const float keep = b1 ? w[j + 2][k] : w[j][k];
            x[j][k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const float send = b0 ? x[0][k] : x[1][k];
        const float keep = b0 ? x[1][k] : x[0][k];
        r[k] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
}

// One CTA per (split s, KV head g, sequence b).  GT >= G query heads are
// computed (heads G..GT-1 get a zero q and zero weight).
//
// Scores: lane = (slice = lane & 7, row-lane rl = lane >> 3).  A slice is
// the float4 chunks {slice + 8c} of a row (interleaved so the 8 slices hit
// 8 different bank groups); a lane accumulates 4 rows (rl + 4k) x GT heads
// over its slice with packed fp32x2 FMAs (even / odd dims), in two passes
// of 2 rows to bound registers; a reduce-scatter over the 8 slices leaves
// lane (slice = j, rl) with query head j's scores, and that lane owns head
// j's softmax state.
// PV: lane = dims; each row adds p_j * v to GT accumulators, two dims per
// packed FMA.
template <int DPL, int GT, bool BIG, int KT>
__global__ void __launch_bounds__(AT_THREADS, 1) k_attn_split(const AttnArgs a) {
    constexpr int ES = kv_es(KT);
    constexpr int HD = 32 * DPL;
    constexpr int HD4 = HD / 4;
    constexpr int VEC = (DPL % 4 == 0) ? 4 : ((DPL % 2 == 0) ? 2 : 1);
    constexpr int NV = DPL / VEC;
    constexpr int PR = at_prow(GT);
    extern __shared__ __align__(128) uint8_t smem[];
    const AttnSmem L = attn_smem(HD);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.off_full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + L.off_empty);
    uint64_t *qbar = reinterpret_cast<uint64_t *>(smem + L.off_qbar);
    uint8_t *stage = smem + L.off_stage;  // cache elements of ES bytes
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

    int T, T0 = 0;  // rows [T0, T) are attended
    if (a.block_tables) {  // paged cache: seq_lens[b] rows, the last `window` of them when window > 0
        T = a.seq_lens[b];
        if (T < 0 || T > a.max_blocks * a.block_size) {
            if (s == 0 && g == 0 && threadIdx.x == 0) flag_error(a.status, FLAG_RANGE);
            T = 0;  // nothing attended: empty records
        }
        if (a.window > 0 && T > a.window) T0 = T - a.window;
    } else if (a.d_pos) {
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
    const int chunk = a.chunk > 0 ? a.chunk : (T - T0 + S - 1) / S;
    const int t0 = T0 + s * chunk;
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
    const bool paged = a.block_tables != nullptr;
    const uint8_t *kc = reinterpret_cast<const uint8_t *>(a.k_caches ? a.k_caches[b] : a.k_cache) +
                        (paged ? 0 : static_cast<size_t>(g) * a.C * HD * ES);
    const uint8_t *vc = reinterpret_cast<const uint8_t *>(a.v_caches ? a.v_caches[b] : a.v_cache) +
                        (paged ? 0 : static_cast<size_t>(g) * a.C * HD * ES);
    // paged: this split's block-table entries (logical blocks lb0 ..) in shared memory
    int *bts = reinterpret_cast<int *>(smem + L.off_bt);
    const int bs = paged ? a.block_size : 1;
    const int lb0 = paged ? t0 / bs : 0;
    const int nbt = paged ? min((t1 - 1) / bs - lb0 + 1, AT_BT_CACHE) : 0;
    if (paged && warp == 0) {
        const int32_t *btr = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
        for (int i = lane; i < nbt; i += 32) bts[i] = btr[lb0 + i];
    }
    const int ntiles = (t1 - t0 + AT_TILE - 1) / AT_TILE;
    constexpr int RS = at_rs(HD, BIG, ES), TPS = RS / AT_TILE, NSS = at_nss(HD, BIG, ES), LA = at_la(HD, BIG, ES);

    if (threadIdx.x < NSS) {  // one barrier pair per thread: a serial loop costs ~0.5 us
        mbar_init(&full[threadIdx.x], 1);
        mbar_init(&empty[threadIdx.x], TPS);  // every tile of the stage releases it
    }
    if (threadIdx.x == AT_THREADS - 1) mbar_init(qbar, 1);
    fence_mbar_init();
    __syncthreads();
    pdl_trigger();

    if (warp == 0) {
        // ---- producer.  Rows before `fresh` are never written by the
        // preceding grid, so they stream before waiting on it; a super-stage
        // holding a row from `fresh` on (the row just stored, or a prefill
        // chunk's rows) waits first.  Super-stage k is issued once
        // super-stage k - LA has arrived and its slot is free.
        if (lane == 0) {
            const int fresh = a.fresh_chunk ? min(a.fresh_from, T - 1) : T - 1;
            const int nss = (t1 - t0 + RS - 1) / RS;
            for (int k = 0; k < nss; ++k) {
                const int sl = k % NSS;
                bool ok = true;
                if (k >= LA) ok = mbar_wait(&full[(k - LA) % NSS], ((k - LA) / NSS) & 1);
                if (ok && k >= NSS) ok = mbar_wait(&empty[sl], ((k / NSS) - 1) & 1);
                if (!ok) {
                    flag_error(a.status, FLAG_TIMEOUT);
                    break;
                }
                const int r = t0 + k * RS;
                const int n = min(RS, t1 - r);
                if (r + n > fresh) pdl_wait();
                uint8_t *dst = stage + static_cast<size_t>(sl) * 2 * RS * HD * ES;
                if (!paged) {
                    const uint32_t bytes = static_cast<uint32_t>(n) * HD * ES;
                    mbar_arrive_expect_tx(&full[sl], 2 * bytes);
                    bulk_g2s(dst, kc + static_cast<size_t>(r) * HD * ES, bytes, &full[sl]);
                    bulk_g2s(dst + RS * HD * ES, vc + static_cast<size_t>(r) * HD * ES, bytes, &full[sl]);
                } else {
                    // rows r .. r + n - 1 as runs inside physical blocks
                    // ([num_blocks][KV][block_size][hd]); an entry out of
                    // range is flagged and its rows are not copied
                    uint32_t total = 0;
                    for (int u = r; u < r + n;) {
                        const int lb = u / bs, o = u - lb * bs, m = min(r + n - u, bs - o);
                        const int pb = lb - lb0 < AT_BT_CACHE ? bts[lb - lb0]
                                                              : a.block_tables[static_cast<size_t>(b) * a.max_blocks + lb];
                        if (pb >= 0 && pb < a.num_blocks) total += static_cast<uint32_t>(m) * HD * ES;
                        u += m;
                    }
                    mbar_arrive_expect_tx(&full[sl], 2 * total);
                    for (int u = r; u < r + n;) {
                        const int lb = u / bs, o = u - lb * bs, m = min(r + n - u, bs - o);
                        const int pb = lb - lb0 < AT_BT_CACHE ? bts[lb - lb0]
                                                              : a.block_tables[static_cast<size_t>(b) * a.max_blocks + lb];
                        if (pb >= 0 && pb < a.num_blocks) {
                            const size_t src = ((static_cast<size_t>(pb) * a.KV + g) * bs + o) * HD * ES;
                            const size_t off = static_cast<size_t>(u - r) * HD * ES;
                            const uint32_t bytes = static_cast<uint32_t>(m) * HD * ES;
                            bulk_g2s(dst + off, kc + src, bytes, &full[sl]);
                            bulk_g2s(dst + RS * HD * ES + off, vc + src, bytes, &full[sl]);
                        } else {
                            flag_error(a.status, FLAG_RANGE);
                        }
                        u += m;
                    }
                }
            }
        }
        return;
    }

    // ---- consumers
    const int cw = warp - 1;
    const int ct = threadIdx.x - 32;
    float *Pw = reinterpret_cast<float *>(smem + L.off_p) + cw * AT_TILE * PR;  // [TILE][PR]
    float *alw = reinterpret_cast<float *>(smem + L.off_alpha) + cw * GMAX;
    float *mlw = reinterpret_cast<float *>(smem + L.off_ml);  // m[NC][GMAX], l[NC][GMAX]
    pdl_wait();  // q is the preceding grid's output
    if (ct == 0) {
        const uint32_t qbytes = static_cast<uint32_t>(G) * HD * 4;
        mbar_arrive_expect_tx(qbar, qbytes);
        bulk_g2s(qs, a.q + (static_cast<size_t>(b) * a.H + static_cast<size_t>(g) * G) * HD, qbytes, qbar);
    }
    for (int idx = G * HD + ct; idx < GT * HD; idx += 32 * AT_CONSUMERS) qs[idx] = 0.0f;
    if (!mbar_wait(qbar, 0)) flag_error(a.status, FLAG_TIMEOUT);
    consumers_sync();

    float scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
    if constexpr (KT == KV_FP8) scale2 *= a.k_scale;  // k = code * k_scale
    const float4 *q4 = reinterpret_cast<const float4 *>(qs);
    const int slice = lane & 7, rl = lane >> 3;
    float mrun = -INFINITY, lrun = 0.0f;  // head `slice`
    float2 acc[GT][DPL / 2 > 0 ? DPL / 2 : 1];
    float accs[GT][DPL % 2 ? DPL : 1];  // unpacked accumulators when DPL is odd
#pragma unroll
    for (int j = 0; j < GT; ++j) {
#pragma unroll
        for (int e = 0; e < (DPL / 2 > 0 ? DPL / 2 : 1); ++e) acc[j][e] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int e = 0; e < (DPL % 2 ? DPL : 1); ++e) accs[j][e] = 0.0f;
    }

    for (int t = cw; t < ntiles; t += AT_CONSUMERS) {
        const int k = t / TPS, st = k % NSS;
        if (!mbar_wait(&full[st], (k / NSS) & 1)) flag_error(a.status, FLAG_TIMEOUT);
        const uint8_t *Kt = stage + (static_cast<size_t>(st) * 2 * RS * HD + (t - k * TPS) * AT_TILE * HD) * ES;
        const uint8_t *Vt = Kt + RS * HD * ES;
        const int n = min(AT_TILE, t1 - (t0 + t * AT_TILE));

        // ---- scores, rows rl + 4k, in passes of k = {2p, 2p + 1}
        float my[AT_RPL];
#pragma unroll
        for (int pass = 0; pass < AT_RPL / 2; ++pass) {
            float2 sp[GT][2];
#pragma unroll
            for (int j = 0; j < GT; ++j)
#pragma unroll
                for (int k = 0; k < 2; ++k) sp[j][k] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int c = 0; c < DPL; ++c) {
                float4 kk[2];
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    kk[k] = kv_load4<KT>(Kt + ((rl + 4 * (2 * pass + k)) * HD + 4 * (slice + 8 * c)) * ES);
#pragma unroll
                for (int j = 0; j < GT; ++j) {
                    const float4 qv = q4[j * HD4 + slice + 8 * c];
                    const float2 qa = make_float2(qv.x, qv.y), qb = make_float2(qv.z, qv.w);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        sp[j][k] = __ffma2_rn(qa, make_float2(kk[k].x, kk[k].y), sp[j][k]);
                        sp[j][k] = __ffma2_rn(qb, make_float2(kk[k].z, kk[k].w), sp[j][k]);
                    }
                }
            }
            float v[8][2];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    v[j][k] = (j < GT) ? sp[j < GT ? j : 0][k].x + sp[j < GT ? j : 0][k].y : 0.0f;
            float r2[2];
            reduce_scatter_heads<2>(v, slice, r2);
            my[2 * pass] = r2[0];
            my[2 * pass + 1] = r2[1];
        }
        const bool live = slice < G;
#pragma unroll
        for (int k = 0; k < AT_RPL; ++k) my[k] = (live && rl + 4 * k < n) ? my[k] * scale2 : -INFINITY;
        float tmax = my[0];
#pragma unroll
        for (int k = 1; k < AT_RPL; ++k) tmax = fmaxf(tmax, my[k]);
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        const float mnew = fmaxf(mrun, tmax);
        const float alpha = (mrun == -INFINITY) ? 0.0f : exp2f(mrun - mnew);
        float psum = 0.0f;
#pragma unroll
        for (int k = 0; k < AT_RPL; ++k) {
            const float p = (my[k] == -INFINITY) ? 0.0f : exp2f(my[k] - mnew);
            if (2 * slice < PR) *reinterpret_cast<float2 *>(Pw + (rl + 4 * k) * PR + 2 * slice) = make_float2(p, p);
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 8);
        psum += __shfl_xor_sync(0xffffffffu, psum, 16);
        if (live) {
            lrun = lrun * alpha + psum;
            mrun = mnew;
        }
        if (rl == 0 && slice < GT) alw[slice] = live ? alpha : 0.0f;
        __syncwarp();

        // ---- acc = alpha * acc + P V
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            const float al = alw[j];
            if constexpr (DPL % 2 == 0) {
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) acc[j][e] = __fmul2_rn(acc[j][e], make_float2(al, al));
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e) accs[j][e] *= al;
            }
        }
        auto row = [&](int r) {
            float2 pp[GT];
#pragma unroll
            for (int j = 0; j < GT; j += 2) {
                const float4 t4 = *reinterpret_cast<const float4 *>(Pw + r * PR + 2 * j);
                pp[j] = make_float2(t4.x, t4.y);
                if (j + 1 < GT) pp[j + 1] = make_float2(t4.z, t4.w);
            }
            if constexpr (DPL % 2 == 0) {
                float2 vv[DPL / 2];
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    const uint8_t *src = Vt + (r * HD + VEC * (lane + 32 * u)) * ES;
                    if constexpr (VEC == 4) {
                        const float4 tv = kv_load4<KT>(src);
                        vv[2 * u] = make_float2(tv.x, tv.y);
                        vv[2 * u + 1] = make_float2(tv.z, tv.w);
                    } else {
                        vv[u] = kv_load2<KT>(src);
                    }
                }
#pragma unroll
                for (int j = 0; j < GT; ++j)
#pragma unroll
                    for (int e = 0; e < DPL / 2; ++e) acc[j][e] = __ffma2_rn(pp[j], vv[e], acc[j][e]);
            } else {
                float vv[DPL];
                static_assert(KT == KV_F32 || DPL % 2 == 0, "bf16 / fp8 caches: head_dim a multiple of 64");
#pragma unroll
                for (int u = 0; u < DPL; ++u) vv[u] = reinterpret_cast<const float *>(Vt)[r * HD + lane + 32 * u];
#pragma unroll
                for (int j = 0; j < GT; ++j)
#pragma unroll
                    for (int e = 0; e < DPL; ++e) accs[j][e] = fmaf(pp[j].x, vv[e], accs[j][e]);
            }
        };
        if (n == AT_TILE) {
#pragma unroll
            for (int r = 0; r < AT_TILE; ++r) row(r);
        } else {
            for (int r = 0; r < n; ++r) row(r);
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
    float *accw = reinterpret_cast<float *>(stage);  // [NC][G][HD]
#pragma unroll
    for (int j = 0; j < GT; ++j) {
        if (j < G) {
            float *dst = accw + (cw * G + j) * HD;
            if constexpr (DPL % 2 == 0) {
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    if constexpr (VEC == 4) {
                        *reinterpret_cast<float4 *>(dst + 4 * (lane + 32 * u)) =
                            make_float4(acc[j][2 * u].x, acc[j][2 * u].y, acc[j][2 * u + 1].x, acc[j][2 * u + 1].y);
                    } else {
                        *reinterpret_cast<float2 *>(dst + 2 * (lane + 32 * u)) = acc[j][u];
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e) dst[lane + 32 * e] = accs[j][e];
            }
        }
    }
    // each warp's weight exp2(m_w - M) per head once (the same values, in the
    // same order, as a per-element evaluation), the record's m and l
    float *scw = reinterpret_cast<float *>(smem + L.off_alpha);  // [NC][GMAX]
    if (ct < G) {
        const int j = ct;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < AT_CONSUMERS; ++w) M = fmaxf(M, mlw[w * GMAX + j]);
        float Ls = 0.0f;
#pragma unroll
        for (int w = 0; w < AT_CONSUMERS; ++w) {
            const float mw = mlw[w * GMAX + j];
            const float sc = (mw != -INFINITY) ? exp2f(mw - M) : 0.0f;
            scw[w * GMAX + j] = sc;
            if (mw != -INFINITY) Ls = fmaf(sc, mlw[(AT_CONSUMERS + w) * GMAX + j], Ls);
        }
        rec[j] = M;
        rec[G + j] = Ls;
    }
    consumers_sync();
    for (int idx = ct; idx < G * HD; idx += 32 * AT_CONSUMERS) {
        const int j = idx / HD;
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < AT_CONSUMERS; ++w) {
            if (mlw[w * GMAX + j] != -INFINITY) t = fmaf(scw[w * GMAX + j], accw[(w * G + j) * HD + (idx - j * HD)], t);
        }
        if constexpr (KT == KV_FP8) t *= a.v_scale;  // v = code * v_scale
        rec[2 * G + idx] = t;
    }
}

// Output block `blk` of query head h of sequence b: the fp32 values, and,
// when requested, the Q8_0 block and its copy in the packed row.
template <int HD>
__device__ __forceinline__ void combine_store(const AttnArgs &a, int b, int h, int blk, int lane, float o) {
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
        if (a.out_img) {  // the block in the tensor-core operand image: one value per lane, hi and lo
            const int bq = h * (HD / 32) + blk;
            __half hi, lo;
            if (!img_split(dq, q, hi, lo)) flag_error(a.status, FLAG_RANGE);
            uint8_t *o = a.out_img + img_code_off(a.img_groups, b, bq, lane >> 3) + (lane & 7) * 2;
            *reinterpret_cast<__half *>(o) = hi;
            *reinterpret_cast<__half *>(o + IMG_CODE_BYTES) = lo;
        }
        if (a.out_pack) {  // the same block in the packed row the O-projection copies
            const int nbo = a.H * (HD / 32), bq = h * (HD / 32) + blk;
            uint8_t *pk = a.out_pack + static_cast<size_t>(b) * xpack_bytes(nbo);
            pk[static_cast<size_t>(xq_chunk(bq, lane >> 4)) * 16 + (lane & 15)] =
                static_cast<uint8_t>(static_cast<int8_t>(q));
            const int sum = warp_isum(q);
            if (lane == 0) {
                reinterpret_cast<float *>(pk + static_cast<size_t>(xq_chunks(nbo)) * 16)[bq] = dq;
                reinterpret_cast<int *>(pk + static_cast<size_t>(xq_chunks(nbo)) * 16 + nbo * 4)[bq] = sum;
            }
        }
    }
}

// Merge of the S partial records of one query head, for one 32-wide slice of
// its dims (= one Q8_0 block of the output).  Each warp loads its splits'
// records in one round, merges them locally, then warp 0 merges the warps.
template <int DPL>
__global__ void __launch_bounds__(256) k_attn_combine(const AttnArgs a) {
    constexpr int HD = 32 * DPL;
    constexpr int NW = 8;
    constexpr int U = 8;  // splits per warp per round
    __shared__ float ared[NW][32];
    __shared__ float mred[NW], lred[NW];
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
    float Mw = -INFINITY, acc = 0.0f, Ls = 0.0f;
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
        float mloc = Mw;
#pragma unroll
        for (int u = 0; u < U; ++u) mloc = fmaxf(mloc, mv[u]);
        if (mloc != -INFINITY) {
            const float sc = (Mw == -INFINITY) ? 0.0f : exp2f(Mw - mloc);
            acc *= sc;
            Ls *= sc;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool live = mv[u] != -INFINITY;
                const float w = live ? exp2f(mv[u] - mloc) : 0.0f;
                Ls = fmaf(w, live ? lv[u] : 0.0f, Ls);
                acc = fmaf(w, live ? av[u] : 0.0f, acc);
            }
            Mw = mloc;
        }
    }
    ared[warp][lane] = acc;
    if (lane == 0) {
        mred[warp] = Mw;
        lred[warp] = Ls;
    }
    __syncthreads();
    if (warp == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mred[w]);
        float t = 0.0f, L = 0.0f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (mred[w] != -INFINITY) {
                const float sc = exp2f(mred[w] - M);
                t = fmaf(sc, ared[w][lane], t);
                L = fmaf(sc, lred[w], L);
            }
        }
        combine_store<HD>(a, b, h, blk, lane, L > 0.0f ? __fdiv_rn(t, L) : 0.0f);  // no rows attended: 0
    }
}

// Few splits (at most AT_COMB_WARP_MAX, the batched step's case): one warp
// per 32-wide output block merges all of its splits itself, in split order,
// with the arithmetic of the second merge level above.  A CTA is 8 warps =
// 8 consecutive blocks; grid ceil(B * H * hd/32 / 8).
constexpr int AT_COMB_WARP_MAX = 8;
template <int DPL>
__global__ void __launch_bounds__(256) k_attn_combine_w(const AttnArgs a, int B) {
    constexpr int HD = 32 * DPL;
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int blk = item % DPL, bh = item / DPL;
    const int h = bh % a.H, b = bh / a.H;
    if (b >= B) {
        pdl_wait();
        return;
    }
    if (a.d_pos) {
        const int pos = a.d_pos[b];
        if (pos < 0 || pos >= a.C) {
            pdl_wait();
            return;
        }
    }
    const int G = a.H / a.KV;
    const int g = h / G, j = h - g * G;
    const int S = a.splits;
    pdl_trigger();
    pdl_wait();
    const size_t ps = part_stride(G, HD);
    const float *base = a.part + (static_cast<size_t>(b) * a.KV + g) * S * ps;
    float mv[AT_COMB_WARP_MAX], lv[AT_COMB_WARP_MAX], av[AT_COMB_WARP_MAX];
#pragma unroll
    for (int s = 0; s < AT_COMB_WARP_MAX; ++s) {
        const bool ok = s < S;
        const float *r = base + static_cast<size_t>(ok ? s : 0) * ps;
        mv[s] = ok ? r[j] : -INFINITY;
        lv[s] = ok ? r[G + j] : 0.0f;
        av[s] = ok ? r[2 * G + j * HD + blk * 32 + lane] : 0.0f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < AT_COMB_WARP_MAX; ++s) M = fmaxf(M, mv[s]);
    float t = 0.0f, L = 0.0f;
#pragma unroll
    for (int s = 0; s < AT_COMB_WARP_MAX; ++s) {
        if (mv[s] != -INFINITY) {
            const float sc = exp2f(mv[s] - M);
            t = fmaf(sc, av[s], t);
            L = fmaf(sc, lv[s], L);
        }
    }
    combine_store<HD>(a, b, h, blk, lane, L > 0.0f ? __fdiv_rn(t, L) : 0.0f);  // no rows attended: 0
}

template <int DPL, int GT, int KT>
static int launch_attn_gt(const AttnArgs &a0, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    AttnArgs a = a0;
    const AttnSmem L = attn_smem(32 * DPL);
    // stage height from the longest split (all splits of a launch share the plan)
    const int T = a.d_pos ? a.C : a.kv_tokens;
    const int chunk = a.chunk > 0 ? a.chunk : (T + a.splits - 1) / a.splits;
    const void *fs = at_big(32 * DPL, chunk, kv_es(KT))
                         ? reinterpret_cast<const void *>(k_attn_split<DPL, GT, true, KT>)
                         : reinterpret_cast<const void *>(k_attn_split<DPL, GT, false, KT>);
    ensure_smem(fs, L.total);
    void *args1[] = {&a};
    cudaError_t e = launch(fs, dim3(a.splits, a.KV, B), dim3(AT_THREADS), L.total, s, pdl_first, args1);
    if (e != cudaSuccess) return -5;
    if (a.splits <= AT_COMB_WARP_MAX) {
        void *args2[] = {&a, &B};
        const int items = B * a.H * DPL;
        e = launch(reinterpret_cast<const void *>(k_attn_combine_w<DPL>), dim3((items + 7) / 8), dim3(256), 0, s,
                   pdl_combine, args2);
    } else {
        void *args2[] = {&a};
        e = launch(reinterpret_cast<const void *>(k_attn_combine<DPL>), dim3(a.H, DPL, B), dim3(256), 0, s,
                   pdl_combine, args2);
    }
    return e == cudaSuccess ? 0 : -5;
}

// Query groups of 1, 2, 4, 7 and 8 heads run exact kernels; 3, 5 and 6 run
// in the next larger one with the extra heads masked.  KT: cache element type.
template <int DPL, int KT>
int launch_attention_dpl(const AttnArgs &a, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    switch (a.H / a.KV) {
        case 1: return launch_attn_gt<DPL, 1, KT>(a, B, s, pdl_first, pdl_combine);
        case 2: return launch_attn_gt<DPL, 2, KT>(a, B, s, pdl_first, pdl_combine);
        case 3:
        case 4: return launch_attn_gt<DPL, 4, KT>(a, B, s, pdl_first, pdl_combine);
        case 5:
        case 6:
        case 7: return launch_attn_gt<DPL, 7, KT>(a, B, s, pdl_first, pdl_combine);
        case 8: return launch_attn_gt<DPL, 8, KT>(a, B, s, pdl_first, pdl_combine);
        default: return -1;
    }
}

}  // namespace ck
