// Split-KV decode attention over bf16 / fp8 E4M3 caches with the scores on
// the 5th-generation tensor cores (head_dim 128, query groups up to 8).
//
// One CTA per (split, KV head, sequence), as the CUDA-core split kernel, and
// the same partial records (m in exp2 units, l, sum of p v), merged by the
// same combine.  A split's rows go in tiles of 128:
//   S^T = K Q^T   (M = 128 rows, N = 16 head slots, K = 128 dims): A = the K
//                 rows in TMEM (each row's lane; bf16 and E4M3 values are
//                 exact in bf16), B = q in shared memory as three bf16 parts
//                 q1 + q2 + q3 (24 significant bits); six independent
//                 accumulators (q part x half of the dims), summed by the rows
//   softmax       one thread per row
//   O^T += V^T P^T (M = 128 dims, N = 16 head slots, K = 128 rows): A = the
//                 tile's V transposed into TMEM (each dim's lane, exact bf16),
//                 B = p in shared memory as bf16 hi + lo parts
// Two groups of four row warps take alternate tiles, each with its own TMEM
// K, S, V^T and O^T buffers and its own softmax state (the four warps agree
// on a running maximum per head through a per-tile exchange; it is raised
// only when a tile's exceeds it by more than 2^8, exp2 units, and O^T and
// the row sums are then rescaled).  A group stores the K rows of its next
// tile as soon as it has read this tile's scores.  K and V rows come in
// separate rings: a slot is free once its rows are in TMEM.  The two groups'
// states merge once at the end.
// Warp roles: 0 copies (lane 0 K rows, lane 1 V rows; contiguous or as runs
// inside paged blocks), 1-8 rows (group (warp - 1) / 4), 9 the score MMAs
// (and TMEM), 10 the P V MMAs.  fp8 caches take P V in fp16 (E4M3 values
// and p's hi / lo parts are exact there), bf16 caches in bf16.
#include <cuda_bf16.h>

#include "ck_attn_kernels.cuh"

namespace ck {
namespace {

constexpr int TA_HD = 128;
constexpr int TA_M = 128;                   // rows per tile
constexpr int TA_N = 16;                    // head slots (MMA N)
constexpr int TA_RW = 8;                    // row warps (two groups of four)
constexpr int TA_THREADS = 32 * (TA_RW + 3);
constexpr int TA_QPART = TA_N * TA_HD * 2;  // one bf16 part of the q image
constexpr int TA_RING = 192 * 1024;         // K and V rings together
// TMEM columns per group gi: K rows (64 columns of bf16 pairs), the six
// partial score accumulators (16 columns each), V^T (64 columns of bf16
// pairs over the tile's rows) and O^T (16 columns)
constexpr int TA_NACC = 6;
constexpr int TA_TMEM_COLS = 512;
constexpr int TC_K = 0, TC_S = 2 * (TA_HD / 2), TC_V = TC_S + 2 * TA_NACC * TA_N, TC_O = TC_V + 2 * (TA_M / 2);
static_assert(TC_O + 2 * TA_N <= TA_TMEM_COLS, "TMEM columns");
constexpr int TA_PPART = TA_N * TA_M * 2;  // one bf16 part of p^T [16 head slots][128 rows]
constexpr float TA_TAU = 8.0f;

template <int KT>
struct TaGeom {
    static constexpr int ES = kv_es(KT);
    static constexpr int ROW = TA_HD * ES;   // bytes of one K (or V) row
    static constexpr int SLOT = TA_M * ROW;  // one tile of K (or V) rows
    static constexpr int NST = TA_RING / (2 * SLOT) > 8 ? 8 : TA_RING / (2 * SLOT);
};

constexpr size_t TA_OFF_RING = 0;                           // K slots, then V slots
constexpr size_t TA_OFF_Q = TA_OFF_RING + TA_RING;
constexpr size_t TA_OFF_P = TA_OFF_Q + 3 * TA_QPART;  // p^T [2 groups][hi, lo][16][128] bf16
// exchange of warp maxima [2 groups][2 tiles][4 warps][8], then the merge:
// l [2 groups][4 warps][8], m [2][8], weights [2][8]
constexpr size_t TA_OFF_RED = TA_OFF_P + 2 * 2 * TA_PPART;
constexpr size_t TA_OFF_BAR = TA_OFF_RED + (2 * 2 * 4 * 8 + 2 * 4 * 8 + 2 * 8 + 2 * 8) * 4;
constexpr size_t TA_OFF_TMEM = TA_OFF_BAR + 64 * 8;
constexpr size_t TA_OFF_BT = TA_OFF_TMEM + 16;  // paged: the split's block-table entries
constexpr size_t TA_SMEM = TA_OFF_BT + static_cast<size_t>(AT_BT_CACHE) * 4;
static_assert(TA_SMEM <= 227 * 1024, "shared memory");
static_assert(2 * 8 * TA_HD * 4 <= TA_RING, "group partials fit the rings");

__device__ __forceinline__ void ta_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void ta_st16(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// Shared-memory descriptor, no swizzle: leading byte offset 128 (next core
// matrix along K), stride byte offset `sbo` (next 8-row group).
__device__ __forceinline__ uint64_t ta_desc(uint32_t saddr, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128u >> 4) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
           (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// Eight 16-byte units of a row (128 bytes at `src`), loaded in the order
// rot, rot + 1, ... (mod 8) so that the eight lanes of a quarter warp, whose
// rows lie a multiple of 128 bytes apart, hit eight different bank groups;
// then put back in order by a three-stage rotation (selects, no dynamic
// register indexing): u[k] = unit k.
__device__ __forceinline__ void load_units_rotated(const uint8_t *src, int rot, uint4 (&u)[8]) {
    uint4 t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = *reinterpret_cast<const uint4 *>(src + 16 * ((k + rot) & 7));
    // t[k] = unit (k + rot) mod 8; rotate right by rot: u[k] = t[(k - rot) mod 8]
#pragma unroll
    for (int b = 1; b < 8; b <<= 1) {
        const bool on = rot & b;
        uint4 n[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 x = t[(k - b) & 7], y = t[k];
            n[k] = make_uint4(on ? x.x : y.x, on ? x.y : y.y, on ? x.z : y.z, on ? x.w : y.w);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = n[k];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) u[k] = t[k];
}

// 16 E4M3 codes -> 8 words of bf16 pairs (E4M3 -> f16 -> f32 -> bf16, exact).
__device__ __forceinline__ void e4m3_unit_words(const uint4 raw, uint32_t *w) {
    const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = e4m3x2_to_float2<KV_FP8>(in[i] & 0xFFFFu);
        const float2 b = e4m3x2_to_float2<KV_FP8>(in[i] >> 16);
        w[2 * i] = bf16x2_bits(a.x, a.y);
        w[2 * i + 1] = bf16x2_bits(b.x, b.y);
    }
}

template <int KT, int GT>
__global__ void __launch_bounds__(TA_THREADS, 1) k_attn_tc(const AttnArgs a) {
    using Geo = TaGeom<KT>;
    constexpr int ROW = Geo::ROW, NST = Geo::NST;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *kring = smem + TA_OFF_RING;
    uint8_t *vring = kring + static_cast<size_t>(NST) * Geo::SLOT;
    uint8_t *qimg = smem + TA_OFF_Q;
    float *red = reinterpret_cast<float *>(smem + TA_OFF_RED);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + TA_OFF_BAR);
    uint64_t *kfull = bars, *kempty = bars + NST, *vfull = bars + 2 * NST, *vempty = bars + 3 * NST;
    uint64_t *kready = bars + 4 * NST, *sfull = kready + 2, *pvready = sfull + 2, *ofull = pvready + 2;
    uint64_t *xch = ofull + 2, *qready = xch + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TA_OFF_TMEM);
    int *bts = reinterpret_cast<int *>(smem + TA_OFF_BT);

    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int S = gridDim.x;
    const int G = a.H / a.KV;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // rows [T0, T) attended; the split's share [t0, t1)
    int T, T0 = 0;
    bool bad = false;
    if (a.block_tables) {
        T = a.seq_lens[b];
        if (T < 0 || T > a.max_blocks * a.block_size) {
            bad = true;
            T = 0;
        }
        if (a.window > 0 && T > a.window) T0 = T - a.window;
    } else if (a.d_pos) {
        const int pos = a.d_pos[b];
        if (pos < 0 || pos >= a.C) {
            bad = true;
            T = 0;
        } else {
            T = pos + 1;
        }
    } else {
        T = a.kv_tokens;
    }
    if (bad && s == 0 && g == 0 && threadIdx.x == 0) flag_error(a.status, FLAG_RANGE);
    const int chunk = a.chunk > 0 ? a.chunk : (T - T0 + S - 1) / S;
    const int t0 = T0 + s * chunk;
    const int t1 = min(T, t0 + chunk);
    float *rec = a.part + ((static_cast<size_t>(b) * a.KV + g) * S + s) * part_stride(G, TA_HD);
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
                        (paged ? 0 : static_cast<size_t>(g) * a.C * ROW);
    const uint8_t *vc = reinterpret_cast<const uint8_t *>(a.v_caches ? a.v_caches[b] : a.v_cache) +
                        (paged ? 0 : static_cast<size_t>(g) * a.C * ROW);
    const int bs = paged ? a.block_size : 1;
    const int lb0 = paged ? t0 / bs : 0;
    const int nbt = paged ? min((t1 - 1) / bs - lb0 + 1, AT_BT_CACHE) : 0;
    if (paged && warp == 0) {
        const int32_t *btr = a.block_tables + static_cast<size_t>(b) * a.max_blocks;
        for (int i = lane; i < nbt; i += 32) bts[i] = btr[lb0 + i];
    }
    const int ntiles = (t1 - t0 + TA_M - 1) / TA_M;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(kfull + i, 1);
            mbar_init(kempty + i, 4);
            mbar_init(vfull + i, 1);
            mbar_init(vempty + i, 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(kready + i, 4);
            mbar_init(sfull + i, 1);
            mbar_init(pvready + i, 4);
            mbar_init(ofull + i, 1);
            mbar_init(xch + i, 4);
        }
        mbar_init(qready, 4);
        fence_mbar_init();
    }
    if (warp == TA_RW + 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sptr(tmem_slot)),
                     "r"(TA_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_trigger();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *tmem_slot;

    if (warp == 0) {
        // ---- copies: lane 0 the K rows of tile k into K slot k % NST, lane 1
        // the V rows into V slot k % NST.  Rows before `fresh` are never
        // written by the preceding grid and stream before waiting on it.
        if (lane < 2) {
            const bool isv = lane == 1;
            const uint8_t *cache = isv ? vc : kc;
            uint8_t *ring = isv ? vring : kring;
            uint64_t *fullb = isv ? vfull : kfull, *emptyb = isv ? vempty : kempty;
            const int fresh = a.fresh_chunk ? min(a.fresh_from, T - 1) : T - 1;
            bool waited = false;
            for (int k = 0; k < ntiles; ++k) {
                const int sl = k % NST;
                if (k >= NST && !mbar_wait(emptyb + sl, ((k / NST) - 1) & 1)) {
                    flag_error(a.status, FLAG_TIMEOUT);
                    break;
                }
                const int r = t0 + k * TA_M;
                const int n = min(TA_M, t1 - r);
                if (!waited && r + n > fresh) {
                    pdl_wait();
                    waited = true;
                }
                uint8_t *dst = ring + static_cast<size_t>(sl) * Geo::SLOT;
                if (!paged) {
                    const uint32_t bytes = static_cast<uint32_t>(n) * ROW;
                    mbar_arrive_expect_tx(fullb + sl, bytes);
                    bulk_g2s(dst, cache + static_cast<size_t>(r) * ROW, bytes, fullb + sl);
                } else {
                    // runs inside physical blocks [num_blocks][KV][block_size][hd];
                    // an entry out of range is flagged and its rows not copied
                    uint32_t total = 0;
                    for (int u = r; u < r + n;) {
                        const int lb = u / bs, o = u - lb * bs, m = min(r + n - u, bs - o);
                        const int pb = lb - lb0 < AT_BT_CACHE
                                           ? bts[lb - lb0]
                                           : a.block_tables[static_cast<size_t>(b) * a.max_blocks + lb];
                        if (pb >= 0 && pb < a.num_blocks) total += static_cast<uint32_t>(m) * ROW;
                        u += m;
                    }
                    mbar_arrive_expect_tx(fullb + sl, total);
                    for (int u = r; u < r + n;) {
                        const int lb = u / bs, o = u - lb * bs, m = min(r + n - u, bs - o);
                        const int pb = lb - lb0 < AT_BT_CACHE
                                           ? bts[lb - lb0]
                                           : a.block_tables[static_cast<size_t>(b) * a.max_blocks + lb];
                        if (pb >= 0 && pb < a.num_blocks) {
                            const size_t src = ((static_cast<size_t>(pb) * a.KV + g) * bs + o) * ROW;
                            bulk_g2s(dst + static_cast<size_t>(u - r) * ROW, cache + src,
                                     static_cast<uint32_t>(m) * ROW, fullb + sl);
                        } else if (!isv) {
                            flag_error(a.status, FLAG_RANGE);
                        }
                        u += m;
                    }
                }
            }
            if (!waited) pdl_wait();
        }
        __syncwarp();
    } else if (warp >= TA_RW + 1) {
        // ---- MMA issue: warp 9 the scores of tiles 0, 1, ... (S(k) once the
        // K rows of tile k are in TMEM), warp 10 the P V of tiles 0, 1, ...
        // (once a tile's p and V^T are ready).  Each commits on its own
        // barriers, so neither waits for the other's progress.
        if (lane == 0) {
            constexpr uint32_t IDS = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(TA_N >> 3) << 17) |
                                     (static_cast<uint32_t>(TA_M >> 4) << 24);
            const uint64_t qd = ta_desc(sptr(qimg), TA_HD * 16);
            const uint64_t pd0 = ta_desc(sptr(smem + TA_OFF_P), TA_M * 16);
            auto issue_s = [&](int k) -> bool {
                const int gi = k & 1;
                if (!mbar_wait(kready + gi, (k >> 1) & 1)) return false;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int kq = 0; kq < TA_HD / 32; ++kq)  // k step within a half of the dims
#pragma unroll
                    for (int part = 0; part < 3; ++part)
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int ks = half * (TA_HD / 32) + kq;
                            const uint32_t at = taddr + TC_K + gi * (TA_HD / 2) + ks * 8;
                            const uint64_t bd = qd + part * (TA_QPART / 16) + ks * 16;
                            const uint32_t dcol = taddr + TC_S + (gi * TA_NACC + 2 * part + half) * TA_N;
                            const uint32_t acc = kq > 0 ? 1u : 0u;
                            asm volatile(
                                "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(dcol),
                                "r"(at), "l"(bd), "r"(IDS), "r"(acc)
                                : "memory");
                        }
                asm volatile(
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sptr(sfull + gi))
                    : "memory");
                return true;
            };
            auto issue_pv = [&](int k) -> bool {
                constexpr uint32_t IDO = KT == KV_FP8 ? ((1u << 4) | (static_cast<uint32_t>(TA_N >> 3) << 17) |
                                                          (static_cast<uint32_t>(TA_M >> 4) << 24))
                                                       : IDS;
                const int gi = k & 1;
                if (!mbar_wait(pvready + gi, (k >> 1) & 1)) return false;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint64_t pd = pd0 + gi * (2 * TA_PPART / 16);
#pragma unroll
                for (int ks = 0; ks < TA_M / 16; ++ks)
#pragma unroll
                    for (int part = 0; part < 2; ++part) {  // p hi, p lo (V^T exact)
                        const uint32_t at = taddr + TC_V + gi * (TA_M / 2) + ks * 8;
                        const uint64_t bd = pd + part * (TA_PPART / 16) + ks * 16;
                        const uint32_t acc = (k >= 2 || ks > 0 || part > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
                                taddr + TC_O + gi * TA_N),
                            "r"(at), "l"(bd), "r"(IDO), "r"(acc)
                            : "memory");
                    }
                asm volatile(
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sptr(ofull + gi))
                    : "memory");
                return true;
            };
            bool ok = true;
            if (warp == TA_RW + 1) {
                ok = mbar_wait(qready, 0);
                for (int k = 0; k < ntiles && ok; ++k) ok = issue_s(k);
            } else {
                for (int k = 0; k < ntiles && ok; ++k) ok = issue_pv(k);
            }
            if (!ok) flag_error(a.status, FLAG_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ---- rows: group gi takes tiles gi, gi + 2, ...; thread r = tile row = TMEM lane
        const int rw = warp - 1, gi = rw >> 2, wq = warp & 3, r = 32 * wq + lane;
        const uint32_t lanes = taddr + (static_cast<uint32_t>(32 * wq) << 16);
        pdl_wait();  // q is the preceding grid's output
        if (gi == 0) {  // q of the group as three bf16 parts [16 head slots][128 dims], K-major core matrices
            const int h = r >> 3, d0 = (r & 7) * 16;
            const float *qrow = a.q + (static_cast<size_t>(b) * a.H + static_cast<size_t>(g) * G + h) * TA_HD + d0;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = h < G ? qrow[i] : 0.0f;
            uint32_t w1[8], w2[8], w3[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float e[2][3];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float v = x[2 * i + u];
                    const float v1 = __bfloat162float(__float2bfloat16_rn(v));
                    const float r1 = v - v1;
                    const float v2 = __bfloat162float(__float2bfloat16_rn(r1));
                    e[u][0] = v1, e[u][1] = v2, e[u][2] = r1 - v2;
                }
                w1[i] = bf16x2_bits(e[0][0], e[1][0]);
                w2[i] = bf16x2_bits(e[0][1], e[1][1]);
                w3[i] = bf16x2_bits(e[0][2], e[1][2]);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {  // dims d0 + 8c .. + 7
                const int off = (h >> 3) * (TA_HD * 16) + ((d0 >> 3) + c) * 128 + (h & 7) * 16;
                *reinterpret_cast<uint4 *>(qimg + off) = make_uint4(w1[4 * c], w1[4 * c + 1], w1[4 * c + 2], w1[4 * c + 3]);
                *reinterpret_cast<uint4 *>(qimg + TA_QPART + off) =
                    make_uint4(w2[4 * c], w2[4 * c + 1], w2[4 * c + 2], w2[4 * c + 3]);
                *reinterpret_cast<uint4 *>(qimg + 2 * TA_QPART + off) =
                    make_uint4(w3[4 * c], w3[4 * c + 1], w3[4 * c + 2], w3[4 * c + 3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(qready);
        }

        float scale2 = 1.4426950408889634f / sqrtf(static_cast<float>(TA_HD));
        if constexpr (KT == KV_FP8) scale2 *= a.k_scale;
        const int rot = lane & 7;
        // K rows of tile k (K slot k % NST) into this group's TMEM K buffer
        auto store_k = [&](int k) -> bool {
            const int sl = k % NST;
            if (!__all_sync(0xffffffffu, mbar_wait(kfull + sl, (k / NST) & 1))) return false;
            const int n = min(TA_M, t1 - (t0 + k * TA_M));
            const uint8_t *krow = kring + static_cast<size_t>(sl) * Geo::SLOT + static_cast<size_t>(r) * ROW;
            const uint32_t kb = lanes + TC_K + gi * (TA_HD / 2);
            constexpr int NW = KT == KV_BF16 ? 32 : 64;  // words of bf16 pairs per 128-byte piece
#pragma unroll
            for (int h = 0; h < ROW / 128; ++h) {  // 128-byte pieces of the row
                uint32_t w[NW];
                if (r < n) {
                    uint4 u[8];
                    load_units_rotated(krow + 128 * h, rot, u);
                    if constexpr (KT == KV_BF16) {
#pragma unroll
                        for (int k2 = 0; k2 < 8; ++k2) {
                            w[4 * k2] = u[k2].x, w[4 * k2 + 1] = u[k2].y, w[4 * k2 + 2] = u[k2].z,
                                   w[4 * k2 + 3] = u[k2].w;
                        }
                    } else {
#pragma unroll
                        for (int k2 = 0; k2 < 8; ++k2) e4m3_unit_words(u[k2], w + 8 * k2);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NW; ++i) w[i] = 0u;
                }
                // a piece is 64 bf16 dims (32 columns) or 128 E4M3 dims (64 columns)
#pragma unroll
                for (int c = 0; c < NW / 16; ++c) ta_st16(kb + 32 * h + 16 * c, w + 16 * c);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(kempty + sl);
                mbar_arrive(kready + gi);
            }
            return true;
        };

        uint8_t *pt = smem + TA_OFF_P + static_cast<size_t>(gi) * 2 * TA_PPART;  // p^T hi, lo of this group
        float *xr = red;                                   // [2 groups][2 tiles][4 warps][8]
        float *lr = red + 2 * 2 * 4 * 8;                   // [2 groups][4 warps][8]
        float *mg = lr + 2 * 4 * 8, *wg = mg + 2 * 8;      // [2 groups][8]
        for (int i = r; i < 2 * TA_PPART / 4; i += 128) reinterpret_cast<uint32_t *>(pt)[i] = 0u;  // head slots >= GT stay 0
        asm volatile("bar.sync 3, 256;" ::: "memory");
        float m[GT], lp[GT], al[GT];
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            m[j] = -INFINITY;
            lp[j] = 0.0f;
        }
        bool ok = gi < ntiles ? store_k(gi) : true;
        int j2 = 0;
        for (int k = gi; k < ntiles && ok; k += 2, ++j2) {
            const int sl = k % NST;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(sfull + gi, j2 & 1)))) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int n = min(TA_M, t1 - (t0 + k * TA_M));
            float sc[GT];
            {
                uint32_t v[TA_NACC][16];
#pragma unroll
                for (int u = 0; u < TA_NACC; ++u) ta_ld16(lanes + TC_S + (gi * TA_NACC + u) * TA_N, v[u]);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < GT; ++j) {
                    const float dot = ((__uint_as_float(v[0][j]) + __uint_as_float(v[1][j])) +
                                       (__uint_as_float(v[2][j]) + __uint_as_float(v[3][j]))) +
                                      (__uint_as_float(v[4][j]) + __uint_as_float(v[5][j]));
                    sc[j] = (r < n && j < G) ? dot * scale2 : -INFINITY;
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            // this tile's scores are in registers: the next tile's K rows may
            // replace the K buffer (its MMAs also overwrite the S buffer)
            if (k + 2 < ntiles && !(ok = store_k(k + 2))) break;
            // the tile maximum of each head over the group's 128 rows
            float *xw = xr + ((gi * 2 + (j2 & 1)) * 4) * 8;
#pragma unroll
            for (int j = 0; j < GT; ++j) {
                const float wm = warp_max(sc[j]);
                if (lane == 0) xw[wq * 8 + j] = wm;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xch + gi);
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(xch + gi, j2 & 1)))) break;
            bool rescale = false;
#pragma unroll
            for (int j = 0; j < GT; ++j) {
                const float tm = fmaxf(fmaxf(xw[j], xw[8 + j]), fmaxf(xw[16 + j], xw[24 + j]));
                al[j] = 1.0f;
                if (tm > m[j] + TA_TAU) {  // the same decision in every thread of the group
                    al[j] = exp2f(m[j] - tm);
                    m[j] = tm;
                    rescale = j2 > 0;
                }
                const float pj = sc[j] == -INFINITY ? 0.0f : exp2f(sc[j] - m[j]);
                lp[j] = lp[j] * al[j] + pj;
                sc[j] = pj;
            }
            // the group's previous P.V is done: O^T is stable, V^T and p^T are free
            if (j2 > 0) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(ofull + gi, (j2 - 1) & 1)))) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            }
            if (rescale) {  // uniform in the group; this thread's lane = dim r of O^T
                uint32_t v[16];
                ta_ld16(lanes + TC_O + gi * TA_N, v);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                for (int j = 0; j < GT; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * al[j]);
                ta_st16(lanes + TC_O + gi * TA_N, v);
            }
            // V^T: this thread's lane takes dim r of the tile's rows (zeros past n)
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(vfull + sl, (k / NST) & 1)))) break;
            {
                const uint8_t *vt = vring + static_cast<size_t>(sl) * Geo::SLOT;
#pragma unroll
                for (int c = 0; c < TA_M / 32; ++c) {  // 32 rows = 16 columns per store
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int k0 = 32 * c + 2 * i;
                        if constexpr (KT == KV_BF16) {
                            const uint32_t lo = k0 < n ? *reinterpret_cast<const uint16_t *>(vt + (k0 * TA_HD + r) * 2) : 0u;
                            const uint32_t hi =
                                k0 + 1 < n ? *reinterpret_cast<const uint16_t *>(vt + ((k0 + 1) * TA_HD + r) * 2) : 0u;
                            w[i] = lo | (hi << 16);
                        } else {  // two E4M3 codes -> an exact f16 pair
                            const uint32_t lo = k0 < n ? vt[k0 * TA_HD + r] : 0u;
                            const uint32_t hi = k0 + 1 < n ? vt[(k0 + 1) * TA_HD + r] : 0u;
                            uint32_t h2;
                            asm("cvt.rn.f16x2.e4m3x2 %0, %1;"
                                : "=r"(h2)
                                : "h"(static_cast<unsigned short>(lo | (hi << 8))));
                            w[i] = h2;
                        }
                    }
                    ta_st16(lanes + TC_V + gi * (TA_M / 2) + 16 * c, w);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(vempty + sl);  // the V rows are in TMEM
            // p^T: row r's probabilities as hi and lo parts (bf16, or f16 for
            // fp8 caches; p <= 2^8 fits f16), K-major [head slot][row]
#pragma unroll
            for (int j = 0; j < GT; ++j) {
                const int off = (j >> 3) * (TA_M * 16) + (r >> 3) * 128 + (j & 7) * 16 + (r & 7) * 2;
                if constexpr (KT == KV_FP8) {
                    const __half ph = __float2half_rn(sc[j]);
                    *reinterpret_cast<__half *>(pt + off) = ph;
                    *reinterpret_cast<__half *>(pt + TA_PPART + off) = __float2half_rn(sc[j] - __half2float(ph));
                } else {
                    const __nv_bfloat16 ph = __float2bfloat16_rn(sc[j]);
                    *reinterpret_cast<__nv_bfloat16 *>(pt + off) = ph;
                    *reinterpret_cast<__nv_bfloat16 *>(pt + TA_PPART + off) =
                        __float2bfloat16_rn(sc[j] - __bfloat162float(ph));
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(pvready + gi);
        }
        const int ntile_g = ntiles > gi ? (ntiles - gi + 1) / 2 : 0;  // this group's tiles
        if (ok && ntile_g > 0) ok = __all_sync(0xffffffffu, mbar_wait(ofull + gi, (ntile_g - 1) & 1));
        if (!ok) flag_error(a.status, FLAG_TIMEOUT);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // ---- the split's record: the two groups' states merged with weights
        // exp2(m_g - M) per head.  After both groups have left their loops
        // the rings are idle (every copy consumed, every MMA done).
        asm volatile("bar.sync 3, 256;" ::: "memory");
        float *accg = reinterpret_cast<float *>(kring);  // [2 groups][8 heads][128 dims]
        {
            uint32_t v[16];
            ta_ld16(lanes + TC_O + gi * TA_N, v);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int j = 0; j < GT; ++j)
                accg[(gi * 8 + j) * TA_HD + r] = (ok && ntile_g > 0) ? __uint_as_float(v[j]) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < GT; ++j) {
            const float ls = warp_sum(lp[j]);
            if (lane == 0) lr[(gi * 4 + wq) * 8 + j] = ls;
        }
#pragma unroll
        for (int j = 0; j < GT; ++j)
            if (r == j) mg[gi * 8 + j] = ntile_g > 0 ? m[j] : -INFINITY;
        asm volatile("bar.sync 3, 256;" ::: "memory");
        const int ct = 128 * gi + r;
        if (ct < G) {
            const float M = fmaxf(mg[ct], mg[8 + ct]);
            float Ls = 0.0f;
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const float mv = mg[g2 * 8 + ct];
                const float sw = mv != -INFINITY ? exp2f(mv - M) : 0.0f;
                wg[g2 * 8 + ct] = sw;
                const float lsum = lr[(g2 * 4) * 8 + ct] + lr[(g2 * 4 + 1) * 8 + ct] + lr[(g2 * 4 + 2) * 8 + ct] +
                                   lr[(g2 * 4 + 3) * 8 + ct];
                Ls = fmaf(sw, lsum, Ls);
            }
            rec[ct] = M;
            rec[G + ct] = Ls;
        }
        asm volatile("bar.sync 3, 256;" ::: "memory");
        for (int idx = ct; idx < G * TA_HD; idx += 256) {
            const int jj = idx / TA_HD, d = idx - jj * TA_HD;
            float t = fmaf(wg[jj], accg[jj * TA_HD + d], wg[8 + jj] * accg[(8 + jj) * TA_HD + d]);
            if constexpr (KT == KV_FP8) t *= a.v_scale;
            rec[2 * G + idx] = t;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == TA_RW + 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TA_TMEM_COLS));
}

template <int KT, int GT>
int launch_tc_gt(const AttnArgs &a0, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    AttnArgs a = a0;
    const void *fs = reinterpret_cast<const void *>(k_attn_tc<KT, GT>);
    ensure_smem(fs, TA_SMEM);
    void *args1[] = {&a};
    cudaError_t e = launch(fs, dim3(a.splits, a.KV, B), dim3(TA_THREADS), TA_SMEM, s, pdl_first, args1);
    if (e != cudaSuccess) return -5;
    if (a.splits <= AT_COMB_WARP_MAX) {
        void *args2[] = {&a, &B};
        const int items = B * a.H * 4;
        e = launch(reinterpret_cast<const void *>(k_attn_combine_w<4>), dim3((items + 7) / 8), dim3(256), 0, s,
                   pdl_combine, args2);
    } else {
        void *args2[] = {&a};
        e = launch(reinterpret_cast<const void *>(k_attn_combine<4>), dim3(a.H, 4, B), dim3(256), 0, s, pdl_combine,
                   args2);
    }
    return e == cudaSuccess ? 0 : -5;
}

}  // namespace

bool attention_tc_ok(int kv_type, int H, int KV, int hd) {
    return (kv_type == KV_BF16 || kv_type == KV_FP8) && hd == TA_HD && H / KV <= 8;
}

int launch_attention_tc(const AttnArgs &a, int B, cudaStream_t s, bool pdl_first, bool pdl_combine) {
    const int G = a.H / a.KV;
    const bool f8 = a.kv_type == KV_FP8;
    if (G <= 1) return f8 ? launch_tc_gt<KV_FP8, 1>(a, B, s, pdl_first, pdl_combine)
                          : launch_tc_gt<KV_BF16, 1>(a, B, s, pdl_first, pdl_combine);
    if (G <= 2) return f8 ? launch_tc_gt<KV_FP8, 2>(a, B, s, pdl_first, pdl_combine)
                          : launch_tc_gt<KV_BF16, 2>(a, B, s, pdl_first, pdl_combine);
    if (G <= 4) return f8 ? launch_tc_gt<KV_FP8, 4>(a, B, s, pdl_first, pdl_combine)
                          : launch_tc_gt<KV_BF16, 4>(a, B, s, pdl_first, pdl_combine);
    return f8 ? launch_tc_gt<KV_FP8, 8>(a, B, s, pdl_first, pdl_combine)
              : launch_tc_gt<KV_BF16, 8>(a, B, s, pdl_first, pdl_combine);
}

}  // namespace ck
