// Batched projections on the 5th-generation tensor cores (tcgen05, kind::f16).
//
// For B activation rows sharing one weight matrix the projection
//   y[s][r] = sum_b d_w[r][b] * sum_i c[r][b][i] * (d_x[s][b] * q[s][b][i])
// is a dense contraction.  The weight codes c are exact in fp16 (Q5_0:
// q - 16 in [-16, 15]; Q8_0: [-127, 127]); each activation value d_x * q is
// held exactly as two fp16 parts (hi + lo) in an operand image written once
// per step; every product is exact in fp32.  The weight scale differs per
// row and per block, so every block of a stage gets its own TMEM accumulator
// (four MMAs: two 16-wide K steps x two parts), read back and folded in with
// acc = fmaf(block sum, d_w, acc) in block order.
//
// CTA = 128 weight rows (MMA M) x NT sequences (MMA N, up to 64: every
// weight row is converted once per 64 sequences) x a range of the K stages
// (4 blocks = 128 codes each).  A tile's K range is split over S CTAs so
// that the grid fills the GPU; the last CTA of a tile to finish sums the S
// partial tiles in split order (deterministic) and runs the epilogue.
//
// Warp roles, linked by mbarrier rings (full / empty) with no CTA-wide
// barrier in the main loop:
//   producers (8 warps)  one pair of a row's blocks per thread and stage:
//                        load (a stage ahead, in registers), decode into the
//                        fp16 A tile (K-major, no swizzle, 8-row x 16-byte
//                        core matrices) and the weight scales; 3 slots.
//   MMA warp (1)         TMEM allocation; bulk copies of the activation
//                        operand (hi and lo parts, written once per step in
//                        the MMA layout by the kernel that produced the
//                        activations; 3 slots); per stage 16 MMAs into 4 TMEM
//                        accumulators of NT columns (2 slots), one commit.
//   read-back (8 warps)  warp w: TMEM lanes 32 (w % 4).. (its rows), half the
//                        columns; acc += block sum * d_w, two lanes per
//                        packed fp32 instruction (each rounded as the scalar
//                        fmaf); then frees the stage's slots.
//
// The epilogue (bias, RoPE at each sequence's position, q / K / V stores, or
// bias + residual) is the one of the dp4a kernel.
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

constexpr int TP_M = 128;                 // weight rows per CTA
constexpr int TP_BPS = IMG_BPS;           // blocks per stage
constexpr int TP_KG = IMG_KG;             // 8-code groups per stage
constexpr uint32_t TP_SBO = TP_KG * 128;  // bytes between 8-row groups (A tiles and activation stages)
constexpr int TP_DWS = TP_M + 4;          // floats per block of the weight scales (bank spread)
constexpr int TP_MAX_SPLITS = 8;
static_assert(TP_SBO == IMG_RG_BYTES, "activation stages share the A tile's core-matrix layout");
// warp roles
constexpr int TW_CONS = 8;                     // read-back warps 0..7
constexpr int TW_PROD = 8;                     // conversion warps 8..15
constexpr int TW_MMA_WARP = TW_CONS + TW_PROD;  // warp 16: TMEM, bulk copies, MMAs
constexpr int TW_THREADS = 32 * (TW_MMA_WARP + 1);
// rings: stage slots (A tile + weight scales + activation stage), TMEM slots
constexpr int TW_NA = 3, TW_NTM = 2;
constexpr size_t TP_A_BYTES = static_cast<size_t>(TP_M) * TP_BPS * 32 * 2;  // 32 KB
constexpr size_t TP_DW_BYTES = static_cast<size_t>(TP_DWS) * TP_BPS * 4;

struct TpSmem {
    size_t a, b, dw, bar, tmem, ticket, total;
};
__host__ __device__ inline TpSmem tp_smem() {
    TpSmem L;
    size_t o = 0;
    L.a = o;  // TW_NA A tiles (later the sums [TP_M][NT + 1])
    o += TW_NA * TP_A_BYTES;
    L.b = o;  // TW_NA activation stages (hi and lo parts)
    o += static_cast<size_t>(TW_NA) * IMG_STAGE_BYTES;
    L.dw = o;  // TW_NA x dw[j][row]
    o += TW_NA * TP_DW_BYTES;
    L.bar = o;
    o += static_cast<size_t>(2 * TW_NA + 2 * TW_NTM) * 8;
    L.tmem = o;
    o += 16;
    L.ticket = o;
    o += 16;
    L.total = (o + 127) / 128 * 128;
    return L;
}

__device__ __forceinline__ uint64_t tp_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((128u >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((TP_SBO >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Four byte codes -> four fp16 values in two words: bytes u (unsigned) map to
// 1024 + u (0x64 as the high byte), then `bias` (1024 + offset) is subtracted.
__device__ __forceinline__ void codes_to_half(uint32_t c, __half2 bias, uint32_t &lo, uint32_t &hi) {
    const uint32_t a = __byte_perm(c, 0x64646464u, 0x5140);
    const uint32_t b = __byte_perm(c, 0x64646464u, 0x7362);
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// One 32-element block (8 words of byte codes, element order) of row r at
// stage block j into the A tile (core-matrix layout).
__device__ __forceinline__ void put_block(uint8_t *tile, int r, int j, const uint32_t (&c)[8], __half2 bias) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {  // 8 elements each
        uint4 v;
        codes_to_half(c[2 * g], bias, v.x, v.y);
        codes_to_half(c[2 * g + 1], bias, v.z, v.w);
        *reinterpret_cast<uint4 *>(tile + ((r >> 3) * TP_KG + 4 * j + g) * 128 + (r & 7) * 16) = v;
    }
}

// Two consecutive blocks of a row (Q5_0: 44 bytes, Q8_0: 68 bytes; 4-byte
// aligned) as raw words.
constexpr int TP_PAIR_WORDS = 17;
__device__ __forceinline__ void load_pair(const uint8_t *src, bool q8, uint32_t (&w)[TP_PAIR_WORDS]) {
    const uint32_t *p = reinterpret_cast<const uint32_t *>(src);
#pragma unroll
    for (int i = 0; i < TP_PAIR_WORDS; ++i) w[i] = (i < 11 || q8) ? __ldg(p + i) : 0u;
}

// Raw Q5_0 pair -> codes q in 0..31 per element and the two scales.
__device__ __forceinline__ void decode_q5_pair(const uint32_t (&w)[TP_PAIR_WORDS], uint32_t (&c0)[8], uint32_t (&c1)[8],
                                               float &d0, float &d1) {
    // block 0 at byte 0: d = w0 low half, qh = bytes 2..5, qs = bytes 6..21
    d0 = half_bits_to_float(w[0]);
    const uint32_t qh0 = __funnelshift_r(w[0], w[1], 16);
    // block 1 at byte 22: d = w5 high half, qh = w6, qs = w7..w10
    d1 = half_bits_to_float(w[5] >> 16);
    const uint32_t qh1 = w[6];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t qs0 = __funnelshift_r(w[1 + i], w[2 + i], 16);
        const uint32_t qs1 = w[7 + i];
        c0[i] = (qs0 & 0x0F0F0F0Fu) | ((((qh0 >> (4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u);
        c0[4 + i] = ((qs0 >> 4) & 0x0F0F0F0Fu) | ((((qh0 >> (16 + 4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u);
        c1[i] = (qs1 & 0x0F0F0F0Fu) | ((((qh1 >> (4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u);
        c1[4 + i] = ((qs1 >> 4) & 0x0F0F0F0Fu) | ((((qh1 >> (16 + 4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u);
    }
}

// Raw Q8_0 pair -> codes with the sign bit flipped (u = q + 128) and scales.
__device__ __forceinline__ void decode_q8_pair(const uint32_t (&w)[TP_PAIR_WORDS], uint32_t (&c0)[8], uint32_t (&c1)[8],
                                               float &d0, float &d1) {
    d0 = half_bits_to_float(w[0]);
    d1 = half_bits_to_float(w[8] >> 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        c0[i] = __funnelshift_r(w[i], w[i + 1], 16) ^ 0x80808080u;  // codes at bytes 2..33
        c1[i] = w[9 + i] ^ 0x80808080u;                             // codes at bytes 36..67
    }
}

// tcgen05.ld of 8 / 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t *v) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// Two fp32 lanes at once (each lane rounded as the scalar operation).
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    return static_cast<uint64_t>(lo) | (static_cast<uint64_t>(hi) << 32);
}

template <bool OPROJ, int NT>
__global__ void __launch_bounds__(TW_THREADS, 1) k_proj_tc(const BatchArgs a, int S) {
    static_assert(NT == 16 || NT == 32 || NT == 64, "MMA N");
    constexpr int TMEM_COLS = TW_NTM * TP_BPS * NT;  // 128, 256 or 512: a power of two
    constexpr int CW = NT / 2;                       // columns per consumer warp
    extern __shared__ __align__(1024) uint8_t smem[];
    const TpSmem L = tp_smem();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nb = OPROJ ? a.H * a.hd / QK : a.D / QK;
    const int nst = nb / TP_BPS;
    const int QD = a.H * a.hd, KD = a.KV * a.hd;
    const int tile = blockIdx.x, split = blockIdx.y, g = blockIdx.z;
    const int G = img_groups(a.B);
    const int R0 = tile * TP_M;  // first global row of the tile
    const int s0 = g * IMG_SEQ;  // first sequence
    const int k0 = static_cast<int>(static_cast<long long>(split) * nst / S);
    const int k1 = static_cast<int>(static_cast<long long>(split + 1) * nst / S);
    const int T = k1 - k0;  // >= 1: S <= nst
    // the tile's matrix (a tile never straddles Q / K / V)
    int kind = 4;  // 0 = Q, 1 = K, 2 = V, 4 = O
    const uint8_t *W = a.wo;
    int rbase = R0, mrows = a.D;
    if (!OPROJ) {
        if (R0 < QD) {
            kind = 0;
            W = a.wq;
            mrows = QD;
        } else if (R0 < QD + KD) {
            kind = 1;
            W = a.wk;
            rbase = R0 - QD;
            mrows = KD;
        } else {
            kind = 2;
            W = a.wv;
            rbase = R0 - QD - KD;
            mrows = KD;
        }
    }
    const bool wq8 = kind == 2;
    const int pb = wq8 ? 2 * Q8B : 2 * Q5B;  // bytes per pair of blocks
    const size_t rb = static_cast<size_t>(nb) * (wq8 ? Q8B : Q5B);
    const uint8_t *img = OPROJ ? a.aimg : a.ximg;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar);
    uint64_t *a_full = bars, *a_empty = bars + TW_NA;
    uint64_t *tm_full = bars + 2 * TW_NA, *tm_empty = tm_full + TW_NTM;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem);
    auto a_tile = [&](int i) { return smem + L.a + static_cast<size_t>(i) * TP_A_BYTES; };
    auto dw_of = [&](int i) { return reinterpret_cast<float *>(smem + L.dw + static_cast<size_t>(i) * TP_DW_BYTES); };
    auto b_stage = [&](int i) { return smem + L.b + static_cast<size_t>(i) * IMG_STAGE_BYTES; };

    // ---- setup: barriers, TMEM (the MMA warp), the producers' first loads
    if (tid == 0) {
        for (int i = 0; i < TW_NA; ++i) {
            mbar_init(a_full + i, TW_PROD);
            mbar_init(a_empty + i, TW_CONS);
        }
        for (int i = 0; i < TW_NTM; ++i) {
            mbar_init(tm_full + i, 1);
            mbar_init(tm_empty + i, TW_CONS);
        }
        fence_mbar_init();
    }
    if (warp == TW_MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sptr(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_trigger();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *tmem_slot;

    float *ep = reinterpret_cast<float *>(smem + L.a);  // [TP_M][NT + 1], after the main loop
    constexpr int EPS = NT + 1;
    // consumer warp w: TMEM lanes 32 (w % 4) .. + 31 (tile rows r), columns
    // c0 .. c0 + NT/2 - 1 (sequences)
    const int r = (warp & 3) * 32 + lane, c0 = (warp >> 2) * CW;
    uint64_t acc[CW / 2];  // pairs of fp32 sums
#pragma unroll
    for (int i = 0; i < CW / 2; ++i) acc[i] = 0;

    if (warp >= TW_CONS && warp < TW_CONS + TW_PROD) {
        // ---- producers: weight pairs -> fp16 A tiles and scales, up to
        // TW_NA stages ahead of the read-back
        const int pt = tid - 32 * TW_CONS, pw = pt >> 5;
        const int cr = 16 * pw + (lane & 7) + 8 * (lane >> 4), cp = (lane >> 3) & 1;
        const uint8_t *wrow = W + static_cast<size_t>(rbase + cr) * rb + static_cast<size_t>(cp) * pb;
        if (pt < TP_M) {  // this CTA's weight bytes into L2, one row each
            const size_t mend = static_cast<size_t>(mrows) * rb;
            size_t lo = static_cast<size_t>(rbase + pt) * rb + static_cast<size_t>(k0) * (TP_BPS / 2) * pb;
            size_t hi = lo + static_cast<size_t>(T) * (TP_BPS / 2) * pb;
            lo &= ~static_cast<size_t>(15);
            hi = (hi + 15) & ~static_cast<size_t>(15);
            if (hi > mend) hi = mend;
            if (hi > lo) prefetch_l2(W + lo, static_cast<uint32_t>(hi - lo));
        }
        const __half2 wbias = __half2half2(__float2half(wq8 ? 1152.0f : 1040.0f));
        auto decode = [&](int i, const uint32_t (&raw)[TP_PAIR_WORDS]) {
            uint32_t c0[8], c1[8];
            float d0, d1;
            if (wq8)
                decode_q8_pair(raw, c0, c1, d0, d1);
            else
                decode_q5_pair(raw, c0, c1, d0, d1);
            uint8_t *tile_a = a_tile(i);
            put_block(tile_a, cr, 2 * cp, c0, wbias);
            put_block(tile_a, cr, 2 * cp + 1, c1, wbias);
            float *dw = dw_of(i);
            dw[(2 * cp) * TP_DWS + cr] = d0;
            dw[(2 * cp + 1) * TP_DWS + cr] = d1;
        };
        // activation stage t (hi and lo parts of NT rows) into slot t % TW_NA:
        // 16-byte async copies, one commit group per stage
        constexpr int BCH = 2 * NT * (IMG_RG_BYTES / 8) / 16;  // 16-byte chunks
        auto copy_b = [&](int t) {
            const uint8_t *src = img + img_stage(G, k0 + t, g);
            uint8_t *dst = b_stage(t % TW_NA);
#pragma unroll
            for (int u = 0; u < BCH / (32 * TW_PROD); ++u) {
                const int c = pt + 32 * TW_PROD * u;
                const int part = c / (BCH / 2), off = (c % (BCH / 2)) * 16;
                cp_async16(dst + part * IMG_CODE_BYTES + off, src + part * IMG_CODE_BYTES + off);
            }
            cp_async_commit();
        };
        uint32_t rc[TP_PAIR_WORDS], rn[TP_PAIR_WORDS];
        load_pair(wrow + static_cast<size_t>(k0) * (TP_BPS / 2) * pb, wq8, rc);
        decode(0, rc);  // the first stage's weights before the wait on the preceding grid
        pdl_wait();     // the activation image is ready
        copy_b(0);
        for (int t = 0; t < T; ++t) {
            const int i = t % TW_NA;
            if (t + 3 < T) {  // three stages ahead into L1: the loads below then hit close by
                const uint8_t *pf = wrow + static_cast<size_t>(k0 + t + 3) * (TP_BPS / 2) * pb;
                prefetch_l1(pf);
                prefetch_l1(pf + 4 * TP_PAIR_WORDS - 1);
            }
            if (t + 1 < T) {
                load_pair(wrow + static_cast<size_t>(k0 + t + 1) * (TP_BPS / 2) * pb, wq8, rn);
                // slot (t + 1) % TW_NA is free once stage t + 1 - TW_NA is read back
                const int n1 = (t + 1) / TW_NA;
                if (n1 >= 1 && !mbar_wait(a_empty + (t + 1) % TW_NA, (n1 - 1) & 1)) flag_error(a.status, FLAG_TIMEOUT);
                copy_b(t + 1);
            }
            if (t > 0) decode(i, rc);
            // this stage's activation copies have landed (the next stage's may be in flight)
            if (t + 1 < T)
                cp_async_wait<1>();
            else
                cp_async_wait<0>();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full + i);
#pragma unroll
            for (int w = 0; w < TP_PAIR_WORDS; ++w) rc[w] = rn[w];
        }
    } else if (warp == TW_MMA_WARP) {
        // ---- MMA warp: the MMAs of each stage into its TMEM slot
        if (lane == 0) {
            const uint32_t idesc =
                (1u << 4) | (static_cast<uint32_t>(NT >> 3) << 17) | (static_cast<uint32_t>(TP_M >> 4) << 24);
            for (int t = 0; t < T; ++t) {
                const int ia = t % TW_NA, ib = ia, im = t % TW_NTM;
                bool ok = mbar_wait(a_full + ia, (t / TW_NA) & 1);
                if (t >= TW_NTM) ok = mbar_wait(tm_empty + im, (t / TW_NTM - 1) & 1) && ok;
                if (!ok) flag_error(a.status, FLAG_TIMEOUT);
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                // descriptors of the stage's tiles; a K step or the lo part is
                // an offset of the 16-byte-unit start address (shared memory
                // addresses stay below 256 KB: no carry out of its 14 bits)
                const uint64_t adesc = tp_desc(sptr(a_tile(ia))), bdesc = tp_desc(sptr(b_stage(ib)));
                const uint32_t dcol = taddr + im * TP_BPS * NT;
                // block j: codes x (hi + lo) over its two 16-wide K steps
#pragma unroll
                for (int j = 0; j < TP_BPS; ++j)
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int h = m >> 1, part = m & 1;
                        const uint64_t ad = adesc + static_cast<uint64_t>((4 * j + 2 * h) * 8);
                        const uint64_t bd = bdesc + static_cast<uint64_t>(part * (IMG_CODE_BYTES / 16) + (4 * j + 2 * h) * 8);
                        asm volatile(
                            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dcol + j * NT),
                            "l"(ad), "l"(bd), "r"(idesc), "r"(m)
                            : "memory");
                    }
                asm volatile(
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sptr(tm_full + im))
                    : "memory");
            }
        }
        __syncwarp();
    } else {
        // ---- consumers: fold each block's exact dots in with its two scales
        for (int t = 0; t < T; ++t) {
            const int ia = t % TW_NA, im = t % TW_NTM;
            // the stage's MMAs are done; the weight scales written by the
            // producers are acquired from their own barrier (whose next phase
            // needs this stage's release, so it is current)
            bool ok = mbar_wait(tm_full + im, (t / TW_NTM) & 1);
            ok = mbar_wait(a_full + ia, (t / TW_NA) & 1) && ok;
            if (!ok) flag_error(a.status, FLAG_TIMEOUT);
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const float *dw = dw_of(ia) + r;
            const uint32_t base = taddr + (static_cast<uint32_t>((warp & 3) * 32) << 16) + im * TP_BPS * NT + c0;
            // 8 columns per TMEM load, software-pipelined:
            // chunk c + 1 loads while chunk c is folded in
            constexpr int CH = 8;
            constexpr int NCH = TP_BPS * (CW / CH);  // chunks per stage
            auto ld_chunk = [&](int c, uint32_t *v) {
                const uint32_t at = base + (c / (CW / CH)) * NT + (c % (CW / CH)) * CH;
                if constexpr (CH == 16)
                    tmem_ld16(at, v);
                else
                    tmem_ld8(at, v);
            };
            uint32_t va[CH], vb[CH];
            ld_chunk(0, va);
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                uint32_t *cur = (c & 1) ? vb : va;
                uint32_t *nxt = (c & 1) ? va : vb;
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (c + 1 < NCH) ld_chunk(c + 1, nxt);
                const int j = c / (CW / CH), h = c % (CW / CH);
                const float dwv = dw[j * TP_DWS];
                const uint64_t dw2 = f2_pack(__float_as_uint(dwv), __float_as_uint(dwv));
#pragma unroll
                for (int p = 0; p < CH / 2; ++p)
                    acc[h * CH / 2 + p] = f2_fma(f2_pack(cur[2 * p], cur[2 * p + 1]), dw2, acc[h * CH / 2 + p]);
            }
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tm_empty + im);
                mbar_arrive(a_empty + ia);
            }
        }
    }
    // Every MMA has completed (the consumers saw the last one) and every A
    // tile has been read: the A tiles take the sums.
    pdl_wait();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == TW_MMA_WARP)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TMEM_COLS));
    if (S == 1) {
        if (warp < TW_CONS) {
#pragma unroll
            for (int p = 0; p < CW / 2; ++p) {
                ep[r * EPS + c0 + 2 * p] = __uint_as_float(static_cast<uint32_t>(acc[p]));
                ep[r * EPS + c0 + 2 * p + 1] = __uint_as_float(static_cast<uint32_t>(acc[p] >> 32));
            }
        }
    } else {
        // publish this split's tile [TP_M][NT] straight from the registers;
        // the last CTA of the tile sums all splits in split order
        float *part = a.proj_part + (static_cast<size_t>(tile) * G + g) * S * (TP_M * NT);
        if (warp < TW_CONS) {
            float4 *dst = reinterpret_cast<float4 *>(part + static_cast<size_t>(split) * (TP_M * NT) + r * NT + c0);
#pragma unroll
            for (int p = 0; p < CW / 4; ++p)
                dst[p] = make_float4(__uint_as_float(static_cast<uint32_t>(acc[2 * p])),
                                     __uint_as_float(static_cast<uint32_t>(acc[2 * p] >> 32)),
                                     __uint_as_float(static_cast<uint32_t>(acc[2 * p + 1])),
                                     __uint_as_float(static_cast<uint32_t>(acc[2 * p + 1] >> 32)));
        }
        __threadfence();
        __syncthreads();
        int *tk = reinterpret_cast<int *>(smem + L.ticket);
        if (tid == 0) *tk = atomicAdd(a.tickets + (OPROJ ? a.tickets_o : 0) + tile * G + g, 1);
        __syncthreads();
        if (*tk != S - 1) return;
        __threadfence();
        // TP_M * NT / 4 float4 per split; thread i takes float4 i, i + 512,
        // ... with every split's loads in flight before the sums
        constexpr int NV = TP_M * NT / 4 / 512;  // 1, 2 or 4
        if (tid < 512) {
            float4 sum[NV];
#pragma unroll
            for (int u = 0; u < NV; ++u) sum[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const float4 *src = reinterpret_cast<const float4 *>(part);
            for (int sp0 = 0; sp0 < S; sp0 += 4) {
                float4 v[4][NV];
#pragma unroll
                for (int d = 0; d < 4; ++d)
#pragma unroll
                    for (int u = 0; u < NV; ++u)
                        if (sp0 + d < S) v[d][u] = __ldcg(src + static_cast<size_t>(sp0 + d) * (TP_M * NT / 4) + tid + 512 * u);
#pragma unroll
                for (int d = 0; d < 4; ++d)
#pragma unroll
                    for (int u = 0; u < NV; ++u)
                        if (sp0 + d < S) {
                            sum[u].x += v[d][u].x;
                            sum[u].y += v[d][u].y;
                            sum[u].z += v[d][u].z;
                            sum[u].w += v[d][u].w;
                        }
            }
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const int e = 4 * (tid + 512 * u), row = e / NT, col = e % NT;
                float *o = ep + row * EPS + col;
                o[0] = sum[u].x;
                o[1] = sum[u].y;
                o[2] = sum[u].z;
                o[3] = sum[u].w;
            }
        }
    }
    __syncthreads();  // the tile's sums are in ep

    // ---- epilogue: thread -> sequence column sl = tid % NT and a group of
    // rows; the sequence's position (and cache rows) once, every load of the
    // thread's rows issued before any is used
    constexpr int NGRP = 512 / NT;  // row groups
    if (tid >= 512) return;
    const int sl = tid % NT, grp = tid / NT;
    const int s = s0 + sl;
    if (s >= a.B) return;
    const int pos = a.d_pos[s];
    if (pos < 0 || pos >= a.C) {
        flag_error(a.status, FLAG_RANGE);
        return;
    }
    const int half = a.hd >> 1;
    if (kind == 0 || kind == 1) {  // RoPE pairs (l, l + hd/2) of the tile's heads
        constexpr int PP = (TP_M / 2) / NGRP;  // pairs per thread
        const float *bias = kind == 0 ? a.bq : a.bk;
        float cv[PP], sv[PP], ba[PP], bb[PP];
#pragma unroll
        for (int u = 0; u < PP; ++u) {
            const int pr = grp + NGRP * u;
            const int l = (pr / half) * a.hd + (pr % half);
            const int ra = rbase + l;
            const int i = ra % a.hd;
            cv[u] = a.rope_cos[static_cast<size_t>(pos) * half + i];
            sv[u] = a.rope_sin[static_cast<size_t>(pos) * half + i];
            ba[u] = bias ? bias[ra] : 0.0f;
            bb[u] = bias ? bias[ra + half] : 0.0f;
        }
        float *krow = nullptr;
        if (kind == 1) krow = a.k_caches[s];
#pragma unroll
        for (int u = 0; u < PP; ++u) {
            const int pr = grp + NGRP * u;
            const int l = (pr / half) * a.hd + (pr % half);
            const int ra = rbase + l, rbb = ra + half;
            const float A = ep[l * EPS + sl] + ba[u];
            const float B = ep[(l + half) * EPS + sl] + bb[u];
            const float A2 = __fsub_rn(__fmul_rn(A, cv[u]), __fmul_rn(B, sv[u]));
            const float B2 = __fadd_rn(__fmul_rn(A, sv[u]), __fmul_rn(B, cv[u]));
            if (kind == 0) {
                a.q[static_cast<size_t>(s) * QD + ra] = A2;
                a.q[static_cast<size_t>(s) * QD + rbb] = B2;
            } else {
                const int head = ra / a.hd, i = ra - head * a.hd;
                float *kr = krow + (static_cast<size_t>(head) * a.C + pos) * a.hd;
                kr[i] = A2;
                kr[i + half] = B2;
            }
        }
    } else {
        constexpr int RR = TP_M / NGRP;  // rows per thread
        float xv[RR], bo[RR];  // O: residual and bias; V: bias
#pragma unroll
        for (int u = 0; u < RR; ++u) {
            const int rr = rbase + grp + NGRP * u;
            if (kind == 4) {
                xv[u] = a.residual[static_cast<size_t>(s) * a.D + rr];
                bo[u] = a.bo ? a.bo[rr] : 0.0f;
            } else {
                xv[u] = a.bv ? a.bv[rr] : 0.0f;
            }
        }
        float *vrow = kind == 2 ? a.v_caches[s] : nullptr;
#pragma unroll
        for (int u = 0; u < RR; ++u) {
            const int l = grp + NGRP * u, rr = rbase + l;
            const float v = ep[l * EPS + sl];
            if (kind == 4) {
                a.out[static_cast<size_t>(s) * a.D + rr] = (v + bo[u]) + xv[u];
            } else {
                const int h = rr / a.hd;
                vrow[(static_cast<size_t>(h) * a.C + pos) * a.hd + (rr - h * a.hd)] = v + xv[u];
            }
        }
    }
}

bool batched_tc_ok(int D, int H, int KV, int hd) {
    const int QD = H * hd, KD = KV * hd;
    return (hd == 64 || hd == 128) && D % TP_M == 0 && QD % TP_M == 0 && KD % TP_M == 0 &&
           tp_smem().total <= device_info().smem_optin;
}

static int tp_nt(int B) { return B > 32 ? 64 : B > 16 ? 32 : 16; }

TpPlan tp_plan(int B, int D, int H, int KV, int hd, bool with_device) {
    TpPlan p{};
    const int G = img_groups(B);
    const int nsm = with_device ? device_info().num_sms : 0;
    const int nt = tp_nt(B);
    const int tiles[2] = {(H + 2 * KV) * hd / TP_M, D / TP_M};
    const int nst[2] = {D / QK / TP_BPS, H * hd / QK / TP_BPS};
    size_t part = 0;
    for (int i = 0; i < 2; ++i) {
        const int smax = nst[i] < TP_MAX_SPLITS ? nst[i] : TP_MAX_SPLITS;
        int S = nsm / (tiles[i] * G);
        p.splits[i] = S < 1 ? 1 : S > smax ? smax : S;
        // scratch for the partial tiles: sized for the most splits (the
        // same on every device)
        const size_t bytes = static_cast<size_t>(tiles[i]) * G * smax * TP_M * nt * 4;
        part = bytes > part ? bytes : part;
    }
    p.part_bytes = part;
    p.tickets_o = tiles[0] * G;
    p.tickets = tiles[0] * G + tiles[1] * G;
    return p;
}

template <bool OPROJ, int NT>
static cudaError_t launch_tp(const BatchArgs &a, int S, cudaStream_t s, bool pdl) {
    const int rows = OPROJ ? a.D : (a.H + 2 * a.KV) * a.hd;
    const dim3 grid(rows / TP_M, S, img_groups(a.B));
    const void *fn = reinterpret_cast<const void *>(k_proj_tc<OPROJ, NT>);
    ensure_smem(fn, tp_smem().total);
    BatchArgs ac = a;
    int Sc = S;
    void *args[] = {&ac, &Sc};
    return launch(fn, grid, dim3(TW_THREADS), tp_smem().total, s, pdl, args);
}

int launch_rows_tc(const BatchArgs &a, bool oproj, cudaStream_t s, bool pdl) {
    const TpPlan p = tp_plan(a.B, a.D, a.H, a.KV, a.hd, true);
    const int S = p.splits[oproj ? 1 : 0];
    cudaError_t e;
    switch (tp_nt(a.B)) {
        case 16: e = oproj ? launch_tp<true, 16>(a, S, s, pdl) : launch_tp<false, 16>(a, S, s, pdl); break;
        case 32: e = oproj ? launch_tp<true, 32>(a, S, s, pdl) : launch_tp<false, 32>(a, S, s, pdl); break;
        default: e = oproj ? launch_tp<true, 64>(a, S, s, pdl) : launch_tp<false, 64>(a, S, s, pdl); break;
    }
    return e == cudaSuccess ? 0 : -5;
}

}  // namespace ck
