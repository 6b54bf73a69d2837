// Batched projections on the 5th-generation tensor cores (tcgen05, kind::f16).
//
// For B activation rows sharing one weight matrix the projection
//   y[s][r] = sum_b d_w[r][b] * d_x[s][b] * isum[r][s][b]
// is a dense contraction.  Codes are exact in fp16 (Q5_0: q - 16 in [-16, 15];
// Q8_0: [-127, 127]), their products and 32-term block sums are exact in the
// fp32 accumulator, so one MMA pair per 32-element block yields the exact
// int32 block dots; the per-block scales differ per row and per sequence, so
// every block gets its own TMEM accumulator, read back and folded in with
// fmaf(isum, d_w * d_x, acc) in block order (the formula of the dp4a GEMVs).
//
// CTA (256 threads): 128 weight rows (MMA M) x 16 sequences (MMA N).  K runs
// in stages of 8 blocks (256 codes): warps 4-7 convert the next stage's
// weights (Q5_0 or Q8_0 rows, read from global memory two blocks at a time)
// and activations (the Q8_0 blocks of each sequence) into fp16 operand tiles
// in shared memory (K-major, no swizzle, 8-row x 16-byte core matrices; the
// leading byte offset is the stride between core matrices along K, the
// stride byte offset the stride between 8-row groups), while thread 0 issues
// the current stage's 16 MMAs into 8 TMEM slots of 16 columns and warps 0-3
// read them back (TMEM lane = weight row).  Operand tiles are double-
// buffered; the TMEM slots are reused every stage.
//
// The epilogue (bias, RoPE at each sequence's position, q / K / V stores, or
// bias + residual) is the one of the dp4a kernel, from the accumulators
// exchanged through shared memory.
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

constexpr int TC_M = 128;              // weight rows per CTA
constexpr int TC_N = 16;               // sequences per CTA
constexpr int TC_BPS = 8;              // blocks per stage
constexpr int TC_KG = 4 * TC_BPS;      // 8-element K groups per stage
constexpr int TC_THREADS = 256;
constexpr int TC_TMEM_COLS = TC_BPS * TC_N;  // 128
constexpr uint32_t TC_SBO = TC_KG * 128;     // bytes between 8-row groups
constexpr int TC_DWS = TC_M + 4;             // floats per block of the weight scales (bank spread)

struct TcSmem {
    size_t a[2], b[2], dw[2], dx[2], ep, bar, tmem, total;
};
__host__ __device__ inline TcSmem tc_smem() {
    TcSmem L;
    size_t o = 0;
    for (int i = 0; i < 2; ++i) {
        L.a[i] = o;
        o += static_cast<size_t>(TC_M) * TC_BPS * 32 * 2;  // 64 KB
    }
    for (int i = 0; i < 2; ++i) {
        L.b[i] = o;
        o += static_cast<size_t>(TC_N) * TC_BPS * 32 * 2;  // 8 KB
    }
    for (int i = 0; i < 2; ++i) {
        L.dw[i] = o;  // dw[j][row], rows padded to TC_DWS
        o += static_cast<size_t>(TC_DWS) * TC_BPS * 4;
    }
    for (int i = 0; i < 2; ++i) {
        L.dx[i] = o;  // 16-byte aligned: read as float4
        o += static_cast<size_t>(TC_N) * TC_BPS * 4;
    }
    L.ep = o;  // accumulators for the epilogue [TC_M][TC_N + 1]
    o += static_cast<size_t>(TC_M) * (TC_N + 1) * 4;
    L.bar = o;
    o += 16;
    L.tmem = o;
    o += 16;
    L.total = (o + 127) / 128 * 128;
    return L;
}

// Offset of double buffer `k & 1` without indexing the layout dynamically
// (which would place it in local memory).
__device__ __forceinline__ size_t buf(const size_t (&b)[2], int k) { return (k & 1) ? b[1] : b[0]; }

__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((128u >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((TC_SBO >> 4) & 0x3FFFu) << 32) | (1ull << 46);
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

// Write one 32-element block (8 words of byte codes, element order) of row r
// at stage block j into the operand tile `tile` (core-matrix layout).
__device__ __forceinline__ void put_block(uint8_t *tile, int r, int j, const uint32_t (&c)[8], __half2 bias) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {  // 8 elements each
        uint4 v;
        codes_to_half(c[2 * g], bias, v.x, v.y);
        codes_to_half(c[2 * g + 1], bias, v.z, v.w);
        *reinterpret_cast<uint4 *>(tile + ((r >> 3) * TC_KG + 4 * j + g) * 128 + (r & 7) * 16) = v;
    }
}

// Two consecutive blocks of a row (Q5_0: 44 bytes, Q8_0: 68 bytes; 4-byte
// aligned) as raw words: every load of a stage is issued before any is used.
constexpr int TC_PAIR_WORDS = 17;
__device__ __forceinline__ void load_pair(const uint8_t *src, bool q8, bool ldg, uint32_t (&w)[TC_PAIR_WORDS]) {
    const uint32_t *p = reinterpret_cast<const uint32_t *>(src);
#pragma unroll
    for (int i = 0; i < TC_PAIR_WORDS; ++i) {
        if (i < 11 || q8) w[i] = ldg ? __ldg(p + i) : __ldcg(p + i);
        else w[i] = 0;
    }
}

// Raw Q5_0 pair -> codes q in 0..31 per element and the two scales.
__device__ __forceinline__ void decode_q5_pair(const uint32_t (&w)[TC_PAIR_WORDS], uint32_t (&c0)[8], uint32_t (&c1)[8],
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
__device__ __forceinline__ void decode_q8_pair(const uint32_t (&w)[TC_PAIR_WORDS], uint32_t (&c0)[8], uint32_t (&c1)[8],
                                               float &d0, float &d1) {
    d0 = half_bits_to_float(w[0]);
    d1 = half_bits_to_float(w[8] >> 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        c0[i] = __funnelshift_r(w[i], w[i + 1], 16) ^ 0x80808080u;  // codes at bytes 2..33
        c1[i] = w[9 + i] ^ 0x80808080u;                             // codes at bytes 36..67
    }
}

template <bool OPROJ>
__global__ void __launch_bounds__(TC_THREADS, 1) k_rows_tc(const BatchArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const TcSmem L = tc_smem();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nb = OPROJ ? a.H * a.hd / QK : a.D / QK;
    const int nst = nb / TC_BPS;
    const int QD = a.H * a.hd, KD = a.KV * a.hd;
    const int R0 = blockIdx.x * TC_M;  // first global row of the tile
    const int s0 = blockIdx.y * TC_N;  // first sequence
    // the tile's matrix (a tile never straddles Q / K / V)
    int kind = 4;  // 0 = Q, 1 = K, 2 = V, 4 = O
    const uint8_t *W = a.wo;
    int rbase = R0;
    if (!OPROJ) {
        if (R0 < QD) {
            kind = 0;
            W = a.wq;
        } else if (R0 < QD + KD) {
            kind = 1;
            W = a.wk;
            rbase = R0 - QD;
        } else {
            kind = 2;
            W = a.wv;
            rbase = R0 - QD - KD;
        }
    }
    const bool wq8 = kind == 2;
    const size_t rb = static_cast<size_t>(nb) * (wq8 ? Q8B : Q5B);
    const uint8_t *xq = OPROJ ? a.aq8 : a.xq8;  // Q8_0 blocks of the activation rows [B][nb]
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L.bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.tmem);
    const __half2 wbias = __half2half2(__float2half(wq8 ? 1152.0f : 1040.0f));
    const __half2 xbias = __half2half2(__float2half(1152.0f));

    // weight half of stage k into buffer k & 1, in two steps so that the
    // loads are in flight while the previous stage is read back: load_w
    // fetches the raw pairs of thread `tid` (TC_WPT pairs of a 256-thread
    // sweep), decode_w writes them to the operand tile.
    // Item `it` of a sweep is row (it & 7) + 8 (it >> 5), pair (it >> 3) & 3:
    // the 8 threads of a quarter-warp write the 8 rows of one core matrix
    // (distinct banks) and a warp reads 8 rows x 4 pairs (contiguous bytes).
    constexpr int TC_WPT = TC_M * (TC_BPS / 2) / TC_THREADS;  // 2
    auto load_w = [&](int k, uint32_t (&raw)[TC_WPT][TC_PAIR_WORDS]) {
#pragma unroll
        for (int u = 0; u < TC_WPT; ++u) {
            const int it = tid + u * TC_THREADS;
            const int r = (it & 7) + 8 * (it >> 5), p = (it >> 3) & 3;
            const int blk = k * TC_BPS + 2 * p;
            load_pair(W + static_cast<size_t>(rbase + r) * rb + static_cast<size_t>(blk) * (wq8 ? Q8B : Q5B), wq8,
                      true, raw[u]);
        }
    };
    auto decode_w = [&](int k, const uint32_t (&raw)[TC_WPT][TC_PAIR_WORDS]) {
        uint8_t *tile = smem + buf(L.a, k);
        float *dw = reinterpret_cast<float *>(smem + buf(L.dw, k));
#pragma unroll
        for (int u = 0; u < TC_WPT; ++u) {
            const int it = tid + u * TC_THREADS;
            const int r = (it & 7) + 8 * (it >> 5), p = (it >> 3) & 3;
            uint32_t c0[8], c1[8];
            float d0, d1;
            if (wq8)
                decode_q8_pair(raw[u], c0, c1, d0, d1);
            else
                decode_q5_pair(raw[u], c0, c1, d0, d1);
            put_block(tile, r, 2 * p, c0, wbias);
            put_block(tile, r, 2 * p + 1, c1, wbias);
            dw[(2 * p) * TC_DWS + r] = d0;
            dw[(2 * p + 1) * TC_DWS + r] = d1;
        }
    };
    // activation half of stage k (after the wait on the preceding grid);
    // scales stored block-major, dx[j][sequence]
    auto convert_x = [&](int k) {
        uint8_t *tile = smem + buf(L.b, k);
        float *dx = reinterpret_cast<float *>(smem + buf(L.dx, k));
        const int it = tid;
        if (it < TC_N * (TC_BPS / 2)) {
            const int sl = (it & 7) + 8 * (it >> 5), p = (it >> 3) & 3;
            const int s = s0 + sl;
            uint32_t c0[8], c1[8];
            float d0 = 0.0f, d1 = 0.0f;
            if (s < a.B) {
                const int blk = k * TC_BPS + 2 * p;
                uint32_t w[TC_PAIR_WORDS];
                load_pair(xq + (static_cast<size_t>(s) * nb + blk) * Q8B, true, false, w);
                decode_q8_pair(w, c0, c1, d0, d1);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) c0[i] = c1[i] = 0x80808080u;  // zero codes
            }
            put_block(tile, sl, 2 * p, c0, xbias);
            put_block(tile, sl, 2 * p + 1, c1, xbias);
            dx[(2 * p) * TC_N + sl] = d0;
            dx[(2 * p + 1) * TC_N + sl] = d1;
        }
    };
    auto issue_mma = [&](int k, uint32_t taddr) {  // thread 0
        const uint32_t abase = sptr(smem + buf(L.a, k)), bbase = sptr(smem + buf(L.b, k));
        const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(TC_N >> 3) << 17) |
                               (static_cast<uint32_t>(TC_M >> 4) << 24);
#pragma unroll
        for (int j = 0; j < TC_BPS; ++j)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint64_t ad = tc_desc(abase + (4 * j + 2 * h) * 128);
                const uint64_t bd = tc_desc(bbase + (4 * j + 2 * h) * 128);
                asm volatile(
                    "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(taddr + j * TC_N),
                    "l"(ad), "l"(bd), "r"(idesc), "r"(h)
                    : "memory");
            }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sptr(bar))
                     : "memory");
    };

    // ---- prologue: the tile's weight rows (contiguous) into L2, barrier,
    // TMEM, the first stage's weights before the wait
    if (warp == 1) {
        const size_t bytes = static_cast<size_t>(TC_M) * rb;
        const uint8_t *base = W + static_cast<size_t>(rbase) * rb;
        for (size_t o = static_cast<size_t>(lane) * 65536; o < bytes; o += 32 * 65536)
            prefetch_l2(base + o, static_cast<uint32_t>(bytes - o < 65536 ? bytes - o : 65536));
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sptr(tmem_slot)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    uint32_t raw[TC_WPT][TC_PAIR_WORDS];
    load_w(0, raw);
    decode_w(0, raw);
    pdl_trigger();
    pdl_wait();  // the activation blocks are ready
    convert_x(0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *tmem_slot;
    if (tid == 0) issue_mma(0, taddr);

    // Every warp reads back half of each stage's blocks: warps w and w + 4
    // share TMEM lanes 32 (w % 4) .. + 31 (the tile rows), blocks
    // jh .. jh + 3.  Their two partial sums meet in the epilogue.
    const int r = (warp & 3) * 32 + lane;
    const int jh = (warp >> 2) * (TC_BPS / 2);
    float acc[TC_N];
#pragma unroll
    for (int i = 0; i < TC_N; ++i) acc[i] = 0.0f;
    for (int k = 0; k < nst; ++k) {
        const bool more = k + 1 < nst;
        if (more) load_w(k + 1, raw);  // in flight during the read-back
        if (!mbar_wait(bar, k & 1)) flag_error(a.status, FLAG_TIMEOUT);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        {
            const float *dw = reinterpret_cast<const float *>(smem + buf(L.dw, k)) + r;
            const float4 *dx = reinterpret_cast<const float4 *>(smem + buf(L.dx, k));
#pragma unroll
            for (int jj = 0; jj < TC_BPS / 2; ++jj) {
                const int j = jh + jj;
                uint32_t v[16];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                      "=r"(v[14]), "=r"(v[15])
                    : "r"(taddr + (static_cast<uint32_t>((warp & 3) * 32) << 16) + j * TC_N)
                    : "memory");
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                const float dwv = dw[j * TC_DWS];
#pragma unroll
                for (int q4 = 0; q4 < TC_N / 4; ++q4) {
                    const float4 d4 = dx[j * (TC_N / 4) + q4];
                    acc[4 * q4 + 0] = fmaf(__uint_as_float(v[4 * q4 + 0]), dwv * d4.x, acc[4 * q4 + 0]);
                    acc[4 * q4 + 1] = fmaf(__uint_as_float(v[4 * q4 + 1]), dwv * d4.y, acc[4 * q4 + 1]);
                    acc[4 * q4 + 2] = fmaf(__uint_as_float(v[4 * q4 + 2]), dwv * d4.z, acc[4 * q4 + 2]);
                    acc[4 * q4 + 3] = fmaf(__uint_as_float(v[4 * q4 + 3]), dwv * d4.w, acc[4 * q4 + 3]);
                }
            }
        }
        if (more) {  // stage k + 1 into the buffers stage k - 1 used
            decode_w(k + 1, raw);
            convert_x(k + 1);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();  // stage k read back, stage k + 1 converted
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (tid == 0 && more) issue_mma(k + 1, taddr);
    }

    // ---- epilogue through shared memory
    float *ep = reinterpret_cast<float *>(smem + L.ep);
    if (warp >= 4) {
#pragma unroll
        for (int s = 0; s < TC_N; ++s) ep[r * (TC_N + 1) + s] = acc[s];
    }
    __syncthreads();
    if (warp < 4) {
#pragma unroll
        for (int s = 0; s < TC_N; ++s) ep[r * (TC_N + 1) + s] += acc[s];
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(TC_TMEM_COLS));
    const int half = a.hd >> 1;
    if (kind == 0 || kind == 1) {  // RoPE pairs (l, l + hd/2) of the tile's heads
        for (int it = tid; it < (TC_M / 2) * TC_N; it += TC_THREADS) {
            const int pr = it / TC_N, sl = it - pr * TC_N;
            const int s = s0 + sl;
            if (s >= a.B) continue;
            const int pos = a.d_pos[s];
            if (pos < 0 || pos >= a.C) {
                flag_error(a.status, FLAG_RANGE);
                continue;
            }
            const int l = (pr / half) * a.hd + (pr % half);  // first row of the pair in the tile
            const int ra = rbase + l, rbb = ra + half;
            const float *bias = kind == 0 ? a.bq : a.bk;
            const float A = ep[l * (TC_N + 1) + sl] + (bias ? bias[ra] : 0.0f);
            const float B = ep[(l + half) * (TC_N + 1) + sl] + (bias ? bias[rbb] : 0.0f);
            const int head = ra / a.hd, i = ra - head * a.hd;
            const float c = a.rope_cos[static_cast<size_t>(pos) * half + i];
            const float sn = a.rope_sin[static_cast<size_t>(pos) * half + i];
            const float A2 = __fsub_rn(__fmul_rn(A, c), __fmul_rn(B, sn));
            const float B2 = __fadd_rn(__fmul_rn(A, sn), __fmul_rn(B, c));
            if (kind == 0) {
                a.q[static_cast<size_t>(s) * QD + ra] = A2;
                a.q[static_cast<size_t>(s) * QD + rbb] = B2;
            } else {
                float *kr = a.k_caches[s] + (static_cast<size_t>(head) * a.C + pos) * a.hd;
                kr[i] = A2;
                kr[i + half] = B2;
            }
        }
    } else {
        for (int it = tid; it < TC_M * TC_N; it += TC_THREADS) {
            const int l = it / TC_N, sl = it - l * TC_N;
            const int s = s0 + sl;
            if (s >= a.B) continue;
            const int pos = a.d_pos[s];
            if (pos < 0 || pos >= a.C) {
                flag_error(a.status, FLAG_RANGE);
                continue;
            }
            const int r = rbase + l;
            const float v = ep[l * (TC_N + 1) + sl];
            if (kind == 4) {
                a.out[static_cast<size_t>(s) * a.D + r] =
                    (v + (a.bo ? a.bo[r] : 0.0f)) + a.residual[static_cast<size_t>(s) * a.D + r];
            } else {
                const int h = r / a.hd;
                a.v_caches[s][(static_cast<size_t>(h) * a.C + pos) * a.hd + (r - h * a.hd)] =
                    v + (a.bv ? a.bv[r] : 0.0f);
            }
        }
    }
}

bool batched_tc_ok(int D, int H, int KV, int hd) {
    const int QD = H * hd, KD = KV * hd;
    return (hd == 64 || hd == 128) && D % TC_M == 0 && QD % TC_M == 0 && KD % TC_M == 0 &&
           (D / QK) % TC_BPS == 0 && (QD / QK) % TC_BPS == 0 && tc_smem().total <= device_info().smem_optin;
}

int launch_rows_tc(const BatchArgs &a0, bool oproj, cudaStream_t s, bool pdl) {
    BatchArgs a = a0;
    const int rows = oproj ? a.D : (a.H + 2 * a.KV) * a.hd;
    const dim3 grid(rows / TC_M, (a.B + TC_N - 1) / TC_N);
    const void *fn = oproj ? reinterpret_cast<const void *>(k_rows_tc<true>)
                           : reinterpret_cast<const void *>(k_rows_tc<false>);
    ensure_smem(fn, tc_smem().total);
    void *args[] = {&a};
    return launch(fn, grid, dim3(TC_THREADS), tc_smem().total, s, pdl, args) == cudaSuccess ? 0 : -5;
}

}  // namespace ck
