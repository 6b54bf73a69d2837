// Device-side building blocks shared by the decode-step kernels (sm_103a).
//
//  - PTX wrappers: mbarrier (init / expect-tx / bounded parity wait), the
//    bulk global->shared copy engine (cp.async.bulk, completion counted in
//    bytes on an mbarrier), L2 prefetch, programmatic dependent launch.
//  - The two block formats of the page "mega_fused_attention_decode_q5_0.c":
//    Q5_0 (22 bytes: fp16 d, u32 qh, 16 bytes of nibbles, weight (q-16)*d)
//    and Q8_0 (34 bytes: fp16 d, 32 x int8, weight q*d), and the exact
//    integer block dots of vec_dot_q5_0_q8_0 / vec_dot_q8_0_q8_0 with dp4a.
//  - The shared-memory layout of a Q8_0 activation row.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ck {

constexpr int QK = 32;
constexpr int Q5B = 22;  // bytes per Q5_0 block
constexpr int Q8B = 34;  // bytes per Q8_0 block

// Device status flags (OR-ed into a status word the host can read).
constexpr unsigned FLAG_RANGE = 1u;    // a position read on the device was out of range
constexpr unsigned FLAG_TIMEOUT = 2u;  // a bounded wait expired

// Upper bound of every wait on an mbarrier: 2 s of %globaltimer.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sptr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sptr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once on the barrier (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sptr(bar)) : "memory");
}

// Arrive once on the barrier and add `bytes` to the transactions it expects.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sptr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(sptr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete; false after
// WAIT_LIMIT_NS (the caller records FLAG_TIMEOUT and skips its work).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sptr(dst)),
        "l"(src), "r"(bytes), "r"(sptr(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared through L2 (both addresses
// 16-byte aligned), its commit groups and the wait for all but N groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sptr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Hint: bring [p, p+bytes) into L2 (16-byte aligned address and size).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait until the preceding grid in the
// stream has completed and its writes are visible (no-op without PDL) /
// allow the following grid to begin launching.
// Bring the cache line holding `p` into L1 (no register result).
__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void flag_error(unsigned *status, unsigned flag) {
    if (status) atomicOr(status, flag);
}

// ---------------------------------------------------------------------------
// fp16 scale fields
// ---------------------------------------------------------------------------
__device__ __forceinline__ float half_bits_to_float(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

// ---------------------------------------------------------------------------
// Exact integer block dots
// ---------------------------------------------------------------------------
// Q5_0 x Q8_0: sum_j (q_j - 16) * x_j with q_j = nibble | (qh bit j) << 4.
// qs[i] holds bytes 4i..4i+3 of the nibble array: its low nibbles are
// elements 4i..4i+3 and its high nibbles elements 16+4i..16+4i+3.  xw[k]
// holds activation codes 4k..4k+3; xsum is the sum of the 32 codes.  The
// four qh bits of a byte-quad are spread to bit 4 of each byte with one
// multiply (t * 0x02040810 places t0..t3 at bits 4, 12, 20, 28).
__device__ __forceinline__ int isum_q5_0(uint32_t qh, const uint32_t (&qs)[4], const int (&xw)[8], int xsum) {
    int s = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t mlo = (((qh >> (4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u;
        const uint32_t mhi = (((qh >> (16 + 4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u;
        s = __dp4a(static_cast<int>((qs[i] & 0x0F0F0F0Fu) | mlo), xw[i], s);
        s = __dp4a(static_cast<int>(((qs[i] >> 4) & 0x0F0F0F0Fu) | mhi), xw[4 + i], s);
    }
    return s - 16 * xsum;
}

// Q8_0 x Q8_0: sum_j w_j * x_j over 32 signed codes.
__device__ __forceinline__ int isum_q8_0(const uint32_t (&qs)[8], const int (&xw)[8]) {
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s = __dp4a(static_cast<int>(qs[i]), xw[i], s);
    return s;
}

// ---------------------------------------------------------------------------
// Q8_0 activation row in shared memory
// ---------------------------------------------------------------------------
// Codes of block b occupy two 16-byte chunks at chunk index 2b + c + b/8
// (c = 0: codes 0-15, c = 1: codes 16-31).  The one-chunk gap after every
// 8 blocks puts blocks 8 apart into different bank groups, so the two
// segment columns that one warp reads at a time never conflict.
__host__ __device__ constexpr int xq_chunk(int b, int c) { return 2 * b + c + (b >> 3); }
__host__ __device__ constexpr int xq_chunks(int nb) { return 2 * nb + nb / 8 + 1; }
// Bytes of a packed row: the XRow image (codes in the chunk layout, then nb
// fp32 scales, then nb int32 code sums), rounded up to 16.
__host__ __device__ constexpr size_t xpack_bytes(int nb) {
    return (static_cast<size_t>(xq_chunks(nb)) * 16 + static_cast<size_t>(nb) * 8 + 15) / 16 * 16;
}

// ---------------------------------------------------------------------------
// Operand image of a batch of Q8_0 activation rows for the tensor-core
// projections.  Each value d * q (d the block's fp16 scale, q its code: at
// most 18 significant bits, exact in fp32) is held exactly as the sum of two
// fp16 values, hi = fp16(d * q) and lo = d * q - hi (at most 7 significant
// bits); |d * q| must stay within the fp16 range.  Rows (sequences) go in
// groups of IMG_SEQ, blocks in stages of IMG_BPS (128 values).  Stage k of
// group g holds 16 KB of the hi parts in the MMA operand layout (core
// matrices of 8 rows x 8 values = 128 bytes, 16 of them along K per 8-row
// group, 8-row groups IMG_RG_BYTES apart), then 16 KB of the lo parts.
// ---------------------------------------------------------------------------
constexpr int IMG_SEQ = 64;
constexpr int IMG_BPS = 4;
constexpr int IMG_KG = IMG_BPS * 4;                         // 8-value groups along K
constexpr int IMG_RG_BYTES = IMG_KG * 128;                  // one 8-row group
constexpr int IMG_CODE_BYTES = IMG_SEQ / 8 * IMG_RG_BYTES;  // 16 KB: one part
constexpr int IMG_STAGE_BYTES = 2 * IMG_CODE_BYTES;         // hi, then lo
__host__ __device__ constexpr int img_groups(int B) { return (B + IMG_SEQ - 1) / IMG_SEQ; }
__host__ __device__ constexpr size_t img_bytes(int nb, int B) {
    return static_cast<size_t>(nb / IMG_BPS) * img_groups(B) * IMG_STAGE_BYTES;
}
__host__ __device__ constexpr size_t img_stage(int G, int k, int g) {
    return (static_cast<size_t>(k) * G + g) * IMG_STAGE_BYTES;
}
// The 16 bytes holding hi parts 8e .. 8e + 7 of block b of row s (the lo
// parts are IMG_CODE_BYTES further).
__host__ __device__ constexpr size_t img_code_off(int G, int s, int b, int e) {
    return img_stage(G, b / IMG_BPS, s / IMG_SEQ) + static_cast<size_t>(((s % IMG_SEQ) >> 3) * IMG_RG_BYTES) +
           static_cast<size_t>(((b % IMG_BPS) * 4 + e) * 128 + (s & 7) * 16);
}
// The exact fp16 pair of d * q (false when it leaves the fp16 range).
__device__ __forceinline__ bool img_split(float d, int q, __half &hi, __half &lo) {
    const float v = d * static_cast<float>(q);  // exact
    hi = __float2half_rn(v);
    lo = __float2half_rn(v - __half2float(hi));  // exact residual
    return fabsf(v) <= 65504.0f;
}

struct XRow {
    int4 *q;     // codes, layout above
    float *d;    // fp16 scale of each block, as float
    int *sum;    // sum of the 32 codes of each block
};

__device__ __forceinline__ void load_x_words(const XRow &x, int b, int (&xw)[8]) {
    const int4 a = x.q[xq_chunk(b, 0)];
    const int4 c = x.q[xq_chunk(b, 1)];
    xw[0] = a.x; xw[1] = a.y; xw[2] = a.z; xw[3] = a.w;
    xw[4] = c.x; xw[5] = c.y; xw[6] = c.z; xw[7] = c.w;
}

// 32-bit little-endian value at an even byte offset `o` of a word array
// (o is a compile-time constant after unrolling).
template <int N>
__device__ __forceinline__ uint32_t at32(const uint32_t (&w)[N], int o) {
    return (o & 3) ? __funnelshift_r(w[o >> 2], w[(o >> 2) + 1], 16) : w[o >> 2];
}
template <int N>
__device__ __forceinline__ uint32_t at16(const uint32_t (&w)[N], int o) {
    return (o & 3) ? (w[o >> 2] >> 16) : (w[o >> 2] & 0xFFFFu);
}

// ---------------------------------------------------------------------------
// Segment dots: 8 consecutive blocks of one weight row (176 bytes = 11
// 16-byte chunks for Q5_0, 272 bytes = 17 chunks for Q8_0), 16-byte aligned.
// Returns sum_j d_w d_x isum_j in fp32; optionally emits the 8 int sums.
// ---------------------------------------------------------------------------
template <bool Q8>
struct SegShape {
    static constexpr int BLK = Q8 ? Q8B : Q5B;
    static constexpr int BYTES = 8 * BLK;
    static constexpr int CHUNKS = BYTES / 16;
    static constexpr int WORDS = BYTES / 4;
};

template <bool Q8>
__device__ __forceinline__ float seg_dot(const uint4 *seg, const XRow &x, int b0, int *isum_out = nullptr) {
    using S = SegShape<Q8>;
    uint32_t w[S::WORDS + 1];
#pragma unroll
    for (int i = 0; i < S::CHUNKS; ++i) {
        const uint4 v = seg[i];
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    w[S::WORDS] = 0;
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int o = S::BLK * j;
        const int b = b0 + j;
        int xw[8];
        load_x_words(x, b, xw);
        int s;
        if constexpr (Q8) {
            uint32_t qs[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) qs[i] = at32(w, o + 2 + 4 * i);
            s = isum_q8_0(qs, xw);
        } else {
            const uint32_t qh = at32(w, o + 2);
            uint32_t qs[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) qs[i] = at32(w, o + 6 + 4 * i);
            s = isum_q5_0(qh, qs, xw, x.sum[b]);
        }
        if (isum_out) isum_out[j] = s;
        const float dw = half_bits_to_float(at16(w, o));
        acc = fmaf(static_cast<float>(s), dw * x.d[b], acc);
    }
    return acc;
}

// ---------------------------------------------------------------------------
// Weight segments decoded ahead of the activation (batched projections): the
// 8 blocks of one row segment as byte codes (Q5_0: q in 0..31 with the high
// bit merged; Q8_0: the signed codes) plus the block scales, held in
// registers and reused for every activation row.
// ---------------------------------------------------------------------------
struct SegCodes {
    uint32_t c[8][8];
    float d[8];
};

template <bool Q8>
__device__ __forceinline__ void seg_decode(const uint8_t *src, SegCodes &R) {
    using S = SegShape<Q8>;
    const uint4 *seg = reinterpret_cast<const uint4 *>(src);
    uint32_t w[S::WORDS + 1];
#pragma unroll
    for (int i = 0; i < S::CHUNKS; ++i) {
        const uint4 v = __ldg(seg + i);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    w[S::WORDS] = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int o = S::BLK * j;
        R.d[j] = half_bits_to_float(at16(w, o));
        if constexpr (Q8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) R.c[j][i] = at32(w, o + 2 + 4 * i);
        } else {
            const uint32_t qh = at32(w, o + 2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t qs = at32(w, o + 6 + 4 * i);
                R.c[j][i] = (qs & 0x0F0F0F0Fu) | ((((qh >> (4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u);
                R.c[j][4 + i] =
                    ((qs >> 4) & 0x0F0F0F0Fu) | ((((qh >> (16 + 4 * i)) & 0xFu) * 0x02040810u) & 0x10101010u);
            }
        }
    }
}

// sum_j d_w d_x isum_j over the decoded segment's blocks b0..b0+7 (fp32, in
// block order, as seg_dot); q5 subtracts the 16 * sum(x) offset of Q5_0.
__device__ __forceinline__ float seg_dot_codes(const SegCodes &R, const XRow &x, int b0, bool q5) {
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int b = b0 + j;
        int xw[8];
        load_x_words(x, b, xw);
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) s = __dp4a(static_cast<int>(R.c[j][i]), xw[i], s);
        if (q5) s -= 16 * x.sum[b];
        acc = fmaf(static_cast<float>(s), R.d[j] * x.d[b], acc);
    }
    return acc;
}

// One block read straight from global memory at byte offset `ob` (even) of
// a 16-byte aligned matrix, without touching bytes outside the block.
template <bool Q8>
__device__ __forceinline__ float block_dot_global(const uint8_t *W, size_t ob, const XRow &x, int b,
                                                  int *isum_out = nullptr) {
    const uint8_t *p = W + ob;
    int xw[8];
    load_x_words(x, b, xw);
    uint32_t dbits;
    int s;
    if constexpr (Q8) {
        uint32_t qs[8];
        if (ob & 3) {  // d at a 2-mod-4 address, codes word aligned
            dbits = __ldg(reinterpret_cast<const unsigned short *>(p));
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p + 2);
#pragma unroll
            for (int i = 0; i < 8; ++i) qs[i] = __ldg(q + i);
        } else {
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
            uint32_t wv[9];
#pragma unroll
            for (int i = 0; i < 8; ++i) wv[i] = __ldg(q + i);
            wv[8] = __ldg(reinterpret_cast<const unsigned short *>(p + 32));
            dbits = wv[0] & 0xFFFFu;
#pragma unroll
            for (int i = 0; i < 8; ++i) qs[i] = __funnelshift_r(wv[i], wv[i + 1], 16);
        }
        s = isum_q8_0(qs, xw);
    } else {
        uint32_t qh, qs[4];
        if (ob & 3) {
            dbits = __ldg(reinterpret_cast<const unsigned short *>(p));
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p + 2);
            qh = __ldg(q);
#pragma unroll
            for (int i = 0; i < 4; ++i) qs[i] = __ldg(q + 1 + i);
        } else {
            const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
            uint32_t wv[6];
#pragma unroll
            for (int i = 0; i < 5; ++i) wv[i] = __ldg(q + i);
            wv[5] = __ldg(reinterpret_cast<const unsigned short *>(p + 20));
            dbits = wv[0] & 0xFFFFu;
            qh = __funnelshift_r(wv[0], wv[1], 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) qs[i] = __funnelshift_r(wv[i + 1], wv[i + 2], 16);
        }
        s = isum_q5_0(qh, qs, xw, x.sum[b]);
    }
    if (isum_out) *isum_out = s;
    return static_cast<float>(s) * (half_bits_to_float(dbits) * x.d[b]);
}

// ---------------------------------------------------------------------------
// Small reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_isum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// quantize_row_q8_0 on one block held one element per lane.  d = amax/127
// and 1/d are IEEE fp32 (correctly rounded), codes round half away from 0.
__device__ __forceinline__ int q8_code(float v, uint32_t &dbits, float &dq) {
    const float amax = warp_max(fabsf(v));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    const __half dh = __float2half_rn(d);
    dbits = __half_as_ushort(dh);
    dq = __half2float(dh);
    return static_cast<int>(roundf(__fmul_rn(v, id)));
}

// Error-free transformation of a + b (Knuth two-sum), round-to-nearest ops
// spelled out so nothing is reassociated.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// ---------------------------------------------------------------------------
// RMSNorm + Q8_0 of an activation row
// ---------------------------------------------------------------------------
// rstd = 1/sqrt(mean + eps) from every thread's (sum, compensation) pair of
// x^2 terms: the pairs are combined with two-sums (warp, then CTA), so the
// total equals the double-precision sum to ~2^-46 relative.  m = sum/D + eps
// is carried as an fp32 pair (hi + lo); rstd is the hardware reciprocal
// square root of hi refined by one Newton-Raphson step for 1/sqrt(m),
// y + y (1 - m y^2) / 2, whose residual is formed with FMAs over the pair
// terms (error ~2^-44), then rounded once to fp32.  (fp64 arithmetic, which
// this replaces, runs at a small fraction of the fp32 rate on this GPU.)
// `red` holds 2*warps + 1 floats.  Every thread of the CTA gets rstd.
__device__ inline float rstd_from_pairs(float s, float c, int D, float eps, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float t, err;
        two_sum(s, s2, t, err);
        s = t;
        c = __fadd_rn(__fadd_rn(c, c2), err);
    }
    if (lane == 0) {
        red[2 * warp] = s;
        red[2 * warp + 1] = c;
    }
    __syncthreads();
    if (warp == 0) {
        s = lane < nw ? red[2 * lane] : 0.0f;
        c = lane < nw ? red[2 * lane + 1] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
            float t, err;
            two_sum(s, s2, t, err);
            s = t;
            c = __fadd_rn(__fadd_rn(c, c2), err);
        }
        if (lane == 0) {
            const float Df = static_cast<float>(D);  // exact: D < 2^24
            const float qh = __fdiv_rn(s, Df);
            const float ql = __fdiv_rn(__fadd_rn(fmaf(-qh, Df, s), c), Df);  // (s - qh D) exactly, plus c
            float mh, e;
            two_sum(qh, eps, mh, e);
            const float ml = __fadd_rn(ql, e);
            const float y = rsqrtf(mh);
            const float p = __fmul_rn(y, y), pl = fmaf(y, y, -p);        // y^2 = p + pl exactly
            const float h = fmaf(-mh, pl, fmaf(-ml, p, fmaf(-mh, p, 1.0f)));  // 1 - m y^2
            red[2 * nw] = fmaf(0.5f * y, h, y);
        }
    }
    __syncthreads();
    return red[2 * nw];
}

// Accumulate v^2 into the unevaluated pair (s, c): two-sum of the rounded
// square plus its exact FMA residual.
__device__ __forceinline__ void sumsq_add(float v, float &s, float &c) {
    const float p = __fmul_rn(v, v);
    const float e = fmaf(v, v, -p);
    float t, err;
    two_sum(s, p, t, err);
    s = t;
    c = __fadd_rn(c, __fadd_rn(err, e));
}

// RMSNorm + quantize_row_q8_0 of the whole input row straight into this
// CTA's shared-memory XRow (the projection prologue): warp w takes blocks
// w, w + W, ... (at most NORM_XPW of them), every load of x is issued before
// any is used, y = (x * rstd) * gamma in fp32, and the Q8_0 codes, scales and
// code sums land in the XRow layout.  `gv` holds the warp's gamma values
// (loaded before the wait on the preceding grid).  When `tap` is set the
// Q8_0 blocks are also written there.
constexpr int NORM_XPW = 8;
__device__ inline void norm_quant_xrow(const float *x, const float (&gv)[NORM_XPW], int nb, int D, float eps, const XRow &xr,
                                float *red, uint8_t *tap) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float xv[NORM_XPW];
    float s = 0.0f, c = 0.0f;
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j) {
        const int b = warp + nw * j;
        xv[j] = b < nb ? x[b * QK + lane] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j) sumsq_add(xv[j], s, c);
    const float rstd = rstd_from_pairs(s, c, D, eps, red);
    // quantize_row_q8_0 of the warp's blocks, all of them at once: amax by
    // one warp reduction over the bit patterns of |y| (non-negative floats
    // order as their bits), d = amax / 127, codes round(y / d), code sums
    float y[NORM_XPW];
    unsigned am[NORM_XPW];
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j) {
        y[j] = __fmul_rn(__fmul_rn(xv[j], rstd), gv[j]);
        am[j] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(y[j])));
    }
    // d = amax / 127, 1 / d and the fp16 scale of block j on lane j, then
    // broadcast (the same values on every lane, computed once per block)
    float myam = 0.0f;
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j)
        if (lane == j) myam = __uint_as_float(am[j]);
    const float dl = __fdiv_rn(myam, 127.0f);
    const float idl = (dl != 0.0f) ? __frcp_rn(dl) : 0.0f;
    const uint32_t dbl = __half_as_ushort(__float2half_rn(dl));
    int q[NORM_XPW];
    float dq[NORM_XPW];
    uint32_t dbits[NORM_XPW];
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j) {
        const float id = __shfl_sync(0xffffffffu, idl, j);
        dbits[j] = __shfl_sync(0xffffffffu, dbl, j);
        dq[j] = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits[j])));
        q[j] = static_cast<int>(roundf(__fmul_rn(y[j], id)));
    }
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j) {
        const int b = warp + nw * j;
        const int sum = __reduce_add_sync(0xffffffffu, q[j]);
        if (b < nb) {  // warp-uniform
            reinterpret_cast<int8_t *>(&xr.q[xq_chunk(b, lane >> 4)])[lane & 15] = static_cast<int8_t>(q[j]);
            if (lane == 0) {
                xr.d[b] = dq[j];
                xr.sum[b] = sum;
            }
            if (tap) {
                uint8_t *o = tap + static_cast<size_t>(b) * Q8B;
                o[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q[j]));
                if (lane == 0) {
                    o[0] = static_cast<uint8_t>(dbits[j] & 0xFF);
                    o[1] = static_cast<uint8_t>(dbits[j] >> 8);
                }
            }
        }
    }
    __syncthreads();
}

}  // namespace ck
