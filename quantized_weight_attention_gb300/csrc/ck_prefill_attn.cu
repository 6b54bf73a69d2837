// Prefill attention on the 5th-generation tensor cores (tcgen05, kind::f16
// with bf16 operands).
//
// For one KV head the chunk's queries (n tokens x G query heads) against the
// cache rows 0 .. pos + n - 1 form a dense contraction with a causal mask:
// token i (position pos + i) sees rows 0 .. pos + i.  One CTA owns a tile of
// 128 query rows (tokens x head slots, the group padded to a power of two) and
// walks the key rows in tiles of 64:
//   S  = Q K^T        (M 128, N 64, K = head_dim 128) into TMEM
//   P  = exp2(S - m)  (one thread per query row, the online softmax)
//   O += P V          (M 128, N 128, K 64) accumulated in TMEM
// Q and P are the A operands and live in TMEM (each query row's lane), K and
// V^T stream through shared memory.  Every fp32 operand x is held as two
// bf16 numbers, x = hi + lo + O(2^-17 |x|); a product takes three MMAs
// (hi.hi, hi.lo, lo.hi) with fp32 accumulation.  The row maximum m is raised only when a
// tile's maximum exceeds it by more than 2^8 (in exp2 units), so O and the
// row sum are rescaled rarely; p stays below 256.
//
// The key / value rows are converted once per call by k_pf_kv_image into
// tiles laid out as the MMA reads them (8-row x 16-byte core matrices,
// K-major, no swizzle): per key tile, K hi, K lo (64 rows x 128 dims), then
// V^T hi, V^T lo (128 dims x 64 keys).  A CTA streams them with one bulk copy
// per tile.  Outputs go through the decode attention's store, so the O
// projection receives the same Q8_0 blocks and operand image.
#include <cuda_bf16.h>

#include "ck_attn_kernels.cuh"

namespace ck {
namespace {

constexpr int PF_M = 128;  // query rows per CTA
constexpr int PF_N = 64;   // key rows per tile
constexpr int PF_HD = 128;
constexpr int PF_K_PART = PF_N * PF_HD * 2;
constexpr int PF_V_PART = PF_HD * PF_N * 2;
constexpr int PF_TILE = 2 * PF_K_PART + 2 * PF_V_PART;  // one key tile of the image
constexpr int PF_NST = 3;                                // key tiles in flight
constexpr int PF_THREADS = 192;                          // warps 0-3 rows, 4 copies, 5 MMA
constexpr float PF_TAU = 8.0f;
// TMEM columns (lane = query row): Q hi / lo as bf16 pairs (64 + 64), the two
// S slots (64 fp32 each), the two P buffers (hi 32 + lo 32 each), O (128 fp32)
constexpr int TC_Q = 0, TC_S = 128, TC_P = 256, TC_O = 384;
constexpr int PF_TMEM_COLS = 512;

constexpr size_t PF_OFF_KV = 0;
constexpr size_t PF_OFF_BAR = PF_OFF_KV + static_cast<size_t>(PF_NST) * PF_TILE;
constexpr size_t PF_OFF_TMEM = PF_OFF_BAR + 16 * 8;
constexpr size_t PF_SMEM = PF_OFF_TMEM + 16;
static_assert(PF_SMEM <= 227 * 1024, "shared memory");
static_assert(PF_M * (PF_HD + 1) * 4 <= PF_NST * PF_TILE, "output staging fits the key stages");

// Byte offset of element (row, k) in a K-major core-matrix tile whose rows
// hold `kdim` elements: 8-row groups of kdim/8 matrices of 8 x 16 bytes.
__host__ __device__ constexpr int cm_off(int row, int k, int kdim) {
    return (row >> 3) * (kdim * 16) + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

// Shared-memory matrix descriptor (no swizzle): start, leading byte offset
// 128 (next core matrix along K), stride byte offset `sbo` (next 8-row group).
__device__ __forceinline__ uint64_t pf_desc(uint32_t saddr, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128u >> 4) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Eight fp32 values -> eight bf16 hi parts and eight bf16 lo parts
// (hi = bf16(x), lo = bf16(x - hi); x - hi is exact in fp32).
__device__ __forceinline__ void bf_split8(const float (&x)[8], uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // packed conversions, two values each
        const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        const float2 hf = __bfloat1622float2(hb);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);
        h[i] = *reinterpret_cast<const uint32_t *>(&hb);
        l[i] = *reinterpret_cast<const uint32_t *>(&lb);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void tm_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tm_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One MMA, D (TMEM) += A x B, A read from TMEM (`a_tmem`: lane = row of A,
// each 32-bit column two consecutive K elements), B from shared memory.
__device__ __forceinline__ void pf_mma_ts(uint32_t dtmem, uint32_t a_tmem, uint64_t bd, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(dtmem),
        "r"(a_tmem), "l"(bd), "r"(idesc), "r"(static_cast<uint32_t>(acc))
        : "memory");
}
__device__ __forceinline__ void pf_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sptr(bar))
                 : "memory");
}

// Instruction descriptor: fp32 accumulator, bf16 A and B, both K-major.
constexpr uint32_t pf_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

struct PfArgs {
    const float *k_cache, *v_cache;  // fp32 [KV, C, 128]
    const float *q;                  // fp32 [n, H * 128], after RoPE
    uint8_t *img;                    // [KV][ntk][PF_TILE]
    int C, ntk;                      // capacity, image tiles per head
    int n, pos, H, KV, G, GP, TPT;   // TPT = 128 / GP tokens per query tile
    const int32_t *d_pos;            // the chunk's first position on the device (or null: pos)
    float scale_log2;                // log2(e) / sqrt(128)
    AttnArgs o;                      // outputs (out, out_q8, out_img, out_pack, img_groups, H, status)
};

// Key tile t of KV head g into the image; rows from pos + n on are zeros.
// A chunk outside the cache converts nothing.
__global__ void __launch_bounds__(256) k_pf_kv_image(const PfArgs a) {
    const int t = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
    uint8_t *dst = a.img + (static_cast<size_t>(g) * a.ntk + t) * PF_TILE;
    const float *kc = a.k_cache + static_cast<size_t>(g) * a.C * PF_HD;
    const float *vc = a.v_cache + static_cast<size_t>(g) * a.C * PF_HD;
    pdl_trigger();
    pdl_wait();  // the chunk's rows were stored by the projection grid
    const int pos = a.d_pos ? *a.d_pos : a.pos;
    if (pos < 0 || pos > a.C - a.n) return;
    const int rows = pos + a.n;
    if (t * PF_N >= rows) return;  // a tile past the chunk (grid sized by the capacity)
    {                              // K: thread -> row tid / 4, dims 32 (tid % 4) ..
        const int r = tid >> 2, d0 = (tid & 3) * 32, row = t * PF_N + r;
        const bool in = row < rows;
        const float4 *src = reinterpret_cast<const float4 *>(kc + static_cast<size_t>(in ? row : 0) * PF_HD + d0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float x[8];
            const float4 u = in ? src[2 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 w = in ? src[2 * c + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
            x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w, x[4] = w.x, x[5] = w.y, x[6] = w.z, x[7] = w.w;
            uint4 hi, lo;
            bf_split8(x, hi, lo);
            const int off = cm_off(r, d0 + 8 * c, PF_HD);
            *reinterpret_cast<uint4 *>(dst + off) = hi;
            *reinterpret_cast<uint4 *>(dst + PF_K_PART + off) = lo;
        }
    }
    {  // V^T: thread -> dim tid % 128, keys 32 (tid / 128) ..
        const int d = tid & 127, c0 = (tid >> 7) * 32;
        uint8_t *vt = dst + 2 * PF_K_PART;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = t * PF_N + c0 + 8 * cc + i;
                x[i] = row < rows ? vc[static_cast<size_t>(row) * PF_HD + d] : 0.0f;
            }
            uint4 hi, lo;
            bf_split8(x, hi, lo);
            const int off = cm_off(d, c0 + 8 * cc, PF_N);
            *reinterpret_cast<uint4 *>(vt + off) = hi;
            *reinterpret_cast<uint4 *>(vt + PF_V_PART + off) = lo;
        }
    }
}

__global__ void __launch_bounds__(PF_THREADS, 1) k_pf_attn(const PfArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *skv = smem + PF_OFF_KV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + PF_OFF_BAR);
    uint64_t *kv_full = bars, *kv_empty = bars + PF_NST, *s_full = bars + 2 * PF_NST, *p_full = s_full + 2,
             *o_full = p_full + 2, *q_ready = o_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PF_OFF_TMEM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y;
    const int tl0 = blockIdx.x * a.TPT;                  // the tile's first token
    const int tl_last = min(a.n - 1, tl0 + a.TPT - 1);  // and its last
    // the chunk's position (a device position was set before the chunk's
    // first kernel, which every later one follows)
    const int pos = a.d_pos ? *a.d_pos : a.pos;
    if (pos < 0 || pos > a.C - a.n) {  // a chunk outside the cache: nothing attended, nothing written
        pdl_trigger();
        pdl_wait();
        return;
    }
    const int nkt = (pos + tl_last + 1 + PF_N - 1) / PF_N;

    if (threadIdx.x == 0) {
        for (int i = 0; i < PF_NST; ++i) {
            mbar_init(kv_full + i, 1);
            mbar_init(kv_empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + i, 1);
            mbar_init(p_full + i, 4);
            mbar_init(o_full + i, 1);
        }
        mbar_init(q_ready, 4);
        fence_mbar_init();
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sptr(tmem_slot)),
                     "r"(PF_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = *tmem_slot;
    pdl_wait();  // q (projection grid) and the image (the grid before this one)

    if (warp < 4) {
        // ---- query rows: row r = TMEM lane r = (token tl0 + r / GP, head slot r % GP)
        const int r = threadIdx.x;
        const int tl = tl0 + r / a.GP, hs = r % a.GP;
        const bool valid = tl < a.n && hs < a.G;
        const int limit = pos + min(tl, a.n - 1);  // the last key row this row sees
        const uint32_t lanes = taddr + (static_cast<uint32_t>(warp * 32) << 16);
        {  // the row's q as bf16 hi / lo into its TMEM lane (the A operand of S)
            const float4 *qr = reinterpret_cast<const float4 *>(
                a.q + (static_cast<size_t>(valid ? tl : 0) * a.H + g * a.G + (valid ? hs : 0)) * PF_HD);
#pragma unroll 1
            for (int ch = 0; ch < PF_HD / 32; ++ch) {
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float x[8];
                    const float4 u = valid ? qr[8 * ch + 2 * c] : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 w = valid ? qr[8 * ch + 2 * c + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w, x[4] = w.x, x[5] = w.y, x[6] = w.z, x[7] = w.w;
                    uint4 hi, lo;
                    bf_split8(x, hi, lo);
                    hw[4 * c] = hi.x, hw[4 * c + 1] = hi.y, hw[4 * c + 2] = hi.z, hw[4 * c + 3] = hi.w;
                    lw[4 * c] = lo.x, lw[4 * c + 1] = lo.y, lw[4 * c + 2] = lo.z, lw[4 * c + 3] = lo.w;
                }
                tm_st16(lanes + TC_Q + 16 * ch, hw);
                tm_st16(lanes + TC_Q + PF_HD / 2 + 16 * ch, lw);
            }
            tm_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);

        float m = -INFINITY, l = 0.0f;  // exp2 units
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            const int b = j & 1;
            // (wait results made warp-uniform: the TMEM accesses are warp-wide)
            if (!__all_sync(0xffffffffu, mbar_wait(s_full + b, (j >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float p[PF_N];
            {
                uint32_t v[PF_N / 16][16];
#pragma unroll
                for (int c = 0; c < PF_N / 16; ++c) tm_ld16(lanes + TC_S + b * PF_N + 16 * c, v[c]);
                tm_wait_ld();
#pragma unroll
                for (int c = 0; c < PF_N / 16; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i) p[16 * c + i] = __uint_as_float(v[c][i]);
            }
            const int k0 = j * PF_N;
            // the causal mask only where a row of this tile may end inside the
            // key tile (the same for the whole CTA: its first token's limit)
            if (k0 + PF_N - 1 > pos + tl0) {
#pragma unroll
                for (int c = 0; c < PF_N; ++c)
                    if (k0 + c > limit) p[c] = -INFINITY;
            }
            // maximum on the raw scores (the scale is positive), then one FMA per exp2
            float mr = -INFINITY;
#pragma unroll
            for (int c = 0; c < PF_N; ++c) mr = fmaxf(mr, p[c]);
            const float mt = mr * a.scale_log2;
            float alpha = 1.0f;
            bool rescale = false;
            if (mt > m + PF_TAU) {
                alpha = exp2f(m - mt);  // 0 on the first tile
                rescale = j > 0;
                l *= alpha;
                m = mt;
            }
            float ps = 0.0f;
            const float nm = -m;
#pragma unroll
            for (int c = 0; c < PF_N; ++c) {
                p[c] = exp2f(fmaf(p[c], a.scale_log2, nm));
                ps += p[c];
            }
            l += ps;
            if (__any_sync(0xffffffffu, rescale)) {  // O must hold every earlier tile's P.V first
                if (!__all_sync(0xffffffffu, mbar_wait(o_full + (b ^ 1), ((j - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[16];
#pragma unroll 1
                for (int c = 0; c < PF_HD / 16; ++c) {
                    tm_ld16(lanes + TC_O + 16 * c, v);
                    tm_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tm_st16(lanes + TC_O + 16 * c, v);
                }
            }
            if (j >= 2) {  // P buffer b was last read by the P.V of tile j - 2
                if (!__all_sync(0xffffffffu, mbar_wait(o_full + b, ((j - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
#pragma unroll
            for (int h = 0; h < PF_N / 32; ++h) {
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = p[32 * h + 8 * c + i];
                    uint4 hi, lo;
                    bf_split8(x, hi, lo);
                    hw[4 * c] = hi.x, hw[4 * c + 1] = hi.y, hw[4 * c + 2] = hi.z, hw[4 * c + 3] = hi.w;
                    lw[4 * c] = lo.x, lw[4 * c + 1] = lo.y, lw[4 * c + 2] = lo.z, lw[4 * c + 3] = lo.w;
                }
                tm_st16(lanes + TC_P + b * PF_N + 16 * h, hw);
                tm_st16(lanes + TC_P + b * PF_N + PF_N / 2 + 16 * h, lw);
            }
            tm_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + b);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_full + ((nkt - 1) & 1), ((nkt - 1) >> 1) & 1));
        if (!ok) flag_error(a.o.status, FLAG_TIMEOUT);
        tc_fence_after();
        // ---- output rows: O / l staged in shared memory (the key stages are
        // free: every MMA has completed), then one warp per row and output
        // block through the decode attention's store
        float *stg = reinterpret_cast<float *>(skv);
        {
            const float inv_ok = ok ? 1.0f : 0.0f;
            uint32_t v[16];
#pragma unroll 1
            for (int c = 0; c < PF_HD / 16; ++c) {
                tm_ld16(lanes + TC_O + 16 * c, v);
                tm_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    stg[r * (PF_HD + 1) + 16 * c + i] = inv_ok * __fdiv_rn(__uint_as_float(v[i]), l);
            }
        }
        tc_fence_before();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int rr = warp; rr < PF_M; rr += 4) {
            const int t2 = tl0 + rr / a.GP, h2 = rr % a.GP;
            if (t2 >= a.n || h2 >= a.G) continue;
#pragma unroll
            for (int blk = 0; blk < PF_HD / 32; ++blk)
                combine_store<PF_HD>(a.o, t2, g * a.G + h2, blk, lane, stg[rr * (PF_HD + 1) + blk * 32 + lane]);
        }
    } else if (warp == 4) {
        // ---- copies: key tile j into stage j % 3 once the MMAs of tile j - 3 are done
        if (lane == 0) {
            const uint8_t *src = a.img + static_cast<size_t>(g) * a.ntk * PF_TILE;
            for (int j = 0; j < nkt; ++j) {
                const int st = j % PF_NST;
                if (j >= PF_NST && !mbar_wait(kv_empty + st, ((j / PF_NST) - 1) & 1)) {
                    flag_error(a.o.status, FLAG_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(kv_full + st, PF_TILE);
                bulk_g2s(skv + static_cast<size_t>(st) * PF_TILE, src + static_cast<size_t>(j) * PF_TILE, PF_TILE,
                         kv_full + st);
            }
        }
        __syncwarp();
    } else {
        // ---- MMA issue: S of tile j + 1 goes in before P.V of tile j.  The A
        // operands (Q, P) are read from TMEM, the B operands (K, V^T) from
        // the stages.
        if (lane == 0) {
            constexpr uint32_t IDS = pf_idesc(PF_M, PF_N), IDO = pf_idesc(PF_M, PF_HD);
            auto issue_s = [&](int j) -> bool {
                const int st = j % PF_NST;
                if (!mbar_wait(kv_full + st, (j / PF_NST) & 1)) return false;
                tc_fence_after();
                const uint64_t kd = pf_desc(sptr(skv + static_cast<size_t>(st) * PF_TILE), PF_HD * 16);
                const uint32_t d = taddr + TC_S + (j & 1) * PF_N;
#pragma unroll
                for (int ks = 0; ks < PF_HD / 16; ++ks)
#pragma unroll
                    for (int term = 0; term < 3; ++term) {  // hi.hi, hi.lo, lo.hi
                        const uint32_t at = taddr + TC_Q + (term == 2 ? PF_HD / 2 : 0) + ks * 8;
                        const uint64_t bd = kd + (term == 1 ? PF_K_PART / 16 : 0) + ks * 16;
                        pf_mma_ts(d, at, bd, IDS, ks > 0 || term > 0);
                    }
                pf_commit(s_full + (j & 1));
                return true;
            };
            bool ok = mbar_wait(q_ready, 0);
            if (ok) {
                tc_fence_after();
                ok = issue_s(0);
            }
            for (int j = 0; j < nkt && ok; ++j) {
                if (j + 1 < nkt && !(ok = issue_s(j + 1))) break;
                const int b = j & 1;
                if (!(ok = mbar_wait(p_full + b, (j >> 1) & 1))) break;
                tc_fence_after();
                const int st = j % PF_NST;
                const uint64_t vd = pf_desc(sptr(skv + static_cast<size_t>(st) * PF_TILE + 2 * PF_K_PART), PF_N * 16);
#pragma unroll
                for (int ks = 0; ks < PF_N / 16; ++ks)
#pragma unroll
                    for (int term = 0; term < 3; ++term) {
                        const uint32_t at = taddr + TC_P + b * PF_N + (term == 2 ? PF_N / 2 : 0) + ks * 8;
                        const uint64_t bd = vd + (term == 1 ? PF_V_PART / 16 : 0) + ks * 16;
                        pf_mma_ts(taddr + TC_O, at, bd, IDO, j > 0 || ks > 0 || term > 0);
                    }
                pf_commit(o_full + b);
                pf_commit(kv_empty + st);
            }
            if (!ok) flag_error(a.o.status, FLAG_TIMEOUT);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(PF_TMEM_COLS));
}

}  // namespace

bool prefill_tc_ok(int H, int KV, int hd) {
    const int G = H / KV;
    return hd == PF_HD && G >= 1 && G <= 16;
}

size_t prefill_img_bytes(int KV, int C) {
    return static_cast<size_t>(KV) * ((C + PF_N - 1) / PF_N) * PF_TILE;
}

int launch_prefill_attn(const AttnArgs &o, const float *q, const float *k_cache, const float *v_cache, uint8_t *img,
                        int n, int pos, const int32_t *d_pos, int H, int KV, int C, cudaStream_t s) {
    PfArgs a{};
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.q = q;
    a.img = img;
    a.C = C;
    a.ntk = (C + PF_N - 1) / PF_N;
    a.n = n;
    a.pos = pos;
    a.d_pos = d_pos;
    a.H = H;
    a.KV = KV;
    a.G = H / KV;
    int gp = 1;
    while (gp < a.G) gp <<= 1;
    a.GP = gp;
    a.TPT = PF_M / gp;
    a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(PF_HD));
    a.o = o;
    void *args[] = {&a};
    // the image's tiles: those of the chunk's rows, or every tile of the
    // capacity when the position is read on the device
    const int tiles = d_pos ? a.ntk : (pos + n + PF_N - 1) / PF_N;
    cudaError_t e = launch(reinterpret_cast<const void *>(k_pf_kv_image), dim3(tiles, KV), dim3(256), 0, s, true, args);
    if (e != cudaSuccess) return -5;
    const void *fn = reinterpret_cast<const void *>(k_pf_attn);
    ensure_smem(fn, PF_SMEM);
    e = launch(fn, dim3((n + a.TPT - 1) / a.TPT, KV), dim3(PF_THREADS), PF_SMEM, s, true, args);
    return e == cudaSuccess ? 0 : -5;
}

}  // namespace ck
