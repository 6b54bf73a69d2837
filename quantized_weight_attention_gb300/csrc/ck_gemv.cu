// Projection kernels of the decode step (sm_103a):
//   - Q8_0 quantization of an fp32 vector (quantize_row_q8_0),
//   - Q5_0 x Q8_0 and Q8_0 x Q8_0 GEMV + bias (gemv_q5_0_from_fp32 /
//     gemv_q8_0_from_fp32 after their quantize step),
//   - the layer's fused Q|K|V projection: RMSNorm + Q8_0 quantization in
//     the prologue, the three GEMVs, bias + RoPE + KV-cache store in the
//     epilogue (page "mega_fused_attention_decode_q5_0.c", STEP 1-6),
//   - the layer's O projection with bias and residual (STEP 8).
//
// Weight streaming.  When a row holds a multiple of 8 blocks (K % 256 == 0)
// every 8-block segment (176 B for Q5_0, 272 B for Q8_0) is 16-byte aligned.
// A CTA then owns a tile of rows, copies each row into padded shared memory
// with the bulk-copy engine at kernel start (all of the CTA's bytes in
// flight at once, before the activation is even known), and each lane
// decodes one whole segment from 16-byte shared loads with compile-time
// byte offsets: lane = (row within a 16-row group, one of two segment
// columns).  Rows of other widths take a direct path: a warp per row, a
// lane per block, aligned 32-bit global loads that never leave the block.
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

// ---------------------------------------------------------------------------
// Shared-memory plan of a projection CTA (identical on host and device)
// ---------------------------------------------------------------------------
struct ProjSmem {
    size_t off_w, off_xq, off_xd, off_xs, off_part, off_rowsum, off_red, off_raw, total;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// R: max rows per CTA; nb: blocks per row; wbytes: bytes of the staged
// weight rows (0 on the direct path).
__host__ __device__ inline ProjSmem proj_smem(int R, int nb, size_t wbytes) {
    ProjSmem s;
    size_t o = 128;  // mbarriers (up to 16)
    s.off_w = o;
    o = align_up(o + wbytes, 16);
    s.off_xq = o;
    o += static_cast<size_t>(xq_chunks(nb)) * 16;
    s.off_xd = o;
    o += static_cast<size_t>(nb) * 4;
    s.off_xs = o;
    o += static_cast<size_t>(nb) * 4;
    o = align_up(o, 16);
    s.off_part = o;
    o += static_cast<size_t>(nb / 8 + 1) * R * 4;
    s.off_rowsum = o;
    o += static_cast<size_t>(R) * 4;
    s.off_red = o;
    o += 64 * 4;
    s.off_raw = o;  // raw bytes of a Q8_0 activation row
    o = align_up(o + static_cast<size_t>(nb) * Q8B + 16, 16);
    s.total = align_up(o, 128);
    return s;
}

__host__ __device__ inline int row_stride(int nb, bool q8) { return nb * (q8 ? Q8B : Q5B) + 16; }

// ---------------------------------------------------------------------------
// Activation prologues
// ---------------------------------------------------------------------------
// Q8_0 blocks already in global memory (4-byte aligned) -> XRow in shared
// memory.  Every global load of the row is issued before any is used (a few
// 32-bit words per thread), then the blocks are unpacked from shared memory.
// `raw` holds nb*34 bytes (+ slack).
__device__ void xrow_from_q8(const uint8_t *xq8, int nb, const XRow &x, uint32_t *raw) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int bytes = nb * Q8B;  // even
    const int words = bytes >> 2;
    const uint32_t *src = reinterpret_cast<const uint32_t *>(xq8);
    constexpr int U = 4;
    for (int base = 0; base < words; base += U * static_cast<int>(blockDim.x)) {
        uint32_t v[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int i = base + k * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
            v[k] = i < words ? __ldg(src + i) : 0u;
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int i = base + k * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
            if (i < words) raw[i] = v[k];
        }
    }
    if ((bytes & 2) && threadIdx.x == 0)
        reinterpret_cast<uint16_t *>(raw)[(bytes >> 1) - 1] =
            __ldg(reinterpret_cast<const unsigned short *>(xq8) + (bytes >> 1) - 1);
    __syncthreads();
    const uint8_t *rb = reinterpret_cast<const uint8_t *>(raw);
    for (int b = warp; b < nb; b += nw) {
        const uint8_t *p = rb + b * Q8B;
        const int c = static_cast<int8_t>(p[2 + lane]);
        const int sum = warp_isum(c);
        reinterpret_cast<int8_t *>(&x.q[xq_chunk(b, lane >> 4)])[lane & 15] = static_cast<int8_t>(c);
        if (lane == 0) {
            x.d[b] = half_bits_to_float(static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8));
            x.sum[b] = sum;
        }
    }
    __syncthreads();  // the row is complete before any warp reads it
}

// rstd of RMSNorm (rmsnorm_forward, T = 1) over x[0..D), for every thread
// of the CTA.  All loads of x are issued before any is used.
__device__ float block_rstd(const float *x, int D, float eps, float *red) {
    constexpr int PE = 8;
    float s = 0.0f, c = 0.0f;
    for (int i0 = 0; i0 < D; i0 += PE * static_cast<int>(blockDim.x)) {
        float v[PE];
#pragma unroll
        for (int k = 0; k < PE; ++k) {
            const int i = i0 + k * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
            v[k] = i < D ? x[i] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < PE; ++k) sumsq_add(v[k], s, c);
    }
    return rstd_from_pairs(s, c, D, eps, red);
}

// A packed activation row (the XRow image, written by its producer kernel)
// copied into the CTA's XRow: one 16-byte load per thread.
__device__ void xrow_from_pack(const uint8_t *pack, int nb, const XRow &xr) {
    const int n16 = static_cast<int>(xpack_bytes(nb) / 16);
    int4 *dst = xr.q;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldcg(reinterpret_cast<const int4 *>(pack) + i);
    __syncthreads();
}

__device__ __forceinline__ XRow xrow_at(uint8_t *smem, const ProjSmem &L) {
    XRow x;
    x.q = reinterpret_cast<int4 *>(smem + L.off_xq);
    x.d = reinterpret_cast<float *>(smem + L.off_xd);
    x.sum = reinterpret_cast<int *>(smem + L.off_xs);
    return x;
}

// ---------------------------------------------------------------------------
// Tile machinery
// ---------------------------------------------------------------------------
// Warp 0 starts the bulk copies of the tile's rows: row i of the tile is
// global row rowof(i); rows are grouped by 16 onto one mbarrier each.
template <typename RowFn>
__device__ void issue_rows(uint8_t *wsm, int rstride, const uint8_t *W, int rb, int rows, uint64_t *bars,
                           RowFn rowof) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        if (lane == 0)
            for (int g = 0; g * 16 < rows; ++g)
                mbar_arrive_expect_tx(&bars[g], static_cast<uint32_t>(min(16, rows - 16 * g) * rb));
        __syncwarp();
        for (int i = lane; i < rows; i += 32)
            bulk_g2s(wsm + static_cast<size_t>(i) * rstride, W + static_cast<size_t>(rowof(i)) * rb,
                     static_cast<uint32_t>(rb), &bars[i >> 4]);
    }
}

__device__ __forceinline__ void init_bars(uint64_t *bars, int n) {
    if (threadIdx.x == 0) {
        for (int g = 0; g < n; ++g) mbar_init(&bars[g], 1);
        fence_mbar_init();
    }
}

// Segment partial sums of the staged rows: part[k * R + i] for row i and
// segment column k.
template <bool Q8>
__device__ void tile_segments(const uint8_t *wsm, int rstride, int rows, int R, int nseg, uint64_t *bars,
                              const XRow &x, float *part, unsigned *status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int npairs = (nseg + 1) >> 1;
    const int ngroups = (rows + 15) >> 4;
    for (int t = warp; t < ngroups * npairs; t += nw) {
        const int g = t / npairs, cp = t - g * npairs;
        const int i = (g << 4) + (lane & 15);
        const int k = (cp << 1) + (lane >> 4);
        if (!mbar_wait(&bars[g], 0)) flag_error(status, FLAG_TIMEOUT);
        if (i < rows && k < nseg)
            part[k * R + i] = seg_dot<Q8>(
                reinterpret_cast<const uint4 *>(wsm + static_cast<size_t>(i) * rstride + k * SegShape<Q8>::BYTES),
                x, k * 8);
    }
}

// rowsum[i] = sum_k part[k * R + i], 8 lanes per row, fixed order.
__device__ void reduce_rows(const float *part, int R, int rows, int nseg, float *rowsum) {
    const int n = (rows * 8 + 31) & ~31;
    for (int it = threadIdx.x; it < n; it += blockDim.x) {
        const int i = it >> 3, sub = it & 7;
        float s = 0.0f;
        if (i < rows)
            for (int k = sub; k < nseg; k += 8) s += part[k * R + i];
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        if (sub == 0 && i < rows) rowsum[i] = s;
    }
}

// Direct path: a warp per row, a lane per block.
template <bool Q8, typename RowFn>
__device__ void tile_direct(const uint8_t *W, int nb, int rows, RowFn rowof, const XRow &x, float *rowsum) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    constexpr int BLK = Q8 ? Q8B : Q5B;
    for (int i = warp; i < rows; i += nw) {
        const size_t r = static_cast<size_t>(rowof(i));
        float acc = 0.0f;
        for (int b = lane; b < nb; b += 32) acc += block_dot_global<Q8>(W, (r * nb + b) * BLK, x, b);
        acc = warp_sum(acc);
        if (lane == 0) rowsum[i] = acc;
    }
}

// ---------------------------------------------------------------------------
// Standalone kernels
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quantize_q8_0(const float *__restrict__ x, uint8_t *__restrict__ y, int nb) {
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= nb) return;
    const int lane = threadIdx.x & 31;
    uint32_t dbits;
    float dq;
    const int q = q8_code(x[static_cast<size_t>(b) * QK + lane], dbits, dq);
    uint8_t *o = y + static_cast<size_t>(b) * Q8B;
    o[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    if (lane == 0) {
        o[0] = static_cast<uint8_t>(dbits & 0xFF);
        o[1] = static_cast<uint8_t>(dbits >> 8);
    }
}

template <bool Q8, bool FAST>
__global__ void __launch_bounds__(512) k_gemv(float *__restrict__ y, const uint8_t *__restrict__ W,
                                              const uint8_t *__restrict__ xq8, const float *__restrict__ bias,
                                              int M, int K, int R, unsigned *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int nb = K / QK, nseg = nb / 8;
    const int rb = nb * (Q8 ? Q8B : Q5B);
    const int rstride = row_stride(nb, Q8);
    const int r0 = blockIdx.x * R;
    const int rows = min(R, M - r0);
    const ProjSmem L = proj_smem(R, nb, FAST ? static_cast<size_t>(R) * rstride : 0);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *wsm = smem + L.off_w;
    float *part = reinterpret_cast<float *>(smem + L.off_part);
    float *rowsum = reinterpret_cast<float *>(smem + L.off_rowsum);
    const XRow x = xrow_at(smem, L);
    auto rowof = [r0](int i) { return r0 + i; };
    if constexpr (FAST) {
        init_bars(bars, (rows + 15) >> 4);
        __syncthreads();
        issue_rows(wsm, rstride, W, rb, rows, bars, rowof);
    }
    xrow_from_q8(xq8, nb, x, reinterpret_cast<uint32_t *>(smem + L.off_raw));
    __syncthreads();
    if constexpr (FAST) {
        tile_segments<Q8>(wsm, rstride, rows, R, nseg, bars, x, part, status);
        __syncthreads();
        reduce_rows(part, R, rows, nseg, rowsum);
    } else {
        tile_direct<Q8>(W, nb, rows, rowof, x, rowsum);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < rows; i += blockDim.x) y[r0 + i] = rowsum[i] + (bias ? bias[r0 + i] : 0.0f);
}

// Per-block int32 dots with the GEMV's own decode path (test access).
template <bool Q8>
__global__ void __launch_bounds__(256) k_block_dots(int32_t *__restrict__ isum, const uint8_t *__restrict__ W,
                                                    const uint8_t *__restrict__ xq8, int M, int K) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int nb = K / QK;
    const ProjSmem L = proj_smem(1, nb, 0);
    const XRow x = xrow_at(smem, L);
    xrow_from_q8(xq8, nb, x, reinterpret_cast<uint32_t *>(smem + L.off_raw));
    __syncthreads();
    constexpr int BLK = Q8 ? Q8B : Q5B;
    if (nb % 8 == 0) {
        const int nseg = nb / 8;
        const long task = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (task >= static_cast<long>(M) * nseg) return;
        const long r = task / nseg, k = task % nseg;
        const uint4 *seg = reinterpret_cast<const uint4 *>(W + (r * nb + k * 8) * BLK);
        int out[8];
        seg_dot<Q8>(seg, x, static_cast<int>(k) * 8, out);
#pragma unroll
        for (int j = 0; j < 8; ++j) isum[r * nb + k * 8 + j] = out[j];
    } else {
        const long task = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
        if (task >= static_cast<long>(M) * nb) return;
        const long r = task / nb, b = task % nb;
        int out;
        block_dot_global<Q8>(W, static_cast<size_t>(r * nb + b) * BLK, x, static_cast<int>(b), &out);
        isum[r * nb + b] = out;
    }
}

// ---------------------------------------------------------------------------
// The layer's projections (STEP 1-6 and STEP 8)
// ---------------------------------------------------------------------------
// K0: RMSNorm + Q8_0 quantization of the layer input into the scratch, for
// every projection CTA to load.  CTA c quantizes blocks [c*W, c*W + W) of the
// W warps it has, one block per warp (y = (x * rstd) * gamma in fp32, then
// quantize_row_q8_0); each CTA recomputes the cheap sum of squares itself.
__global__ void __launch_bounds__(512) k_norm_q8(const QkvArgs a) {
    __shared__ float red[64];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int pos = a.d_pos ? *a.d_pos : a.pos;
    if (pos < 0 || pos >= a.C) {  // nothing of the step is written
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.status, FLAG_RANGE);
        pdl_wait();  // completion of this grid still implies completion of the one before
        return;
    }
    pdl_trigger();
    pdl_wait();  // x may be the previous layer's output
    const int b = blockIdx.x * nw + warp;
    const int nb = a.D / QK;
    float xv = 0.0f, gv = 0.0f;
    if (b < nb) {
        xv = a.x[b * QK + lane];
        gv = a.gamma[b * QK + lane];
    }
    const float rstd = block_rstd(a.x, a.D, a.eps, red);
    if (b >= nb) return;  // warp-uniform
    const float y = __fmul_rn(__fmul_rn(xv, rstd), gv);
    uint32_t dbits;
    float dq;
    const int q = q8_code(y, dbits, dq);
    uint8_t *o = a.xq8 + static_cast<size_t>(b) * Q8B;
    o[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    if (lane == 0) {
        o[0] = static_cast<uint8_t>(dbits & 0xFF);
        o[1] = static_cast<uint8_t>(dbits >> 8);
    }
}

// Warp tasks.  A warp owns two weight rows: a RoPE pair (rows h*hd + i and
// h*hd + hd/2 + i) for Q and K, two consecutive rows for V and O.  Its lane
// 0 copies both rows into the warp's own shared-memory slot with the
// bulk-copy engine at kernel start (before waiting on the preceding grid);
// lanes 0-15 decode the segments of the first row and lanes 16-31 those of
// the second, a shuffle tree sums them, and lane 0 runs the epilogue.  No
// CTA-wide barrier follows the activation prologue.
struct QkvTask {
    int kind;  // 0 = Q, 1 = K, 2 = V, 3 = none
    int ra, rb, head, i;
};

__device__ __forceinline__ QkvTask qkv_task(const QkvArgs &a, int t) {
    QkvTask T{};
    const int half = a.hd >> 1;
    const int nq = a.H * half, nk = a.KV * half, nv = (a.KV * a.hd) >> 1;
    if (t < nq) {
        T.kind = 0;
        T.head = t / half;
        T.i = t - T.head * half;
    } else if (t < nq + nk) {
        T.kind = 1;
        T.head = (t - nq) / half;
        T.i = (t - nq) - T.head * half;
    } else if (t < nq + nk + nv) {
        T.kind = 2;
        T.ra = 2 * (t - nq - nk);
        T.rb = T.ra + 1;
        return T;
    } else {
        T.kind = 3;
        return T;
    }
    T.ra = T.head * a.hd + T.i;
    T.rb = T.ra + half;
    return T;
}

__host__ __device__ int qkv_tasks(const QkvArgs &a) { return (a.H + a.KV) * (a.hd >> 1) + ((a.KV * a.hd) >> 1); }

// Bulk copy of `bytes` (a multiple of 16) in pieces of at most 64 KB.  The
// copy engine of an SM takes one bulk copy per few hundred cycles whatever its
// size, so weight rows are staged in as few, large copies as possible.
__device__ void bulk_g2s_run(uint8_t *dst, const uint8_t *src, uint32_t bytes, uint64_t *bar) {
    for (uint32_t o = 0; o < bytes; o += 65536u) bulk_g2s(dst + o, src + o, bytes - o < 65536u ? bytes - o : 65536u, bar);
}

// Shared-memory rows of warp w's task: Q/K pairs go to an A block (row ra of
// warp w at slot w) and a B block (row rb at slot nw + w), so that the rows
// of consecutive RoPE pairs of one head are contiguous in both places; V
// pairs (rows 2u, 2u + 1) sit side by side.
__device__ __forceinline__ uint8_t *qkv_slot(uint8_t *wst, int kind, int w, int nw, int second, int rb5, int rb8) {
    if (kind == 2) return wst + static_cast<size_t>(2 * w + second) * rb8;
    return wst + static_cast<size_t>(second ? nw + w : w) * rb5;
}

// Thread 0: stage this CTA's Q/K/V rows, completing on `bar`.  When the
// CTA's tasks are consecutive pairs of one head (or all V pairs), that is
// two copies (one); otherwise two copies per task.
__device__ void stage_qkv_rows(const QkvArgs &a, int nw, uint8_t *wst, uint64_t *bar, int rb5, int rb8) {
    const int t0 = blockIdx.x * nw;
    const int nt = min(nw, qkv_tasks(a) - t0);
    mbar_init(bar, 1);
    fence_mbar_init();
    const QkvTask f = qkv_task(a, t0), l = qkv_task(a, t0 + nt - 1);
    const uint8_t *Wf = f.kind == 0 ? a.wq : (f.kind == 1 ? a.wk : a.wv);
    if (f.kind == 2 && l.kind == 2) {
        const uint32_t bytes = static_cast<uint32_t>(2 * nt * rb8);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_run(wst, Wf + static_cast<size_t>(f.ra) * rb8, bytes, bar);
        return;
    }
    if (f.kind == l.kind && f.kind < 2 && f.head == l.head && l.i - f.i == nt - 1) {
        const uint32_t bytes = static_cast<uint32_t>(nt * rb5);
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s_run(wst, Wf + static_cast<size_t>(f.ra) * rb5, bytes, bar);
        bulk_g2s_run(wst + static_cast<size_t>(nw) * rb5, Wf + static_cast<size_t>(f.rb) * rb5, bytes, bar);
        return;
    }
    uint32_t total = 0;
    for (int w = 0; w < nt; ++w) total += static_cast<uint32_t>(2 * (qkv_task(a, t0 + w).kind == 2 ? rb8 : rb5));
    mbar_arrive_expect_tx(bar, total);
    for (int w = 0; w < nt; ++w) {
        const QkvTask T = qkv_task(a, t0 + w);
        const uint8_t *W = T.kind == 0 ? a.wq : (T.kind == 1 ? a.wk : a.wv);
        const int rb = T.kind == 2 ? rb8 : rb5;
        bulk_g2s(qkv_slot(wst, T.kind, w, nw, 0, rb5, rb8), W + static_cast<size_t>(T.ra) * rb, rb, bar);
        bulk_g2s(qkv_slot(wst, T.kind, w, nw, 1, rb5, rb8), W + static_cast<size_t>(T.rb) * rb, rb, bar);
    }
}

// Sum over the segments [li, li + 16, ...) of one staged row, then over the
// 16 lanes of each half-warp (lane 0: first row, lane 16: second row).
template <bool Q8>
__device__ __forceinline__ float warp_row_dot(const uint8_t *row, int nseg, int li, const XRow &x) {
    float acc = 0.0f;
    for (int k = li; k < nseg; k += 16)
        acc += seg_dot<Q8>(reinterpret_cast<const uint4 *>(row + k * SegShape<Q8>::BYTES), x, k * 8);
    acc += __shfl_xor_sync(0xffffffffu, acc, 8);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    return acc;
}

__global__ void __launch_bounds__(512, 1) k_qkv_w(const QkvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int nb = a.D / QK, nseg = nb / 8;
    const int rb5 = nb * Q5B, rb8 = nb * Q8B;
    const ProjSmem L = proj_smem(1, nb, static_cast<size_t>(nw) * 2 * rb8);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);  // the CTA's weight rows
    uint8_t *wst = smem + L.off_w;
    const XRow x = xrow_at(smem, L);
    const QkvTask T = qkv_task(a, blockIdx.x * nw + warp);
    const int pos = a.d_pos ? *a.d_pos : a.pos;
    if (pos < 0 || pos >= a.C) {  // nothing of the step is written
        if (a.fused_norm && blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.status, FLAG_RANGE);
        pdl_wait();
        return;
    }
    const bool q8 = T.kind == 2;
    if (threadIdx.x == 0) stage_qkv_rows(a, nw, wst, bar, rb5, rb8);  // the weights do not depend on earlier grids
    // the epilogue's constant operands (biases, RoPE table entries) before the wait
    const int half = a.hd >> 1;
    float ea = 0.0f, eb = 0.0f, ec = 1.0f, es = 0.0f;
    if (lane == 0 && T.kind != 3) {
        const float *bias = T.kind == 0 ? a.bq : T.kind == 1 ? a.bk : a.bv;
        ea = bias ? bias[T.ra] : 0.0f;
        eb = bias ? bias[T.rb] : 0.0f;
        if (T.kind != 2) {
            ec = a.rope_cos[static_cast<size_t>(pos) * half + T.i];
            es = a.rope_sin[static_cast<size_t>(pos) * half + T.i];
        }
    }
    pdl_trigger();
    if (a.fused_norm) {
        float gv[NORM_XPW];  // gamma does not depend on the preceding grid
#pragma unroll
        for (int j = 0; j < NORM_XPW; ++j) {
            const int b = warp + nw * j;
            gv[j] = b < nb ? __ldg(a.gamma + b * QK + lane) : 0.0f;
        }
        pdl_wait();  // x may be the previous layer's output
        norm_quant_xrow(a.x, gv, nb, a.D, a.eps, x, reinterpret_cast<float *>(smem + L.off_red),
                        blockIdx.x == 0 ? a.xq8 : nullptr);
    } else {
        pdl_wait();  // the quantized input is ready
        xrow_from_q8(a.xq8, nb, x, reinterpret_cast<uint32_t *>(smem + L.off_raw));
    }
    if (T.kind == 3) return;
    if (!mbar_wait(bar, 0)) flag_error(a.status, FLAG_TIMEOUT);
    const uint8_t *row = qkv_slot(wst, T.kind, warp, nw, lane >> 4, rb5, rb8);
    const float acc = q8 ? warp_row_dot<true>(row, nseg, lane & 15, x) : warp_row_dot<false>(row, nseg, lane & 15, x);
    const float sb = __shfl_sync(0xffffffffu, acc, 16);
    if (lane != 0) return;
    if (T.kind == 2) {
        const float va = acc + ea;
        const float vb = sb + eb;
        int h = T.ra / a.hd;
        a.v_cache[(static_cast<size_t>(h) * a.C + pos) * a.hd + (T.ra - h * a.hd)] = va;
        h = T.rb / a.hd;
        a.v_cache[(static_cast<size_t>(h) * a.C + pos) * a.hd + (T.rb - h * a.hd)] = vb;
        return;
    }
    // bias, then rotate-half RoPE of the pair (i, i + hd/2) at row `pos`
    const float A = acc + ea;
    const float B = sb + eb;
    const float A2 = __fsub_rn(__fmul_rn(A, ec), __fmul_rn(B, es));
    const float B2 = __fadd_rn(__fmul_rn(A, es), __fmul_rn(B, ec));
    if (T.kind == 0) {
        a.q_out[T.ra] = A2;
        a.q_out[T.rb] = B2;
    } else {
        float *kr = a.k_cache + (static_cast<size_t>(T.head) * a.C + pos) * a.hd;
        kr[T.i] = A2;
        kr[T.i + half] = B2;
    }
}

__global__ void __launch_bounds__(512, 1) k_oproj_w(const OprojArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int nb = a.QD / QK, nseg = nb / 8;
    const int rb = nb * Q5B;
    const ProjSmem L = proj_smem(1, nb, static_cast<size_t>(nw) * 2 * rb);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);  // the CTA's rows of Wo
    uint8_t *slot = smem + L.off_w + static_cast<size_t>(warp) * 2 * rb;
    const XRow x = xrow_at(smem, L);
    const int r0 = 2 * (blockIdx.x * nw + warp);
    const bool valid = r0 < a.D;
    if (a.d_pos) {
        const int pos = *a.d_pos;
        if (pos < 0 || pos >= a.C) {
            pdl_wait();
            return;
        }
    }
    if (threadIdx.x == 0) {  // the CTA's rows are contiguous: one run of copies
        const int rw0 = 2 * blockIdx.x * nw, rw1 = min(a.D, rw0 + 2 * nw);
        const uint32_t bytes = static_cast<uint32_t>(rw1 - rw0) * rb;
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_run(smem + L.off_w, a.wo + static_cast<size_t>(rw0) * rb, bytes, bar);
    }
    // the bias (a constant input) before the wait; the residual may be the
    // previous layer's output, so it is loaded after the wait, ahead of the dot
    float ba = 0.0f, bb = 0.0f, ra = 0.0f, rbv = 0.0f;
    if (lane == 0 && valid && a.bo) {
        ba = a.bo[r0];
        bb = a.bo[r0 + 1];
    }
    pdl_trigger();
    pdl_wait();  // the attention output is ready
    if (lane == 0 && valid) {
        ra = a.residual[r0];
        rbv = a.residual[r0 + 1];
    }
    if (a.apack)
        xrow_from_pack(a.apack, nb, x);
    else
        xrow_from_q8(a.aq8, nb, x, reinterpret_cast<uint32_t *>(smem + L.off_raw));
    if (!valid) return;
    if (!mbar_wait(bar, 0)) flag_error(a.status, FLAG_TIMEOUT);
    const float acc = warp_row_dot<false>(slot + (lane >> 4) * rb, nseg, lane & 15, x);
    const float sb = __shfl_sync(0xffffffffu, acc, 16);
    if (lane == 0) {
        a.out[r0] = (acc + ba) + ra;
        a.out[r0 + 1] = (sb + bb) + rbv;
    }
}

// ---------------------------------------------------------------------------
// Direct path of the layer (rows whose block count is not a multiple of 8)
// ---------------------------------------------------------------------------
// Tiles: Q and K tiles hold 16 RoPE pairs of one head (rows h*hd + i0 + i
// and h*hd + hd/2 + i0 + i, i < 16), so the epilogue rotates without a
// second pass; V tiles hold rv consecutive rows.  A warp per row, a lane per
// block, aligned 32-bit global loads that never leave the block.
struct QkvTile {
    int kind;  // 0 = Q, 1 = K, 2 = V
    int head, i0, v0, rows;
};

__device__ __forceinline__ QkvTile qkv_tile(const QkvArgs &a, int t) {
    QkvTile T{};
    const int sub = a.hd >> 5;  // RoPE pair-tiles per head
    if (t < a.n_q_tiles) {
        T.kind = 0;
        T.head = t / sub;
        T.i0 = (t % sub) << 4;
        T.rows = 32;
    } else if (t < a.n_q_tiles + a.n_k_tiles) {
        const int u = t - a.n_q_tiles;
        T.kind = 1;
        T.head = u / sub;
        T.i0 = (u % sub) << 4;
        T.rows = 32;
    } else {
        T.kind = 2;
        T.v0 = (t - a.n_q_tiles - a.n_k_tiles) * a.rv;
        T.rows = min(a.rv, a.KV * a.hd - T.v0);
    }
    return T;
}

__global__ void __launch_bounds__(256) k_qkv_direct(const QkvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const QkvTile T = qkv_tile(a, blockIdx.x);
    const int half = a.hd >> 1;
    const int nb = a.D / QK;
    const bool q8 = T.kind == 2;
    const uint8_t *W = T.kind == 0 ? a.wq : (T.kind == 1 ? a.wk : a.wv);
    const ProjSmem L = proj_smem(max(32, a.rv), nb, 0);
    float *rowsum = reinterpret_cast<float *>(smem + L.off_rowsum);
    const XRow x = xrow_at(smem, L);
    auto rowof = [&](int i) {
        return T.kind == 2 ? T.v0 + i : T.head * a.hd + (i < 16 ? T.i0 + i : half + T.i0 + i - 16);
    };
    const int pos = a.d_pos ? *a.d_pos : a.pos;
    if (pos < 0 || pos >= a.C) {
        pdl_wait();
        return;
    }
    pdl_trigger();
    pdl_wait();  // the quantized input is ready
    xrow_from_q8(a.xq8, nb, x, reinterpret_cast<uint32_t *>(smem + L.off_raw));
    if (q8)
        tile_direct<true>(W, nb, T.rows, rowof, x, rowsum);
    else
        tile_direct<false>(W, nb, T.rows, rowof, x, rowsum);
    __syncthreads();
    if (T.kind == 2) {
        for (int i = threadIdx.x; i < T.rows; i += blockDim.x) {
            const int r = T.v0 + i;
            const float v = rowsum[i] + (a.bv ? a.bv[r] : 0.0f);
            const int h = r / a.hd, d = r - h * a.hd;
            a.v_cache[(static_cast<size_t>(h) * a.C + pos) * a.hd + d] = v;
        }
    } else if (threadIdx.x < 16) {
        const int i = threadIdx.x, d = T.i0 + i;
        const int ra = rowof(i), rb2 = rowof(16 + i);
        const float *bias = T.kind == 0 ? a.bq : a.bk;
        const float A = rowsum[i] + (bias ? bias[ra] : 0.0f);
        const float B = rowsum[16 + i] + (bias ? bias[rb2] : 0.0f);
        const float c = a.rope_cos[static_cast<size_t>(pos) * half + d];
        const float s = a.rope_sin[static_cast<size_t>(pos) * half + d];
        const float A2 = __fsub_rn(__fmul_rn(A, c), __fmul_rn(B, s));
        const float B2 = __fadd_rn(__fmul_rn(A, s), __fmul_rn(B, c));
        if (T.kind == 0) {
            a.q_out[ra] = A2;
            a.q_out[rb2] = B2;
        } else {
            float *kr = a.k_cache + (static_cast<size_t>(T.head) * a.C + pos) * a.hd;
            kr[d] = A2;
            kr[d + half] = B2;
        }
    }
}

__global__ void __launch_bounds__(256) k_oproj_direct(const OprojArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int nb = a.QD / QK;
    const int R = a.rows_per_cta;
    const int r0 = blockIdx.x * R;
    const int rows = min(R, a.D - r0);
    const ProjSmem L = proj_smem(R, nb, 0);
    float *rowsum = reinterpret_cast<float *>(smem + L.off_rowsum);
    const XRow x = xrow_at(smem, L);
    auto rowof = [r0](int i) { return r0 + i; };
    if (a.d_pos) {
        const int pos = *a.d_pos;
        if (pos < 0 || pos >= a.C) {
            pdl_wait();
            return;
        }
    }
    pdl_trigger();
    pdl_wait();  // the attention output is ready
    xrow_from_q8(a.aq8, nb, x, reinterpret_cast<uint32_t *>(smem + L.off_raw));
    tile_direct<false>(a.wo, nb, rows, rowof, x, rowsum);
    __syncthreads();
    for (int i = threadIdx.x; i < rows; i += blockDim.x) {
        const int r = r0 + i;
        a.out[r] = (rowsum[i] + (a.bo ? a.bo[r] : 0.0f)) + a.residual[r];
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
static int cuda_status(cudaError_t e) { return e == cudaSuccess ? 0 : -5; }

template <typename F>
static void set_smem(F *fn, size_t bytes) {
    ensure_smem(reinterpret_cast<const void *>(fn), bytes);
}

int launch_quantize_q8_0(const float *x, void *y, int n, cudaStream_t s) {
    const int nb = n / QK;
    const int wpb = 8;
    k_quantize_q8_0<<<(nb + wpb - 1) / wpb, 32 * wpb, 0, s>>>(x, static_cast<uint8_t *>(y), nb);
    return cuda_status(cudaGetLastError());
}

// Rows per CTA for a standalone GEMV: about one CTA per SM, at most 64 rows
// (4 mbarrier groups) and at most ~200 KB of staged rows.
static int gemv_rows_per_cta(int M, int nb, bool q8) {
    const DeviceInfo &di = device_info();
    int R = (M + di.num_sms - 1) / di.num_sms;
    const int rs = row_stride(nb, q8);
    const int cap = static_cast<int>((di.smem_optin - 16384) / static_cast<size_t>(rs));
    R = R < 1 ? 1 : R;
    R = R > 64 ? 64 : R;
    return R > cap ? cap : R;
}

int launch_gemv(bool q8, float *y, const void *W, const void *xq8, const float *bias, int M, int K, cudaStream_t s) {
    const int nb = K / QK;
    const uint8_t *w = static_cast<const uint8_t *>(W);
    const uint8_t *x = static_cast<const uint8_t *>(xq8);
    const bool fast = (nb % 8 == 0) && gemv_rows_per_cta(M, nb, q8) >= 1;
    if (fast) {
        const int R = gemv_rows_per_cta(M, nb, q8);
        const ProjSmem L = proj_smem(R, nb, static_cast<size_t>(R) * row_stride(nb, q8));
        const int grid = (M + R - 1) / R;
        const int tasks = ((R + 15) / 16) * ((nb / 8 + 1) / 2);
        const int threads = 32 * (tasks < 1 ? 1 : (tasks > 16 ? 16 : tasks));
        if (q8) {
            set_smem(k_gemv<true, true>, L.total);
            k_gemv<true, true><<<grid, threads, L.total, s>>>(y, w, x, bias, M, K, R, status_word());
        } else {
            set_smem(k_gemv<false, true>, L.total);
            k_gemv<false, true><<<grid, threads, L.total, s>>>(y, w, x, bias, M, K, R, status_word());
        }
    } else {
        const int R = 8;
        const ProjSmem L = proj_smem(R, nb, 0);
        const int grid = (M + R - 1) / R;
        if (q8) {
            set_smem(k_gemv<true, false>, L.total);
            k_gemv<true, false><<<grid, 256, L.total, s>>>(y, w, x, bias, M, K, R, status_word());
        } else {
            set_smem(k_gemv<false, false>, L.total);
            k_gemv<false, false><<<grid, 256, L.total, s>>>(y, w, x, bias, M, K, R, status_word());
        }
    }
    return cuda_status(cudaGetLastError());
}

int launch_block_dots(bool q8, int32_t *isum, const void *W, const void *xq8, int M, int K, cudaStream_t s) {
    const int nb = K / QK;
    const ProjSmem L = proj_smem(1, nb, 0);
    const long tasks = (nb % 8 == 0) ? static_cast<long>(M) * (nb / 8) : static_cast<long>(M) * nb;
    const int grid = static_cast<int>((tasks + 255) / 256);
    const uint8_t *w = static_cast<const uint8_t *>(W);
    const uint8_t *x = static_cast<const uint8_t *>(xq8);
    if (q8) {
        set_smem(k_block_dots<true>, L.total);
        k_block_dots<true><<<grid, 256, L.total, s>>>(isum, w, x, M, K);
    } else {
        set_smem(k_block_dots<false>, L.total);
        k_block_dots<false><<<grid, 256, L.total, s>>>(isum, w, x, M, K);
    }
    return cuda_status(cudaGetLastError());
}

void plan_qkv(QkvArgs &a) {
    const DeviceInfo &di = device_info();
    const int sub = a.hd / 32;
    a.n_q_tiles = a.H * sub;
    a.n_k_tiles = a.KV * sub;
    const int KD = a.KV * a.hd;
    const int rem = di.num_sms - a.n_q_tiles - a.n_k_tiles;
    int rv = rem > 0 ? (KD + rem - 1) / rem : 32;
    rv = rv < 8 ? 8 : (rv > 48 ? 48 : rv);
    a.rv = rv;
}

// Warps per CTA of a warp-task GEMV whose slots hold two rows of `rb` bytes:
// 16, fewer when the slots would not fit in shared memory, 0 if one does not.
static int task_warps(int nb, int rb) {
    const size_t other = proj_smem(1, nb, 0).total;
    const size_t avail = device_info().smem_optin;
    int w = 16;
    while (w > 0 && other + static_cast<size_t>(w) * 2 * rb > avail) w >>= 1;
    return w;
}

int launch_norm_q8(const QkvArgs &a0, cudaStream_t s, bool pdl) {
    QkvArgs a = a0;
    const int warps = 16;
    const int grid = (a.D / QK + warps - 1) / warps;
    void *args[] = {&a};
    return cuda_status(launch(reinterpret_cast<const void *>(k_norm_q8), dim3(grid), dim3(32 * warps), 0, s, pdl, args));
}

bool qkv_fused_norm_ok(const QkvArgs &a) {
    const int nb = a.D / QK;
    if (nb % 8 != 0) return false;
    const int warps = task_warps(nb, nb * Q8B);
    return warps > 0 && warps * NORM_XPW >= nb;
}

int launch_qkv(const QkvArgs &a0, cudaStream_t s, bool pdl) {
    QkvArgs a = a0;
    const int nb = a.D / QK;
    const int warps = (nb % 8 == 0) ? task_warps(nb, nb * Q8B) : 0;
    void *args[] = {&a};
    if (warps > 0) {
        const size_t smem = proj_smem(1, nb, static_cast<size_t>(warps) * 2 * nb * Q8B).total;
        const int grid = (qkv_tasks(a) + warps - 1) / warps;
        const void *fn = reinterpret_cast<const void *>(k_qkv_w);
        ensure_smem(fn, smem);
        return cuda_status(launch(fn, dim3(grid), dim3(32 * warps), smem, s, pdl, args));
    }
    plan_qkv(a);
    const size_t smem = proj_smem(a.rv > 32 ? a.rv : 32, nb, 0).total;
    if (smem > device_info().smem_optin) return -1;
    const int grid = a.n_q_tiles + a.n_k_tiles + (a.KV * a.hd + a.rv - 1) / a.rv;
    const void *fn = reinterpret_cast<const void *>(k_qkv_direct);
    ensure_smem(fn, smem);
    return cuda_status(launch(fn, dim3(grid), dim3(256), smem, s, pdl, args));
}

int launch_oproj(const OprojArgs &a0, cudaStream_t s, bool pdl) {
    OprojArgs a = a0;
    const int nb = a.QD / QK;
    const int warps = (nb % 8 == 0) ? task_warps(nb, nb * Q5B) : 0;
    void *args[] = {&a};
    if (warps > 0) {
        const size_t smem = proj_smem(1, nb, static_cast<size_t>(warps) * 2 * nb * Q5B).total;
        const int grid = (a.D / 2 + warps - 1) / warps;
        const void *fn = reinterpret_cast<const void *>(k_oproj_w);
        ensure_smem(fn, smem);
        return cuda_status(launch(fn, dim3(grid), dim3(32 * warps), smem, s, pdl, args));
    }
    a.rows_per_cta = 8;
    const size_t smem = proj_smem(8, nb, 0).total;
    const int grid = (a.D + 7) / 8;
    const void *fn = reinterpret_cast<const void *>(k_oproj_direct);
    ensure_smem(fn, smem);
    return cuda_status(launch(fn, dim3(grid), dim3(256), smem, s, pdl, args));
}

}  // namespace ck
