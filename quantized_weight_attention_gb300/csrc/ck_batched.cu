// The decode step for a batch of B sequences that share one layer's weights,
// each with its own KV cache and position (ragged lengths): the same step as
// ck_decode_layer applied to every sequence (STEP 1-8 of the page
// "mega_fused_attention_decode_q5_0.c", MAIN KERNEL), with the projections
// computed for all B activation rows while each weight segment sits decoded
// in registers, so the weights are read once per step instead of B times.
//
//   k_norm_pack    grid B: RMSNorm + Q8_0 quantization of sequence s's row
//                  into a packed row in the scratch (and its Q8_0 blocks).
//   k_rows_batched warp task = two weight rows (a RoPE pair of Q or K, two V
//                  rows, or two Wo rows); lane l < 16 decodes segment l of the
//                  first row, lane 16 + l segment l of the second, once, before
//                  waiting on the preceding grid; then for every sequence the
//                  lanes dot their segment with its activation row (staged
//                  in shared memory 16 rows at a time) and lane 0 runs the
//                  epilogue: bias, RoPE at the sequence's
//                  position and the q / K-row / V-row stores (Q/K/V), or bias
//                  plus residual (O).
//   attention      the split kernel of ck_attn_kernels.cuh with per-sequence
//                  cache pointers and positions (grid (S, KV, B)), and its
//                  combine, which also writes the packed rows the O
//                  projection reads.
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {

// Sequence s = blockIdx.x: RMSNorm + Q8_0 of x[s] into shared memory, then
// the packed image to xpack[s] (and the Q8_0 blocks to xq8[s]).
__global__ void __launch_bounds__(512) k_norm_pack(const BatchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float red[64];
    const int s = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nb = a.D / QK;
    XRow xr;
    xr.q = reinterpret_cast<int4 *>(smem);
    xr.d = reinterpret_cast<float *>(smem + static_cast<size_t>(xq_chunks(nb)) * 16);
    xr.sum = reinterpret_cast<int *>(smem + static_cast<size_t>(xq_chunks(nb)) * 16 + static_cast<size_t>(nb) * 4);
    float gv[NORM_XPW];
#pragma unroll
    for (int j = 0; j < NORM_XPW; ++j) {
        const int b = warp + nw * j;
        gv[j] = b < nb ? __ldg(a.gamma + b * QK + lane) : 0.0f;
    }
    pdl_trigger();
    pdl_wait();  // x may be the previous layer's output
    if (s == 0 && a.tickets)  // the tensor-core projections' tile tickets of this step
        for (int i = threadIdx.x; i < a.n_tickets; i += blockDim.x) a.tickets[i] = 0;
    norm_quant_xrow(a.x + static_cast<size_t>(s) * a.D, gv, nb, a.D, a.eps, xr, red,
                    a.xq8 + static_cast<size_t>(s) * nb * Q8B);
    const int n16 = static_cast<int>(xpack_bytes(nb) / 16);
    int4 *dst = reinterpret_cast<int4 *>(a.xpack + static_cast<size_t>(s) * xpack_bytes(nb));
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = xr.q[i];
    if (a.ximg) {  // the row in the tensor-core operand image: 8 values per item, hi and lo parts
        const int G = img_groups(a.B);
        bool in_range = true;
        for (int i = threadIdx.x; i < nb * 4; i += blockDim.x) {
            const int b = i >> 2, e = i & 3;
            const int8_t *c = reinterpret_cast<const int8_t *>(&xr.q[xq_chunk(b, e >> 1)]) + (e & 1) * 8;
            const float d = xr.d[b];
            __align__(16) __half hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) in_range = img_split(d, c[k], hi[k], lo[k]) && in_range;
            uint8_t *o = a.ximg + img_code_off(G, s, b, e);
            *reinterpret_cast<uint4 *>(o) = *reinterpret_cast<const uint4 *>(hi);
            *reinterpret_cast<uint4 *>(o + IMG_CODE_BYTES) = *reinterpret_cast<const uint4 *>(lo);
        }
        if (!in_range) flag_error(a.status, FLAG_RANGE);
    }
}

// Rows of warp task t.  Q/K/V: the tasks of the single-sequence projection
// (Q pairs, K pairs, V row pairs); O: Wo rows 2t, 2t + 1.
struct RowTask {
    int kind;  // 0 = Q, 1 = K, 2 = V, 3 = none, 4 = O
    int ra, rb, head, i;
};
__device__ __forceinline__ RowTask row_task(const BatchArgs &a, bool oproj, int t) {
    RowTask T{};
    if (oproj) {
        T.kind = 2 * t < a.D ? 4 : 3;
        T.ra = 2 * t;
        T.rb = 2 * t + 1;
        return T;
    }
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

// Activation rows pass through shared memory in groups of BG sequences (two
// buffers, filled by bulk copies while the other is in use), so each CTA
// reads the batch's packed rows from L2 once instead of once per warp.
constexpr int BG = 16;

template <bool OPROJ>
__global__ void __launch_bounds__(512, 1) k_rows_batched(const BatchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int li = lane & 15;
    const int nb = OPROJ ? a.H * a.hd / QK : a.D / QK;  // blocks per weight row
    const int nseg = nb / 8;
    const uint32_t pstride = static_cast<uint32_t>(xpack_bytes(nb));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);  // one per buffer
    uint8_t *buf0 = smem + 128;
    const RowTask T = row_task(a, OPROJ, blockIdx.x * nw + warp);
    const bool q8 = T.kind == 2;
    SegCodes R;
    if (T.kind != 3 && li < nseg) {  // the weights do not depend on earlier grids
        const int row = lane < 16 ? T.ra : T.rb;
        const uint8_t *W = OPROJ ? a.wo : (T.kind == 0 ? a.wq : (T.kind == 1 ? a.wk : a.wv));
        if (q8)
            seg_decode<true>(W + (static_cast<size_t>(row) * nb + li * 8) * Q8B, R);
        else
            seg_decode<false>(W + (static_cast<size_t>(row) * nb + li * 8) * Q5B, R);
    }
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();  // the packed activation rows are ready
    const uint8_t *pack = OPROJ ? a.apack : a.xpack;
    const int ngroups = (a.B + BG - 1) / BG;
    auto fill = [&](int g) {  // thread 0: group g into buffer g % 2
        const int n = min(BG, a.B - g * BG);
        const uint32_t bytes = static_cast<uint32_t>(n) * pstride;
        uint8_t *dst = buf0 + static_cast<size_t>(g & 1) * BG * pstride;
        const uint8_t *src = pack + static_cast<size_t>(g) * BG * pstride;
        mbar_arrive_expect_tx(&bar[g & 1], bytes);
        for (uint32_t o = 0; o < bytes; o += 65536u)
            bulk_g2s(dst + o, src + o, bytes - o < 65536u ? bytes - o : 65536u, &bar[g & 1]);
    };
    if (threadIdx.x == 0) {
        fill(0);
        if (ngroups > 1) fill(1);
    }
    const int QD = a.H * a.hd, half = a.hd >> 1;
    for (int g = 0; g < ngroups; ++g) {
        if (!mbar_wait(&bar[g & 1], (g >> 1) & 1)) flag_error(a.status, FLAG_TIMEOUT);
        const uint8_t *gb = buf0 + static_cast<size_t>(g & 1) * BG * pstride;
        const int n = min(BG, a.B - g * BG);
        for (int j = 0; j < n && T.kind != 3; ++j) {
            const int s = g * BG + j;
            const int pos = a.d_pos[s];
            XRow x;
            x.q = reinterpret_cast<int4 *>(const_cast<uint8_t *>(gb) + static_cast<size_t>(j) * pstride);
            x.d = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(x.q) + static_cast<size_t>(xq_chunks(nb)) * 16);
            x.sum = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(x.d) + static_cast<size_t>(nb) * 4);
            float acc = li < nseg ? seg_dot_codes(R, x, li * 8, !q8) : 0.0f;
            acc += __shfl_xor_sync(0xffffffffu, acc, 8);
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            const float sb = __shfl_sync(0xffffffffu, acc, 16);
            if (lane != 0) continue;
            if (pos < 0 || pos >= a.C) {  // this sequence's step writes nothing
                flag_error(a.status, FLAG_RANGE);
                continue;
            }
            if (OPROJ) {
                float *o = a.out + static_cast<size_t>(s) * a.D;
                const float *res = a.residual + static_cast<size_t>(s) * a.D;
                o[T.ra] = (acc + (a.bo ? a.bo[T.ra] : 0.0f)) + res[T.ra];
                o[T.rb] = (sb + (a.bo ? a.bo[T.rb] : 0.0f)) + res[T.rb];
                continue;
            }
            if (q8) {
                float *vc = a.v_caches[s];
                const float va = acc + (a.bv ? a.bv[T.ra] : 0.0f);
                const float vb = sb + (a.bv ? a.bv[T.rb] : 0.0f);
                int h = T.ra / a.hd;
                vc[(static_cast<size_t>(h) * a.C + pos) * a.hd + (T.ra - h * a.hd)] = va;
                h = T.rb / a.hd;
                vc[(static_cast<size_t>(h) * a.C + pos) * a.hd + (T.rb - h * a.hd)] = vb;
                continue;
            }
            const float *bias = T.kind == 0 ? a.bq : a.bk;
            const float A = acc + (bias ? bias[T.ra] : 0.0f);
            const float B = sb + (bias ? bias[T.rb] : 0.0f);
            const float c = a.rope_cos[static_cast<size_t>(pos) * half + T.i];
            const float sn = a.rope_sin[static_cast<size_t>(pos) * half + T.i];
            const float A2 = __fsub_rn(__fmul_rn(A, c), __fmul_rn(B, sn));
            const float B2 = __fadd_rn(__fmul_rn(A, sn), __fmul_rn(B, c));
            if (T.kind == 0) {
                a.q[static_cast<size_t>(s) * QD + T.ra] = A2;
                a.q[static_cast<size_t>(s) * QD + T.rb] = B2;
            } else {
                float *kr = a.k_caches[s] + (static_cast<size_t>(T.head) * a.C + pos) * a.hd;
                kr[T.i] = A2;
                kr[T.i + half] = B2;
            }
        }
        __syncthreads();  // every warp is done with this buffer
        if (threadIdx.x == 0 && g + 2 < ngroups) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // reads before the copy's writes
            fill(g + 2);
        }
    }
}

bool batched_shape_ok(int D, int H, int hd) {
    const int nb = D / QK, nbo = H * hd / QK;
    return D % 256 == 0 && nb <= 128 && nbo % 8 == 0 && nbo <= 128;
}

// The multi-token (prefill) form runs as a batch whose entries are the chunk's
// tokens: every entry names the one cache, entry i sits at position pos + i.
__global__ void k_prefill_setup(float **kcs, float **vcs, int32_t *pos_of, float *k_cache, float *v_cache, int pos,
                                const int32_t *d_pos, int n, int C, unsigned *status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int p0 = d_pos ? *d_pos : pos;
    const bool fits = p0 >= 0 && p0 <= C - n;
    if (!fits && i == 0) flag_error(status, FLAG_RANGE);
    if (i < n) {
        kcs[i] = k_cache;
        vcs[i] = v_cache;
        pos_of[i] = fits ? p0 + i : C;
    }
}

int launch_prefill_setup(float **kcs, float **vcs, int32_t *pos_of, float *k_cache, float *v_cache, int pos,
                         const int32_t *d_pos, int n, int C, unsigned *status, cudaStream_t s) {
    void *args[] = {&kcs, &vcs, &pos_of, &k_cache, &v_cache, &pos, &d_pos, &n, &C, &status};
    return launch(reinterpret_cast<const void *>(k_prefill_setup), dim3((n + 255) / 256), dim3(256), 0, s, false,
                  args) == cudaSuccess
               ? 0
               : -5;
}

int launch_norm_pack(const BatchArgs &a0, cudaStream_t s, bool pdl) {
    BatchArgs a = a0;
    const size_t smem = xpack_bytes(a.D / QK);
    void *args[] = {&a};
    return launch(reinterpret_cast<const void *>(k_norm_pack), dim3(a.B), dim3(512), smem, s, pdl, args) ==
                   cudaSuccess
               ? 0
               : -5;
}

int launch_rows_batched(const BatchArgs &a0, bool oproj, cudaStream_t s, bool pdl) {
    BatchArgs a = a0;
    const int warps = 16;
    const int tasks = oproj ? a.D / 2 : (a.H + a.KV) * (a.hd / 2) + (a.KV * a.hd) / 2;
    void *args[] = {&a};
    const void *fn = oproj ? reinterpret_cast<const void *>(k_rows_batched<true>)
                           : reinterpret_cast<const void *>(k_rows_batched<false>);
    const int nb = oproj ? a.H * a.hd / QK : a.D / QK;
    const size_t smem = 128 + 2 * static_cast<size_t>(BG) * xpack_bytes(nb);
    ensure_smem(fn, smem);
    return launch(fn, dim3((tasks + warps - 1) / warps), dim3(32 * warps), smem, s, pdl, args) == cudaSuccess ? 0
                                                                                                             : -5;
}

}  // namespace ck
