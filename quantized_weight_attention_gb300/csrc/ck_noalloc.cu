// ck_attn_decode_gqa_noalloc: the split-KV decode attention of
// ck_attn_decode_gqa for callers that cannot allocate device memory.
//
// Who needs it: code whose device memory is owned entirely by someone else
// (a host framework with its own pooling allocator, or a fixed memory budget
// agreed up front) and code that must never pay for a cudaMalloc, which can
// synchronize the whole device, in the middle of a latency-critical decode
// loop.  Such a caller can hand us its inputs and outputs but no scratch
// buffer.  This entry point keeps the split-KV partial results in a buffer
// compiled into the library instead, so the call allocates nothing.
//
// The buffer is a file-scope __device__ array of CK_ATTN_NOALLOC_MAX_BYTES:
// every GPU that loads the library holds it until the process exits.  All
// calls share it and it keeps the last call's contents; nothing in it has to
// start at zero (every record the merge reads is written by the same call).
// Two calls whose work overlaps on the GPU (different streams, or different
// host threads on the same device) race on it.
#include <mutex>

#include "../../include/ck_decode.h"
#include "ck_device.cuh"
#include "ck_internal.h"

namespace ck {
namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[CK_ATTN_NOALLOC_MAX_BYTES];

std::mutex g_noalloc_mu;

// Device address of g_attn_scratch on the current device.  In host code the
// array's name only stands in for the symbol; the address the kernels need
// comes from cudaGetSymbolAddress, looked up once per device with that
// device current, on its first call.
float *noalloc_scratch() {
    static float *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return nullptr;
        cache[dev] = static_cast<float *>(p);
    }
    return cache[dev];
}

}  // namespace
}  // namespace ck

using namespace ck;

extern "C" int ck_attn_decode_gqa_noalloc(const float *q, const float *k_cache, const float *v_cache, float *out,
                                          int num_heads, int num_kv_heads, int kv_tokens, int cache_capacity,
                                          int head_dim, void *stream) {
    for (const void *p : {static_cast<const void *>(q), static_cast<const void *>(k_cache),
                          static_cast<const void *>(v_cache), static_cast<const void *>(out)}) {
        if (!p) return CK_EINVAL;
        if (reinterpret_cast<uintptr_t>(p) & 15u) return CK_EALIGN;
    }
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return CK_EINVAL;
    if (num_heads / num_kv_heads > 8) return CK_EINVAL;
    const int dpl = head_dim / 32;
    if (head_dim % 32 != 0 || (dpl != 1 && dpl != 2 && dpl != 3 && dpl != 4 && dpl != 8)) return CK_EINVAL;
    if (cache_capacity <= 0) return CK_EINVAL;
    if (kv_tokens < 1 || kv_tokens > cache_capacity) return CK_ERANGE;
    const int S = attn_splits(1, num_kv_heads, kv_tokens);
    if (attn_part_bytes(1, num_heads, num_kv_heads, head_dim, S) > CK_ATTN_NOALLOC_MAX_BYTES) return CK_ESCRATCH;
    float *part = noalloc_scratch();
    unsigned *st = status_word();
    if (!part || !st) return CK_ECUDA;
    AttnArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.kv_tokens = kv_tokens;
    a.H = num_heads;
    a.KV = num_kv_heads;
    a.hd = head_dim;
    a.C = cache_capacity;
    a.splits = S;
    a.part = part;
    a.out = out;
    a.status = st;
    return launch_attention(a, 1, static_cast<cudaStream_t>(stream), false, false) ? CK_ECUDA : CK_OK;
}
