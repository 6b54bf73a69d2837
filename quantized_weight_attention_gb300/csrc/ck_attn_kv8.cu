// Decode attention kernels over fp8 E4M3 caches with per-tensor scales, head_dim 64 and 128
// (see ck_attn_kernels.cuh).
#include "ck_attn_kernels.cuh"

namespace ck {
template int launch_attention_dpl<2, KV_FP8>(const AttnArgs &, int, cudaStream_t, bool, bool);
template int launch_attention_dpl<4, KV_FP8>(const AttnArgs &, int, cudaStream_t, bool, bool);
}  // namespace ck
