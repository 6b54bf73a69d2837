// Decode attention kernels over bf16 caches, head_dim 64 and 128 (see ck_attn_kernels.cuh).
#include "ck_attn_kernels.cuh"

namespace ck {
template int launch_attention_dpl<2, KV_BF16>(const AttnArgs &, int, cudaStream_t, bool, bool);
template int launch_attention_dpl<4, KV_BF16>(const AttnArgs &, int, cudaStream_t, bool, bool);
}  // namespace ck
