// Decode attention kernels for head_dim = 64 (see ck_attn_kernels.cuh).
#include "ck_attn_kernels.cuh"

namespace ck {
template int launch_attention_dpl<2, KV_F32>(const AttnArgs &, int, cudaStream_t, bool, bool);
}  // namespace ck
