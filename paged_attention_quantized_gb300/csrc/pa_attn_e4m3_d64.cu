// Attention kernel instantiations for E4M3 KV codes, head dim 64.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_E4M3, 64)
}  // namespace pa
