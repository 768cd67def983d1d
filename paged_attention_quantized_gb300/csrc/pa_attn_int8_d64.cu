// Attention kernel instantiations for INT8 KV codes, head dim 64.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT8, 64)
}  // namespace pa
