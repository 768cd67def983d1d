// Attention kernel instantiations for INT4 KV codes, head dim 128.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT4, 128)
}  // namespace pa
