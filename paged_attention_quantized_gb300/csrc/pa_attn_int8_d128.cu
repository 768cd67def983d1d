// Attention kernel instantiations for INT8 KV codes, head dim 128.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT8, 128)
}  // namespace pa
