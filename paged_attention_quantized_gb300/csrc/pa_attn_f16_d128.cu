// Attention kernel instantiations for F16 KV codes, head dim 128.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_F16, 128)
}  // namespace pa
