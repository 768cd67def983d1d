// Attention kernel instantiations for BF16 KV codes, head dim 128.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_BF16, 128)
}  // namespace pa
