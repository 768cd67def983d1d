// Attention kernel instantiations for INT8 KV codes, head dim 64, work pages of
// several consecutive blocks.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN_MERGED(PA_INT8, 64)
}  // namespace pa
