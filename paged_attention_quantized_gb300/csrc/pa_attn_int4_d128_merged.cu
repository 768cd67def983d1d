// Attention kernel instantiations for INT4 KV codes, head dim 128, work pages of
// several consecutive blocks.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN_MERGED(PA_INT4, 128)
}  // namespace pa
