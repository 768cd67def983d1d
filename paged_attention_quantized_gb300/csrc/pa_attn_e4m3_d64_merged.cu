// Attention kernel instantiations for FP8 E4M3 KV codes, head dim 64, work pages of
// several consecutive blocks.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN_MERGED(PA_E4M3, 64)
}  // namespace pa
