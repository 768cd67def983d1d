// Attention kernel instantiations for INT8 KV codes, head dim 64, blocks handled as
// several work pages.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN_SPLIT(PA_INT8, 64)
}  // namespace pa
