// Attention kernel instantiations for INT8 KV codes, head dim 128, blocks handled as
// several work pages.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN_SPLIT(PA_INT8, 128)
}  // namespace pa
