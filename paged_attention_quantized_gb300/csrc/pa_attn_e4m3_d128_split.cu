// Attention kernel instantiations for E4M3 KV codes, head dim 128, blocks handled as
// several work pages.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN_SPLIT(PA_E4M3, 128)
}  // namespace pa
