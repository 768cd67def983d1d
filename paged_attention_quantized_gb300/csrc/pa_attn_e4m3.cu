// Split-KV attention kernel instantiations for E4M3 KV codes.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_E4M3, 64)
PA_DEFINE_ATTN(PA_E4M3, 128)
PA_DEFINE_ATTN(PA_E4M3, 256)
}  // namespace pa
