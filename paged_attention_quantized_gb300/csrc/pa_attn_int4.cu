// Split-KV attention kernel instantiations for INT4 KV codes.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT4, 128)
PA_DEFINE_ATTN(PA_INT4, 256)
}  // namespace pa
