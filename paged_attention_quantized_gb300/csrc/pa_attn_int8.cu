// Split-KV attention kernel instantiations for INT8 KV codes.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT8, 64)
PA_DEFINE_ATTN(PA_INT8, 128)
PA_DEFINE_ATTN(PA_INT8, 256)
}  // namespace pa
