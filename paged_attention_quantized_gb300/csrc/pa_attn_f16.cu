// Split-KV attention kernel instantiations for F16 KV codes.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_F16, 64)
PA_DEFINE_ATTN(PA_F16, 128)
PA_DEFINE_ATTN(PA_F16, 256)
}  // namespace pa
