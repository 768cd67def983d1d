// Split-KV attention kernel instantiations for BF16 KV codes.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_BF16, 64)
PA_DEFINE_ATTN(PA_BF16, 128)
PA_DEFINE_ATTN(PA_BF16, 256)
}  // namespace pa
