// Attention kernel instantiations for F16 KV codes, head dim 128.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_F16, 128)
PA_DEFINE_ATTN_MERGED(PA_F16, 128)  // rows too long to merge: reports cudaErrorNotSupported
}  // namespace pa
