// Attention kernel instantiations for INT4 KV codes, head dim 256.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT4, 256)
PA_DEFINE_ATTN_MERGED(PA_INT4, 256)  // rows too long to merge: reports cudaErrorNotSupported
}  // namespace pa
