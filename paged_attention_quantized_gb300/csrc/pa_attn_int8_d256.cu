// Attention kernel instantiations for INT8 KV codes, head dim 256.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_INT8, 256)
PA_DEFINE_ATTN_MERGED(PA_INT8, 256)  // rows too long to merge: reports cudaErrorNotSupported
}  // namespace pa
