// Attention kernel instantiations for E4M3 KV codes, head dim 256.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_E4M3, 256)
PA_DEFINE_ATTN_MERGED(PA_E4M3, 256)  // rows too long to merge: reports cudaErrorNotSupported
}  // namespace pa
