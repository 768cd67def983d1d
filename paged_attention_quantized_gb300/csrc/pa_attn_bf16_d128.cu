// Attention kernel instantiations for BF16 KV codes, head dim 128.
#include "pa_attn_launch.cuh"

namespace pa {
PA_DEFINE_ATTN(PA_BF16, 128)
PA_DEFINE_ATTN_MERGED(PA_BF16, 128)  // rows too long to merge: reports cudaErrorNotSupported
}  // namespace pa
