// Instantiations of the multi-token decode kernel (several query tokens per
// sequence) for head_dim 64.
#include "pa_attn.cuh"

namespace pa {
cudaError_t launch_attn_d64_multi(const AttnLaunch& L, cudaStream_t stream) {
    return launch_attn_for_d<64, true>(L, stream);
}
}  // namespace pa
