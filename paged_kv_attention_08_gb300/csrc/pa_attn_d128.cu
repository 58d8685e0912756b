// Instantiations of the one-token decode kernel for head_dim 128 (kept in
// their own translation unit so that the library builds in parallel).
#include "pa_attn.cuh"

namespace pa {
cudaError_t launch_attn_d128(const AttnLaunch& L, cudaStream_t stream) {
    if (L.p.q_len > 1) return launch_attn_d128_multi(L, stream);
    return launch_attn_for_d<128, false>(L, stream);
}
int attn_max_clusters_d128(int block_size, int kv_dtype, int cluster, int threads,
                          uint32_t smem_bytes) {
    return attn_max_clusters_for_d<128>(block_size, kv_dtype, cluster, threads, smem_bytes);
}
}  // namespace pa
