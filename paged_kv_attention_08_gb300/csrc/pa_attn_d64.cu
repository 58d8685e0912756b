// Instantiations of the one-token decode kernel for head_dim 64 (kept in
// their own translation unit so that the library builds in parallel).
#include "pa_attn.cuh"

namespace pa {
cudaError_t launch_attn_d64(const AttnLaunch& L, cudaStream_t stream) {
    if (L.p.q_len > 1) return launch_attn_d64_multi(L, stream);
    return launch_attn_for_d<64, false>(L, stream);
}
int attn_max_clusters_d64(int block_size, int kv_dtype, int cluster, int threads,
                          uint32_t smem_bytes) {
    return attn_max_clusters_for_d<64>(block_size, kv_dtype, cluster, threads, smem_bytes);
}
}  // namespace pa
