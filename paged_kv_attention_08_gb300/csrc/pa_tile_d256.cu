// Instantiations of the tcgen05 tile kernel (several query tokens per
// sequence) for head_dim 256.
#include "pa_tile.cuh"

namespace pa {
cudaError_t launch_tile_d256(const AttnLaunch& L, cudaStream_t stream) {
    return launch_tile_for_d<256, kTileRows>(L, stream);
}
int tile_max_clusters_d256(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes) {
    return tile_max_clusters_for_d<256, kTileRows>(block_size, kv_dtype, cluster, smem_bytes);
}
}  // namespace pa
