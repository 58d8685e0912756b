// Instantiations of the tcgen05 tile kernel (several query tokens per
// sequence) for head_dim 128.
#include "pa_tile.cuh"

namespace pa {
cudaError_t launch_tile_d128(const AttnLaunch& L, cudaStream_t stream) {
    return launch_tile_for_d<128, kTileRows>(L, stream);
}
int tile_max_clusters_d128(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes) {
    return tile_max_clusters_for_d<128, kTileRows>(block_size, kv_dtype, cluster, smem_bytes);
}
}  // namespace pa
