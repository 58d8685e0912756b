// Instantiations of the tcgen05 tile kernel for head_dim 256 with a compact
// Q tile (units of at most 16 rows, e.g. one-token MQA with a group of 16
// heads): three stages per K / V ring instead of two.
#include "pa_tile.cuh"

namespace pa {
cudaError_t launch_tile_d256_compact(const AttnLaunch& L, cudaStream_t stream) {
    return launch_tile_for_d<256, kTileCompactQRows>(L, stream);
}
int tile_max_clusters_d256_compact(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes) {
    return tile_max_clusters_for_d<256, kTileCompactQRows>(block_size, kv_dtype, cluster, smem_bytes);
}
}  // namespace pa
