// Internal host/device declarations shared by the decode library's translation
// units: the kernel parameter block, the shared-memory layout of the attention
// kernel, and the per-head_dim launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa_decode.h"

namespace pa {


struct AttnParams {
    const void* q;            // [B, Q, H, D] kv dtype
    void* out;                // [B, Q, H, D] out dtype (final mode)
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* part_acc;          // [B, Hkv, P, Q*G, D] fp32 (split mode)
    float* part_ml;           // [B, Hkv, P, Q*G, 2] fp32 (split mode): running max (log2 units), normaliser
    int32_t* err;             // device error word
    int32_t batch, num_heads, num_kv_heads, group, max_blocks;
    int32_t q_len;            // Q: query tokens per sequence (1 for a one-token decode)
    int32_t q_chunk;          // query tokens per CTA (q_chunk * group <= 16 MMA rows);
                              // gridDim.y = num_kv_heads * ceil(Q / q_chunk)
    int32_t unit_rows;        // Q * group: workspace rows of one (sequence, kv head, partition)
    int64_t num_blocks;
    float qscale;             // scale * log2(e): scores are kept in base-2 units
    int32_t part_pages;       // pages per partition
    int32_t num_parts;        // partitions per (sequence, kv head) = gridDim.x
    int32_t nt;               // token streams (independent page rings) per CTA
    int32_t nh;               // warps per stream, each producing a slice of the output columns
    int32_t ns;               // pipeline stages per stream
    int32_t out_dtype;        // pa_dtype
    int32_t final_out;        // 1: write out (one partition); 0: partitions reduce elsewhere
    int32_t balanced;         // 1: CTA c takes pages [c*W/C, (c+1)*W/C) of the flattened
                              //    (sequence, kv head, page) order; units it covers whole are
                              //    written out, pieces become records [C][2][G] in part_acc/ml
    int32_t cluster_reduce;   // 1: the num_parts partitions of a (sequence, kv head) form one
                              //    thread-block cluster and reduce through distributed shared
                              //    memory; 0: partials go to the workspace for the combine kernel
    uint64_t timeout_ns;      // bound on every wait of the copy pipeline
};

struct CombineParams {
    void* out;
    const int32_t* context_lens;
    const float* part_acc;
    const float* part_ml;
    int32_t batch, num_heads, num_kv_heads, group, max_blocks, block_size;
    int32_t q_len;     // query tokens per sequence; gridDim.x = q_len * num_heads
    int32_t part_pages, num_parts, out_dtype;
    int32_t num_ctas;  // balanced split: CTAs of the attention kernel (records [C][2][G])
};

// Largest batch the balanced split handles (its per-sequence page counts live
// in shared memory).
constexpr int kMaxBalancedBatch = 512;

// Shared-memory layout of the attention kernel, identical on host and device.
// Each stage holds one page of one kv head: the K tile then the V tile, each
// head_dim/64 column blocks of [block_size rows][128 bytes], written by TMA
// with the 128-byte swizzle.  After the page loop the stage area is reused
// for the final merge of the warps' partial results.
struct AttnSmem {
    uint32_t tile_bytes;    // one K (or V) page tile: block_size * head_dim * 2
    uint32_t stage_bytes;   // K tile + V tile
    uint32_t stages_off;    // [nt][ns] stages (1024-byte aligned)
    uint32_t full_off;      // [nt][ns] uint64 mbarriers: page landed
    uint32_t empty_off;     // [nt][ns] uint64 mbarriers: page consumed
    uint32_t phys_off;      // [nt][ns] int32 physical block of the staged page (-1 = masked)
    uint32_t seq_off;       // balanced split: pages of each sequence, then the total
    uint32_t total;         // bytes, excluding the alignment slack
};



__host__ __device__ inline uint32_t pa_align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline AttnSmem attn_smem_layout(int D, int BS, int nt, int ns) {
    AttnSmem L;
    L.tile_bytes = (uint32_t)BS * D * 2u;
    L.stage_bytes = 2u * L.tile_bytes;
    L.stages_off = 0;
    uint32_t o = L.stage_bytes * nt * ns;
    L.full_off = o;
    o += 8u * nt * ns;
    L.empty_off = o;
    o += 8u * nt * ns;
    L.phys_off = o;
    o = pa_align_up(o + 4u * nt * ns, 16);
    L.seq_off = o;
    o += 4u * (kMaxBalancedBatch + 1);
    L.total = pa_align_up(o, 16);
    return L;
}

// Floats the final merge needs in the stage area for R rows (query token,
// head pairs): per warp, acc rows over that warp's output columns, m and l per
// row, the streams' weights and per-row totals; then the CTA's merged partial
// (acc [R][D], m [R], l [R]) that the other CTAs of a cluster read, and the
// cluster's per-rank statistics.
__host__ __device__ inline uint32_t merge_floats(int nw, int G, int cols_per_warp) {
    return (uint32_t)nw * G * cols_per_warp + 3u * nw * G + 4u * G;
}
__host__ __device__ inline uint32_t cluster_part_floats(int G, int D) {
    return (uint32_t)G * D + 2u * G + 3u * 8u * G;
}

// Most partitions of one (sequence, kv head) reduced inside a cluster.
constexpr int kMaxClusterParts = 8;

// Slack added to the dynamic shared-memory request so that the kernel can
// align its base to 1024 bytes (TMA destinations).
constexpr uint32_t kSmemAlignSlack = 1024;

struct AttnLaunch {
    AttnParams p;
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    int head_dim, block_size, kv_dtype;
    bool pdl;     // launch with programmatic stream serialization
    int cluster;  // > 1: cluster size along x (= partitions per sequence and kv head)
    dim3 grid;
    int threads;
    uint32_t smem_bytes;
};

// Per-head_dim launchers (one translation unit each, compiled in parallel);
// with q_len > 1 they hand over to the multi-token instantiations.
cudaError_t launch_attn_d64(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_d128(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_d256(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_d64_multi(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_d128_multi(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_d256_multi(const AttnLaunch& L, cudaStream_t stream);

cudaError_t launch_combine(const CombineParams& p, int head_dim, dim3 grid, bool pdl,
                           cudaStream_t stream);
cudaError_t launch_combine_balanced(const CombineParams& p, int head_dim, dim3 grid, bool pdl,
                                    cudaStream_t stream);
cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* block_tables, const int32_t* positions, int32_t batch,
                          int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                          int32_t row_bytes, bool pdl, cudaStream_t stream);
cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_resolve(int32_t* out_phys, const int32_t* block_tables,
                           const int32_t* context_lens, int32_t batch, int32_t max_blocks,
                           int32_t block_size, int64_t num_blocks, cudaStream_t stream);

}  // namespace pa
