// Internal host/device declarations shared by the decode library's translation
// units: the kernel parameter block, the shared-memory layout of the attention
// kernel, and the per-head_dim launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

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
    int32_t persistent;       // tile kernel: 1: CTA c takes the units c, c + C, c + 2C, ... whole
                              //    (C = gridDim.x; units = (sequence, kv head, 128-row tile))
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

// Most partitions of one (sequence, kv head) reduced inside a cluster: 8 is
// the portable cluster size; the one-token kernel may use clusters of up to
// 16 (a non-portable size) where the device can hold all of a call's
// clusters at once.
constexpr int kMaxClusterParts = 8;
constexpr int kMaxDecodeClusterParts = 16;

// Slack added to the dynamic shared-memory request so that the kernel can
// align its base to 1024 bytes (TMA destinations).
constexpr uint32_t kSmemAlignSlack = 1024;

// Tile kernel (several query tokens, tcgen05).  A CTA walks its pages in
// KV blocks of BN tokens (128, or 64 at head_dim 256): the pages of a block
// are copied into consecutive rows of one stage, so that one MMA covers the
// whole block.  Shared memory: the Q tile (128 rows x head_dim, 128-byte
// swizzle, head_dim/64 column blocks of 16 KB), `ns` stages of a block's K
// and V tiles (head_dim/64 column blocks of BN rows x 128 bytes each), then
// the mbarriers and the physical block of every staged page.  K and V have
// rings of their own (a K stage is free once S is computed, long before P V
// has read the V stage), each fed by its own copy warp.
constexpr int kTileRows = 128;
constexpr int kTileThreads = 384;  // warp 0 copies K, warp 3 copies V, warp 1 issues
                                   // MMAs, warp 2 owns tensor memory, warps 4-11 softmax
                                   // (two warpgroups, one half of a block's columns each)

__host__ __device__ constexpr int tile_block_tokens(int D) { return D == 256 ? 64 : 128; }
// S / P buffers in tensor memory: S of block j + 2 may be computed while P of
// block j still waits for its P V MMA.
constexpr int kTileSBufs = 3;
// Q rows staged in shared memory: a tile's 128, or -- at head_dim 256, for
// units of at most 16 rows (one-token MQA: a group of 16 heads) -- only 16:
// the MMA still runs M = 128, its rows past 16 read whatever follows the
// compact Q tile (their results are never used), and the 56 KB saved buy a
// third stage for each of the K and V rings.
constexpr int kTileCompactQRows = 16;
__host__ __device__ constexpr int tile_stages(int D, int qr = kTileRows) {
    return D == 64 ? 4 : (D == 256 && qr == kTileCompactQRows ? 3 : 2);
}

// Q tiles in shared memory: two (a unit's Q while the next one's is staged)
// where they fit beside the rings -- compact tiles, and whole tiles up to
// head_dim 128 -- else one.
__host__ __device__ constexpr int tile_q_bufs(int D, int qr = kTileRows) {
    return (qr == kTileCompactQRows || D <= 128) ? 2 : 1;
}

struct TileSmem {
    uint32_t tile_bytes;   // one K (or V) block tile: BN * head_dim * 2
    uint32_t q_off;        // Q tiles: [head_dim / 64] column blocks of qr rows x 128 bytes each;
                           // tile_q_bufs of them
    uint32_t k_off;        // [ns] K stages
    uint32_t v_off;        // [ns] V stages
    uint32_t bar_off;      // mbarriers: k_full[ns], k_empty[ns], v_full[ns], v_empty[ns],
                           // s_full[3], p_full[2][3], pv_done[3], final, q_ready, q_full[2],
                           // q_free[2], o_free
    uint32_t phys_off;     // [ns][BN / block_size] int32 physical block of each K stage's pages,
                           // then [ns] int32: V stage holds a page
    uint32_t xchg_off;     // softmax exchange: row maxima [2][2][128], normalisers [2][128] (fp32),
                           // then mbarriers xchg[2]
    uint32_t misc_off;     // tensor-memory base address, abort flag
    uint32_t seq_off;      // compact units, balanced split: pages of each sequence [512]
    uint32_t walk_off;     // compact units, balanced split: the CTA's share (4 x int64)
    uint32_t total;
    int ns;
};

__host__ __device__ inline TileSmem tile_smem_layout(int D, int BS, int qr = kTileRows) {
    TileSmem L;
    const int BN = tile_block_tokens(D);
    L.ns = tile_stages(D, qr);
    L.tile_bytes = (uint32_t)BN * D * 2u;
    const bool compact = qr == kTileCompactQRows;
    L.q_off = 0;
    // a multiple of 1024 (qr and D multiples of 16 and 64)
    L.k_off = (uint32_t)tile_q_bufs(D, qr) * 2u * qr * D;
    L.v_off = L.k_off + L.tile_bytes * L.ns;
    uint32_t o = L.v_off + L.tile_bytes * L.ns;
    L.bar_off = o;
    o += 8u * (4 * L.ns + 4 * kTileSBufs + 2 + 5);  // p_full: one set per softmax warpgroup
    L.phys_off = o;
    o += 4u * L.ns * (BN / BS + 1);
    L.xchg_off = pa_align_up(o, 16);
    o = L.xchg_off + 4u * (2 * 2 * 128 + 2 * 128) + 16;
    L.misc_off = pa_align_up(o, 16);
    o = L.misc_off + 16;
    L.seq_off = o;
    if (compact) o += 4u * kMaxBalancedBatch;
    L.walk_off = pa_align_up(o, 16);
    o = L.walk_off + (compact ? 32u : 0u);
    L.total = pa_align_up(o, 16);
    return L;
}

// Cluster reduction of the tile kernel: after its pages, a CTA leaves its
// partial in its own (then idle) operand buffers at offset 0 -- O rows
// [128][head_dim + 4] fp32, m [128], l [128] -- and the merge weights of its
// share of the rows [128][8] follow.
__host__ __device__ constexpr uint32_t tile_cluster_bytes(int D) {
    return 4u * (kTileRows * (D + 4) + 2 * kTileRows + kTileRows * 8);
}

// Tensor-memory columns of the tile kernel: O [head_dim] (two of them, one per
// softmax warpgroup, at head_dim <= 128), then the S buffers of BN fp32
// columns (P, as 16-bit high and low parts, overwrites S) in what is left.
__host__ __device__ constexpr uint32_t tile_tmem_cols(int D) {
    return (uint32_t)D + kTileSBufs * tile_block_tokens(D) <= 256u ? 256u : 512u;
}

// ---------------------------------------------------------------------------
// Host: kernel attributes set once per device.  A kernel's dynamic
// shared-memory limit only caps what a launch may request (occupancy follows
// the bytes a launch actually asks for), so it is raised once per device to
// all the device offers a block -- by the launch and the occupancy paths
// alike, so that neither ever lowers it under the other -- and the
// non-portable cluster permission is granted once where a launch needs it;
// later calls skip the runtime calls.  `done` is the kernel's own flag array.
// ---------------------------------------------------------------------------
constexpr int kMaxAttrDevices = 64;
using AttrFlags = std::atomic<int>[kMaxAttrDevices];

template <typename Kern>
cudaError_t raise_smem_limit_once(Kern kern, AttrFlags& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

template <typename Kern>
cudaError_t allow_nonportable_clusters_once(Kern kern, AttrFlags& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
}

struct AttnLaunch {
    AttnParams p;
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    CUtensorMap tmap_q;  // tile kernel, several segments per CTA: the Q tiles of later segments
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
// Clusters of `cluster` one-token attention CTAs (tune: `threads`, `smem_bytes`)
// resident at once on the current device (0 if the query fails).
int attn_max_clusters_d64(int block_size, int kv_dtype, int cluster, int threads, uint32_t smem_bytes);
int attn_max_clusters_d128(int block_size, int kv_dtype, int cluster, int threads, uint32_t smem_bytes);
int attn_max_clusters_d256(int block_size, int kv_dtype, int cluster, int threads, uint32_t smem_bytes);
cudaError_t launch_attn_d128_multi(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_d256_multi(const AttnLaunch& L, cudaStream_t stream);

// Tile kernel (tcgen05) launchers, one translation unit per head_dim.
cudaError_t launch_tile_d64(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_tile_d128(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_tile_d256(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_tile_d256_compact(const AttnLaunch& L, cudaStream_t stream);
// Clusters of `cluster` tile-kernel CTAs resident at once on the current device.
int tile_max_clusters_d64(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes);
int tile_max_clusters_d128(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes);
int tile_max_clusters_d256(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes);
int tile_max_clusters_d256_compact(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes);

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
