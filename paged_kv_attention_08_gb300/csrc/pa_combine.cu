// Split-KV combine and page-walk export.
//
// Combine (flash-decoding-bench "design.md": each chunk's local max, sum and
// weighted values are reduced into the final output): for query head h of
// sequence b, with partitions p holding (m_p, l_p, acc_p) in base-2 units,
//     M = max_p m_p,   L = sum_p 2^(m_p - M) l_p,
//     out = sum_p 2^(m_p - M) acc_p / L.
// Partitions past the sequence's context are never read; an empty partition
// (m = -inf, l = 0, acc = 0) contributes nothing; a sequence with no attended
// token gets zeros.  One CTA per (query head, sequence), one thread per
// output element: the reads of acc are coalesced along head_dim.
#include "pa_device.cuh"

namespace pa {

namespace {

// One CTA per (query head, sequence); each warp computes the partition
// weights itself (lanes stride over partitions, shuffles reduce), then every
// thread accumulates VEC output columns over the partitions with up to eight
// independent loads in flight.  Two dependent memory round trips in all.
template <int D>
__global__ void __launch_bounds__(64) combine_kernel(const CombineParams p) {
    constexpr int VEC = D <= 128 ? D / 32 : 4;
    constexpr float NEG_INF = -INFINITY;
    extern __shared__ float weight_all[];  // [warps][num_parts]
    grid_dependency_wait();                // partials come from the attention kernel
    grid_launch_dependents();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* weight = weight_all + (size_t)warp * p.num_parts;
    const int h = blockIdx.x, b = blockIdx.y;
    const int kvh = h / p.group, g = h % p.group;
    const int T = reachable_tokens(p.context_lens, b, p.max_blocks, p.block_size);
    const int npages = (T + p.block_size - 1) / p.block_size;
    const int nparts = min((npages + p.part_pages - 1) / p.part_pages, p.num_parts);

    const size_t row0 = ((size_t)b * p.num_kv_heads + kvh) * p.num_parts;  // partition 0 of (b, kvh)
    const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
    auto ml_at = [&](int part) { return ml[(row0 + part) * p.group + g]; };

    float mx = NEG_INF;
    for (int q = lane; q < nparts; q += 32) mx = fmaxf(mx, ml_at(q).x);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
    float ls = 0.f;
    for (int q = lane; q < nparts; q += 32) {
        const float2 v = ml_at(q);
        const float w = (v.x == NEG_INF) ? 0.f : exp2f(v.x - mx);
        weight[q] = w;
        ls = fmaf(w, v.y, ls);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ls += __shfl_xor_sync(kFullMask, ls, m);
    __syncwarp();

    const int d0 = threadIdx.x * VEC;
    float a[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) a[v] = 0.f;
    const bool empty = (mx == NEG_INF) || !(ls > 0.f);
    if (!empty) {
        const float* src = p.part_acc + (row0 * p.group + g) * D + d0;
        const size_t stride = (size_t)p.group * D;
#pragma unroll 8
        for (int q = 0; q < nparts; ++q) {
            const float w = weight[q];
            if constexpr (VEC == 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + (size_t)q * stride);
                a[0] = fmaf(w, x.x, a[0]);
                a[1] = fmaf(w, x.y, a[1]);
                a[2] = fmaf(w, x.z, a[2]);
                a[3] = fmaf(w, x.w, a[3]);
            } else {
                const float2 x = *reinterpret_cast<const float2*>(src + (size_t)q * stride);
                a[0] = fmaf(w, x.x, a[0]);
                a[1] = fmaf(w, x.y, a[1]);
            }
        }
    }
    const size_t o = ((size_t)b * p.num_heads + h) * D + d0;
#pragma unroll
    for (int v = 0; v < VEC; ++v) store_out(p.out, o + v, empty ? 0.f : a[v] / ls, p.out_dtype);
}

__global__ void resolve_kernel(int32_t* out_phys, const int32_t* block_tables,
                               const int32_t* context_lens, int32_t batch, int32_t max_blocks,
                               int32_t block_size, int64_t num_blocks) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)batch * max_blocks) return;
    const int b = (int)(idx / max_blocks), j = (int)(idx % max_blocks);
    const int T = reachable_tokens(context_lens, b, max_blocks, block_size);
    const int npages = (T + block_size - 1) / block_size;
    out_phys[idx] = page_phys(block_tables + (size_t)b * max_blocks, j, npages, num_blocks);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int head_dim, dim3 grid, bool pdl,
                           cudaStream_t stream) {
    void (*kern)(const CombineParams);
    switch (head_dim) {
        case 64: kern = combine_kernel<64>; break;
        case 128: kern = combine_kernel<128>; break;
        default: kern = combine_kernel<256>; break;
    }
    const int threads = head_dim <= 128 ? 32 : 64;
    const uint32_t smem = (uint32_t)(threads / 32) * p.num_parts * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_resolve(int32_t* out_phys, const int32_t* block_tables,
                           const int32_t* context_lens, int32_t batch, int32_t max_blocks,
                           int32_t block_size, int64_t num_blocks, cudaStream_t stream) {
    const int64_t n = (int64_t)batch * max_blocks;
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    resolve_kernel<<<blocks, threads, 0, stream>>>(out_phys, block_tables, context_lens, batch,
                                                   max_blocks, block_size, num_blocks);
    return cudaGetLastError();
}

}  // namespace pa
