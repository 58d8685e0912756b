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

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) {
        const float o = __shfl_xor_sync(kFullMask, v, mask);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    __syncthreads();  // `red` may still be read from a previous reduction
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < nw; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p, int D) {
    extern __shared__ float weight[];  // [num_parts]
    __shared__ float red[32];
    constexpr float NEG_INF = -INFINITY;

    const int h = blockIdx.x, b = blockIdx.y;
    const int kvh = h / p.group, g = h % p.group;
    const int T = reachable_tokens(p.context_lens, b, p.max_blocks, p.block_size);
    const int npages = (T + p.block_size - 1) / p.block_size;
    int nparts = (npages + p.part_pages - 1) / p.part_pages;
    nparts = min(nparts, p.num_parts);

    const size_t row0 = ((size_t)b * p.num_kv_heads + kvh) * p.num_parts;  // partition 0 of (b, kvh)
    auto ml_at = [&](int part) { return p.part_ml + ((row0 + part) * p.group + g) * 2; };

    float mx = NEG_INF;
    for (int q = threadIdx.x; q < nparts; q += blockDim.x) mx = fmaxf(mx, ml_at(q)[0]);
    const float M = block_reduce(mx, true, red);

    float ls = 0.f;
    for (int q = threadIdx.x; q < nparts; q += blockDim.x) {
        const float mq = ml_at(q)[0];
        const float w = (mq == NEG_INF) ? 0.f : exp2f(mq - M);
        weight[q] = w;
        ls = fmaf(w, ml_at(q)[1], ls);
    }
    const float Ls = block_reduce(ls, false, red);  // its barriers also publish `weight`

    const bool empty = (M == NEG_INF) || !(Ls > 0.f);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float a = 0.f;
        if (!empty) {
            const float* src = p.part_acc + (row0 * p.group + g) * D + d;
            const size_t stride = (size_t)p.group * D;
            int q = 0;
            for (; q + 4 <= nparts; q += 4) {
                const float a0 = src[(size_t)q * stride], a1 = src[(size_t)(q + 1) * stride];
                const float a2 = src[(size_t)(q + 2) * stride], a3 = src[(size_t)(q + 3) * stride];
                a = fmaf(weight[q], a0, a);
                a = fmaf(weight[q + 1], a1, a);
                a = fmaf(weight[q + 2], a2, a);
                a = fmaf(weight[q + 3], a3, a);
            }
            for (; q < nparts; ++q) a = fmaf(weight[q], src[(size_t)q * stride], a);
        }
        store_out(p.out, ((size_t)b * p.num_heads + h) * D + d, empty ? 0.f : a / Ls, p.out_dtype);
    }
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

cudaError_t launch_combine(const CombineParams& p, int head_dim, dim3 grid, int threads,
                           uint32_t smem_bytes, cudaStream_t stream) {
    if (smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(combine_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_bytes);
        if (e != cudaSuccess) return e;
    }
    combine_kernel<<<grid, threads, smem_bytes, stream>>>(p, head_dim);
    return cudaGetLastError();
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
