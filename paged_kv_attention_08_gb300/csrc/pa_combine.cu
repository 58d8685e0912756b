// Split-KV combine and page-walk export.
//
// Combine (flash-decoding-bench "design.md": each chunk's local max, sum and
// weighted values are reduced into the final output): for query head h of
// query token qi of sequence b, with partitions p holding (m_p, l_p, acc_p)
// in base-2 units,
//     M = max_p m_p,   L = sum_p 2^(m_p - M) l_p,
//     out = sum_p 2^(m_p - M) acc_p / L.
// Partitions past the sequence's context are never read; an empty partition
// (m = -inf, l = 0, acc = 0) contributes nothing; a sequence with no attended
// token gets zeros.
#include "pa_device.cuh"

namespace pa {

namespace {

// One CTA of 256 threads per (query token and head, sequence).  Every thread loads the
// (m, l) of a few partitions; two block reductions give the maximum and the
// weighted normaliser.  The threads then form PGRP groups over the
// partitions, each thread a 16-byte slice of the head dimension, so that all
// acc loads of a head are in flight at once; a shared-memory sum over the
// groups finishes the head.  Two dependent memory round trips in all.
constexpr int kCombineThreads = 256;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
    constexpr int SLICES = D / 4;                      // float4 slices of one row
    constexpr int PGRP = kCombineThreads / SLICES;     // partition groups
    constexpr float NEG_INF = -INFINITY;
    extern __shared__ float weight[];                  // [num_parts]
    __shared__ float red[kCombineThreads / 32];
    __shared__ float4 part[PGRP][SLICES];
    grid_dependency_wait();                            // partials come from the attention kernel
    grid_launch_dependents();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = (int)blockIdx.x % p.num_heads, qi = (int)blockIdx.x / p.num_heads;
    const int b = blockIdx.y;
    const int kvh = h / p.group;
    const int U = p.q_len * p.group, u = qi * p.group + h % p.group;  // rows of a unit; this row
    const int T = reachable_tokens(p.context_lens, b, p.max_blocks, p.block_size);
    const int npages = (T + p.block_size - 1) / p.block_size;
    const int nparts = min((npages + p.part_pages - 1) / p.part_pages, p.num_parts);

    const size_t row0 = ((size_t)b * p.num_kv_heads + kvh) * p.num_parts;  // partition 0 of (b, kvh)
    const float2* ml = reinterpret_cast<const float2*>(p.part_ml);

    float mx = NEG_INF;
    for (int q = tid; q < nparts; q += kCombineThreads) mx = fmaxf(mx, ml[(row0 + q) * U + u].x);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();

    float ls = 0.f;
    for (int q = tid; q < nparts; q += kCombineThreads) {
        const float2 v = ml[(row0 + q) * U + u];
        const float w = (v.x == NEG_INF) ? 0.f : exp2f(v.x - mx);
        weight[q] = w;
        ls = fmaf(w, v.y, ls);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ls += __shfl_xor_sync(kFullMask, ls, m);
    if (lane == 0) red[warp] = ls;
    __syncthreads();  // also publishes `weight`
    ls = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) ls += red[w];

    const bool empty = (mx == NEG_INF) || !(ls > 0.f);
    const int pg = tid / SLICES, sl = tid % SLICES;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
        const float4* src = reinterpret_cast<const float4*>(p.part_acc + (row0 * U + u) * D) + sl;
        const size_t stride = (size_t)U * SLICES;  // float4s between partitions
#pragma unroll 4
        for (int q = pg; q < nparts; q += PGRP) {
            const float w = weight[q];
            const float4 x = src[(size_t)q * stride];
            a.x = fmaf(w, x.x, a.x);
            a.y = fmaf(w, x.y, a.y);
            a.z = fmaf(w, x.z, a.z);
            a.w = fmaf(w, x.w, a.w);
        }
    }
    part[pg][sl] = a;
    __syncthreads();
    if (pg == 0) {
        for (int k = 1; k < PGRP; ++k) {
            const float4 x = part[k][sl];
            a.x += x.x;
            a.y += x.y;
            a.z += x.z;
            a.w += x.w;
        }
        const float inv = empty ? 0.f : 1.f / ls;
        const size_t o = (((size_t)b * p.q_len + qi) * p.num_heads + h) * D + sl * 4;
        store_out(p.out, o, a.x * inv, p.out_dtype);
        store_out(p.out, o + 1, a.y * inv, p.out_dtype);
        store_out(p.out, o + 2, a.z * inv, p.out_dtype);
        store_out(p.out, o + 3, a.w * inv, p.out_dtype);
    }
}

// Combine for the balanced split: the attention kernel's CTA c covered pages
// [c*W/C, (c+1)*W/C) of the flattened (sequence, kv head, page) order and
// wrote every unit it covered whole; a unit spread over CTAs c0..c1 left one
// record in each: slot 1 of c0 when the unit began inside c0's range (slot 0
// when exactly at its start), slot 0 of every later CTA whose share is not
// empty (with more CTAs than pages, some CTAs take no page and write nothing).  One CTA per (query
// head, sequence) finds its unit's CTAs from the same arithmetic and merges
// their records as the partition combine does.  Records hold every row of a
// unit: [C][2][Q * G].
template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_balanced_kernel(const CombineParams p) {
    constexpr int SLICES = D / 4;
    constexpr int PGRP = kCombineThreads / SLICES;
    constexpr float NEG_INF = -INFINITY;
    extern __shared__ float weight[];                  // [records]
    __shared__ float red[kCombineThreads / 32];
    __shared__ float4 part[PGRP][SLICES];
    __shared__ long long span[2];                      // W, flat start of sequence b
    grid_dependency_wait();
    grid_launch_dependents();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = (int)blockIdx.x % p.num_heads, qi = (int)blockIdx.x / p.num_heads;
    const int b = blockIdx.y;
    const int Hkv = p.num_kv_heads;
    const int kvh = h / p.group;
    const int U = p.q_len * p.group, u = qi * p.group + h % p.group;
    if (warp == 0) {
        long long all = 0, before = 0;
        for (int b0 = lane; b0 < p.batch; b0 += 32) {
            const int T = reachable_tokens(p.context_lens, b0, p.max_blocks, p.block_size);
            const int np = (T + p.block_size - 1) / p.block_size;
            all += np;
            if (b0 < b) before += np;
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            all += __shfl_xor_sync(kFullMask, all, m);
            before += __shfl_xor_sync(kFullMask, before, m);
        }
        if (lane == 0) {
            span[0] = all * Hkv;
            span[1] = before * Hkv;
        }
    }
    __syncthreads();
    const long long W = span[0];
    const int T = reachable_tokens(p.context_lens, b, p.max_blocks, p.block_size);
    const int np = (T + p.block_size - 1) / p.block_size;
    const size_t o = (((size_t)b * p.q_len + qi) * p.num_heads + h) * D;
    if (np == 0) {  // no page, no CTA: the empty-context result
        for (int d = tid; d < D; d += kCombineThreads) store_out(p.out, o + d, 0.f, p.out_dtype);
        return;
    }
    const long long Cn = p.num_ctas;
    const long long A = span[1] + (long long)kvh * np, E = A + np;
    const long long c0 = ((A + 1) * Cn - 1) / W, c1 = (E * Cn - 1) / W;
    if (c0 == c1) return;  // one CTA covered the unit and wrote it
    const int nrec = (int)(c1 - c0 + 1);
    const bool c0_tail = A != c0 * W / Cn;
    auto rec_row = [&](int k) -> size_t {
        const long long c = c0 + k;
        const int slotk = (k == 0 && c0_tail) ? 1 : 0;
        return ((size_t)c * 2 + slotk) * U + u;
    };
    // CTA c0 + k wrote a record only if its share [c*W/C, (c+1)*W/C) is not empty
    auto live = [&](int k) -> bool {
        const long long c = c0 + k;
        return (c + 1) * W / Cn > c * W / Cn;
    };
    const float2* ml = reinterpret_cast<const float2*>(p.part_ml);

    float mx = NEG_INF;
    for (int k = tid; k < nrec; k += kCombineThreads)
        if (live(k)) mx = fmaxf(mx, ml[rec_row(k)].x);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, m));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();
    float ls = 0.f;
    for (int k = tid; k < nrec; k += kCombineThreads) {
        float w = 0.f;
        if (live(k)) {
            const float2 v = ml[rec_row(k)];
            w = (v.x == NEG_INF) ? 0.f : exp2f(v.x - mx);
            ls = fmaf(w, v.y, ls);
        }
        weight[k] = w;
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ls += __shfl_xor_sync(kFullMask, ls, m);
    if (lane == 0) red[warp] = ls;
    __syncthreads();  // also publishes `weight`
    ls = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) ls += red[w];

    const bool empty = (mx == NEG_INF) || !(ls > 0.f);
    const int pg = tid / SLICES, sl = tid % SLICES;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
        for (int k = pg; k < nrec; k += PGRP) {
            const float w = weight[k];
            if (w == 0.f) continue;  // no record (or an empty one): nothing to add
            const float4 x = reinterpret_cast<const float4*>(p.part_acc + rec_row(k) * D)[sl];
            a.x = fmaf(w, x.x, a.x);
            a.y = fmaf(w, x.y, a.y);
            a.z = fmaf(w, x.z, a.z);
            a.w = fmaf(w, x.w, a.w);
        }
    }
    part[pg][sl] = a;
    __syncthreads();
    if (pg == 0) {
        for (int k = 1; k < PGRP; ++k) {
            const float4 x = part[k][sl];
            a.x += x.x;
            a.y += x.y;
            a.z += x.z;
            a.w += x.w;
        }
        const float inv = empty ? 0.f : 1.f / ls;
        store_out(p.out, o + sl * 4, a.x * inv, p.out_dtype);
        store_out(p.out, o + sl * 4 + 1, a.y * inv, p.out_dtype);
        store_out(p.out, o + sl * 4 + 2, a.z * inv, p.out_dtype);
        store_out(p.out, o + sl * 4 + 3, a.w * inv, p.out_dtype);
    }
}

// Append of one new token per sequence (MiniVLLM docs "Decoding Benchmark":
// each decode step stores the new token's keys/values in the block the table
// assigns, at slot position % block_size).  One CTA per sequence copies the
// token's row for all kv heads (contiguous in both the new-token array and
// the cache slot) with 16-byte vectors.  Positions outside the table row and
// masked entries write nothing.
__global__ void __launch_bounds__(128) append_kernel(uint4* k_cache, uint4* v_cache,
                                                    const uint4* k_new, const uint4* v_new,
                                                    const int32_t* block_tables,
                                                    const int32_t* positions, int32_t max_blocks,
                                                    int32_t block_size, int64_t num_blocks,
                                                    int32_t row_vecs) {
    grid_dependency_wait();  // the new rows may come from the previous kernel
    grid_launch_dependents();
    const int b = blockIdx.x;
    const int pos = __ldg(positions + b);
    if (pos < 0 || pos >= max_blocks * block_size) return;
    const int e = __ldg(block_tables + (size_t)b * max_blocks + pos / block_size);
    if (e < 0 || (int64_t)e >= num_blocks) return;
    const size_t dst = ((size_t)e * block_size + pos % block_size) * row_vecs;
    const size_t src = (size_t)b * row_vecs;
    for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        k_cache[dst + i] = __ldg(k_new + src + i);
        v_cache[dst + i] = __ldg(v_new + src + i);
    }
}

// Self-test of the bounded wait: an mbarrier that nothing ever arrives at.
// The wait gives up after `timeout_ns` and records PA_ERR_TIMEOUT, exactly as
// the decode kernels do when their copy pipeline stops delivering.
__global__ void wait_timeout_kernel(int32_t* err, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_init_fence();
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(smem_u32(&bar), 0u, timeout_ns);
    if (!ok && threadIdx.x == 0) record_error(err, PA_ERR_TIMEOUT);
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
    const uint32_t smem = (uint32_t)p.num_parts * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_combine_balanced(const CombineParams& p, int head_dim, dim3 grid, bool pdl,
                                    cudaStream_t stream) {
    void (*kern)(const CombineParams);
    switch (head_dim) {
        case 64: kern = combine_balanced_kernel<64>; break;
        case 128: kern = combine_balanced_kernel<128>; break;
        default: kern = combine_balanced_kernel<256>; break;
    }
    const uint32_t smem = (uint32_t)(p.num_ctas + 1) * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* block_tables, const int32_t* positions, int32_t batch,
                          int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                          int32_t row_bytes, bool pdl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)batch);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, append_kernel, static_cast<uint4*>(k_cache),
                              static_cast<uint4*>(v_cache), static_cast<const uint4*>(k_new),
                              static_cast<const uint4*>(v_new), block_tables, positions,
                              max_blocks, block_size, num_blocks, row_bytes / 16);
}

cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
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
