// Paged-attention decode kernel for sm_103a: one CTA per (sequence, kv head,
// partition of the sequence's pages).
//
// What it computes ("benchmark_decoding.py", reference_output and the Triton
// (new) kernel; MiniVLLM docs "Decoding Benchmark", "Why CUDA chunk processing
// matters"): for every query head h of the kv head's group,
//     out[b, h] = sum_t softmax_t(scale * q[b, h] . K_t) V_t
// over the partition's tokens, with a running max m and normaliser l (the
// online softmax) so that no score array is ever stored.  In split mode the
// CTA writes (m, l, unnormalised acc) for its partition instead
// (flash-decoding-bench "design.md": per-chunk local max, sum and weighted
// values), and a second kernel combines the partitions.
//
// How it maps to GB300:
//   - K/V are read once per (sequence, kv head): every query head of the GQA
//     group is served from the same staged page, so the group does not re-read
//     it (the Triton kernel launches one program per query head instead).
//   - The CTA's warps form `nt` independent token streams.  Each stream owns a
//     ring of `ns` shared-memory stages; one lane issues a 4-D TMA copy per K
//     and V page (a single block-table read per page, not per token) and an
//     mbarrier signals its arrival.  A stream's `nh` warps split the head group
//     (at most 4 heads each) and release a stage through a second mbarrier.
//   - Inside a warp, LPT = head_dim/8 lanes cover one token row with 16-byte
//     vectors (8 elements each) and 32/LPT rows are processed side by side.
//     Partial q.K dot products of a chunk (8 row steps x up to 4 heads) are
//     summed across the LPT lanes with a transposing butterfly: each level
//     halves the values a lane carries, so a chunk costs ~STEPS*GW shuffles
//     instead of STEPS*GW*log2(LPT).
//   - Scores are kept in base-2 units (q is pre-multiplied by
//     scale*log2(e)); softmax uses exp2.  All arithmetic is fp32.
//   - Tokens past the context (and pages whose table entry is masked) are
//     excluded by select, never by multiplying by zero, so poison in unused
//     slots cannot leak into the result.
//   - Every mbarrier wait is bounded; on timeout the kernel records
//     PA_ERR_TIMEOUT in the device error word and abandons its work.
// No tensor cores: with one query token per sequence the contraction is a
// matrix-vector product, bound by HBM bandwidth, not by math throughput.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int D, int BS, int GW>
struct AttnCfg {
    static constexpr int LPT = D / 8;                               // lanes per token row
    static constexpr int TPS = 32 / LPT;                            // rows per warp step
    static constexpr int STEPS = (8 * TPS <= BS) ? 8 : BS / TPS;    // row steps per chunk
    static constexpr int CHUNK = STEPS * TPS;                       // tokens per chunk
    static constexpr int NVAL = STEPS * GW;                         // partial dots per lane
    static constexpr int NOUT = NVAL >= LPT ? NVAL / LPT : 1;       // reduced dots per lane
    static constexpr int DUP = NVAL >= LPT ? 1 : LPT / NVAL;        // lanes holding one dot
    static constexpr int HL = LPT / GW;                             // lanes per head in a row group
    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    static_assert(BS % CHUNK == 0, "a chunk must not straddle a page");
    static_assert(STEPS % NOUT == 0, "a lane's reduced dots belong to one head");
};

// Sum each of N per-lane values over the LPT lanes of a row group (xor masks
// LPT/2 .. 1).  While a lane carries two or more values, each level keeps half
// of them and trades the other half with its partner, so after log2(N) levels
// a lane holds the full sums of its own values; remaining levels (N < LPT)
// are plain butterflies that leave duplicates.  On return vals[0..NOUT) hold
// the sums of original indices [lig*NOUT, lig*NOUT + NOUT) when N >= LPT, or
// of index lig / (LPT/N) otherwise (lig = lane % LPT).
template <int N, int LPT>
__device__ __forceinline__ void transpose_reduce(float (&vals)[N], int lane) {
    int n = N;
#pragma unroll
    for (int mask = LPT / 2; mask >= 1; mask >>= 1) {
        if (n >= 2) {
            const int half = n / 2;
            const bool upper = (lane & mask) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (i < half) {
                    const float lo = vals[i], hi = vals[i + half];
                    const float send = upper ? lo : hi;
                    const float keep = upper ? hi : lo;
                    vals[i] = keep + __shfl_xor_sync(kFullMask, send, mask);
                }
            }
            n = half;
        } else {
            vals[0] += __shfl_xor_sync(kFullMask, vals[0], mask);
        }
    }
}

template <int D, int BS, typename KV, int GW>
__global__ void __launch_bounds__(256, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    using C = AttnCfg<D, BS, GW>;
    constexpr int LPT = C::LPT, TPS = C::TPS, STEPS = C::STEPS, CHUNK = C::CHUNK;
    constexpr int NVAL = C::NVAL, NOUT = C::NOUT, DUP = C::DUP, HL = C::HL;
    constexpr float NEG_INF = -INFINITY;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + (kSmemAlignSlack - 1)) &
        ~uintptr_t(kSmemAlignSlack - 1));
    const AttnSmem L = attn_smem_layout(D, BS, (int)sizeof(KV), GW, TPS, STEPS, p.nt, p.nh, p.ns);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stream = warp / p.nh, hg = warp % p.nh;
    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int G = p.group;

    const int T = reachable_tokens(p.context_lens, b, p.max_blocks, BS);
    const int npages = (T + BS - 1) / BS;
    const int pb = part * p.part_pages;
    const int pe = min(pb + p.part_pages, npages);
    if (pb >= pe) {
        // Nothing of this sequence falls in the partition.  The single pass
        // writes the empty-context result; the combine kernel never reads
        // partitions past the context.
        if (p.final_out) {
            for (int idx = tid; idx < G * D; idx += blockDim.x) {
                const int h = kvh * G + idx / D;
                store_out(p.out, ((size_t)b * p.num_heads + h) * D + idx % D, 0.f, p.out_dtype);
            }
        }
        return;
    }

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty_off);
    int32_t* phys_of = reinterpret_cast<int32_t*>(smem + L.phys_off);
    float* pbuf = reinterpret_cast<float*>(smem + L.pbuf_off);
    float* mrg = reinterpret_cast<float*>(smem + L.mrg_off);

    if (tid == 0) {
        for (int i = 0; i < p.nt * p.ns; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), p.nh);
        }
        mbar_init_fence();
    }
    __syncthreads();

    const int32_t* table_row = p.block_tables + (size_t)b * p.max_blocks;
    const int span = pe - pb;
    const int n_s = span > stream ? (span - stream + p.nt - 1) / p.nt : 0;  // pages of this stream
    const bool leader = hg == 0 && lane == 0;
    const uint64_t policy = l2_policy_evict_first();
    int n_issued = 0;

    // Stage local page i of this stream: one table read, then one TMA copy
    // each for the K and V page of this kv head (bs rows of head_dim).
    auto issue = [&](int i) {
        const int sidx = stream * p.ns + i % p.ns;
        const int j = pb + stream + i * p.nt;
        const int phys = page_phys(table_row, j, npages, p.num_blocks);
        phys_of[sidx] = phys;
        const uint32_t bar = smem_u32(full + sidx);
        if (phys >= 0) {
            mbar_arrive_expect_tx(bar, L.stage_bytes);
            const uint32_t dst = smem_u32(smem + L.stages_off + (size_t)sidx * L.stage_bytes);
            tma_load_4d(dst, &tmap_k, 0, kvh, 0, phys, bar, policy);
            tma_load_4d(dst + L.stage_bytes / 2, &tmap_v, 0, kvh, 0, phys, bar, policy);
        } else {
            mbar_arrive(bar);
        }
    };

    if (leader) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
        const int pro = n_s < p.ns ? n_s : p.ns;
        for (int i = 0; i < pro; ++i) issue(i);
        n_issued = pro;
    }

    // This warp's query heads, pre-scaled into base-2 score units.
    const int lig = lane & (LPT - 1);  // 16-byte slice of the head dimension
    const int ts = lane / LPT;         // row within a step
    float qf[GW][8];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
        const int h = kvh * G + hg * GW + g;
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
            static_cast<const KV*>(p.q) + ((size_t)b * p.num_heads + h) * D + lig * 8));
        Vec8<KV>::to_float(raw, qf[g]);
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[g][e] *= p.qscale;
    }

    float m[GW], acc[GW][8];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
        m[g] = NEG_INF;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    }
    float l_own = 0.f;  // normaliser share of this lane's head

    const int vbase = (NVAL >= LPT) ? lig * NOUT : lig / DUP;  // first reduced dot of this lane
    const int gown = vbase / STEPS;                            // its head
    const bool designated = (DUP == 1) || (lig % DUP) == 0;
    float* pw_base = pbuf + (size_t)(warp * TPS + ts) * STEPS * GW;

    bool aborted = false;
    int i = 0;
    for (; i < n_s; ++i) {
        const int sidx = stream * p.ns + i % p.ns;
        const uint32_t par = (uint32_t)(i / p.ns) & 1u;
        const bool ok = __all_sync(kFullMask, mbar_wait_bounded(smem_u32(full + sidx), par,
                                                                p.timeout_ns));
        if (!ok) {
            if (lane == 0) record_error(p.err, PA_ERR_TIMEOUT);
            aborted = true;
            break;
        }
        const int phys = phys_of[sidx];
        if (phys >= 0) {
            const int j = pb + stream + i * p.nt;
            const int nvalid = min(BS, T - j * BS);
            const KV* Kt = reinterpret_cast<const KV*>(smem + L.stages_off +
                                                       (size_t)sidx * L.stage_bytes);
            const KV* Vt = Kt + BS * D;

            for (int c0 = 0; c0 < nvalid; c0 += CHUNK) {
                // ---- q.K partial dots over this lane's 8 dims ----
                float v[NVAL];
#pragma unroll
                for (int st = 0; st < STEPS; ++st) {
                    const int row = c0 + st * TPS + ts;
                    const uint4 raw = *reinterpret_cast<const uint4*>(Kt + row * D + lig * 8);
                    float kf[8];
                    Vec8<KV>::to_float(raw, kf);
#pragma unroll
                    for (int g = 0; g < GW; ++g) {
                        float a = qf[g][0] * kf[0];
#pragma unroll
                        for (int e = 1; e < 8; ++e) a = fmaf(qf[g][e], kf[e], a);
                        v[g * STEPS + st] = a;
                    }
                }
                transpose_reduce<NVAL, LPT>(v, lane);

                // ---- chunk max per head, online-softmax rescale ----
                float cmax = NEG_INF;
#pragma unroll
                for (int k = 0; k < NOUT; ++k) {
                    const int row = c0 + ((vbase + k) % STEPS) * TPS + ts;
                    v[k] = row < nvalid ? v[k] : NEG_INF;
                    cmax = fmaxf(cmax, v[k]);
                }
#pragma unroll
                for (int mask = 1; mask < HL; mask <<= 1)
                    cmax = fmaxf(cmax, __shfl_xor_sync(kFullMask, cmax, mask));
#pragma unroll
                for (int mask = LPT; mask < 32; mask <<= 1)
                    cmax = fmaxf(cmax, __shfl_xor_sync(kFullMask, cmax, mask));

                float alpha_own = 1.f, m_own = NEG_INF;
#pragma unroll
                for (int g = 0; g < GW; ++g) {
                    const float cm = __shfl_sync(kFullMask, cmax, g * HL);
                    const float mn = fmaxf(m[g], cm);
                    const float alpha = (m[g] == mn) ? 1.f : exp2f(m[g] - mn);
                    m[g] = mn;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
                    if (g == gown) {
                        alpha_own = alpha;
                        m_own = mn;
                    }
                }

                // ---- probabilities of this lane's dots ----
                float psum = 0.f;
#pragma unroll
                for (int k = 0; k < NOUT; ++k) {
                    const float pk = exp2f(v[k] - m_own);  // exp2(-inf) = 0 for masked rows
                    psum += pk;
                    if (designated) pw_base[((vbase + k) % STEPS) * GW + gown] = pk;
                }
                l_own = l_own * alpha_own + (designated ? psum : 0.f);
                __syncwarp();

                // ---- acc += p * V over the chunk's rows ----
#pragma unroll
                for (int st = 0; st < STEPS; ++st) {
                    const int row = c0 + st * TPS + ts;
                    if (row < nvalid) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(Vt + row * D + lig * 8);
                        float vf[8];
                        Vec8<KV>::to_float(raw, vf);
                        float pw[GW];
#pragma unroll
                        for (int g = 0; g < GW; ++g) pw[g] = pw_base[st * GW + g];
#pragma unroll
                        for (int g = 0; g < GW; ++g)
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pw[g], vf[e], acc[g][e]);
                    }
                }
                __syncwarp();
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + sidx));
        // Refill the stage just released with this stream's page i + ns.
        int refill_failed = 0;
        if (leader && i + p.ns < n_s) {
            if (mbar_wait_bounded(smem_u32(empty + sidx), par, p.timeout_ns)) {
                fence_proxy_async_smem();
                issue(i + p.ns);
                ++n_issued;
            } else {
                record_error(p.err, PA_ERR_TIMEOUT);
                refill_failed = 1;
            }
        }
        if (__shfl_sync(kFullMask, refill_failed, 0)) {
            aborted = true;
            ++i;
            break;
        }
    }
    if (aborted && leader) {
        // Let copies this stream still has in flight land before the CTA exits.
        for (int k = i; k < n_issued; ++k)
            (void)mbar_wait_bounded(smem_u32(full + stream * p.ns + k % p.ns),
                                    (uint32_t)(k / p.ns) & 1u, p.timeout_ns);
    }

    // ---- per-warp totals: rows of a step share m, so plain sums ----
#pragma unroll
    for (int mask = LPT; mask < 32; mask <<= 1)
#pragma unroll
        for (int g = 0; g < GW; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(kFullMask, acc[g][e], mask);
#pragma unroll
    for (int mask = 1; mask < HL; mask <<= 1) l_own += __shfl_xor_sync(kFullMask, l_own, mask);
#pragma unroll
    for (int mask = LPT; mask < 32; mask <<= 1) l_own += __shfl_xor_sync(kFullMask, l_own, mask);

    const uint32_t MS = merge_stride(D, GW);
    float* wm = mrg + (size_t)warp * MS;  // acc [GW][D], then m [GW], l [GW]
#pragma unroll
    for (int g = 0; g < GW; ++g) {
        const float lg = __shfl_sync(kFullMask, l_own, g * HL);
        if (lane < LPT) {
            float4* dst = reinterpret_cast<float4*>(wm + g * D + lig * 8);
            dst[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
            dst[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
        }
        if (lane == 0) {
            wm[GW * D + g] = m[g];
            wm[GW * D + GW + g] = lg;
        }
    }
    __syncthreads();

    // ---- merge the token streams (log-sum-exp), then write ----
    for (int idx = tid; idx < G * D; idx += blockDim.x) {
        const int gfull = idx / D, d = idx % D;
        const int hgx = gfull / GW, gi = gfull % GW;
        float M = NEG_INF;
        for (int s2 = 0; s2 < p.nt; ++s2)
            M = fmaxf(M, mrg[(size_t)(s2 * p.nh + hgx) * MS + GW * D + gi]);
        float A = 0.f, Ls = 0.f;
        if (M != NEG_INF) {
            for (int s2 = 0; s2 < p.nt; ++s2) {
                const float* w2 = mrg + (size_t)(s2 * p.nh + hgx) * MS;
                const float ms = w2[GW * D + gi];
                if (ms != NEG_INF) {
                    const float f = exp2f(ms - M);
                    A = fmaf(f, w2[gi * D + d], A);
                    Ls = fmaf(f, w2[GW * D + GW + gi], Ls);
                }
            }
        }
        const int h = kvh * G + gfull;
        if (p.final_out) {
            store_out(p.out, ((size_t)b * p.num_heads + h) * D + d, Ls > 0.f ? A / Ls : 0.f,
                      p.out_dtype);
        } else {
            const size_t row = (((size_t)b * p.num_kv_heads + kvh) * p.num_parts + part) * G + gfull;
            p.part_acc[row * D + d] = A;
            if (d == 0) {
                p.part_ml[row * 2] = M;
                p.part_ml[row * 2 + 1] = Ls;
            }
        }
    }
}

template <int D, int BS, typename KV, int GW>
cudaError_t launch_attn_inst(const AttnLaunch& L, cudaStream_t stream) {
    auto kern = attn_kernel<D, BS, KV, GW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L.smem_bytes);
    if (e != cudaSuccess) return e;
    kern<<<L.grid, L.threads, L.smem_bytes, stream>>>(L.tmap_k, L.tmap_v, L.p);
    return cudaGetLastError();
}

template <int D, int BS, typename KV>
cudaError_t launch_attn_gw(const AttnLaunch& L, cudaStream_t stream) {
    switch (L.heads_per_warp) {
        case 1: return launch_attn_inst<D, BS, KV, 1>(L, stream);
        case 2: return launch_attn_inst<D, BS, KV, 2>(L, stream);
        case 4: return launch_attn_inst<D, BS, KV, 4>(L, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_attn_for_d(const AttnLaunch& L, cudaStream_t stream) {
    const bool bf = L.kv_dtype == PA_BF16;
    if (L.block_size == 16)
        return bf ? launch_attn_gw<D, 16, __nv_bfloat16>(L, stream)
                  : launch_attn_gw<D, 16, __half>(L, stream);
    if (L.block_size == 32)
        return bf ? launch_attn_gw<D, 32, __nv_bfloat16>(L, stream)
                  : launch_attn_gw<D, 32, __half>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
