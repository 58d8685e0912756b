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
//   - K/V are read from HBM once per (sequence, kv head): the whole GQA group
//     (up to 16 query heads) is served from the same staged page.
//   - The CTA's warps form `nt` independent token streams.  Each stream owns a
//     ring of `ns` shared-memory stages; one lane reads one block-table entry
//     per page and issues 4-D TMA copies of the page's K and V tiles (column
//     blocks of 64 elements, 128-byte swizzle), and an mbarrier signals their
//     arrival.  The stream's warps release a stage through a second mbarrier.
//   - The two contractions of a page run on the tensor cores as warp-level
//     m16n8k16 MMAs with fp32 accumulation: the group's query heads are the 16
//     rows (padded with zero rows when the group is smaller), tokens and head
//     dims the other two dimensions.  S = Q K^T takes K fragments straight
//     from the swizzled tile with ldmatrix; O += P V takes V fragments with
//     ldmatrix.trans and P from the S accumulators, split into a high and a
//     low 16-bit part (two MMAs) so that P keeps ~16 significant bits.  This
//     replaces ~2*G*D multiply-adds per token on the CUDA cores, which at the
//     GB300's bandwidth-to-FP32 ratio would consume the SM's whole issue budget.
//   - Online softmax in base-2 units with conditional rescaling: the running
//     max of a head only moves (and acc, l are rescaled) when a page's max
//     exceeds it by more than 2^8; the result acc/l is the same for any such
//     reference value.
//   - Tokens past the context are excluded by select; the V rows of a partial
//     last page are zeroed in shared memory before the MMA (0 * NaN would
//     otherwise leak poison), masked pages are never read.
//   - Every mbarrier wait is bounded; on timeout the kernel records
//     PA_ERR_TIMEOUT in the device error word and abandons its work.
#pragma once

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

template <int D, int BS>
struct AttnCfg {
    static constexpr int DS = (D == 256) ? 2 : 1;  // warps that split one page's output columns
    static constexpr int DW = D / DS;              // output columns per warp
    static constexpr int KSTEPS = D / 16;          // k-steps of S = Q K^T
    static constexpr int NT = BS / 8;              // token n-tiles of S per page
    static constexpr int PKS = BS / 16;            // k-steps of O += P V per page
    static constexpr int ONT = DW / 8;             // output n-tiles per warp
    static constexpr int DBLK = D / 64;            // 128-byte column blocks per tile
    static_assert(D == 64 || D == 128 || D == 256, "head_dim");
    static_assert(BS == 16 || BS == 32, "block_size");
};

// Byte offset of (row t, 16-byte chunk c) in a tile written by TMA with the
// 128-byte swizzle: chunk c & 7 of a 128-byte row lands at (c & 7) ^ (t & 7).
template <int BS>
__device__ __forceinline__ uint32_t swz(int t, int c) {
    return (uint32_t)((c >> 3) * BS * 128 + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

constexpr float kRescaleSlack = 8.0f;  // log2 units: p may reach 2^8 before a rescale

// Where the merged result of a segment goes.
enum SegOut { kOutFinal = 0, kOutPartial = 1, kOutCluster = 2, kOutRecord = 3 };

// MULTI: several query tokens per sequence (rows are (query token, head)
// pairs with a causal limit each); otherwise one token, rows = the group's heads.
template <int D, int BS, typename KV, bool MULTI>
__global__ void __launch_bounds__(256, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    using C = AttnCfg<D, BS>;
    constexpr int DS = C::DS, DW = C::DW, KSTEPS = C::KSTEPS, NT = C::NT, PKS = C::PKS;
    constexpr int ONT = C::ONT, DBLK = C::DBLK;
    constexpr float NEG_INF = -INFINITY;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + (kSmemAlignSlack - 1)) &
        ~uintptr_t(kSmemAlignSlack - 1));
    const AttnSmem L = attn_smem_layout(D, BS, p.nt, p.ns);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int stream = warp / DS, ds = warp % DS;
    const int G = p.group, Hkv = p.num_kv_heads;
    const int Q = MULTI ? p.q_len : 1;
    const int gshift = __ffs(G) - 1;  // the group is a power of two
    // MMA rows are (query token, head) pairs: row r is query token qi0 + r / G
    // and head kvh * G + r % G.  A CTA takes the query tokens of one chunk.
    const int qi0 = MULTI ? ((int)blockIdx.y / Hkv) * p.q_chunk : 0;
    const int R = MULTI ? min(p.q_chunk, Q - qi0) * G : G;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full_off);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty_off);
    int32_t* phys_of = reinterpret_cast<int32_t*>(smem + L.phys_off);
    int32_t* seq_pages = reinterpret_cast<int32_t*>(smem + L.seq_off);  // balanced split only
    if (tid == 0) {
        for (int i = 0; i < p.nt * p.ns; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), DS);
        }
        mbar_init_fence();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    // Inputs may come from the previous kernel in the stream.
    grid_dependency_wait();
    grid_launch_dependents();

    const int g = lane >> 2, tig = lane & 3;
    const bool real0 = g < R, real1 = g + 8 < R;
    const float qscale = p.qscale;
    const int ldsm_t = lane & 7;         // row supplied to ldmatrix
    const int ldsm_m = lane >> 3;        // matrix supplied to ldmatrix
    const int col0 = ds * (DW / 8);      // first 16-byte output chunk of this warp
    const int nw = p.nt * DS;
    // After a segment's pages are consumed the stage area holds the merge data.
    float* macc = reinterpret_cast<float*>(smem + L.stages_off);   // [nw][R][DW]
    float* mm = macc + (size_t)nw * R * DW;                         // [nw][R] running max
    float* mls = mm + nw * R;                                       // [nw][R] normaliser
    float* cpart = mls + nw * R;  // this CTA's partial when the cluster reduces: acc [R][D], m [R], l [R]

    // Element offset of row r's query (and output) vector: [B, Q, H, D].
    auto row_off = [&](int b, int kvh, int r) -> size_t {
        if constexpr (MULTI)
            return (((size_t)b * Q + qi0 + (r >> gshift)) * p.num_heads + kvh * G +
                    (r & (G - 1))) * D;
        else
            return ((size_t)b * p.num_heads + kvh * G + r) * D;
    };

    // Pipeline state of this warp's stream, carried across segments.
    int slot = 0;
    uint32_t par = 0;
    bool aborted = false;

    // Table entries of this stream's pages of the current segment, 32 at a
    // time, one per lane of the leader warp.
    const int32_t* table_row = nullptr;
    int seg_pb = 0, seg_fetch_end = 0;
    int ent_cur = -1, ent_next = -1, cur_chunk = 0;
    auto fetch = [&](int chunk) -> int {
        const int li = chunk * 32 + lane;
        const int j = seg_pb + stream + li * p.nt;
        return j < seg_fetch_end ? __ldg(table_row + j) : -1;
    };
    auto start_fetch = [&](int b, int pb, int fetch_end) {
        table_row = p.block_tables + (size_t)b * p.max_blocks;
        seg_pb = pb;
        seg_fetch_end = fetch_end;
        cur_chunk = 0;
        if (ds == 0) {
            ent_cur = fetch(0);
            ent_next = fetch(1);
        }
    };

    // Pages [pb, pe) of (sequence b, kv head kvh), whose table reaches T
    // tokens; the leader warp has already called start_fetch(b, pb, >= pe).
    // The streams take the pages in turn; the merged (m, l, acc) of every
    // row is handed to emit(idx = r*D + d, A, M, L).  Query token qi sits at
    // position ctx - Q + qi and attends to the tokens before and at it.
    auto run_segment = [&](int b, int kvh, int pb, int pe, int T, auto&& emit) {
        const int npages = (T + BS - 1) / BS;
        const int span = pe - pb;
        const int n_s = span > stream ? (span - stream + p.nt - 1) / p.nt : 0;
        const int slot0 = slot;
        const uint32_t par0 = par;
        int n_issued = 0;

        // Stage local page i of this stream (whole leader warp): its table
        // entry, then one TMA copy per 64-column block of its K and V tiles.
        auto issue = [&](int i, int sidx) {
            if ((i >> 5) != cur_chunk) {  // slide the prefetched window
                cur_chunk = i >> 5;
                ent_cur = ent_next;
                ent_next = fetch(cur_chunk + 1);
            }
            const int e = __shfl_sync(kFullMask, ent_cur, i & 31);
            const int j = pb + stream + i * p.nt;
            const int phys = (j < npages && e >= 0 && (int64_t)e < p.num_blocks) ? e : -1;
            if (lane == 0) {
                phys_of[sidx] = phys;
                const uint32_t bar = smem_u32(full + sidx);
                if (phys >= 0) {
                    const uint64_t policy = l2_policy_evict_first();
                    mbar_arrive_expect_tx(bar, L.stage_bytes);
                    const uint32_t dst =
                        smem_u32(smem + L.stages_off + (size_t)sidx * L.stage_bytes);
#pragma unroll
                    for (int blk = 0; blk < DBLK; ++blk) {
                        tma_load_4d(dst + blk * BS * 128, &tmap_k, blk * 64, kvh, 0, phys, bar,
                                    policy);
                        tma_load_4d(dst + L.tile_bytes + blk * BS * 128, &tmap_v, blk * 64, kvh,
                                    0, phys, bar, policy);
                    }
                } else {
                    mbar_arrive(bar);
                }
            }
        };

        if (ds == 0 && !aborted) {
            const int pro = n_s < p.ns ? n_s : p.ns;
            int sl = slot0;
            for (int i = 0; i < pro; ++i) {
                issue(i, stream * p.ns + sl);
                if (++sl == p.ns) sl = 0;
            }
            n_issued = pro;
        }

        // ---- Q fragments (A operand of S = Q K^T): rows g and g + 8 ----
        uint32_t qa[KSTEPS][4];
        {
            // (the rows of padded lanes are never loaded)
            const KV* q = static_cast<const KV*>(p.q);
            const uint32_t* q0 = reinterpret_cast<const uint32_t*>(q + row_off(b, kvh, g));
            const uint32_t* q1 = reinterpret_cast<const uint32_t*>(q + row_off(b, kvh, g + 8));
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int w = (kk * 16 + tig * 2) >> 1;  // 32-bit word index of the element pair
                qa[kk][0] = real0 ? __ldg(q0 + w) : 0u;
                qa[kk][1] = real1 ? __ldg(q1 + w) : 0u;
                qa[kk][2] = real0 ? __ldg(q0 + w + 4) : 0u;
                qa[kk][3] = real1 ? __ldg(q1 + w + 4) : 0u;
            }
        }

        // Tokens each row attends: the causal limit of its query token, inside
        // the table's reach (with one query token, every row attends T).
        int lim0 = T, lim1 = T;
        if constexpr (MULTI) {
            const int ctx = max(__ldg(p.context_lens + b), 0);
            lim0 = min(T, ctx - Q + qi0 + (g >> gshift) + 1);
            lim1 = min(T, ctx - Q + qi0 + ((g + 8) >> gshift) + 1);
        }

        // Running state of rows g and g+8 (padded rows stay at m = 0, p = 0).
        float m0 = real0 ? NEG_INF : 0.f, m1 = real1 ? NEG_INF : 0.f;
        float l0 = 0.f, l1 = 0.f;  // this lane's share of the normalisers
        float acc[ONT][4];
#pragma unroll
        for (int n = 0; n < ONT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

        int i = 0;
        for (; i < n_s && !aborted; ++i) {
            const int sidx = stream * p.ns + slot;
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
                uint8_t* kt = smem + L.stages_off + (size_t)sidx * L.stage_bytes;
                uint8_t* vt = kt + L.tile_bytes;
                const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);

                if (nvalid < BS) {
                    // Zero this warp's columns of the V rows past the context.
                    const int rows = BS - nvalid;
                    for (int idx = lane; idx < rows * 8 * (DW / 64); idx += 32) {
                        const int blk = ds * (DW / 64) + idx / (rows * 8);
                        const int rem = idx % (rows * 8);
                        *reinterpret_cast<uint4*>(vt + blk * BS * 128 + (nvalid + rem / 8) * 128 +
                                                  (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }

                // ---- S = Q K^T (fp32), even and odd k-steps in separate chains ----
                float s[NT][4], s2[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
                    s2[nt][0] = s2[nt][1] = s2[nt][2] = s2[nt][3] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < KSTEPS; kk += 2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kbase + swz<BS>(nt * 8 + ldsm_t, 2 * kk + ldsm_m), b0, b1, b2, b3);
                        Mma<KV>::mma(s[nt], qa[kk], b0, b1);
                        Mma<KV>::mma(s2[nt], qa[kk + 1], b2, b3);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
                }

                // ---- page max per row, conditional rescale ----
                // this page's attended tokens of rows g and g + 8
                const int v0 = MULTI ? lim0 - j * BS : nvalid;
                const int v1 = MULTI ? lim1 - j * BS : nvalid;
                float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = nt * 8 + tig * 2 + e;
                        s[nt][e] = c < v0 ? s[nt][e] : NEG_INF;
                        s[nt][2 + e] = c < v1 ? s[nt][2 + e] : NEG_INF;
                        mx0 = fmaxf(mx0, s[nt][e]);
                        mx1 = fmaxf(mx1, s[nt][2 + e]);
                    }
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, 2));
                const float ms0 = mx0 * qscale, ms1 = mx1 * qscale;
                const bool need = (real0 && ms0 > m0 + kRescaleSlack) ||
                                  (real1 && ms1 > m1 + kRescaleSlack);
                if (__any_sync(kFullMask, need)) {
                    const float n0 = real0 ? fmaxf(m0, ms0) : m0;
                    const float n1 = real1 ? fmaxf(m1, ms1) : m1;
                    const float a0 = (n0 == m0) ? 1.f : fast_exp2(m0 - n0);
                    const float a1 = (n1 == m1) ? 1.f : fast_exp2(m1 - n1);
                    m0 = n0;
                    m1 = n1;
                    l0 *= a0;
                    l1 *= a1;
#pragma unroll
                    for (int n = 0; n < ONT; ++n) {
                        acc[n][0] *= a0;
                        acc[n][1] *= a0;
                        acc[n][2] *= a1;
                        acc[n][3] *= a1;
                    }
                }

                // ---- P = 2^(S*scale*log2e - m), and its hi/lo 16-bit split ----
                // (with several query tokens, a row that has attended nothing
                // yet still has m = -inf and only -inf scores; its P must come
                // out 0, not NaN.  With one token every real row has a finite
                // max once a page is read.)
                const float e0 = (MULTI && m0 == NEG_INF) ? 0.f : m0;
                const float e1 = (MULTI && m1 == NEG_INF) ? 0.f : m1;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        s[nt][e] = real0 ? fast_exp2(fmaf(s[nt][e], qscale, -e0)) : 0.f;
                        s[nt][2 + e] = real1 ? fast_exp2(fmaf(s[nt][2 + e], qscale, -e1)) : 0.f;
                        l0 += s[nt][e];
                        l1 += s[nt][2 + e];
                    }

                // ---- O += P V on this warp's columns ----
#pragma unroll
                for (int ks = 0; ks < PKS; ++ks) {
                    uint32_t ph[4], pl[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        // a0: n-tile 2ks rows g; a1: rows g+8; a2/a3: n-tile 2ks+1
                        const float x0 = s[2 * ks + (r >> 1)][(r & 1) * 2];
                        const float x1 = s[2 * ks + (r >> 1)][(r & 1) * 2 + 1];
                        ph[r] = Mma<KV>::pack(x0, x1);
                        float h0, h1;
                        Mma<KV>::unpack(ph[r], h0, h1);
                        pl[r] = Mma<KV>::pack(x0 - h0, x1 - h1);
                    }
#pragma unroll
                    for (int n = 0; n < ONT; n += 2) {
                        uint32_t b0, b1, b2, b3;
                        const int t = ks * 16 + ((ldsm_m & 1) << 3) + ldsm_t;
                        ldsm_x4_trans(vbase + swz<BS>(t, col0 + n + (ldsm_m >> 1)), b0, b1, b2,
                                      b3);
                        Mma<KV>::mma(acc[n], ph, b0, b1);
                        Mma<KV>::mma(acc[n], pl, b0, b1);
                        Mma<KV>::mma(acc[n + 1], ph, b2, b3);
                        Mma<KV>::mma(acc[n + 1], pl, b2, b3);
                    }
                }
            }
            __syncwarp();
            // A stream of one warp frees its own stage; with two, both must be done.
            if (DS > 1 && lane == 0) mbar_arrive(smem_u32(empty + sidx));
            // Refill the stage just released with this stream's page i + ns.
            int refill_failed = 0;
            if (ds == 0 && i + p.ns < n_s) {
                const bool freed = DS == 1 || __all_sync(kFullMask,
                                                         mbar_wait_bounded(smem_u32(empty + sidx),
                                                                           par, p.timeout_ns));
                if (freed) {
                    fence_proxy_async_smem();
                    issue(i + p.ns, sidx);
                    ++n_issued;
                } else {
                    if (lane == 0) record_error(p.err, PA_ERR_TIMEOUT);
                    refill_failed = 1;
                }
            }
            if (++slot == p.ns) {
                slot = 0;
                par ^= 1u;
            }
            if (__shfl_sync(kFullMask, refill_failed, 0)) {
                aborted = true;
                ++i;
                break;
            }
        }
        if (aborted && ds == 0 && lane == 0) {
            // Let copies this stream still has in flight land before moving on.
            for (int k = i; k < n_issued; ++k) {
                const int ks = (slot0 + k) % p.ns;
                const uint32_t kp = par0 ^ (uint32_t)(((slot0 + k) / p.ns) & 1);
                (void)mbar_wait_bounded(smem_u32(full + stream * p.ns + ks), kp, p.timeout_ns);
            }
        }

        // ---- per-warp normalisers: sum the quad's shares ----
        l0 += __shfl_xor_sync(kFullMask, l0, 1);
        l1 += __shfl_xor_sync(kFullMask, l1, 1);
        l0 += __shfl_xor_sync(kFullMask, l0, 2);
        l1 += __shfl_xor_sync(kFullMask, l1, 2);

        // Every stage of the segment has been consumed: the stage area now
        // holds the merge data.
        __syncthreads();
#pragma unroll
        for (int n = 0; n < ONT; ++n) {
            const int c = n * 8 + tig * 2;
            if (real0)
                *reinterpret_cast<float2*>(macc + ((size_t)warp * R + g) * DW + c) =
                    make_float2(acc[n][0], acc[n][1]);
            if (real1)
                *reinterpret_cast<float2*>(macc + ((size_t)warp * R + g + 8) * DW + c) =
                    make_float2(acc[n][2], acc[n][3]);
        }
        if (tig == 0) {
            if (real0) {
                mm[warp * R + g] = m0;
                mls[warp * R + g] = l0;
            }
            if (real1) {
                mm[warp * R + g + 8] = m1;
                mls[warp * R + g + 8] = l1;
            }
        }
        __syncthreads();

        // ---- merge the token streams (log-sum-exp) ----
        for (int idx = tid; idx < R * D; idx += blockDim.x) {
            const int r = idx / D, d = idx % D;
            const int dsx = d / DW, dd = d % DW;
            float M = NEG_INF;
            for (int s2 = 0; s2 < p.nt; ++s2) M = fmaxf(M, mm[(s2 * DS + dsx) * R + r]);
            float A = 0.f, Ls = 0.f;
            for (int s2 = 0; s2 < p.nt; ++s2) {
                const int w2 = s2 * DS + dsx;
                const float ms = mm[w2 * R + r];
                const float f = (ms == NEG_INF) ? 0.f : fast_exp2(ms - M);
                A = fmaf(f, macc[((size_t)w2 * R + r) * DW + dd], A);
                Ls = fmaf(f, mls[w2 * R + r], Ls);
            }
            emit(idx, A, M, Ls);
        }
        __syncthreads();  // the next segment's copies may now reuse the stage area
    };

    auto emit_final = [&](int b, int kvh) {
        return [&, b, kvh](int idx, float A, float M, float Ls) {
            store_out(p.out, row_off(b, kvh, idx / D) + idx % D, Ls > 0.f ? A / Ls : 0.f,
                      p.out_dtype);
        };
    };
    // (m, l, acc) of the CTA's rows into workspace row `row0 + r`.
    auto emit_rows = [&](size_t row0) {
        return [&, row0](int idx, float A, float M, float Ls) {
            const int r = idx / D, d = idx % D;
            p.part_acc[(row0 + r) * D + d] = A;
            if (d == 0) {
                p.part_ml[(row0 + r) * 2] = M;
                p.part_ml[(row0 + r) * 2 + 1] = Ls;
            }
        };
    };

    if (p.balanced) {
        // ---- balanced split: CTA c takes pages [c*W/C, (c+1)*W/C) of the
        // flattened (sequence, kv head, page) order, W pages in all; every
        // query token of a unit is in the CTA's rows ----
        int* totals = seq_pages + p.batch;  // [0]: W
        if (warp == 0) {
            int w = 0;
            for (int b0 = lane; b0 < p.batch; b0 += 32) {
                const int T = reachable_tokens(p.context_lens, b0, p.max_blocks, BS);
                const int np = (T + BS - 1) / BS;
                seq_pages[b0] = np;
                w += np;
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) w += __shfl_xor_sync(kFullMask, w, m);
            if (lane == 0) totals[0] = w * Hkv;
        }
        __syncthreads();
        const int64_t W = totals[0];
        const int64_t Cn = gridDim.x, c = blockIdx.x;
        const int64_t start = c * W / Cn, end = (c + 1) * W / Cn;
        if (start >= end) return;
        // locate the sequence holding flat page `start` (each thread of the
        // warp scans the same prefix, 32 sequences at a time)
        int b = 0;
        int64_t base = 0;  // flat index of sequence b's first page
        for (;;) {
            const int bb = b + lane;
            const int64_t v = bb < p.batch ? (int64_t)seq_pages[bb] * Hkv : 0;
            int64_t incl = v;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int64_t o = __shfl_up_sync(kFullMask, incl, m);
                if (lane >= m) incl += o;
            }
            const unsigned hit = __ballot_sync(kFullMask, bb < p.batch && base + incl > start);
            if (hit) {
                const int k = __ffs(hit) - 1;
                base += __shfl_sync(kFullMask, incl - v, k);
                b += k;
                break;
            }
            base += __shfl_sync(kFullMask, incl, 31);
            b += 32;
        }
        int64_t cur = start;
        bool first = true;
        while (cur < end) {
            const int np = seq_pages[b];
            const int kvh = (int)((cur - base) / np);
            const int j = (int)((cur - base) % np);
            const int64_t room = np - j;
            const int len = (int)((end - cur) < room ? (end - cur) : room);
            const int T = reachable_tokens(p.context_lens, b, p.max_blocks, BS);
            start_fetch(b, j, j + len);
            const bool whole = j == 0 && len == np;
            const bool last = cur + len >= end;
            if (whole) {
                run_segment(b, kvh, j, j + len, T, emit_final(b, kvh));
            } else {
                const size_t row0 = ((size_t)c * 2 + (first ? 0 : 1)) * R;
                run_segment(b, kvh, j, j + len, T, emit_rows(row0));
            }
            (void)last;
            cur += len;
            first = false;
            if (cur - base >= (int64_t)np * Hkv) {  // next sequence with pages
                base += (int64_t)np * Hkv;
                ++b;
                while (b < p.batch && seq_pages[b] == 0) ++b;
            }
        }
        return;
    }

    // ---- one CTA per (sequence, query chunk and kv head, partition) ----
    const int part = blockIdx.x, b = blockIdx.z;
    const int kvh = MULTI ? (int)blockIdx.y % Hkv : (int)blockIdx.y;
    const int pb = part * p.part_pages;
    // the table entries are fetched before the context length is known
    // (every index stays inside the table row); those past it are masked
    start_fetch(b, pb, min(pb + p.part_pages, p.max_blocks));
    const int T = reachable_tokens(p.context_lens, b, p.max_blocks, BS);
    const int npages = (T + BS - 1) / BS;
    const int pe = min(pb + p.part_pages, npages);
    if (pb >= pe && !p.cluster_reduce) {
        // Nothing of this sequence falls in the partition.  The single pass
        // writes the empty-context result; the combine kernel never reads
        // partitions past the context.  (Inside a cluster every CTA takes
        // part in the reduction, so an empty one carries on with no pages.)
        if (p.final_out) {
            for (int idx = tid; idx < R * D; idx += blockDim.x)
                store_out(p.out, row_off(b, kvh, idx / D) + idx % D, 0.f, p.out_dtype);
        }
        return;
    }
    __syncthreads();  // barrier initialisation visible to every warp

    if (p.final_out) {
        run_segment(b, kvh, pb, max(pb, pe), T, emit_final(b, kvh));
    } else if (p.cluster_reduce) {
        run_segment(b, kvh, pb, max(pb, pe), T, [&](int idx, float A, float M, float Ls) {
            cpart[idx] = A;
            if (idx % D == 0) {
                cpart[R * D + idx / D] = M;
                cpart[R * D + R + idx / D] = Ls;
            }
        });
    } else {
        // workspace rows [B][Hkv][P][Q * G]: this CTA's rows start at qi0 * G
        run_segment(b, kvh, pb, max(pb, pe), T,
                    emit_rows((((size_t)b * Hkv + kvh) * p.num_parts + part) *
                                  (MULTI ? p.unit_rows : G) + (size_t)qi0 * G));
    }

    if (p.cluster_reduce) {
        // Log-sum-exp over the cluster's partitions through distributed shared
        // memory: each CTA finalises a 1/P share of the outputs; for an
        // element, the (m, l, acc) of every rank are loaded at once.
        cluster_sync_release_acquire();  // every CTA's partial is in place
        const int P = p.num_parts;
        const uint32_t rank = (uint32_t)blockIdx.x;  // the cluster spans grid x
        const uint32_t cp = smem_u32(cpart);
        const int chunk = (R * D + P - 1) / P;
        const int i1 = min(((int)rank + 1) * chunk, R * D);
        // unrolled for the cluster's size class: up to 8 ranks (portable
        // clusters, the common case) or up to 16
        auto merge = [&](auto maxp) {
            constexpr int MAXP = decltype(maxp)::value;
            uint32_t rbase[MAXP];
#pragma unroll
            for (int q = 0; q < MAXP; ++q)
                rbase[q] = q < P ? map_cluster_rank(cp, (uint32_t)q) : cp;
            for (int idx = (int)rank * chunk + tid; idx < i1; idx += blockDim.x) {
                const int r = idx / D;
                float m[MAXP], l[MAXP], a[MAXP];
#pragma unroll
                for (int q = 0; q < MAXP; ++q) {
                    if (q < P) {
                        m[q] = ld_cluster_f32(rbase[q] + 4u * (R * D + r));
                        l[q] = ld_cluster_f32(rbase[q] + 4u * (R * D + R + r));
                        a[q] = ld_cluster_f32(rbase[q] + 4u * idx);
                    }
                }
                float M = NEG_INF;
#pragma unroll
                for (int q = 0; q < MAXP; ++q)
                    if (q < P) M = fmaxf(M, m[q]);
                float A = 0.f, Ls = 0.f;
#pragma unroll
                for (int q = 0; q < MAXP; ++q) {
                    if (q < P && m[q] != NEG_INF) {
                        const float f = fast_exp2(m[q] - M);
                        A = fmaf(f, a[q], A);
                        Ls = fmaf(f, l[q], Ls);
                    }
                }
                store_out(p.out, row_off(b, kvh, r) + idx % D, Ls > 0.f ? A / Ls : 0.f,
                          p.out_dtype);
            }
        };
        if (P <= kMaxClusterParts)
            merge(std::integral_constant<int, kMaxClusterParts>{});
        else
            merge(std::integral_constant<int, kMaxDecodeClusterParts>{});
        cluster_sync_relaxed();  // no CTA leaves while others still read its shared memory
    }
}

// Per-instantiation flags of the attributes set once per device.
template <int D, int BS, typename KV, bool MULTI>
struct AttnAttrs {
    static inline AttrFlags smem;
    static inline AttrFlags nonportable;
};

template <int D, int BS, typename KV, bool MULTI>
cudaError_t launch_attn_inst(const AttnLaunch& L, cudaStream_t stream) {
    auto kern = attn_kernel<D, BS, KV, MULTI>;
    using Attrs = AttnAttrs<D, BS, KV, MULTI>;
    cudaError_t e = raise_smem_limit_once(kern, Attrs::smem);
    if (e != cudaSuccess) return e;
    if (L.cluster > kMaxClusterParts) {
        e = allow_nonportable_clusters_once(kern, Attrs::nonportable);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = dim3(L.threads);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (L.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (L.cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)L.cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_k, L.tmap_v, L.p);
}

// Clusters of `cluster` CTAs of the one-token instantiation resident at once
// on the current device (0 if the query fails).
template <int D, int BS, typename KV>
int attn_max_clusters_inst(int cluster, int threads, uint32_t smem_bytes) {
    auto kern = attn_kernel<D, BS, KV, false>;
    using Attrs = AttnAttrs<D, BS, KV, false>;
    if (raise_smem_limit_once(kern, Attrs::smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (cluster > kMaxClusterParts &&
        allow_nonportable_clusters_once(kern, Attrs::nonportable) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster, 1, 1);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

template <int D>
int attn_max_clusters_for_d(int block_size, int kv_dtype, int cluster, int threads,
                            uint32_t smem_bytes) {
    const bool bf = kv_dtype == PA_BF16;
    if (block_size == 16)
        return bf ? attn_max_clusters_inst<D, 16, __nv_bfloat16>(cluster, threads, smem_bytes)
                  : attn_max_clusters_inst<D, 16, __half>(cluster, threads, smem_bytes);
    return bf ? attn_max_clusters_inst<D, 32, __nv_bfloat16>(cluster, threads, smem_bytes)
              : attn_max_clusters_inst<D, 32, __half>(cluster, threads, smem_bytes);
}

template <int D, bool MULTI>
cudaError_t launch_attn_for_d(const AttnLaunch& L, cudaStream_t stream) {
    const bool bf = L.kv_dtype == PA_BF16;
    if (L.block_size == 16)
        return bf ? launch_attn_inst<D, 16, __nv_bfloat16, MULTI>(L, stream)
                  : launch_attn_inst<D, 16, __half, MULTI>(L, stream);
    if (L.block_size == 32)
        return bf ? launch_attn_inst<D, 32, __nv_bfloat16, MULTI>(L, stream)
                  : launch_attn_inst<D, 32, __half, MULTI>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
