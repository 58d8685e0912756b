// Paged attention for many query rows per kv head on the Blackwell tensor
// cores (tcgen05): several query tokens per sequence, causal over the new
// tokens, where the rows of a (sequence, kv head) -- query token x head of
// the group -- fill 128-row tiles.
//
// What it computes is the multi-token decode step (each query token i of
// sequence b sits at position T - Q + i and attends to the cached tokens at
// and before it; "benchmark_decoding.py" reference_output for the attention
// itself, MiniVLLM docs "Decoding Benchmark" for the paged layout and the
// online softmax, flash-decoding-bench "design.md" for the split into
// partitions with a (max, sum, weighted values) partial each).
//
// One CTA per (sequence, 128-row tile and kv head, partition of pages), or a
// CTA taking a list of such segments in turn (persistent CTAs, the balanced
// split); pages are taken in KV blocks of BN tokens (128; 64 at head_dim 256):
//   - warps 0 and 3 stream the blocks, K and V in rings of their own: one
//     lane per page reads its block-table entry and issues a 4-D TMA copy per
//     64-column block of the page's tile (128-byte swizzle) into consecutive
//     rows of a stage, so that a block's pages form one BN-row operand; the V
//     warp also loads later segments' Q tiles through a Q tensor map;
//   - warp 1 (one lane) issues S = Q K^T for a block (M = 128 rows, N = BN
//     tokens, K = head_dim; Q and K from shared memory) into an S buffer in
//     tensor memory as soon as the buffer's previous P V is done; warp 2
//     (one lane, after allocating tensor memory) issues O += P V (M = 128,
//     N = head_dim, K = BN; P from tensor memory, V from shared memory,
//     MN-major) as soon as the block's P is in tensor memory;
//   - warps 4-11 (two warpgroups, one half of a block's columns each) own one
//     row per thread (a tensor-memory lane): they read the row's scores, mask
//     them (table reach and the row's causal limit), keep the running max m
//     and normaliser l in base-2 units, rescale O in tensor memory when the
//     max moves by more than 2^8, and write P over S (bf16: a high and a low
//     16-bit part, two MMAs, ~16 significant bits; fp16: one part, 11 bits),
//     zero the V rows that P weights with 0 (slots past the last token, pages
//     the table does not reach: 0 * NaN would reach O), and write the final
//     O / l or the partial (m, l, O) for the combine.  Whole tiles up to
//     head_dim 128 give each warpgroup an O accumulator of its own (its half
//     of the keys, whose V rows it zeroes itself; the two are merged once per
//     segment); otherwise the two share O and exchange row maxima every block.
// Units of at most 16 rows at head_dim 256 (one-token MQA) stage only those
// rows of Q (QR = 16): the 56 KB saved give each K / V ring a third stage,
// and the MMAs run at M = 64.
// Every mbarrier wait is bounded: on timeout the kernel records
// PA_ERR_TIMEOUT, the roles stop, and tensor memory is released.
#pragma once

#include <type_traits>

#include "pa_device.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr float kTileRescaleSlack = 8.0f;  // log2 units: P may reach 2^8 before a rescale

// QR: Q rows staged in shared memory (kTileRows, or kTileCompactQRows for
// units of at most 16 rows at head_dim 256, which buys a third ring stage).
//
// Work of a CTA: one segment -- (sequence, kv head, 128-row tile) and a range
// of its pages -- from the grid position; or, for the balanced split of
// compact units, the CTA's equal share [c W / C, (c + 1) W / C) of the
// flattened (sequence, kv head, page) order, W pages in all, walked as a list
// of segments (a whole unit is written out; a piece at either end of the
// share becomes a record [C][2][unit rows] for the balanced combine kernel).
// Every role walks the same segments and numbers the KV blocks of all of them
// in one sequence, so that the rings, the S / P buffers and their barrier
// phases run on across segment boundaries; Q is double-buffered (the V copy
// warp loads the Q of segment s >= 1 by TMA once the last S MMA of segment
// s - 2 has completed), and the first P V MMA of a segment waits until the
// previous segment's O has been read out.
template <int D, int BS, typename KV, int QR>
__global__ void __launch_bounds__(kTileThreads, 1)
    tile_kernel(const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_v,
                const __grid_constant__ CUtensorMap tmap_q, const AttnParams p) {
    constexpr int BN = tile_block_tokens(D);  // tokens per KV block
    constexpr int NPB = BN / BS;              // pages per KV block
    constexpr int NS = tile_stages(D, QR);
    static_assert(QR == kTileRows || (QR == kTileCompactQRows && D == 256), "staged Q rows");
    constexpr int DBLK = D / 64;
    constexpr int KSTEPS = D / 16;
    constexpr float NEG_INF = -INFINITY;
    constexpr bool kBF = std::is_same<KV, __nv_bfloat16>::value;
    // P enters the P V MMA as 16-bit values.  bf16 keeps 8 significant bits,
    // so P is split into a high and a low part (two MMAs, ~16 bits); fp16
    // keeps 11, a relative rounding of at most 2^-11 per weight, and is used
    // alone, with the normaliser summed from the rounded weights so that the
    // result stays a weighted mean of the V rows.
    constexpr bool kSplitP = kBF;
    constexpr bool kCanBalance = QR == kTileCompactQRows;  // the balanced split: compact units
    constexpr bool kTwoQ = tile_q_bufs(D, QR) == 2;         // several segments per CTA possible
    constexpr uint32_t kCols = tile_tmem_cols(D);
    // Whole tiles up to head_dim 128 give each softmax warpgroup an O of its
    // own: warpgroup h keeps the running max, the normaliser and O of its half
    // of every block's keys, so the two never wait on each other inside the
    // block loop; the halves are merged once, in the epilogue.  Otherwise the
    // warpgroups share one O and exchange their row maxima every block.
    constexpr bool kHalfO = QR == kTileRows && D <= 128;
    constexpr int NB = kHalfO ? (512 - 2 * D) / BN : kTileSBufs;  // S / P buffers
    // O (h) at O_COL + h * D; S buffer b at S_COL + b*BN; P (hi, lo) over it
    constexpr uint32_t O_COL = 0, S_COL = kHalfO ? 2 * D : D;
    static_assert(NB >= 2 && NB <= kTileSBufs, "S / P buffers");
    static_assert(S_COL + NB * BN <= 512, "tensor memory");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + (kSmemAlignSlack - 1)) &
        ~uintptr_t(kSmemAlignSlack - 1));
    const TileSmem L = tile_smem_layout(D, BS, QR);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
    uint64_t* k_full = bars;
    uint64_t* k_empty = bars + NS;
    uint64_t* v_full = bars + 2 * NS;
    uint64_t* v_empty = bars + 3 * NS;
    uint64_t* s_full = bars + 4 * NS;
    uint64_t* p_full = s_full + kTileSBufs;  // [2][3]: per softmax warpgroup with kHalfO
    uint64_t* pv_done = p_full + 2 * kTileSBufs;
    uint64_t* final_bar = pv_done + kTileSBufs;
    uint64_t* q_ready = final_bar + 1;  // the first segment's Q tile is in shared memory
    uint64_t* q_full = q_ready + 1;     // [2] Q buffer b holds a later segment's Q
    uint64_t* q_free = q_full + 2;      // [2] the S MMAs of buffer b's segment have completed
    uint64_t* o_free = q_free + 2;      // a segment's O has been read out
    int32_t* phys_of = reinterpret_cast<int32_t*>(smem + L.phys_off);  // [NS][NPB] of K stages
    int32_t* v_live = phys_of + NS * NPB;  // [NS]: V stage's block holds a page
    float* xmax = reinterpret_cast<float*>(smem + L.xchg_off);    // [2][2][128]
    float* xl = xmax + 2 * 2 * 128;                                   // [2][128]
    uint64_t* xchg = reinterpret_cast<uint64_t*>(xl + 2 * 128);     // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    int32_t* seq_pages = reinterpret_cast<int32_t*>(smem + L.seq_off);  // balanced: [B] pages
    long long* walk0 = reinterpret_cast<long long*>(smem + L.walk_off);  // share start, end, base, b

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.group, Q = p.q_len, Hkv = p.num_kv_heads, U = p.unit_rows;
    const int gshift = __ffs(G) - 1;
    const bool bal = kCanBalance && p.balanced;
    const bool pers = kTwoQ && !bal && p.persistent;
    const bool multi = bal || pers;  // the CTA may take several segments
    const int part = blockIdx.x;
    const int tiles = (U + kTileRows - 1) / kTileRows;  // 128-row tiles of a unit

    grid_dependency_wait();
    grid_launch_dependents();

    // Element offset of unit row u's query / output vector ([B, Q, H, D]).
    auto row_off = [&](int b, int kvh, int u) -> size_t {
        return (((size_t)b * Q + (u >> gshift)) * p.num_heads + kvh * G + (u & (G - 1))) * D;
    };

    // ---- the CTA's segments ----
    struct Seg {
        int b, kvh, tile, pb, pe, T, np;  // pages [pb, pe) of the np of (b, kvh); T tokens
                                          // reach the table; rows of `tile`
        bool whole;                       // the segment is the whole unit
    };
    struct Walk {
        long long cur, end, base;  // balanced: flat position, end of the share, flat start of b
        int b;
        long long x;               // persistent: the next unit index
    };
    if (bal) {
        // pages of every sequence, their total W (times the kv heads), and the
        // sequence holding the first page of this CTA's share
        if (warp == 0) {
            long long w = 0;
            for (int b0 = lane; b0 < p.batch; b0 += 32) {
                const int T = reachable_tokens(p.context_lens, b0, p.max_blocks, BS);
                const int np = (T + BS - 1) / BS;
                seq_pages[b0] = np;
                w += np;
            }
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) w += __shfl_xor_sync(kFullMask, w, m);
            const long long W = w * Hkv, Cn = gridDim.x, c = blockIdx.x;
            const long long start = c * W / Cn, end = (c + 1) * W / Cn;
            __syncwarp();
            // scan the sequences 32 at a time for the one that holds `start`
            int b = 0;
            long long base = 0;
            if (start < end) {
                for (;;) {
                    const int bb = b + lane;
                    const long long v = bb < p.batch ? (long long)seq_pages[bb] * Hkv : 0;
                    long long incl = v;
#pragma unroll
                    for (int m = 1; m < 32; m <<= 1) {
                        const long long o = __shfl_up_sync(kFullMask, incl, m);
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
            }
            if (lane == 0) {
                walk0[0] = start;
                walk0[1] = end;
                walk0[2] = base;
                walk0[3] = b;
            }
        }
        __syncthreads();
        if (walk0[0] >= walk0[1]) return;  // an empty share (fewer pages than CTAs)
    }
    auto walk_init = [&](Walk& w) {
        if (pers) {
            w.x = blockIdx.x;
            return;
        }
        w.cur = walk0[0];
        w.end = walk0[1];
        w.base = walk0[2];
        w.b = (int)walk0[3];
    };
    // unit x of the persistent order: tiles of a (sequence, kv head) in turn,
    // so that the CTAs working at once share each page through L2
    auto unit_of = [&](long long x, Seg& g) {
        g.tile = (int)(x % tiles);
        const long long bk = x / tiles;
        g.kvh = (int)(bk % Hkv);
        g.b = (int)(bk / Hkv);
        g.T = reachable_tokens(p.context_lens, g.b, p.max_blocks, BS);
        g.np = (g.T + BS - 1) / BS;
        g.pb = 0;
        g.pe = g.np;
        g.whole = true;
    };
    const long long nunits = (long long)p.batch * Hkv * tiles;
    auto walk_next = [&](Walk& w, Seg& g) -> bool {
        if (pers) {  // the CTA's units with pages (empty ones are written out apart)
            while (w.x < nunits) {
                unit_of(w.x, g);
                w.x += gridDim.x;
                if (g.np > 0) return true;
            }
            return false;
        }
        if (w.cur >= w.end) return false;
        const int np = seq_pages[w.b];
        const long long off = w.cur - w.base;
        const int j = (int)(off % np);
        const int len = (int)min(w.end - w.cur, (long long)(np - j));
        g.b = w.b;
        g.kvh = (int)(off / np);
        g.tile = 0;
        g.pb = j;
        g.pe = j + len;
        g.np = np;
        g.whole = j == 0 && len == np;
        g.T = reachable_tokens(p.context_lens, w.b, p.max_blocks, BS);
        w.cur += len;
        if (w.cur - w.base >= (long long)np * Hkv) {  // past this sequence's pages
            w.base += (long long)np * Hkv;
            ++w.b;
            while (w.b < p.batch && seq_pages[w.b] == 0) ++w.b;
        }
        return true;
    };
    // the segment of a grid-position CTA
    Seg seg0;
    if (!multi) {
        seg0.b = blockIdx.z;
        seg0.kvh = (int)blockIdx.y % Hkv;
        seg0.tile = (int)blockIdx.y / Hkv;
        seg0.T = reachable_tokens(p.context_lens, seg0.b, p.max_blocks, BS);
        seg0.np = (seg0.T + BS - 1) / BS;
        seg0.pb = part * p.part_pages;
        seg0.pe = min(seg0.pb + p.part_pages, seg0.np);
        seg0.whole = false;
    }
    // calls fn(segment, index) for each of the CTA's segments until fn returns false
    auto for_segments = [&](auto&& fn) {
        if (!multi) {
            (void)fn(seg0, 0);
            return;
        }
        Walk w;
        walk_init(w);
        Seg g;
        for (int s = 0; walk_next(w, g); ++s)
            if (!fn(g, s)) return;
    };
    auto nblk_of = [&](const Seg& g) { return (g.pe - g.pb + NPB - 1) / NPB; };

    // ---- cluster reduction (at most 8 partitions of a unit form one cluster
    // along grid x): every CTA has left its partial at offset 0 of its shared
    // memory; CTA `rank` merges rows [rank*rpc, (rank+1)*rpc) of all of them
    // through distributed shared memory and writes the output ----
    constexpr int CL = D + 4;  // row stride of the parked O rows (floats)
    float* cl_o = reinterpret_cast<float*>(smem);
    float* cl_m = cl_o + kTileRows * CL;
    float* cl_l = cl_m + kTileRows;
    float* cl_w = cl_l + kTileRows;  // [rpc][8] merge weights of this CTA's rows
    auto cluster_merge = [&]() {
        cluster_sync_release_acquire();  // every CTA's partial is in place
        const int P = p.num_parts;
        const int rank = (int)blockIdx.x;
        // the tile's rows that hold unit rows, shared out among the cluster
        const int nr = min(U - seg0.tile * kTileRows, kTileRows);
        const int rpc = (nr + P - 1) / P;
        const int r0 = min(rank * rpc, nr), r1 = min(r0 + rpc, nr);
        uint32_t rb_m[kMaxClusterParts], rb_l[kMaxClusterParts], rb_o[kMaxClusterParts];
#pragma unroll
        for (int q = 0; q < kMaxClusterParts; ++q) {
            const uint32_t qq = (uint32_t)(q < P ? q : 0);
            rb_m[q] = map_cluster_rank(smem_u32(cl_m), qq);
            rb_l[q] = map_cluster_rank(smem_u32(cl_l), qq);
            rb_o[q] = map_cluster_rank(smem_u32(cl_o), qq);
        }
        for (int t = tid; t < r1 - r0; t += kTileThreads) {
            const int r = r0 + t;
            float mq[kMaxClusterParts];
            float M = NEG_INF;
#pragma unroll
            for (int q = 0; q < kMaxClusterParts; ++q) {
                mq[q] = q < P ? ld_cluster_f32(rb_m[q] + 4u * r) : NEG_INF;
                M = fmaxf(M, mq[q]);
            }
            float w[kMaxClusterParts], Ls = 0.f;
#pragma unroll
            for (int q = 0; q < kMaxClusterParts; ++q) {
                w[q] = mq[q] == NEG_INF ? 0.f : fast_exp2(mq[q] - M);
                if (w[q] != 0.f) Ls = fmaf(w[q], ld_cluster_f32(rb_l[q] + 4u * r), Ls);
            }
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
            for (int q = 0; q < kMaxClusterParts; ++q) cl_w[t * 8 + q] = w[q] * inv;
        }
        __syncthreads();
        for (int idx = tid; idx < (r1 - r0) * (D / 4); idx += kTileThreads) {
            const int t = idx / (D / 4), c4 = idx % (D / 4);
            const int r = r0 + t, u = seg0.tile * kTileRows + r;
            if (u >= U) continue;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kMaxClusterParts; ++q) {
                const float w = cl_w[t * 8 + q];
                if (w == 0.f) continue;  // an empty partial: nothing parked there
                const float4 v = ld_cluster_v4f32(rb_o[q] + 4u * (r * CL + 4 * c4));
                a.x = fmaf(w, v.x, a.x);
                a.y = fmaf(w, v.y, a.y);
                a.z = fmaf(w, v.z, a.z);
                a.w = fmaf(w, v.w, a.w);
            }
            const size_t o = row_off(seg0.b, seg0.kvh, u) + 4 * c4;
            if (p.out_dtype == PA_F32) {
                *reinterpret_cast<float4*>(static_cast<float*>(p.out) + o) = a;
            } else {
                *reinterpret_cast<uint2*>(static_cast<KV*>(p.out) + o) =
                    make_uint2(Mma<KV>::pack(a.x, a.y), Mma<KV>::pack(a.z, a.w));
            }
        }
        cluster_sync_relaxed();  // no CTA leaves while others still read its partial
    };

    if (!multi && seg0.pe <= seg0.pb) {
        if (p.cluster_reduce) {
            // no pages here, but the cluster's merge needs this CTA: an empty partial
            for (int r = tid; r < kTileRows; r += kTileThreads) {
                cl_m[r] = NEG_INF;
                cl_l[r] = 0.f;
            }
            cluster_merge();
            return;
        }
        // Nothing of this sequence in the partition: the single pass writes the
        // empty-context result; the combine never reads such partitions.
        if (p.final_out) {
            for (int idx = tid; idx < kTileRows * D; idx += kTileThreads) {
                const int u = seg0.tile * kTileRows + idx / D;
                if (u < U) store_out(p.out, row_off(seg0.b, seg0.kvh, u) + idx % D, 0.f, p.out_dtype);
            }
        }
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(k_full + i), 1);
            mbar_init(smem_u32(k_empty + i), 1);
            mbar_init(smem_u32(v_full + i), 1);
            mbar_init(smem_u32(v_empty + i), 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(smem_u32(s_full + i), 1);
            mbar_init(smem_u32(p_full + i), kHalfO ? 128 : 256);
            mbar_init(smem_u32(p_full + kTileSBufs + i), 128);
            mbar_init(smem_u32(pv_done + i), 1);
        }
        mbar_init(smem_u32(final_bar), 2);  // the S and the P V issuer
        mbar_init(smem_u32(q_ready), kTileThreads - 64);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(q_full + i), 1);
            mbar_init(smem_u32(q_free + i), 1);
        }
        mbar_init(smem_u32(o_free), 8);
        mbar_init(smem_u32(xchg), 256);
        mbar_init(smem_u32(xchg + 1), 256);
        *abort_flag = 0;
        mbar_init_fence();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
        if (multi) prefetch_tensormap(&tmap_q);
    }
    if (warp == 2) {  // tensor memory for O and the S / P buffers
        tc::tmem_alloc(smem_u32(tmem_slot), kCols);
        tc::tmem_relinquish();
    }

    tc::fence_before_sync();
    __syncthreads();  // barriers initialised, tensor memory allocated
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // ---- Q tile of a segment into Q buffer `qb`: rows u = tile*128 + r for
    // r < QR, zero rows past the unit's rows; written with the 128-byte
    // swizzle the MMA descriptors expect, threads `t0, t0 + step, ...`.  With a
    // compact Q tile the S MMA's rows past QR read whatever follows it: those
    // rows lie past the unit's rows, their scores are masked or never read,
    // and their P and O rows are never used ----
    auto stage_q = [&](const Seg& g, int qb, int t0, int step) {
        uint8_t* qs = smem + L.q_off + (size_t)qb * (2u * QR * D);
#pragma unroll 4
        for (int i = t0; i < QR * (D / 8); i += step) {
            const int r = i / (D / 8), c = i % (D / 8);
            const int u = g.tile * kTileRows + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (u < U)
                v = __ldg(reinterpret_cast<const uint4*>(static_cast<const KV*>(p.q) +
                                                         row_off(g.b, g.kvh, u)) + c);
            *reinterpret_cast<uint4*>(qs + (c >> 3) * (QR * 128) + r * 128 +
                                      (((c & 7) ^ (r & 7)) << 4)) = v;
        }
    };
    // the first segment's Q: every thread outside the two copy warps (which
    // already stream K and V); the MMA issuer waits for q_ready
    if (warp != 0 && warp != 3) {
        const int qt = (warp < 3 ? (warp - 1) * 32 : 64 + (warp - 4) * 32) + lane;  // 0..319
        for_segments([&](const Seg& g, int s) {
            stage_q(g, 0, qt, kTileThreads - 64);
            return false;  // the first segment only
        });
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(q_ready));
    }

    auto fail = [&]() {
        if (lane == 0) record_error(p.err, PA_ERR_TIMEOUT);
        *abort_flag = 1;
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const bool ok = mbar_wait_bounded(smem_u32(bar), parity, p.timeout_ns);
        if (!ok) fail();
        return ok;
    };
    // does KV block k (in stage st) hold at least one page?
    auto block_live = [&](int st) -> bool {
        bool any = false;
#pragma unroll
        for (int q = 0; q < NPB; ++q) any |= phys_of[st * NPB + q] >= 0;
        return any;
    };

    if (warp == 0 || warp == 3) {
        // ============ producers: warp 0 the K ring, warp 3 the V ring ============
        // lane q < NPB reads the table entry of page q of a block and copies it
        const bool is_k = warp == 0;
        uint64_t* full = is_k ? k_full : v_full;
        uint64_t* empty = is_k ? k_empty : v_empty;
        const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
        const uint32_t ring = smem_u32(smem + (is_k ? L.k_off : L.v_off));
        // a unit of several tiles has each page read by all of them, by CTAs
        // working on it at the same time: keep the pages in L2 at the default
        // priority then (prefill chunk 181.4 -> 178.8 us), else evict them first
        const uint64_t policy = tiles > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
        int issued = 0;  // blocks issued, over all segments (the ring's position)
        int q_last = 0;  // V warp: the last segment whose Q copy was issued (0: none)
        for_segments([&](const Seg& g, int s) {
            if (!is_k && multi && s >= 1) {
                // Q of segment s into buffer s & 1 once the S MMAs of segment
                // s - 2 (the buffer's previous user) are done.  The box is the
                // tile's rows (G heads x QR / G query tokens, or QR heads of one
                // token when the group is larger), 64 columns at a time, in the
                // 128-byte swizzle the S MMA reads; rows past the unit's rows
                // hold the next tokens' queries or the fill value, and are
                // masked like the zero rows of a staged tile
                bool qok = true;
                if (lane == 0) {
                    const int qb = s & 1;
                    if (s >= 2) qok = wait(q_free + qb, ((s - 2) >> 1) & 1);
                    if (qok) {
                        const int r0 = g.tile * kTileRows;  // the tile's first row
                        const int hc = G >= QR ? g.kvh * G + (r0 & (G - 1)) : g.kvh * G;
                        const int qc = g.b * Q + (r0 >> gshift);
                        const uint32_t qbar = smem_u32(q_full + qb);
                        const uint32_t qdst = smem_u32(smem + L.q_off) + (uint32_t)qb * (2u * QR * D);
                        mbar_arrive_expect_tx(qbar, 2u * QR * D);
#pragma unroll
                        for (int blk = 0; blk < DBLK; ++blk)
                            tma_load_3d(qdst + blk * (QR * 128), &tmap_q, blk * 64, hc, qc, qbar);
                        q_last = s;
                    }
                }
                if (!__shfl_sync(kFullMask, qok ? 1 : 0, 0)) return false;
            }
            const int32_t* table_row = p.block_tables + (size_t)g.b * p.max_blocks;
            const int nblk = nblk_of(g);
            // the segment's table entries, 32 pages at a time (one per lane),
            // fetched one window ahead so that no block waits for its entries
            auto fetch = [&](int w) -> int {
                const int jj = g.pb + w * 32 + lane;
                return jj < g.pe ? __ldg(table_row + jj) : -1;
            };
            int ent_cur = fetch(0), ent_next = fetch(1), win = 0;
            for (int k = 0; k < nblk && !*abort_flag; ++k) {
                const int st = issued % NS, round = issued / NS;
                const int first = k * NPB;  // page index of the block within the segment
                if ((first >> 5) != win) {  // NPB divides 32: a block never straddles windows
                    win = first >> 5;
                    ent_cur = ent_next;
                    ent_next = fetch(win + 1);
                }
                const int e0 = __shfl_sync(kFullMask, ent_cur, (first & 31) + (lane < NPB ? lane : 0));
                const int e = lane < NPB ? e0 : -1;
                const int phys = (e >= 0 && (int64_t)e < p.num_blocks) ? e : -1;
                bool ok = true;
                if (round > 0 && lane == 0) ok = wait(empty + st, (round - 1) & 1);
                if (!__shfl_sync(kFullMask, ok ? 1 : 0, 0)) return false;
                if (is_k && lane < NPB) phys_of[st * NPB + lane] = phys;
                const unsigned live = __ballot_sync(kFullMask, lane < NPB && phys >= 0);
                if (!is_k && lane == 0) v_live[st] = live != 0u;
                const uint32_t bar = smem_u32(full + st);
                if (lane == 0) {
                    if (live) mbar_arrive_expect_tx(bar, (uint32_t)__popc(live) * 2u * BS * D);
                    else mbar_arrive(bar);
                }
                __syncwarp();
                if (lane < NPB && phys >= 0) {
                    const uint32_t dst = ring + (uint32_t)st * L.tile_bytes + (uint32_t)lane * BS * 128;
#pragma unroll
                    for (int blk = 0; blk < DBLK; ++blk)
                        tma_load_4d(dst + blk * BN * 128, map, blk * 64, g.kvh, 0, phys, bar, policy);
                }
                ++issued;
            }
            return !*abort_flag;
        });
        if (*abort_flag && lane == 0) {
            // let copies still in flight land before the CTA may exit (no one
            // else arrives on q_full, so its phase stays complete once it is)
            for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
                (void)mbar_wait_bounded(smem_u32(full + k % NS), (k / NS) & 1, p.timeout_ns);
            if (q_last > 0)
                (void)mbar_wait_bounded(smem_u32(q_full + (q_last & 1)), ((q_last - 1) >> 1) & 1,
                                        p.timeout_ns);
        }
    } else if (warp == 2) {
        // ======= P V issuer (one lane): O += P_j V_j as soon as block j's P
        // is in tensor memory, apart from the S issuer so that neither waits
        // behind the other's MMAs being accepted =======
        if (lane == 0) {
            constexpr int kType = kBF ? 1 : 0;
            // (compact Q tiles: M = 64, rows 0..15 in lanes 0..15 as at M = 128)
            constexpr int kM = QR == kTileCompactQRows ? 64 : kTileRows;
            constexpr uint32_t id_o = tc::idesc_f16(kType, true, kM, D);
            int j = 0;  // blocks over all segments
            bool ok = true;
            for_segments([&](const Seg& g, int s) {
                bool started = false;  // O holds this segment's sum
                if (s >= 1) {
                    // the previous segment's O must have been read out
                    if (!wait(o_free, (s - 1) & 1)) return ok = false;
                    tc::fence_after_sync();
                }
                const int nblk = nblk_of(g);
                for (int k = 0; k < nblk && !*abort_flag; ++k, ++j) {
                    const int st = j % NS;
                    if (!wait(v_full + st, (j / NS) & 1)) return ok = false;
                    const bool live = v_live[st] != 0;  // the block holds a page
                    const uint32_t v_base = smem_u32(smem + L.v_off) + (uint32_t)st * L.tile_bytes;
                    // V: MN-major, 64-column blocks BN*128 bytes apart, 8-row
                    // groups 1024 bytes apart; rows ks*16 .. +15 per step
                    const uint64_t vd0 = tc::smem_desc(v_base, BN * 128, 1024, tc::kSwizzle128B);
                    if constexpr (kHalfO) {
                        // each warpgroup's half of the keys into its own O, as soon as
                        // that half's P is in tensor memory
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (!wait(p_full + h * kTileSBufs + j % NB, (j / NB) & 1)) return ok = false;
                            tc::fence_after_sync();
                            if (live) {
                                // half h's P: hi at columns h*BN/2 .., lo BN/4 after it
                                const uint32_t ph = tmem + S_COL + (j % NB) * BN + h * (BN / 2);
#pragma unroll
                                for (int kk = 0; kk < BN / 32; ++kk) {
                                    const int ks = h * (BN / 32) + kk;  // token rows of V
                                    const uint64_t vd = vd0 + (uint64_t)((ks * 16 * 128) >> 4);
                                    tc::mma_ts(tmem + O_COL + h * D, ph + kk * 8, vd, id_o,
                                               (started || kk > 0) ? 1u : 0u);
                                    if (kSplitP)
                                        tc::mma_ts(tmem + O_COL + h * D, ph + BN / 4 + kk * 8, vd, id_o, 1u);
                                }
                            }
                        }
                        if (live) started = true;
                    } else {
                        if (!wait(p_full + j % NB, (j / NB) & 1)) return ok = false;
                        tc::fence_after_sync();
                        if (live) {
                            // P of all BN keys: hi at columns 0 .., lo BN/2 after it
                            const uint32_t p_hi = tmem + S_COL + (j % NB) * BN;
                            const uint32_t p_lo = p_hi + BN / 2;
#pragma unroll
                            for (int ks = 0; ks < BN / 16; ++ks) {
                                const uint64_t vd = vd0 + (uint64_t)((ks * 16 * 128) >> 4);
                                tc::mma_ts(tmem + O_COL, p_hi + ks * 8, vd, id_o,
                                           (started || ks > 0) ? 1u : 0u);
                                if (kSplitP) tc::mma_ts(tmem + O_COL, p_lo + ks * 8, vd, id_o, 1u);
                            }
                            started = true;
                        }
                    }
                    tc::commit(smem_u32(pv_done + j % NB));
                    tc::commit(smem_u32(v_empty + st));
                }
                return ok && !*abort_flag;
            });
            // every MMA issued has completed before tensor memory is released
            tc::commit(smem_u32(final_bar));
            (void)mbar_wait_bounded(smem_u32(final_bar), 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= S issuer (one lane) =================
        if (lane == 0) {
            constexpr int kType = kBF ? 1 : 0;
            // a compact Q tile (at most 16 live rows) runs the MMAs at M = 64:
            // rows 0..15 of an M = 64 result (and of an M = 64 operand in
            // tensor memory) sit in lanes 0..15, as they do at M = 128 (on
            // GB300 the tensor pipe takes as long for M = 64 as for 128: the
            // MMAs of a block cost the same either way)
            constexpr int kM = QR == kTileCompactQRows ? 64 : kTileRows;
            constexpr uint32_t id_s = tc::idesc_f16(kType, false, kM, BN);
            int i = 0;  // blocks over all segments
            bool ok = true;
            for_segments([&](const Seg& g, int s) {
                // this segment's Q: buffer s & 1
                if (s == 0) ok = wait(q_ready, 0);
                else ok = wait(q_full + (s & 1), ((s - 1) >> 1) & 1);
                if (!ok) return false;
                const uint32_t q_base = smem_u32(smem + L.q_off) + (uint32_t)(s & 1) * (2u * QR * D);
                // Operand descriptors: a shared-memory descriptor holds (address >> 4)
                // in its low 14 bits, and every address here is below 2^18, so the
                // descriptor of base + offset is base's plus offset >> 4.  Q's are
                // fixed for the segment; K's are one add from their stage's.
                uint64_t qd[KSTEPS];
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks)
                    qd[ks] = tc::smem_desc(q_base + (ks >> 2) * (QR * 128) + (ks & 3) * 32, 16, 1024,
                                           tc::kSwizzle128B);
                const int nblk = nblk_of(g);
                for (int k = 0; k < nblk && !*abort_flag; ++k, ++i) {
                    // S_i = Q K_i^T into buffer i % NB, once P_{i-NB} there has been consumed
                    const int st = i % NS;
                    if (!wait(k_full + st, (i / NS) & 1)) return ok = false;
                    if (i >= NB && !wait(pv_done + i % NB, ((i - NB) / NB) & 1)) return ok = false;
                    tc::fence_after_sync();
                    if (block_live(st)) {
                        const uint32_t k_base = smem_u32(smem + L.k_off) + (uint32_t)st * L.tile_bytes;
                        const uint64_t kd = tc::smem_desc(k_base, 16, 1024, tc::kSwizzle128B);
#pragma unroll
                        for (int ks = 0; ks < KSTEPS; ++ks)
                            tc::mma_ss(tmem + S_COL + (i % NB) * BN, qd[ks],
                                       kd + (uint64_t)(((ks >> 2) * (BN * 128) + (ks & 3) * 32) >> 4),
                                       id_s, ks > 0);
                    }
                    tc::commit(smem_u32(s_full + i % NB));
                    tc::commit(smem_u32(k_empty + st));
                    // the segment's last S: its Q buffer is free once these complete
                    if (multi && k == nblk - 1) tc::commit(smem_u32(q_free + (s & 1)));
                }
                return ok && !*abort_flag;
            });
            // every MMA issued has completed before tensor memory is released
            tc::commit(smem_u32(final_bar));
            (void)mbar_wait_bounded(smem_u32(final_bar), 0, p.timeout_ns);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ============ softmax: two warpgroups, one row per thread each ============
        // warpgroup wg takes columns [wg*BH, (wg+1)*BH) of every block and
        // output columns [wg*D/2, (wg+1)*D/2); with a shared O the two exchange
        // row maxima every block, with an O each (kHalfO) only at the end of a
        // segment, with their normalisers, through shared memory
        constexpr int BH = BN / 2;
        const int wg = (warp - 4) >> 2, w4 = warp & 3;
        const int r = w4 * 32 + lane;
        const int sr = wg * 128 + r;  // 0 .. 255 among the softmax threads
        const uint32_t lane_base = tmem + ((uint32_t)(w4 * 32) << 16);
        const float qscale = p.qscale;
        // exchange round nx: publish v, return the other warpgroup's value
        int nx = 0;
        auto exchange = [&](float* buf, float v, float& other) -> bool {
            buf[wg * 128 + r] = v;
            mbar_arrive(smem_u32(xchg + (nx & 1)));
            const bool ok = __all_sync(kFullMask, wait(xchg + (nx & 1), (nx >> 1) & 1));
            other = buf[(1 - wg) * 128 + r];
            ++nx;
            return ok;
        };
        if (pers) {
            // the CTA's units without a page: an all-zero output
            for (long long x = blockIdx.x; x < nunits; x += gridDim.x) {
                Seg g;
                unit_of(x, g);
                if (g.np > 0) continue;
                for (int idx = sr; idx < kTileRows * D; idx += 256) {
                    const int uu = g.tile * kTileRows + idx / D;
                    if (uu < U) store_out(p.out, row_off(g.b, g.kvh, uu) + idx % D, 0.f, p.out_dtype);
                }
            }
        }
        int j = 0;  // blocks over all segments
        for_segments([&](const Seg& g, int s) {
            const int u = g.tile * kTileRows + r;
            // a warp whose 32 rows all lie past the unit's rows (a partial tile)
            // only keeps the barriers going: its P and O rows are never used
            const bool dead = g.tile * kTileRows + w4 * 32 >= U;
            const int nblk = nblk_of(g);
            const int jb = j;  // the segment's first block
            const int tend = min(g.T, g.pe * BS);  // tokens of this segment end here
            const int ctx = max(__ldg(p.context_lens + g.b), 0);
            // tokens t < lim: the row's causal limit, the table's reach, the segment's end
            const int lim = u < U ? min(tend, ctx - Q + (u >> gshift) + 1) : 0;
            const int32_t* table_row = p.block_tables + (size_t)g.b * p.max_blocks;
            // which pages of the segment's block k hold data: bit q for page q
            // (read from the table here; the K stage's record may already
            // describe a later block)
            auto page_bits = [&](int k) -> unsigned {
                const int jj = g.pb + k * NPB + lane;
                const int e = (lane < NPB && jj < g.pe && k < nblk) ? __ldg(table_row + jj) : -1;
                return __ballot_sync(kFullMask, e >= 0 && (int64_t)e < p.num_blocks);
            };
            float m = NEG_INF, l = 0.f;  // l: this half's share of the normaliser
            unsigned bits_next = page_bits(0);
            int k = 0;
            for (; k < nblk && !*abort_flag; ++k, ++j) {
                const int st = j % NS;
                const unsigned bits = bits_next;
                bits_next = page_bits(k + 1);
                // (waits are decided warp-wide: the tensor-memory accesses below
                // are warp-collective)
                if (!__all_sync(kFullMask, wait(s_full + j % NB, (j / NB) & 1))) break;
                tc::fence_after_sync();
                if (bits) {
                    const int t0 = (g.pb + k * NPB) * BS + wg * BH;  // first token of this half
                    const uint32_t sb = lane_base + S_COL + (j % NB) * BN;
                    float sc[BH];
                    float mx = NEG_INF;
                    if (!dead) {
                        uint32_t x[32];
#pragma unroll
                        for (int c0 = 0; c0 < BH; c0 += 32) {
                            tc::ld_32x32b_x32(sb + wg * BH + c0, x);
                            tc::wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c) sc[c0 + c] = __uint_as_float(x[c]);
                        }
                        // masked unless every page is live and the whole half lies
                        // inside every row's limit; then the row maximum, three at a time
                        if (!__all_sync(kFullMask, bits == (1u << NPB) - 1u && t0 + BH <= lim)) {
#pragma unroll
                            for (int c = 0; c < BH; ++c) {
                                const bool pl = (bits >> ((wg * BH + c) / BS)) & 1u;
                                sc[c] = (pl && t0 + c < lim) ? sc[c] : NEG_INF;
                            }
                        }
#pragma unroll
                        for (int c = 0; c < BH; c += 2) mx = fmax3(mx, sc[c], sc[c + 1]);
                    }
                    float ms;
                    if constexpr (kHalfO) {
                        ms = mx * qscale;  // this warpgroup's half of the keys alone
                    } else {
                        float mo;
                        if (!exchange(xmax + (nx & 1) * 256, mx, mo)) break;
                        ms = fmaxf(mx, mo) * qscale;
                    }
                    const bool need = ms > m + kTileRescaleSlack;
                    float alpha = 1.f;
                    if (need) {
                        alpha = (m == NEG_INF) ? 1.f : fast_exp2(m - ms);
                        l *= alpha;
                        m = ms;
                    }
                    // O holds earlier blocks' sums only if this row had attended a token;
                    // each warpgroup rescales its own O (kHalfO) or its half of the
                    // shared O's columns
                    if (__any_sync(kFullMask, need && alpha != 1.f)) {
                        if (j > jb && !__all_sync(kFullMask, wait(pv_done + (j - 1) % NB,
                                                                   ((j - 1) / NB) & 1)))
                            break;
                        tc::fence_after_sync();
                        constexpr int kRC = kHalfO ? D : D / 2;  // columns rescaled
                        const uint32_t ob = lane_base + O_COL + (kHalfO ? wg * D : wg * (D / 2));
                        uint32_t x[16];
#pragma unroll 1
                        for (int c0 = 0; c0 < kRC; c0 += 16) {
                            tc::ld_32x32b_x16(ob + c0, x);
                            tc::wait_ld();
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                x[c] = __float_as_uint(__uint_as_float(x[c]) * alpha);
                            tc::st_32x32b_x16(ob + c0, x);
                        }
                        tc::wait_st();
                    }
                    // P = 2^(s*scale*log2e - m) over S, as 16-bit values: for bf16 a
                    // high and a low part, hi in columns [0, BN/2) and lo in [BN/2, BN)
                    // of the buffer; for fp16 the high part alone
                    const float me = (m == NEG_INF) ? 0.f : m;
                    if (!dead) {
#pragma unroll
                        for (int c0 = 0; c0 < BH; c0 += 16) {
                            uint32_t ph[8], pl[8];
#pragma unroll
                            for (int c = 0; c < 16; c += 2) {
                                const float x0 = fast_exp2(fmaf(sc[c0 + c], qscale, -me));
                                const float x1 = fast_exp2(fmaf(sc[c0 + c + 1], qscale, -me));
                                const uint32_t h = Mma<KV>::pack(x0, x1);
                                ph[c / 2] = h;
                                if constexpr (kSplitP) {
                                    float h0, h1;
                                    Mma<KV>::unpack(h, h0, h1);
                                    l += x0 + x1;
                                    pl[c / 2] = Mma<KV>::pack(x0 - h0, x1 - h1);
                                } else {
                                    l = Mma<KV>::add2(h, l);  // the weights the MMA uses
                                }
                            }
                            // kHalfO: the warpgroup's P inside its own S columns
                            // (hi then lo), which it alone reads; otherwise hi in
                            // [0, BN/2) and lo in [BN/2, BN) of the buffer (the
                            // per-block exchange has seen both halves' S loaded)
                            const uint32_t col_hi = kHalfO ? (uint32_t)(wg * BH + c0 / 2)
                                                           : (uint32_t)(wg * BH + c0) / 2;
                            const uint32_t col_lo = kHalfO ? col_hi + BH / 2 : col_hi + BN / 2;
                            tc::st_32x32b_x8(sb + col_hi, ph);
                            if (kSplitP) tc::st_32x32b_x8(sb + col_lo, pl);
                        }
                    }
                    tc::wait_st();
                    // zero the V rows of masked pages and past the segment's last
                    // token (0 * NaN would otherwise reach O), once the stage's
                    // copies have landed.  With an O per warpgroup, half h's P V
                    // MMAs wait for warpgroup h's arrival alone, so each
                    // warpgroup zeroes the rows of its own half of the keys;
                    // otherwise the two share all BN rows
                    const int tb = (g.pb + k * NPB) * BS;
                    const bool holes = tb + BN > tend || bits != (1u << NPB) - 1u;
                    if (holes) {
                        if (!__all_sync(kFullMask, wait(v_full + st, (j / NS) & 1))) break;
                        uint8_t* vt = smem + L.v_off + (size_t)st * L.tile_bytes;
                        constexpr int kZRows = kHalfO ? BH : BN, kZThreads = kHalfO ? 128 : 256;
                        const int zrow0 = kHalfO ? wg * BH : 0, zt = kHalfO ? r : sr;
                        for (int idx = zt; idx < kZRows * DBLK * 8; idx += kZThreads) {
                            const int row = zrow0 + idx / (DBLK * 8), rem = idx % (DBLK * 8);
                            if (!((bits >> (row / BS)) & 1u) || tb + row >= tend)
                                *reinterpret_cast<uint4*>(vt + (rem >> 3) * BN * 128 + row * 128 +
                                                          (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tc::fence_before_sync();
                mbar_arrive(smem_u32(p_full + (kHalfO ? wg * kTileSBufs : 0) + j % NB));
            }
            // ---- epilogue of the segment: O / l, or the partial (m, l, O);
            // each warpgroup its half of the columns ----
            bool have_o = __all_sync(kFullMask, k == nblk && !*abort_flag);
            if (have_o)
                have_o = __all_sync(kFullMask, wait(pv_done + (j - 1) % NB, ((j - 1) / NB) & 1));
            // the rows' normaliser (and, with an O per warpgroup, their max and
            // the weights of the two O's)
            float w_own = 1.f, w_oth = 0.f;
            if constexpr (kHalfO) {
                float m_oth = NEG_INF, l_oth = 0.f;
                if (have_o) have_o = exchange(xmax + (nx & 1) * 256, m, m_oth);
                if (have_o) have_o = exchange(xl, l, l_oth);
                const float M = fmaxf(m, m_oth);
                w_own = m == NEG_INF ? 0.f : fast_exp2(m - M);
                w_oth = m_oth == NEG_INF ? 0.f : fast_exp2(m_oth - M);
                l = l * w_own + l_oth * w_oth;
                m = M;
            } else {
                float lo_half = 0.f;
                if (have_o) have_o = exchange(xl, l, lo_half);
                if (have_o) l += lo_half;
            }
            tc::fence_after_sync();
            // the row's (unnormalised) O for columns c0 .. c0 + 15
            auto load_o = [&](int c0, float (&v)[16]) {
                uint32_t x[16];
                if constexpr (kHalfO) {
                    uint32_t y[16];
                    tc::ld_32x32b_x16(lane_base + O_COL + wg * D + c0, x);
                    tc::ld_32x32b_x16(lane_base + O_COL + (1 - wg) * D + c0, y);
                    tc::wait_ld();
                    // (an O never written holds garbage, but then its weight is 0)
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        v[c] = (w_own != 0.f ? __uint_as_float(x[c]) * w_own : 0.f) +
                               (w_oth != 0.f ? __uint_as_float(y[c]) * w_oth : 0.f);
                } else {
                    tc::ld_32x32b_x16(lane_base + O_COL + c0, x);
                    tc::wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(x[c]);
                }
            };
            if (p.cluster_reduce) {
                // park this CTA's partial in its own shared memory (the operand
                // buffers are idle: every copy and MMA has completed)
                const bool rows_ok = have_o && !dead;
                if (wg == 0) {
                    cl_m[r] = rows_ok && l > 0.f ? m : NEG_INF;
                    cl_l[r] = rows_ok ? l : 0.f;
                }
                if (rows_ok) {
                    float v[16];
#pragma unroll 1
                    for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 16) {
                        load_o(c0, v);
#pragma unroll
                        for (int c = 0; c < 16; c += 4)
                            *reinterpret_cast<float4*>(cl_o + r * CL + c0 + c) =
                                l > 0.f ? make_float4(v[c], v[c + 1], v[c + 2], v[c + 3])
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            } else if (have_o && !dead) {
                // a grid-position CTA: out (one partition) or its partition's
                // workspace rows; the balanced split: out for a whole unit, else
                // the CTA's record slot -- 0 for its first segment, 1 for a later one
                const bool fin = bal ? g.whole : (pers || p.final_out);
                const bool live = u < U;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                size_t orow = 0;
                if (live) {
                    if (fin)
                        orow = row_off(g.b, g.kvh, u);
                    else if (bal)
                        orow = (((size_t)blockIdx.x * 2 + (s == 0 ? 0 : 1)) * U + u) * D;
                    else
                        orow = ((((size_t)g.b * Hkv + g.kvh) * p.num_parts + part) * U + u) * D;
                    if (!fin && wg == 0) {
                        p.part_ml[(orow / D) * 2] = l > 0.f ? m : NEG_INF;
                        p.part_ml[(orow / D) * 2 + 1] = l;
                    }
                }
#pragma unroll 1
                for (int c0 = wg * (D / 2); c0 < (wg + 1) * (D / 2); c0 += 16) {
                    float v[16];
                    load_o(c0, v);
                    if (!live) continue;
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = l > 0.f ? v[c] * (fin ? inv : 1.f) : 0.f;
                    if (!fin || p.out_dtype == PA_F32) {
                        float* base = fin ? static_cast<float*>(p.out) : p.part_acc;
                        float* dst = base + orow + c0;
                        // rows start at multiples of head_dim floats and c0 at multiples
                        // of 16: a 32-byte aligned base gives whole-sector stores
                        if ((reinterpret_cast<uintptr_t>(base) & 31) == 0) {
                            st_global_v8(dst, v);
                            st_global_v8(dst + 8, v + 8);
                        } else {
#pragma unroll
                            for (int c = 0; c < 16; c += 4)
                                *reinterpret_cast<float4*>(dst + c) =
                                    make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
                        }
                    } else {
                        uint32_t w[8];
#pragma unroll
                        for (int c = 0; c < 16; c += 2) w[c / 2] = Mma<KV>::pack(v[c], v[c + 1]);
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<KV*>(p.out) + orow + c0);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
            if (multi) {
                // O of this segment has been read out: the next segment's first
                // P V may overwrite it
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(o_free));
            }
            return have_o && !*abort_flag;
        });
    }

    // ---- release tensor memory once every role is done with it ----
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kCols);
    }
    if (p.cluster_reduce) cluster_merge();
}

// Per-instantiation flag of the shared-memory limit set once per device.
template <int D, int BS, typename KV, int QR>
struct TileAttrs {
    static inline AttrFlags smem;
};

template <int D, int BS, typename KV, int QR>
cudaError_t launch_tile_inst(const AttnLaunch& L, cudaStream_t stream) {
    auto kern = tile_kernel<D, BS, KV, QR>;
    cudaError_t e = raise_smem_limit_once(kern, TileAttrs<D, BS, KV, QR>::smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    cfg.blockDim = dim3(kTileThreads);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (L.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (L.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)L.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, L.tmap_k, L.tmap_v, L.tmap_q, L.p);
}

// Clusters of `cluster` CTAs of this instantiation that can be resident at
// once on the current device (0 if the query fails).
template <int D, int BS, typename KV, int QR>
int tile_max_clusters_inst(int cluster, uint32_t smem_bytes) {
    auto kern = tile_kernel<D, BS, KV, QR>;
    if (raise_smem_limit_once(kern, TileAttrs<D, BS, KV, QR>::smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cluster, 1, 1);
    cfg.blockDim = dim3(kTileThreads);
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

template <int D, int QR>
int tile_max_clusters_for_d(int block_size, int kv_dtype, int cluster, uint32_t smem_bytes) {
    const bool bf = kv_dtype == PA_BF16;
    if (block_size == 16)
        return bf ? tile_max_clusters_inst<D, 16, __nv_bfloat16, QR>(cluster, smem_bytes)
                  : tile_max_clusters_inst<D, 16, __half, QR>(cluster, smem_bytes);
    return bf ? tile_max_clusters_inst<D, 32, __nv_bfloat16, QR>(cluster, smem_bytes)
              : tile_max_clusters_inst<D, 32, __half, QR>(cluster, smem_bytes);
}

template <int D, int QR>
cudaError_t launch_tile_for_d(const AttnLaunch& L, cudaStream_t stream) {
    const bool bf = L.kv_dtype == PA_BF16;
    if (L.block_size == 16)
        return bf ? launch_tile_inst<D, 16, __nv_bfloat16, QR>(L, stream)
                  : launch_tile_inst<D, 16, __half, QR>(L, stream);
    if (L.block_size == 32)
        return bf ? launch_tile_inst<D, 32, __nv_bfloat16, QR>(L, stream)
                  : launch_tile_inst<D, 32, __half, QR>(L, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
