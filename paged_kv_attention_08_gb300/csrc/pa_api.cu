// Host side of the C ABI in include/pa_decode.h, in this order: shape and
// argument validation; the device state (SM count, error word); the launch
// shape of the warp-level kernel (pick_tune) and the occupancy of its
// clusters; the split plans -- auto_plan (warp-level kernel), balanced_plan,
// tile_plan (tcgen05 tile kernel) and make_plan, which picks among them;
// workspace sizing; TMA descriptors (cached per host thread); the launches;
// and the exported entry points.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pa_internal.h"

// One error word per device; kernels set it when a bounded wait runs out.
__device__ int32_t pa_device_error_word;

// Fixed split-KV scratch for pa_decode_splitkv_noalloc: 16 MiB of fp32 per
// device that loads this library, held until the process exits.  In host code
// this name is only a stand-in for the symbol, never a device address: the
// address is looked up per device with cudaGetSymbolAddress.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) float pa_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace pa {
namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int32_t*> g_err_word[kMaxDevices];

std::atomic<void*> g_noalloc_scratch[kMaxDevices];

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Tuning and test switches.  The environment is read once, when the library
// is loaded (static initialisation), never by a call:
//   PA_TUNE_STREAMS, PA_TUNE_STAGES  warp-level kernel's streams per CTA and
//                                    stages per stream
//   PA_NO_PDL=1                      launch without programmatic dependent launch
//   PA_NO_CLUSTER=1                  never reduce partitions inside a cluster
//   PA_BALANCED=1|2                  let the automatic plan pick the balanced split
//   PA_NO_PERSIST=1                  tile kernel: one CTA per unit instead of persistent CTAs
//   PA_MULTI_KERNEL=mma|tile         initial value of PA_SWITCH_MULTI_KERNEL
//   PA_TILE_COMPACT_Q=0              initial value of PA_SWITCH_TILE_COMPACT_Q
// The last two can also be changed at run time through pa_set_switch.  None
// changes a result beyond rounding order.
int env_value(const char* name, int fallback, int (*parse)(const char*)) {
    const char* v = std::getenv(name);
    return (v && *v) ? parse(v) : fallback;
}
int parse_positive(const char* v) {
    const int x = std::atoi(v);
    return x > 0 ? x : 0;
}
int parse_flag(const char* v) { return std::atoi(v) > 0 ? 1 : 0; }
int parse_balanced(const char* v) {
    const int x = std::atoi(v);
    return x < 0 ? 0 : (x > 2 ? 2 : x);
}
int parse_kernel(const char* v) {
    if (std::strcmp(v, "tile") == 0) return PA_KERNEL_TILE;
    if (std::strcmp(v, "mma") == 0) return PA_KERNEL_MMA;
    return PA_KERNEL_AUTO;
}
int parse_compact(const char* v) { return std::atoi(v) == 0 ? 0 : 1; }

struct LoadTimeEnv {
    int tune_streams, tune_stages, no_pdl, no_cluster, balanced, no_persist;
};
const LoadTimeEnv g_env = {env_value("PA_TUNE_STREAMS", 0, parse_positive),
                           env_value("PA_TUNE_STAGES", 0, parse_positive),
                           env_value("PA_NO_PDL", 0, parse_flag),
                           env_value("PA_NO_CLUSTER", 0, parse_flag),
                           env_value("PA_BALANCED", 0, parse_balanced),
                           env_value("PA_NO_PERSIST", 0, parse_flag)};
std::atomic<int> g_switch_multi_kernel{env_value("PA_MULTI_KERNEL", PA_KERNEL_AUTO, parse_kernel)};
std::atomic<int> g_switch_compact_q{env_value("PA_TILE_COMPACT_Q", 1, parse_compact)};

int elem_size(int dtype) { return dtype == PA_F32 ? 4 : 2; }

bool aligned(const void* ptr, size_t a) { return reinterpret_cast<uintptr_t>(ptr) % a == 0; }

bool pow2_group_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

pa_status check_shape(const pa_shape* s) {
    if (!s) return PA_ERR_INVALID_ARG;
    if (s->batch < 0 || s->num_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0 ||
        s->block_size <= 0 || s->max_blocks_per_seq <= 0 || s->num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (s->num_heads % s->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (s->kv_dtype != PA_F16 && s->kv_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (s->out_dtype != PA_F32 && s->out_dtype != s->kv_dtype) return PA_ERR_UNSUPPORTED;
    if (!pow2_group_ok(s->num_heads / s->num_kv_heads)) return PA_ERR_UNSUPPORTED;
    if (s->head_dim != 64 && s->head_dim != 128 && s->head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (s->block_size != 16 && s->block_size != 32) return PA_ERR_UNSUPPORTED;
    if (s->batch > 65535 || s->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (s->num_blocks >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
    if ((int64_t)s->max_blocks_per_seq * s->block_size >= (int64_t(1) << 31))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// The scores are scaled by `scale` before the softmax; the kernels take the
// running maximum of the unscaled scores, which needs scale > 0.
bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

// Query tokens one CTA serves: q_chunk * group rows fill at most the 16 rows
// of the MMA tile.
int q_chunk_for(const pa_shape* s, int32_t q_len) {
    const int per = 16 / (s->num_heads / s->num_kv_heads);
    return q_len < per ? q_len : per;
}
int q_chunks_for(const pa_shape* s, int32_t q_len) {
    const int c = q_chunk_for(s, q_len);
    return (q_len + c - 1) / c;
}

pa_status check_ptrs(const void* out, const void* q, const void* k, const void* v,
                     const int32_t* bt, const int32_t* lens) {
    if (!out || !q || !k || !v || !bt || !lens) return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
        return PA_ERR_INVALID_ARG;
    if (!aligned(bt, 4) || !aligned(lens, 4)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// SM count of the current device (cached).
pa_status device_sms(int* sms, int* device) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return PA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return PA_ERR_CUDA;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    *sms = n;
    if (device) *device = dev;
    return PA_OK;
}

// SM count for the size and plan queries: the current device's, as the calls
// themselves plan with it (it picks the CTA shape, and with it whether a
// cluster split fits on the device, explicit partition sizes included).  An
// explicit partition size may also be queried without a device: the plan is
// then made for one SM (the split itself does not depend on the count).
pa_status query_sms(int32_t partition_tokens, int* sms) {
    *sms = 1;
    const pa_status st = device_sms(sms, nullptr);
    if (st == PA_OK) return PA_OK;
    *sms = 1;
    return partition_tokens > 0 ? PA_OK : st;
}

// SM count and error-word address of the current device (cached).
pa_status device_state(int* sms, int32_t** err) {
    int dev = 0, n = 0;
    const pa_status st = device_sms(&n, &dev);
    if (st != PA_OK) return st;
    int32_t* e = g_err_word[dev].load(std::memory_order_acquire);
    if (!e) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, pa_device_error_word) != cudaSuccess || !ptr)
            return PA_ERR_CUDA;
        e = static_cast<int32_t*>(ptr);
        g_err_word[dev].store(e, std::memory_order_release);
    }
    if (sms) *sms = n;
    if (err) *err = e;
    return PA_OK;
}

// Launch shape of the attention kernel for one problem: warps per stream
// (head_dim 256 splits a page's output columns over two warps), streams per
// CTA and stages per stream.
struct Tune {
    int nh, nt, ns;
};

Tune pick_tune(const pa_shape* s, bool many_ctas) {
    Tune t;
    t.nh = s->head_dim == 256 ? 2 : 1;
    const uint32_t stage = 2u * s->block_size * s->head_dim * 2u;
    if (many_ctas) {
        // grids of several waves: four warps, ~96 KB of pages, two CTAs per SM
        t.nt = 4 / t.nh;
        const int ns = (96 * 1024) / (t.nt * (int)stage);
        t.ns = ns < 2 ? 2 : (ns > 8 ? 8 : ns);
    } else {
        // grids of at most one wave: eight warps, one CTA per SM, two pages in
        // flight per stream; fewer streams when the pages are too large
        t.nt = 8 / t.nh;
        t.ns = 2;
        while (t.nt > 1 && (uint32_t)t.nt * t.ns * stage > 200u * 1024u) --t.nt;
    }
    if (g_env.tune_streams > 0 && g_env.tune_streams * t.nh <= 8) t.nt = g_env.tune_streams;
    if (g_env.tune_stages > 0 && g_env.tune_stages <= 16) t.ns = g_env.tune_stages;
    // never ask for more shared memory than a CTA may have
    while (t.ns > 1 && attn_smem_layout(s->head_dim, s->block_size, t.nt, t.ns).total +
                               kSmemAlignSlack > 227u * 1024u)
        --t.ns;
    return t;
}

// CTAs of this tune resident per SM: by shared memory, and by registers
// (the kernels use about 200 registers a thread).
int ctas_per_sm(const pa_shape* s, const Tune& t) {
    const AttnSmem L = attn_smem_layout(s->head_dim, s->block_size, t.nt, t.ns);
    int by_smem = (int)((227u * 1024u) / (L.total + kSmemAlignSlack));
    const int threads = 32 * t.nt * t.nh;
    int by_regs = 65536 / (200 * threads);
    int n = by_smem < by_regs ? by_smem : by_regs;
    return n < 1 ? 1 : (n > 8 ? 8 : n);
}

// Programmatic dependent launch lets each kernel's launch overlap the tail
// of the previous one in the stream; PA_NO_PDL=1 launches plainly instead.
bool use_pdl() { return !g_env.no_pdl; }


int pages_for(const pa_shape* s, int32_t max_context_len) {
    int64_t t = max_context_len < 1 ? 1 : max_context_len;
    const int64_t cap = (int64_t)s->max_blocks_per_seq * s->block_size;
    if (t > cap) t = cap;
    return (int)((t + s->block_size - 1) / s->block_size);
}

// How a call is split: pages per partition, partitions per (sequence, kv
// head), and whether the partitions reduce inside a thread-block cluster
// (no workspace, no combine launch) or through the workspace and the combine
// kernel.
struct Plan {
    int part_pages, num_parts;
    bool cluster;
    bool many_ctas;  // the grid spans several waves: pick the two-CTAs-per-SM tune
    bool balanced;   // one CTA per SM, equal shares of the flattened page order
    int num_ctas;    // balanced: grid size
    bool tile;       // several query tokens on the tcgen05 tile kernel (128-row tiles)
    int tile_qr;     // tile kernel: Q rows staged in shared memory (128, or 16: compact)
    bool persistent; // tile kernel, one pass: num_ctas CTAs take the units in turn, whole
};

Plan plan_with(const pa_shape* s, int pages, int pp, bool cluster_ok,
               int max_cluster = kMaxClusterParts) {
    Plan p;
    p.many_ctas = false;
    p.balanced = false;
    p.num_ctas = 0;
    p.tile = false;
    p.tile_qr = kTileRows;
    p.persistent = false;
    if (pp < 1) pp = 1;
    p.num_parts = (pages + pp - 1) / pp;
    if (p.num_parts < 1) p.num_parts = 1;
    p.part_pages = p.num_parts <= 1 ? s->max_blocks_per_seq : pp;
    p.cluster = cluster_ok && p.num_parts > 1 && p.num_parts <= max_cluster;
    return p;
}

// Automatic split (the design notes only say the chunk size follows the KV
// length; these rules are this library's own, fitted to GB300 timings of the
// workloads it is measured on).  With units = batch * kv heads CTAs unsplit
// and `slots` CTAs resident at once:
//  - a grid already a third full or more (at two CTAs per SM) runs in one
//    pass when every unit is resident at once, and is otherwise split only
//    into partitions of about 64 pages, so that long and ragged sequences
//    balance across waves; no cluster (the grid spans several waves);
//  - a smaller grid is split to fill about 85% of one wave, either into at
//    most 8 partitions of at least 4 pages reduced inside a cluster (up to 16
//    where the device holds all of the call's clusters at once), or, when
//    that gives less parallelism, into partitions of at least 16 pages
//    combined through the workspace.
// The longest context stands for every sequence: the host reads no lengths.
// The automatic choice does not pick the balanced split (on GB300 it was
// slower than equal partitions for every workload measured: once ~128 CTAs
// stream, HBM is the limit and the split's extra reduction costs more than
// the idle SMs); PA_BALANCED=1 lets it pick the balanced split where equal
// partitions leave SMs idle, PA_BALANCED=2 wherever the batch allows.  A
// tuning switch; results agree.
int balanced_mode() { return g_env.balanced; }

Plan balanced_plan(const pa_shape* s, int pages, int num_sms) {
    Plan p = plan_with(s, pages, pages, false);
    p.balanced = true;
    p.num_ctas = num_sms;
    p.many_ctas = false;
    return p;
}

// Clusters of `cluster` one-token attention CTAs of tune `t` that fit on the
// current device at once (cached per device and shape class; 0 when unknown,
// e.g. without a device).
int attn_max_clusters(const pa_shape* s, const Tune& t, int cluster) {
    static std::atomic<int> cache[kMaxDevices][3][2][2][2][kMaxDecodeClusterParts + 1];  // n+1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return 0;
    }
    const int di = s->head_dim == 64 ? 0 : (s->head_dim == 128 ? 1 : 2);
    const int threads = 32 * t.nt * t.nh;  // the tune: 8-warp (one per SM) or 4-warp CTAs
    std::atomic<int>& slot =
        cache[dev][di][s->block_size == 32][s->kv_dtype == PA_BF16][threads >= 256][cluster];
    int v = slot.load(std::memory_order_relaxed);
    if (v == 0) {
        const uint32_t smem =
            attn_smem_layout(s->head_dim, s->block_size, t.nt, t.ns).total + kSmemAlignSlack;
        int n = 0;
        switch (s->head_dim) {
            case 64: n = attn_max_clusters_d64(s->block_size, s->kv_dtype, cluster, threads, smem); break;
            case 128: n = attn_max_clusters_d128(s->block_size, s->kv_dtype, cluster, threads, smem); break;
            default: n = attn_max_clusters_d256(s->block_size, s->kv_dtype, cluster, threads, smem); break;
        }
        v = n + 1;
        slot.store(v, std::memory_order_relaxed);
    }
    return v - 1;
}

bool clusters_enabled();

Plan auto_plan(const pa_shape* s, int32_t max_context_len, int num_sms, int q_chunks = 1) {
    const int pages = pages_for(s, max_context_len);
    const int64_t units = (int64_t)s->batch * s->num_kv_heads * q_chunks;
    auto ceil_div = [](int64_t a, int64_t b) { return (a + b - 1) / b; };
    const bool can_balance =
        s->batch <= kMaxBalancedBatch && q_chunks == 1 && balanced_mode() > 0;
    // enough pages that every SM gets at least eight
    const bool big = units * pages >= 8LL * num_sms;
    const int64_t wide_slots = (int64_t)num_sms * ctas_per_sm(s, pick_tune(s, true));
    if (units * 3 >= wide_slots) {
        if (can_balance && balanced_mode() == 2 && big) return balanced_plan(s, pages, num_sms);
        // every unit resident at once: one pass, no split (B=16, T=2048:
        // 24.5 us against 29.3 us in 64-page partitions through the
        // workspace; B=16, T=8192: 82.9 against 98.0 us)
        if (units <= wide_slots) {
            Plan p = plan_with(s, pages, pages, false);
            p.many_ctas = units > num_sms;
            return p;
        }
        const int parts = (int)ceil_div(pages, 64);
        Plan p = plan_with(s, pages, (int)ceil_div(pages, parts), false);
        p.many_ctas = units * p.num_parts > num_sms;
        return p;
    }
    const int64_t slots = (int64_t)num_sms * ctas_per_sm(s, pick_tune(s, false));
    int64_t fill = (int64_t)(0.85 * (double)slots / (double)units);
    if (fill < 1) fill = 1;
    // The largest cluster (up to 16 CTAs) of which the device holds every
    // unit's copy at once: one cluster more than fits runs as a second wave
    // (at ~133 KB per CTA the device holds 15 clusters of 8, so 16 units in
    // clusters of 8 took 13.9 us at B=2, T=2048, against 8.9 us in clusters
    // of 6).  Without a device to ask (the host-only partition query),
    // clusters of up to 8 are assumed to fit.
    int64_t cap = 1;
    const int64_t want = std::min<int64_t>(std::min<int64_t>(kMaxDecodeClusterParts, fill),
                                           ceil_div(pages, 4));
    if (clusters_enabled()) {
        const Tune tall = pick_tune(s, false);
        for (int64_t c = want; c >= 2; --c) {
            const int n = attn_max_clusters(s, tall, (int)c);
            if (n > 0 ? units <= n : c <= kMaxClusterParts) {
                cap = c;
                break;
            }
        }
    }
    const int64_t p_cl = std::min<int64_t>(std::min<int64_t>(cap, fill), ceil_div(pages, 4));
    const int64_t p_ws = std::min<int64_t>(fill, ceil_div(pages, 16));
    // a cluster split with fewer partitions than the workspace split still
    // wins when partitions are short (latency-bound: the combine launch costs
    // more than the lost parallelism), e.g. B=1, T=8K: 12 in clusters 11.6 us,
    // 16 through the workspace 12.5 us; at T=32K/128K the workspace split wins
    const bool short_parts = ceil_div(pages, p_cl) <= 64;
    const bool use_cluster = p_cl >= p_ws || (short_parts && p_cl * 4 >= p_ws * 3);
    Plan p = use_cluster ? plan_with(s, pages, (int)ceil_div(pages, p_cl), true, (int)cap)
                         : plan_with(s, pages, (int)ceil_div(pages, p_ws), false);
    // Equal partitions of few units leave SMs idle (e.g. 32 units x 4 = 128
    // CTAs on 152 SMs); the balanced split gives every SM the same share.
    const double coverage = (double)(units * p.num_parts) / (double)slots;
    if (can_balance && big && (balanced_mode() == 2 || coverage < 0.9))
        return balanced_plan(s, pages, (int)slots);
    return p;
}

// PA_NO_CLUSTER=1 turns the in-cluster reduction off (partitions then always
// go through the workspace); a tuning switch, results are the same.
bool clusters_enabled() { return !g_env.no_cluster; }

// Which kernel serves several query tokens: the tcgen05 tile kernel once
// the rows of a (sequence, kv head) -- q_len * group -- exceed the 16 rows
// of the warp-level MMA path (which would otherwise read the pages once per
// 16 rows), and for 16 rows at head_dim 256.  The PA_SWITCH_MULTI_KERNEL
// switch forces the warp-level path for every q_len > 1 (PA_KERNEL_MMA) or
// the tile kernel for every split-KV call, one query token included
// (PA_KERNEL_TILE); results agree.
bool use_tile(const pa_shape* s, int32_t q_len, int32_t partition_tokens) {
    const int64_t rows = (int64_t)q_len * (s->num_heads / s->num_kv_heads);
    // the balanced split is honoured by the warp-level kernel up to 16 rows,
    // and by the tile kernel for units of at most 16 rows at head_dim 256
    if (partition_tokens == PA_PARTITION_BALANCED && rows <= 16)
        return s->head_dim == 256 && s->batch <= kMaxBalancedBatch;
    const int force = g_switch_multi_kernel.load(std::memory_order_relaxed);
    if (force == PA_KERNEL_TILE) return true;
    if (force == PA_KERNEL_MMA && q_len > 1) return false;
    // 16 rows at head_dim 256 too: the warp-level path needs two warps per
    // page there and spills registers; the tile kernel was 6-23 % faster
    return rows > 16 || (rows == 16 && s->head_dim == 256);
}

// Q rows the tile kernel stages: 16 at head_dim 256 when a unit has at most 16
// rows (its other 112 would be zeros), which buys a third stage per K / V
// ring; otherwise a whole tile.  PA_SWITCH_TILE_COMPACT_Q = 0 stages whole
// tiles always (results agree).
int tile_q_rows(const pa_shape* s, int32_t q_len) {
    if (g_switch_compact_q.load(std::memory_order_relaxed) == 0) return kTileRows;
    const int64_t rows = (int64_t)q_len * (s->num_heads / s->num_kv_heads);
    return s->head_dim == 256 && rows <= kTileCompactQRows ? kTileCompactQRows : kTileRows;
}

bool tile_cluster_fits(const pa_shape* s, int qr) {
    return tile_cluster_bytes(s->head_dim) <=
           tile_smem_layout(s->head_dim, s->block_size, qr).bar_off;
}

int tile_ctas_per_sm(const pa_shape* s, int qr) {
    const TileSmem L = tile_smem_layout(s->head_dim, s->block_size, qr);
    int n = (int)((227u * 1024u) / (L.total + kSmemAlignSlack));
    const int by_tmem = (int)(512u / tile_tmem_cols(s->head_dim));
    n = n < by_tmem ? n : by_tmem;
    n = n < 2 ? n : 2;  // registers: 256 threads of up to ~128
    return n < 1 ? 1 : n;
}

// Clusters of `cluster` tile-kernel CTAs that fit on the current device at
// once (cached per device and instantiation; 0 when unknown).
int tile_max_clusters(const pa_shape* s, int cluster, int qr) {
    // n + 1; 0 = unset
    static std::atomic<int> cache[kMaxDevices][3][2][2][2][kMaxClusterParts + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int di = s->head_dim == 64 ? 0 : (s->head_dim == 128 ? 1 : 2);
    const bool compact = qr == kTileCompactQRows && s->head_dim == 256;
    std::atomic<int>& slot =
        cache[dev][di][s->block_size == 32][s->kv_dtype == PA_BF16][compact][cluster];
    int v = slot.load(std::memory_order_relaxed);
    if (v == 0) {
        const uint32_t smem =
            tile_smem_layout(s->head_dim, s->block_size, compact ? qr : kTileRows).total +
            kSmemAlignSlack;
        int n = 0;
        switch (s->head_dim) {
            case 64: n = tile_max_clusters_d64(s->block_size, s->kv_dtype, cluster, smem); break;
            case 128: n = tile_max_clusters_d128(s->block_size, s->kv_dtype, cluster, smem); break;
            default:
                n = compact ? tile_max_clusters_d256_compact(s->block_size, s->kv_dtype, cluster, smem)
                            : tile_max_clusters_d256(s->block_size, s->kv_dtype, cluster, smem);
                break;
        }
        v = n + 1;
        slot.store(v, std::memory_order_relaxed);
    }
    return v - 1;
}

// Tile kernel split: units = B * Hkv * ceil(q_len*G / 128) CTAs unsplit; cut
// each unit's pages into as many partitions (of at least 4 pages) as fit in
// one wave of resident CTAs.  Partitions reduce inside a cluster through
// distributed shared memory when every unit's cluster (at most 8 CTAs) fits
// on the device at once and the cluster split keeps at least 2/3 of those
// partitions (the workspace round trip and the combine launch cost more than
// the rest); otherwise through the workspace.
Plan tile_plan(const pa_shape* s, int32_t max_context_len, int32_t partition_tokens, int num_sms,
               int32_t q_len) {
    const int pages = pages_for(s, max_context_len);
    const int qr = tile_q_rows(s, q_len);
    int pp;
    if (partition_tokens > 0) {
        pp = partition_tokens / s->block_size;
    } else {
        const int64_t rows = (int64_t)q_len * (s->num_heads / s->num_kv_heads);
        const int64_t units = (int64_t)s->batch * s->num_kv_heads * ((rows + kTileRows - 1) / kTileRows);
        const int64_t slots = (int64_t)num_sms * tile_ctas_per_sm(s, qr);
        int64_t parts = slots / units;  // whole waves: one partition more would add a wave
        const int64_t max_parts = (pages + 3) / 4;
        if (parts > max_parts) parts = max_parts;
        if (parts < 1) parts = 1;
        int best_c = 0;  // largest cluster split whose clusters are all resident at once
        for (int c = (int)std::min<int64_t>(kMaxClusterParts, max_parts); c >= 2; --c)
            if (units <= tile_max_clusters(s, c, qr)) {
                best_c = c;
                break;
            }
        // the parked partial must fit in the operand buffers
        const bool fits = tile_cluster_fits(s, qr);
        // (B=2, T=4096, 64 query tokens of 16 heads: 6 partitions in clusters
        // 32.0 us against 9 through the workspace 35.6 us)
        const bool cluster =
            fits && parts >= 2 && best_c >= 2 && (int64_t)best_c * 3 >= parts * 2;
        if (cluster) parts = std::min<int64_t>(best_c, parts);
        pp = (int)((pages + parts - 1) / parts);
        Plan p = plan_with(s, pages, pp, cluster);
        p.tile = true;
        p.tile_qr = qr;
        // one pass over more units than fit at once: persistent CTAs, one
        // per resident slot, take the units in turn, so that a unit's start
        // (its Q, the first K / V blocks) overlaps the previous unit's end
        if (p.num_parts <= 1 && units > slots && tile_q_bufs(s->head_dim, qr) == 2 &&
            !g_env.no_persist) {
            p.persistent = true;
            p.num_ctas = (int)slots;
        }
        return p;
    }
    // an explicit partition count: a cluster when its partial fits in shared
    // memory and the device holds every unit's cluster at once
    Plan p = plan_with(s, pages, pp, tile_cluster_fits(s, qr));
    if (p.cluster) {
        const int64_t rows = (int64_t)q_len * (s->num_heads / s->num_kv_heads);
        const int64_t units =
            (int64_t)s->batch * s->num_kv_heads * ((rows + kTileRows - 1) / kTileRows);
        const int n = tile_max_clusters(s, p.num_parts, qr);
        if (n > 0 && units > n) p.cluster = false;
    }
    p.tile = true;
    p.tile_qr = qr;
    return p;
}

// The balanced split keeps every query token of a (sequence, kv head) in
// one CTA: it needs q_len * group <= 16, and batch <= kMaxBalancedBatch.
Plan make_plan(const pa_shape* s, int32_t max_context_len, int32_t partition_tokens, int num_sms,
               int32_t q_len = 1) {
    if (use_tile(s, q_len, partition_tokens) && partition_tokens == PA_PARTITION_BALANCED &&
        tile_q_rows(s, q_len) == kTileCompactQRows && s->batch <= kMaxBalancedBatch) {
        // the balanced split of compact units on the tile kernel: one CTA per
        // SM, each an equal share of the flattened (sequence, kv head, page)
        // order, pieces that straddle shares combined afterwards
        Plan p = balanced_plan(s, pages_for(s, max_context_len),
                               num_sms * tile_ctas_per_sm(s, kTileCompactQRows));
        p.tile = true;
        p.tile_qr = kTileCompactQRows;
        return p;
    }
    if (use_tile(s, q_len, partition_tokens)) {
        Plan tp = tile_plan(s, max_context_len,
                            partition_tokens == PA_PARTITION_BALANCED ? 0 : partition_tokens,
                            num_sms, q_len);
        if (!clusters_enabled()) tp.cluster = false;
        return tp;
    }
    Plan plan;
    const int q_chunks = q_chunks_for(s, q_len);
    if (partition_tokens == PA_PARTITION_BALANCED && s->batch <= kMaxBalancedBatch &&
        q_chunks == 1) {
        plan = balanced_plan(s, pages_for(s, max_context_len),
                             num_sms * ctas_per_sm(s, pick_tune(s, false)));
    } else if (partition_tokens <= 0) {
        plan = auto_plan(s, max_context_len, num_sms, q_chunks);
    } else {
        plan = plan_with(s, pages_for(s, max_context_len), partition_tokens / s->block_size, true);
        plan.many_ctas =
            (int64_t)s->batch * s->num_kv_heads * q_chunks * plan.num_parts > num_sms;
        if (plan.cluster) {
            // the partition count is honoured; its reduction goes through the
            // workspace when the device cannot hold every cluster at once
            const int n = attn_max_clusters(s, pick_tune(s, plan.many_ctas), plan.num_parts);
            if (n > 0 && (int64_t)s->batch * s->num_kv_heads * q_chunks > n) plan.cluster = false;
        }
    }
    if (!clusters_enabled()) plan.cluster = false;
    return plan;
}

bool partition_arg_ok(const pa_shape* s, int32_t partition_tokens) {
    return partition_tokens == PA_PARTITION_BALANCED ||
           (partition_tokens >= 0 && partition_tokens % s->block_size == 0);
}

// Workspace: part_acc [B, Hkv, P, Q*G, D] fp32, then part_ml [B, Hkv, P, Q*G, 2]
// fp32 (rows of a (sequence, kv head, partition): query token, then head).
// Workspace bytes of a plan; SIZE_MAX (which no buffer satisfies, so the call
// is refused with PA_ERR_WORKSPACE) when the size does not fit in a size_t.
size_t workspace_bytes_for(const pa_shape* s, const Plan& plan, size_t* ml_offset,
                           int32_t q_len = 1) {
    const size_t kTooBig = SIZE_MAX;
    size_t rows = 1;  // (m, l, acc) rows
    auto mul = [&](size_t f) { return !__builtin_mul_overflow(rows, f, &rows); };
    bool ok;
    if (plan.balanced) {  // [C][2][Q*G]
        ok = mul((size_t)plan.num_ctas) && mul(2) &&
             mul((size_t)(s->num_heads / s->num_kv_heads)) && mul((size_t)q_len);
    } else {
        if (plan.num_parts <= 1 || plan.cluster) return 0;  // one pass, or reduced in a cluster
        ok = mul((size_t)s->batch) && mul((size_t)s->num_heads) && mul((size_t)q_len) &&
             mul((size_t)plan.num_parts);  // [B][Hkv][P][Q*G]
    }
    size_t acc = 0, ml = 0;
    if (!ok || __builtin_mul_overflow(rows, (size_t)s->head_dim * sizeof(float), &acc) ||
        __builtin_mul_overflow(rows, 2 * sizeof(float), &ml) || acc > kTooBig - 255 - ml)
        return kTooBig;
    const size_t off = (acc + 255) / 256 * 256;
    if (ml_offset) *ml_offset = off;
    return off + ml;
}

// The last few tensor-map pairs this host thread encoded, by everything a map
// encodes (addresses and dimensions; no contents), so a hit is exact.  A call
// on the same cache buffers as a recent one skips the two driver encodes.
struct MapCacheEntry {
    const void* k;
    const void* v;
    int64_t num_blocks;
    int32_t head_dim, num_kv_heads, block_size, kv_dtype;
    bool valid;
    CUtensorMap mk, mv;
};
constexpr int kMapCacheEntries = 4;
thread_local MapCacheEntry tl_maps[kMapCacheEntries];
thread_local int tl_maps_next = 0;

pa_status encode_maps_uncached(const pa_shape* s, const void* k, const void* v, CUtensorMap* mk,
                               CUtensorMap* mv);

pa_status encode_maps(const pa_shape* s, const void* k, const void* v, CUtensorMap* mk,
                      CUtensorMap* mv) {
    for (int i = 0; i < kMapCacheEntries; ++i) {
        const MapCacheEntry& c = tl_maps[i];
        if (c.valid && c.k == k && c.v == v && c.num_blocks == s->num_blocks &&
            c.head_dim == s->head_dim && c.num_kv_heads == s->num_kv_heads &&
            c.block_size == s->block_size && c.kv_dtype == s->kv_dtype) {
            *mk = c.mk;
            *mv = c.mv;
            return PA_OK;
        }
    }
    const pa_status st = encode_maps_uncached(s, k, v, mk, mv);
    if (st != PA_OK) return st;
    MapCacheEntry& c = tl_maps[tl_maps_next];
    tl_maps_next = (tl_maps_next + 1) % kMapCacheEntries;
    c.k = k;
    c.v = v;
    c.num_blocks = s->num_blocks;
    c.head_dim = s->head_dim;
    c.num_kv_heads = s->num_kv_heads;
    c.block_size = s->block_size;
    c.kv_dtype = s->kv_dtype;
    c.mk = *mk;
    c.mv = *mv;
    c.valid = true;
    return PA_OK;
}

pa_status encode_maps_uncached(const pa_shape* s, const void* k, const void* v, CUtensorMap* mk,
                               CUtensorMap* mv) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return PA_ERR_CUDA;
    const cuuint64_t e = elem_size(s->kv_dtype);
    // dims innermost first: head_dim, kv head, slot in block, block
    const cuuint64_t dims[4] = {(cuuint64_t)s->head_dim, (cuuint64_t)s->num_kv_heads,
                                (cuuint64_t)s->block_size, (cuuint64_t)s->num_blocks};
    const cuuint64_t strides[3] = {e * s->head_dim, e * s->head_dim * s->num_kv_heads,
                                   e * s->head_dim * s->num_kv_heads * s->block_size};
    // one 64-column block (128 bytes) of one kv head's block_size rows, written
    // to shared memory with the 128-byte swizzle that ldmatrix reads conflict-free
    const cuuint32_t box[4] = {64u, 1u, (cuuint32_t)s->block_size, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUtensorMapDataType dt =
        s->kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    for (int which = 0; which < 2; ++which) {
        CUresult r = g_encode(which ? mv : mk, dt, 4, const_cast<void*>(which ? v : k), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return PA_ERR_CUDA;
    }
    return PA_OK;
}

// The Q tiles of the tile kernel's later segments: q [batch * q_len, heads,
// head_dim] read in boxes of 64 columns x (G heads x qr / G tokens), or x qr
// heads of one token when the group has qr or more heads -- a tile's rows in
// order -- with the 128-byte swizzle; past the last token the fill value (0).
pa_status encode_q_map(const pa_shape* s, const void* q, int32_t q_len, int qr, CUtensorMap* mq) {
    if (!g_encode) return PA_ERR_CUDA;  // set up by the K / V maps' first encode
    const int G = s->num_heads / s->num_kv_heads;
    const cuuint64_t e = elem_size(s->kv_dtype);
    const cuuint64_t dims[3] = {(cuuint64_t)s->head_dim, (cuuint64_t)s->num_heads,
                                (cuuint64_t)s->batch * (cuuint64_t)q_len};
    const cuuint64_t strides[2] = {e * s->head_dim, e * s->head_dim * s->num_heads};
    const cuuint32_t box[3] = {64u, (cuuint32_t)(G >= qr ? qr : G), (cuuint32_t)(G >= qr ? 1 : qr / G)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapDataType dt =
        s->kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = g_encode(mq, dt, 3, const_cast<void*>(q), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

pa_status launch_attention(void* out, const void* q, const void* k, const void* v,
                           const int32_t* bt, const int32_t* lens, const pa_shape* s, float scale,
                           const Plan& plan, float* part_acc, float* part_ml, int32_t* err,
                           cudaStream_t stream, int32_t q_len = 1) {
    AttnLaunch L;
    std::memset(&L, 0, sizeof L);
    const int G = s->num_heads / s->num_kv_heads;
    const int q_chunk = q_chunk_for(s, q_len);
    const int64_t grid_y = (int64_t)s->num_kv_heads * q_chunks_for(s, q_len);
    if (grid_y > 65535) return PA_ERR_UNSUPPORTED;
    const Tune t = pick_tune(s, plan.many_ctas);
    const AttnSmem sm = attn_smem_layout(s->head_dim, s->block_size, t.nt, t.ns);
    const int rows = q_chunk * G;  // MMA rows in use
    if (4u * (merge_floats(t.nt * t.nh, rows, s->head_dim / t.nh) +
              cluster_part_floats(rows, s->head_dim)) > sm.stage_bytes * t.nt * t.ns)
        return PA_ERR_UNSUPPORTED;  // the final merge must fit in the stage area
    pa_status st = encode_maps(s, k, v, &L.tmap_k, &L.tmap_v);
    if (st != PA_OK) return st;
    AttnParams& p = L.p;
    p.q = q;
    p.out = out;
    p.block_tables = bt;
    p.context_lens = lens;
    p.part_acc = part_acc;
    p.part_ml = part_ml;
    p.err = err;
    p.batch = s->batch;
    p.num_heads = s->num_heads;
    p.num_kv_heads = s->num_kv_heads;
    p.group = G;
    p.q_len = q_len;
    p.q_chunk = q_chunk;
    p.unit_rows = q_len * G;
    p.max_blocks = s->max_blocks_per_seq;
    p.num_blocks = s->num_blocks;
    p.qscale = scale * 1.4426950408889634f;  // log2(e)
    p.part_pages = plan.part_pages;
    p.num_parts = plan.num_parts;
    p.nt = t.nt;
    p.nh = t.nh;
    p.ns = t.ns;
    p.out_dtype = s->out_dtype;
    p.final_out = plan.num_parts <= 1 ? 1 : 0;
    p.cluster_reduce = plan.cluster ? 1 : 0;
    p.balanced = plan.balanced ? 1 : 0;
    if (plan.balanced) p.final_out = 0;
    p.timeout_ns = kDefaultTimeoutNs;
    L.head_dim = s->head_dim;
    L.block_size = s->block_size;
    L.kv_dtype = s->kv_dtype;
    L.pdl = use_pdl();
    L.cluster = p.cluster_reduce ? plan.num_parts : 1;
    L.grid = plan.balanced ? dim3((unsigned)plan.num_ctas)
                           : dim3((unsigned)plan.num_parts, (unsigned)grid_y,
                                  (unsigned)s->batch);
    L.threads = 32 * t.nt * t.nh;
    L.smem_bytes = sm.total + kSmemAlignSlack;
    cudaError_t e;
    switch (s->head_dim) {
        case 64: e = launch_attn_d64(L, stream); break;
        case 128: e = launch_attn_d128(L, stream); break;
        default: e = launch_attn_d256(L, stream); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status launch_tile(void* out, const void* q, const void* k, const void* v, const int32_t* bt,
                      const int32_t* lens, const pa_shape* s, float scale, const Plan& plan,
                      float* part_acc, float* part_ml, int32_t* err, cudaStream_t stream,
                      int32_t q_len) {
    AttnLaunch L;
    std::memset(&L, 0, sizeof L);
    const int G = s->num_heads / s->num_kv_heads;
    const int64_t rows = (int64_t)q_len * G;
    const int64_t grid_y = (int64_t)s->num_kv_heads * ((rows + kTileRows - 1) / kTileRows);
    if (grid_y > 65535 || rows > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    pa_status st = encode_maps(s, k, v, &L.tmap_k, &L.tmap_v);
    if (st != PA_OK) return st;
    AttnParams& p = L.p;
    p.q = q;
    p.out = out;
    p.block_tables = bt;
    p.context_lens = lens;
    p.part_acc = part_acc;
    p.part_ml = part_ml;
    p.err = err;
    p.batch = s->batch;
    p.num_heads = s->num_heads;
    p.num_kv_heads = s->num_kv_heads;
    p.group = G;
    p.q_len = q_len;
    p.q_chunk = kTileRows / G;
    p.unit_rows = (int32_t)rows;
    p.max_blocks = s->max_blocks_per_seq;
    p.num_blocks = s->num_blocks;
    p.qscale = scale * 1.4426950408889634f;  // log2(e)
    p.part_pages = plan.part_pages;
    p.num_parts = plan.num_parts;
    p.out_dtype = s->out_dtype;
    p.final_out = plan.num_parts <= 1 ? 1 : 0;
    p.cluster_reduce = plan.cluster ? 1 : 0;
    p.timeout_ns = kDefaultTimeoutNs;
    L.head_dim = s->head_dim;
    L.block_size = s->block_size;
    L.kv_dtype = s->kv_dtype;
    L.pdl = use_pdl();
    L.cluster = plan.cluster ? plan.num_parts : 1;
    const bool compact = plan.tile_qr == kTileCompactQRows;
    if (compact && (s->head_dim != 256 || rows > kTileCompactQRows)) return PA_ERR_UNSUPPORTED;
    if (plan.cluster && !tile_cluster_fits(s, plan.tile_qr)) return PA_ERR_UNSUPPORTED;
    p.balanced = plan.balanced ? 1 : 0;
    p.persistent = plan.persistent ? 1 : 0;
    if (plan.balanced) {
        if (!compact || plan.cluster) return PA_ERR_UNSUPPORTED;
        p.final_out = 0;
        L.grid = dim3((unsigned)plan.num_ctas);
    } else if (plan.persistent) {
        if (plan.cluster || plan.num_parts > 1 || tile_q_bufs(s->head_dim, plan.tile_qr) != 2)
            return PA_ERR_UNSUPPORTED;
        p.final_out = 1;
        L.grid = dim3((unsigned)plan.num_ctas);
    } else {
        L.grid = dim3((unsigned)plan.num_parts, (unsigned)grid_y, (unsigned)s->batch);
    }
    if (plan.balanced || plan.persistent) {
        st = encode_q_map(s, q, q_len, plan.tile_qr, &L.tmap_q);
        if (st != PA_OK) return st;
    }
    L.threads = kTileThreads;
    L.smem_bytes = tile_smem_layout(s->head_dim, s->block_size, plan.tile_qr).total + kSmemAlignSlack;
    cudaError_t e;
    switch (s->head_dim) {
        case 64: e = launch_tile_d64(L, stream); break;
        case 128: e = launch_tile_d128(L, stream); break;
        default: e = compact ? launch_tile_d256_compact(L, stream) : launch_tile_d256(L, stream); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_set_switch(int32_t which, int32_t value) {
    switch (which) {
        case PA_SWITCH_MULTI_KERNEL:
            if (value != PA_KERNEL_AUTO && value != PA_KERNEL_MMA && value != PA_KERNEL_TILE)
                return PA_ERR_INVALID_ARG;
            g_switch_multi_kernel.store(value, std::memory_order_relaxed);
            return PA_OK;
        case PA_SWITCH_TILE_COMPACT_Q:
            if (value != 0 && value != 1) return PA_ERR_INVALID_ARG;
            g_switch_compact_q.store(value, std::memory_order_relaxed);
            return PA_OK;
    }
    return PA_ERR_INVALID_ARG;
}

int32_t pa_get_switch(int32_t which) {
    switch (which) {
        case PA_SWITCH_MULTI_KERNEL: return g_switch_multi_kernel.load(std::memory_order_relaxed);
        case PA_SWITCH_TILE_COMPACT_Q: return g_switch_compact_q.load(std::memory_order_relaxed);
    }
    return -1;
}

const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_TIMEOUT: return "kernel wait timed out";
    }
    return "unknown status";
}

int32_t pa_choose_partition_tokens(const pa_shape* shape, int32_t max_context_len,
                                   int32_t num_sms) {
    if (check_shape(shape) != PA_OK || max_context_len < 0 || num_sms <= 0) return 0;
    const Plan plan = auto_plan(shape, max_context_len, num_sms);
    if (plan.balanced) return PA_PARTITION_BALANCED;
    return plan.part_pages * shape->block_size;
}

size_t pa_workspace_size(const pa_shape* shape, int32_t max_context_len,
                         int32_t partition_tokens) {
    return pa_workspace_size_multi(shape, 1, max_context_len, partition_tokens);
}

pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens,
                    const pa_shape* shape, float scale, void* stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!scale_ok(scale)) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    st = check_ptrs(out, q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    int32_t* err = nullptr;
    int sms = 0;
    st = device_state(&sms, &err);
    if (st != PA_OK) return st;
    Plan plan{shape->max_blocks_per_seq, 1, false,
              (int64_t)shape->batch * shape->num_kv_heads > sms, false, 0, false, kTileRows, false};
    return launch_attention(out, q, k_cache, v_cache, block_tables, context_lens, shape, scale,
                            plan, nullptr, nullptr, err, static_cast<cudaStream_t>(stream));
}

pa_status pa_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          const pa_shape* shape, int32_t q_len, float scale,
                          int32_t max_context_len, int32_t partition_tokens, void* workspace,
                          size_t workspace_bytes, void* stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (q_len < 1 || !scale_ok(scale)) return PA_ERR_INVALID_ARG;
    if (max_context_len < 0 || !partition_arg_ok(shape, partition_tokens)) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    st = check_ptrs(out, q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    int sms = 0;
    int32_t* err = nullptr;
    st = device_state(&sms, &err);
    if (st != PA_OK) return st;
    const Plan plan = make_plan(shape, max_context_len, partition_tokens, sms, q_len);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (plan.tile && !plan.balanced && (plan.num_parts <= 1 || plan.cluster))
        return launch_tile(out, q, k_cache, v_cache, block_tables, context_lens, shape, scale, plan,
                           nullptr, nullptr, err, cs, q_len);
    if (!plan.tile && !plan.balanced && (plan.num_parts <= 1 || plan.cluster))
        return launch_attention(out, q, k_cache, v_cache, block_tables, context_lens, shape, scale,
                                plan, nullptr, nullptr, err, cs, q_len);

    size_t ml_off = 0;
    const size_t need = workspace_bytes_for(shape, plan, &ml_off, q_len);
    if (!workspace || !aligned(workspace, 16) || workspace_bytes < need) return PA_ERR_WORKSPACE;
    if ((size_t)plan.num_parts * 2 * sizeof(float) > 200u * 1024u) return PA_ERR_UNSUPPORTED;
    if ((int64_t)q_len * shape->num_heads > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    float* part_acc = static_cast<float*>(workspace);
    float* part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ml_off);
    st = plan.tile ? launch_tile(out, q, k_cache, v_cache, block_tables, context_lens, shape, scale,
                                 plan, part_acc, part_ml, err, cs, q_len)
                   : launch_attention(out, q, k_cache, v_cache, block_tables, context_lens, shape,
                                      scale, plan, part_acc, part_ml, err, cs, q_len);
    if (st != PA_OK) return st;
    CombineParams c;
    c.out = out;
    c.context_lens = context_lens;
    c.part_acc = part_acc;
    c.part_ml = part_ml;
    c.batch = shape->batch;
    c.num_heads = shape->num_heads;
    c.num_kv_heads = shape->num_kv_heads;
    c.group = shape->num_heads / shape->num_kv_heads;
    c.max_blocks = shape->max_blocks_per_seq;
    c.block_size = shape->block_size;
    c.q_len = q_len;
    c.part_pages = plan.part_pages;
    c.num_parts = plan.num_parts;
    c.out_dtype = shape->out_dtype;
    c.num_ctas = plan.num_ctas;
    const dim3 cgrid((unsigned)(q_len * shape->num_heads), (unsigned)shape->batch);
    const cudaError_t e = plan.balanced ? launch_combine_balanced(c, shape->head_dim, cgrid,
                                                                  use_pdl(), cs)
                                        : launch_combine(c, shape->head_dim, cgrid, use_pdl(), cs);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_splitkv(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            const pa_shape* shape, float scale, int32_t max_context_len,
                            int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                            void* stream) {
    return pa_decode_multi(out, q, k_cache, v_cache, block_tables, context_lens, shape, 1, scale,
                           max_context_len, partition_tokens, workspace, workspace_bytes, stream);
}

pa_status pa_plan_info(const pa_shape* shape, int32_t q_len, int32_t max_context_len,
                       int32_t partition_tokens, pa_plan_desc* desc) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!desc || q_len < 1 || max_context_len < 0 || !partition_arg_ok(shape, partition_tokens))
        return PA_ERR_INVALID_ARG;
    int sms = 1;
    st = query_sms(partition_tokens, &sms);
    if (st != PA_OK) return st;
    const Plan plan = make_plan(shape, max_context_len, partition_tokens, sms, q_len);
    const int64_t G = shape->num_heads / shape->num_kv_heads;
    desc->kernel = plan.tile ? 1 : 0;
    desc->partitions = plan.num_parts;
    desc->partition_tokens =
        plan.num_parts <= 1 ? pages_for(shape, max_context_len) * shape->block_size
                            : plan.part_pages * shape->block_size;
    desc->reduce = plan.balanced ? 3 : (plan.num_parts <= 1 ? 0 : (plan.cluster ? 1 : 2));
    if (plan.tile) {
        const int64_t tiles = ((int64_t)q_len * G + kTileRows - 1) / kTileRows;
        desc->ctas = (plan.balanced || plan.persistent) ? plan.num_ctas
                                   : (int32_t)((int64_t)shape->batch * shape->num_kv_heads * tiles *
                                               plan.num_parts);
        desc->threads = kTileThreads;
    } else {
        const Tune t = pick_tune(shape, plan.many_ctas);
        desc->ctas = (plan.balanced || plan.persistent) ? plan.num_ctas
                                   : (int32_t)((int64_t)shape->batch * shape->num_kv_heads *
                                               q_chunks_for(shape, q_len) * plan.num_parts);
        desc->threads = 32 * t.nt * t.nh;
    }
    return PA_OK;
}

size_t pa_workspace_size_multi(const pa_shape* shape, int32_t q_len, int32_t max_context_len,
                               int32_t partition_tokens) {
    if (check_shape(shape) != PA_OK || max_context_len < 0 || q_len < 1) return 0;
    if (!partition_arg_ok(shape, partition_tokens)) return 0;
    int sms = 1;
    if (query_sms(partition_tokens, &sms) != PA_OK) return 0;
    const Plan plan = make_plan(shape, max_context_len, partition_tokens, sms, q_len);
    return workspace_bytes_for(shape, plan, nullptr, q_len);
}

pa_status pa_resolve_blocks(int32_t* out_phys, const int32_t* block_tables,
                            const int32_t* context_lens, const pa_shape* shape, void* stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (!out_phys || !block_tables || !context_lens || !aligned(out_phys, 4) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_resolve(out_phys, block_tables, context_lens, shape->batch,
                                         shape->max_blocks_per_seq, shape->block_size,
                                         shape->num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_append_kv(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                       const int32_t* block_tables, const int32_t* positions,
                       const pa_shape* shape, void* stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !block_tables || !positions)
        return PA_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(block_tables, 4) || !aligned(positions, 4))
        return PA_ERR_INVALID_ARG;
    int sms = 0;
    st = device_state(&sms, nullptr);
    if (st != PA_OK) return st;
    const int32_t row_bytes = shape->num_kv_heads * shape->head_dim * 2;
    return launch_append(k_cache, v_cache, k_new, v_new, block_tables, positions, shape->batch,
                         shape->max_blocks_per_seq, shape->block_size, shape->num_blocks,
                         row_bytes, use_pdl(), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 5000000000ull) return PA_ERR_INVALID_ARG;
    int32_t* err = nullptr;
    pa_status st = device_state(nullptr, &err);
    if (st != PA_OK) return st;
    return launch_wait_timeout(err, timeout_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_device_error(int32_t* code, void* stream) {
    if (!code) return PA_ERR_INVALID_ARG;
    int32_t* err = nullptr;
    pa_status st = device_state(nullptr, &err);
    if (st != PA_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), cs) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return PA_ERR_CUDA;
    *code = v;
    return PA_OK;
}

pa_status pa_decode_splitkv_noalloc(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, const pa_shape* shape,
                                    float scale, int32_t max_context_len,
                                    int32_t partition_tokens, void* stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (!scale_ok(scale)) return PA_ERR_INVALID_ARG;
    if (max_context_len < 0 || !partition_arg_ok(shape, partition_tokens)) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    st = check_ptrs(out, q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    int sms = 0;
    st = device_state(&sms, nullptr);
    if (st != PA_OK) return st;
    const Plan plan = make_plan(shape, max_context_len, partition_tokens, sms);
    if (workspace_bytes_for(shape, plan, nullptr) > kNoAllocScratchBytes)
        return PA_ERR_WORKSPACE;  // more partials than the fixed scratch holds

    // Device address of this device's copy of the scratch array, looked up
    // once per device with that device current (the caller's current device).
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    void* scratch = g_noalloc_scratch[dev].load(std::memory_order_acquire);
    if (!scratch) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, pa_noalloc_scratch) != cudaSuccess || !ptr)
            return PA_ERR_CUDA;
        g_noalloc_scratch[dev].store(ptr, std::memory_order_release);
        scratch = ptr;
    }
    // The partials need no clearing: every partition inside a sequence's
    // context writes its (m, l, acc) before the combine reads it, and the
    // combine never reads partitions past the context.
    return pa_decode_splitkv(out, q, k_cache, v_cache, block_tables, context_lens, shape, scale,
                             max_context_len, partition_tokens, scratch, kNoAllocScratchBytes,
                             stream);
}

}  // extern "C"
