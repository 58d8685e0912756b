// Device helpers of the decode library: the page walk, mbarrier / TMA /
// cluster inline PTX with bounded waits, and the warp-level MMA pieces.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Page walk (MiniVLLM docs "Decoding Benchmark", "Block table lookup
// mechanics"): logical page j of a sequence lives in physical block
// block_tables[b][j].  A page holds attended tokens only if j < npages; an
// entry that is -1 or outside [0, num_blocks) is masked and never read.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int reachable_tokens(const int32_t* context_lens, int b, int max_blocks,
                                                int block_size) {
    int t = __ldg(context_lens + b);
    const int cap = max_blocks * block_size;
    t = t < 0 ? 0 : t;
    return t > cap ? cap : t;
}

__device__ __forceinline__ int page_phys(const int32_t* table_row, int j, int npages,
                                         int64_t num_blocks) {
    if (j >= npages) return -1;
    const int e = __ldg(table_row + j);
    return (e >= 0 && (int64_t)e < num_blocks) ? e : -1;
}

// ---------------------------------------------------------------------------
// mbarrier / TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `timeout_ns`.
// Returns false on timeout; the caller records the error and abandons work.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && global_timer_ns() - start > timeout_ns) return false;
    }
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-D tiled TMA load into shared memory; completion is signalled on `bar`
// as transaction bytes.  Coordinates are innermost first.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
        "l"(policy)
        : "memory");
}

// 3-D tiled TMA load into shared memory (no L2 policy); completion is
// signalled on `bar` as transaction bytes.  Coordinates are innermost first.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// Eight floats in one 32-byte store (sm_100 and later): a whole L2 sector per
// lane.  dst must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(float* dst, const float* v) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "f"(v[0]),
                 "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

// L2 policy for data read exactly once per step: evict it first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for data that other CTAs read again shortly: the default priority.
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor in the stream
// is finishing; it must wait here before touching memory the predecessor may
// write.  Without that attribute the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel in the stream to begin launching (it still waits for
// this grid's completion before it reads anything this grid writes).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void record_error(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core pieces: ldmatrix from shared memory and the
// m16n8k16 MMA with fp32 accumulation, for fp16 and bf16 operands.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// 2^x on the special-function unit (relative error ~2^-22; -inf -> +0).
// max(a, b, c) in one instruction (three-operand max, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Thread-block cluster barrier.  arrive.release / wait.acquire publishes this
// CTA's shared-memory writes to the cluster; the relaxed form only waits.
__device__ __forceinline__ void cluster_sync_release_acquire() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::
                     : "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster,
// and a load through it (distributed shared memory).
__device__ __forceinline__ uint32_t map_cluster_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_cluster_v4f32(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

template <typename KV>
struct Mma;

template <>
struct Mma<__half> {
    // c += a (16x16, row major) * b (16x8, column major)
    static __device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // x0 in the low half, x1 in the high half, round to nearest even
    static __device__ __forceinline__ uint32_t pack(float x0, float x1) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x1), "f"(x0));
        return r;
    }
    static __device__ __forceinline__ void unpack(uint32_t v, float& x0, float& x1) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
        x0 = f.x;
        x1 = f.y;
    }
    // (l + x0) + x1 for the two packed values, each widened exactly inside a
    // mixed-precision add (f16 operand, f32 sum: one instruction apiece)
    static __device__ __forceinline__ float add2(uint32_t v, float l) {
        asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
            "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %0, hi, %0;\n\t}"
            : "+f"(l)
            : "r"(v));
        return l;
    }
};

template <>
struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float x0, float x1) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x1), "f"(x0));
        return r;
    }
    static __device__ __forceinline__ void unpack(uint32_t v, float& x0, float& x1) {
        x0 = __uint_as_float(v << 16);
        x1 = __uint_as_float(v & 0xffff0000u);
    }
};

// Store one fp32 value as the output dtype.
__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int out_dtype) {
    if (out_dtype == PA_F32) {
        static_cast<float*>(out)[idx] = v;
    } else if (out_dtype == PA_F16) {
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
    } else {
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    }
}

}  // namespace pa
