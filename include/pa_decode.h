/*
 * pa_decode.h -- C ABI of the GB300 (sm_103a) paged-attention decode library
 * (libpa_decode.so).
 *
 * The operation.  One decode step: every sequence b of a batch has one query
 * token q[b, h, :] per query head h; it attends over the keys and values of
 * its context_lens[b] cached tokens, which live in a pool of fixed-size
 * physical blocks reached through a per-sequence block table:
 *
 *   out[b, h, :] = sum_t softmax_t(scale * q[b, h, :] . K_t) * V_t
 *   K_t = k_cache[block_tables[b][t / block_size], t % block_size, kvh, :]
 *   kvh = h / (num_heads / num_kv_heads)       (grouped-query heads)
 *
 * Sources: MiniVLLM docs "Decoding Benchmark" (sections "What paged attention
 * decode does" and "Block table lookup mechanics"); "benchmark_decoding.py"
 * (reference_output: the float32 definition; setup_test_data: the layouts;
 * the Triton (new) kernel: head grouping and masking of -1 entries);
 * flash-decoding-bench "design.md" (Flash-Decoding: split the KV sequence into
 * chunks processed in parallel, each producing a local max, sum and weighted
 * value sum, then reduce the partials into the output).
 *
 * Layouts (all row-major, contiguous, device memory owned by the caller):
 *   q            [batch, num_heads, head_dim]                      kv_dtype
 *   k_cache      [num_blocks, block_size, num_kv_heads, head_dim]  kv_dtype
 *   v_cache      same shape and dtype as k_cache
 *   block_tables [batch, max_blocks_per_seq]                       int32, -1 = unallocated
 *   context_lens [batch]                                           int32
 *   out          [batch, num_heads, head_dim]                      out_dtype
 *
 * Semantics at the edges (the pages are silent or disagree; this library and
 * its tests take these readings):
 *   - tokens t >= max_blocks_per_seq * block_size are unreachable and ignored;
 *     a negative context length counts as 0;
 *   - a table entry inside the used range that is -1 or outside
 *     [0, num_blocks) excludes its tokens from the softmax (never read);
 *   - a sequence with no attended token gets an all-zero output row.
 *
 * Arithmetic: scores, the online softmax (running max m and normaliser l) and
 * the value accumulation are fp32; K/V/q are fp16 or bf16.  `scale` must be
 * finite and > 0 (PA_ERR_INVALID_ARG otherwise).
 *
 * Calls.  All entry points validate on the host and either launch work on
 * `stream` (a cudaStream_t; NULL = the legacy default stream) and return
 * PA_OK immediately, or return an error status and launch nothing.  A
 * PA_ERR_CUDA status means the launch itself failed.  The library allocates no
 * device memory.  Entry points may be called from several host threads; the
 * shared state is a per-device cache of the SM count, of the device error
 * word's address and of which cluster sizes fit, per-thread caches of tensor
 * maps, and the two test switches of pa_set_switch.  No call reads the
 * environment (the tuning variables are read once, when the library loads).
 *
 * Supported shapes: head_dim in {64, 128, 256}; block_size in {16, 32};
 * num_heads / num_kv_heads in {1, 2, 4, 8, 16}; kv_dtype fp16 or bf16; out_dtype
 * fp32 or equal to kv_dtype; every pointer 16-byte aligned.  Anything else
 * returns PA_ERR_UNSUPPORTED (or PA_ERR_INVALID_ARG for inconsistent values).
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null pointer, inconsistent or negative sizes */
    PA_ERR_UNSUPPORTED = 2, /* a shape or dtype this library has no kernel for */
    PA_ERR_WORKSPACE = 3,   /* split-KV workspace missing, misaligned or too small */
    PA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    PA_ERR_TIMEOUT = 5      /* a kernel gave up waiting on its own copy pipeline */
} pa_status;

typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2 } pa_dtype;

/* partition_tokens value requesting the balanced split: one CTA per SM, each
 * taking an equal share of all (sequence, kv head, page) triples in order,
 * pieces of a (sequence, kv head) that straddle CTAs combined afterwards.
 * Needs batch <= 512 (otherwise the automatic choice is used). */
#define PA_PARTITION_BALANCED (-1)

typedef struct pa_shape {
    int32_t batch;              /* B >= 0 (B = 0 launches nothing) */
    int32_t num_heads;          /* H, query heads */
    int32_t num_kv_heads;       /* Hkv, H % Hkv == 0 */
    int32_t head_dim;           /* D */
    int32_t block_size;         /* tokens per physical block */
    int32_t max_blocks_per_seq; /* columns of block_tables */
    int64_t num_blocks;         /* physical blocks in the pool, < 2^31 */
    int32_t kv_dtype;           /* pa_dtype of q, k_cache, v_cache: PA_F16 or PA_BF16 */
    int32_t out_dtype;          /* pa_dtype of out: PA_F32 or kv_dtype */
} pa_shape;

/*
 * Single-pass decode ("benchmark_decoding.py", reference_output and the
 * Triton (new) kernel; MiniVLLM docs "Decoding Benchmark", "Why CUDA chunk
 * processing matters"): one CTA per (sequence, kv head) walks all of that
 * sequence's pages, one block-table read per page, with an fp32 online
 * softmax, and writes out[b, h, :] for the head group.
 * Arguments: device pointers as laid out above; `scale` multiplies q.K
 * (1/sqrt(head_dim) in the pages' set-up); `stream` is a cudaStream_t.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens,
                    const pa_shape* shape, float scale, void* stream);

/*
 * Bytes of device workspace pa_decode_splitkv needs for this shape, longest
 * context `max_context_len` and partition size `partition_tokens` (tokens per
 * split, a multiple of block_size; 0 = choose automatically for the current
 * device; PA_PARTITION_BALANCED = the balanced split).  Returns 0 for invalid
 * arguments and when no workspace is needed (one partition, or partitions
 * reduced inside a thread-block cluster: see pa_decode_splitkv).  The answer
 * is for the current device, as the call plans with its SM count (which picks
 * the CTA shape and with it whether a cluster split fits); an explicit
 * partition size may be queried without a device, and is then sized as for
 * one SM.  A size that does not fit in a size_t is reported as SIZE_MAX, which
 * no workspace satisfies (the call is then refused with PA_ERR_WORKSPACE).
 */
size_t pa_workspace_size(const pa_shape* shape, int32_t max_context_len,
                         int32_t partition_tokens);

/*
 * Partition size (tokens) the automatic choice picks for `num_sms`
 * multiprocessors: a multiple of block_size (a result >= max_context_len
 * means "no split"), or PA_PARTITION_BALANCED when it picks the balanced
 * split; 0 for invalid arguments.  A function of its arguments, exported so
 * that the choice can be checked without a GPU, with one exception: which
 * cluster sizes fit on the device at once is asked of the current device
 * when there is one (cached per device); without a device, clusters of up to
 * 8 CTAs are assumed to fit.  Launches nothing.
 * The rules are this library's own, fitted to GB300 timings: the
 * flash-decoding-bench design notes only say that the chunk size is picked
 * from the KV length.
 */
int32_t pa_choose_partition_tokens(const pa_shape* shape, int32_t max_context_len,
                                   int32_t num_sms);

/*
 * Flash-Decoding split-KV decode (flash-decoding-bench "design.md": the KV
 * cache is split into chunks, one thread block each, each computing its local
 * max, sum and weighted value sum, followed by a reduction of the partials).
 * Each (sequence, kv head) is cut into partitions of `partition_tokens` tokens
 * (or, with PA_PARTITION_BALANCED, the flattened pages of all of them are cut
 * into one equal share per SM, and a piece that straddles two shares leaves
 * a partial record for the combine kernel);
 * one CTA per partition computes fp32 partials (m, l, acc[head_dim]) for each
 * query head of the group.  The partitions of a (sequence, kv head) are
 * launched as one thread-block cluster and reduced through distributed
 * shared memory inside the same kernel (no workspace needed) when there are
 * at most 8 of them (up to 16 for the automatic choice) and the device can
 * hold every cluster of the call at once; otherwise they write their
 * partials to `workspace` and a second kernel combines them with a
 * log-sum-exp reduction into out.  pa_workspace_size reports which.  `max_context_len` must be >= every context_lens[b] that
 * should be attended in full (tokens beyond it are dropped; no device->host
 * read is made); `partition_tokens` = 0 chooses the split automatically, and a
 * choice of one partition runs the single pass.  `workspace` (device, 16-byte
 * aligned) must hold at least pa_workspace_size(shape, max_context_len,
 * partition_tokens) bytes (may be NULL when that is 0); it is scratch owned by
 * the caller and may be reused once the stream has passed this call.
 * Kernel choice: groups of 16 query heads at head_dim 256 run on the tcgen05
 * tile kernel described at pa_decode_multi (its own split, from the device's
 * resident clusters); every other shape on the warp-level kernel, whose split
 * pa_choose_partition_tokens reports.  PA_PARTITION_BALANCED always runs the
 * warp-level kernel.
 */
pa_status pa_decode_splitkv(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            const pa_shape* shape, float scale, int32_t max_context_len,
                            int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * Several query tokens per sequence in one call: the decode step of
 * speculative decoding's verification, or a short chunk of new tokens (the
 * pages define only the one-token decode; this is its causal extension, the
 * q_len > 1 attention that the flash-decoding-bench design notes contrast
 * with the q_len = 1 decode).  Layouts:
 *   q    [batch, q_len, num_heads, head_dim]  kv_dtype
 *   out  [batch, q_len, num_heads, head_dim]  out_dtype
 * context_lens[b] counts the q_len new tokens, whose keys and values are
 * already in the cache at positions T - q_len .. T - 1 (T = context_lens[b]).
 * Query token i sits at position T - q_len + i and attends to the tokens
 * t <= T - q_len + i that the table reaches, with the same masking as
 * pa_decode; a query token with no such token gets zeros.  With q_len = 1
 * this is pa_decode_splitkv.
 *
 * Rows.  A (sequence, kv head) has q_len * group rows, one per (query token,
 * head) pair.  Up to 16 rows (except exactly 16 at head_dim 256) the
 * warp-level kernel serves them: its MMA tile's 16 rows hold the pairs, one
 * CTA per floor(16 / group) query tokens of a kv head and partition.  Beyond
 * that the tcgen05 tile kernel serves them: 384-thread CTAs of 128 rows (one
 * per ceil(q_len * group / 128) tiles of a kv head and partition) with
 * Q K^T and P V on the tensor cores (operands staged by TMA in shared memory,
 * S and O accumulated in tensor memory), the online softmax on two
 * warpgroups, and its partitions sized from the device's resident clusters.
 * Either way every CTA of a (sequence, kv head) reads that sequence's pages
 * again, and num_kv_heads times the CTA count per kv head must be <= 65535
 * (else PA_ERR_UNSUPPORTED).  Partitions, workspace and max_context_len as in
 * pa_decode_splitkv; PA_PARTITION_BALANCED is honoured only when
 * q_len * group <= 16 (otherwise the automatic choice is used).  The
 * workspace must hold pa_workspace_size_multi(shape, q_len, ...) bytes.
 * pa_plan_info reports the kernel and split a call will use.
 */
pa_status pa_decode_multi(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens,
                          const pa_shape* shape, int32_t q_len, float scale,
                          int32_t max_context_len, int32_t partition_tokens, void* workspace,
                          size_t workspace_bytes, void* stream);

/* How a split-KV call (pa_decode_splitkv / pa_decode_multi) with these
 * arguments runs on the current device; filled by pa_plan_info. */
typedef struct pa_plan_desc {
    int32_t kernel;           /* 0: warp-level m16n8k16 kernel; 1: tcgen05 tile kernel */
    int32_t partitions;       /* partitions per (sequence, kv head[, query chunk / tile]) */
    int32_t partition_tokens; /* tokens per partition (the longest context for one) */
    int32_t reduce;           /* 0: none (one pass); 1: cluster (distributed shared
                                 memory); 2: workspace + combine kernel; 3: balanced split */
    int32_t ctas;             /* CTAs of the attention kernel */
    int32_t threads;          /* threads per CTA */
} pa_plan_desc;

/* Describes, without launching anything, the plan a split-KV call with these
 * arguments would use on the current device (no counterpart in the pages: a
 * diagnostic of this library's own choices).  Automatic and balanced choices
 * need the device, as the calls do; an explicit partition size may be
 * queried without one (planned as for one SM).  Returns PA_ERR_INVALID_ARG /
 * PA_ERR_UNSUPPORTED like the calls, else PA_OK. */
pa_status pa_plan_info(const pa_shape* shape, int32_t q_len, int32_t max_context_len,
                       int32_t partition_tokens, pa_plan_desc* desc);

/* Workspace bytes of pa_decode_multi (0 for invalid arguments or when none is
 * needed); pa_workspace_size(shape, ...) is this with q_len = 1. */
size_t pa_workspace_size_multi(const pa_shape* shape, int32_t q_len, int32_t max_context_len,
                               int32_t partition_tokens);

/*
 * Append of each sequence's new token to the paged cache, the step that
 * precedes attention in every decode iteration (MiniVLLM docs "Decoding
 * Benchmark", "What paged attention decode does": the cache is a pool of
 * blocks allocated on demand, token t of sequence b in block
 * block_tables[b][t / block_size] at slot t % block_size).  For each b with
 * 0 <= positions[b] < max_blocks_per_seq * block_size and a table entry in
 * [0, num_blocks): k_cache[entry][positions[b] % block_size][:][:] =
 * k_new[b][:][:], and likewise v_cache from v_new.  Other sequences (padding:
 * a negative position; a masked entry) write nothing.  k_new, v_new:
 * [batch, num_kv_heads, head_dim] in kv_dtype, 16-byte aligned; positions:
 * [batch] int32.  Launched with programmatic stream serialization, so a
 * decode call queued right after it overlaps its launch and still sees every
 * write.  Bit-exact (a copy).
 */
pa_status pa_append_kv(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                       const int32_t* block_tables, const int32_t* positions,
                       const pa_shape* shape, void* stream);

/*
 * Test export of the page walk (MiniVLLM docs "Decoding Benchmark", "Block
 * table lookup mechanics"): out_phys[b][j] (device, int32, [batch,
 * max_blocks_per_seq]) = the physical block the decode kernels read for
 * logical page j of sequence b, or -1 where that page holds no attended token
 * (beyond the context, or a masked entry).  Uses the kernels' own page-walk
 * code.
 */
pa_status pa_resolve_blocks(int32_t* out_phys, const int32_t* block_tables,
                            const int32_t* context_lens, const pa_shape* shape, void* stream);

/*
 * Reads and clears the current device's error word, which a kernel sets when
 * a bounded wait on its own copy pipeline runs out (it then abandons the
 * work and returns instead of hanging).  Synchronises `stream`.  *code is 0
 * or the pa_status the kernel recorded.
 */
pa_status pa_device_error(int32_t* code, void* stream);

/*
 * pa_decode_splitkv without a caller-supplied workspace, for callers that
 * cannot allocate device memory: for instance code that runs inside a host
 * application which hands it only fixed input/output buffers and forbids
 * further allocation, or a latency-critical loop that must not pay for
 * cudaMalloc's device-wide synchronisation.  (The pages have no counterpart;
 * this is a convenience of this library.)
 *
 * The split-KV partials go to a fixed scratch array inside the library, 16 MiB
 * of device memory on every GPU that loads it, held until the process exits.
 * A call whose partials need more than that -- batch * num_heads * partitions
 * * (head_dim + 2) * 4 bytes, plus alignment -- returns PA_ERR_WORKSPACE and
 * launches nothing; use pa_decode_splitkv with your own workspace then.  The
 * call allocates nothing and needs no clearing of the scratch.
 *
 * The first call on a device looks up that device's scratch address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * All calls on a device share the one array, which keeps the last call's
 * contents: two calls that can run at the same time on the GPU (different
 * streams without ordering between them) race on it and both results are then
 * undefined.  Other arguments and behaviour are those of pa_decode_splitkv.
 */
pa_status pa_decode_splitkv_noalloc(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, const pa_shape* shape,
                                    float scale, int32_t max_context_len,
                                    int32_t partition_tokens, void* stream);

/*
 * Test export of the kernels' failure path (no counterpart in the pages): one
 * CTA waits, with the decode kernels' bounded wait, on an mbarrier that nothing
 * ever completes; after `timeout_ns` (1 ns .. 5 s) it gives up and records
 * PA_ERR_TIMEOUT in the device error word, which pa_device_error then returns.
 * The context stays usable.  Asynchronous on `stream`.
 */
pa_status pa_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Test and tuning switches (no counterpart in the pages: they choose between
 * this library's own kernels, whose results agree up to rounding order).
 *   PA_SWITCH_MULTI_KERNEL    PA_KERNEL_AUTO (default): the library's choice;
 *                             PA_KERNEL_MMA: the warp-level kernel for every
 *                             q_len > 1 call; PA_KERNEL_TILE: the tcgen05 tile
 *                             kernel for every split-KV / multi-token call
 *   PA_SWITCH_TILE_COMPACT_Q  1 (default): the tile kernel stages only 16 Q rows
 *                             for units of at most 16 rows at head_dim 256;
 *                             0: it stages whole 128-row tiles
 * The initial values come from the environment variables PA_MULTI_KERNEL
 * (mma | tile) and PA_TILE_COMPACT_Q (0), read once when the library is
 * loaded; no call reads the environment.  pa_set_switch changes a switch for
 * every later call of the process (a relaxed atomic store: set it while no
 * other host thread is between a pa_workspace_size query and the call it
 * sizes).  Returns PA_ERR_INVALID_ARG for an unknown switch or value.
 * pa_get_switch returns the current value, -1 for an unknown switch.
 */
enum { PA_SWITCH_MULTI_KERNEL = 0, PA_SWITCH_TILE_COMPACT_Q = 1 };
enum { PA_KERNEL_AUTO = 0, PA_KERNEL_MMA = 1, PA_KERNEL_TILE = 2 };
pa_status pa_set_switch(int32_t which, int32_t value);
int32_t pa_get_switch(int32_t which);

/* Static, human-readable name of a status. */
const char* pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
