/*
 * carat.h -- C ABI of libcarat.so: sliding-window ring-buffer KV cache and
 * grouped-query attention for Gemma-4-style decoding and speculative verify,
 * written for one NVIDIA GB300 (sm_103a).
 *
 * Two parts, as the pages describe them:
 *
 *  1. Sliding-window layers keep each request's K and V history in a fixed
 *     ring of `window` slots (1024 for Gemma 4).  A token's slot is its
 *     absolute position modulo the window, and a new token overwrites the
 *     slot of the token one window older, with nothing shifted
 *     ("Announcing Carat: An inference engine designed for Gemma 4", section
 *     "Replacing page lookups with a ring buffer").  K and V are written in
 *     lockstep, so both rings share one rotation, and attention reads the
 *     rotated rings in place: attention does not depend on a common
 *     reordering of K and V ("Improving Decode Throughput on Intel Gaudi 3",
 *     section "Our approach").
 *
 *  2. Global layers keep the full history in a zero-initialised cache.  Their
 *     speculative-verify attention groups the query heads that share one KV
 *     head together with all proposal positions into one tile of rows
 *     (8 heads x 4 positions = 32 rows for Gemma 4), computes QK^T, a causal
 *     softmax and PV, and masks the key tail past key_count
 *     ("Announcing Carat ...", sections "More FLOPs can be faster" and
 *     "Doing it all in one kernel can be slower").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers on the current CUDA device and
 *    must be 16-byte aligned.  `stream` is a cudaStream_t passed as void*
 *    (NULL = the legacy default stream).  Every call is asynchronous on that
 *    stream; nothing synchronises the host.
 *  - bf16 tensors are raw IEEE bfloat16; outputs are fp32.  Layouts are dense
 *    row-major in the order written next to each argument.
 *  - The caller owns every buffer, including the workspace; the library
 *    allocates no device memory and keeps no state across calls except one
 *    device status word per GPU (carat_get_device_status), whose device
 *    address is looked up on a device's first call and kept: after
 *    cudaDeviceReset on a device, do not call the library on it again in the
 *    same process.
 *  - Positions.  For request b, context_lengths[b] tokens are in the cache
 *    BEFORE this step; the step's proposal_count new tokens sit at positions
 *    context_lengths[b] + j, j = 0 .. proposal_count-1, and
 *    key_count = context_length + proposal_count (the "More FLOPs" section's
 *    key_count).  Query j of request b is the token at position
 *    context_lengths[b] + j.  Plain decode is proposal_count = 1.
 *  - Grouping.  Query head h reads KV head h / (q_heads / kv_heads).
 *  - Errors.  Nothing aborts and nothing throws across the ABI.  Argument
 *    checks run on the host before any launch and return a status without
 *    touching the GPU.  Values that live in device memory (context lengths,
 *    ring ids) are checked by the kernels: a request with a bad value is
 *    skipped, its outputs are written as NaN, and a bit is set in the device
 *    status word (CARAT_DEV_*).  A failed launch returns CARAT_ERR_CUDA.
 *  - batch == 0 is valid and launches nothing.
 */
#ifndef CARAT_H
#define CARAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum carat_status {
    CARAT_OK = 0,
    CARAT_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, inconsistent sizes */
    CARAT_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, rows per tile */
    CARAT_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    CARAT_ERR_CUDA = 4           /* a CUDA runtime call or launch failed */
} carat_status;

/* Bits of the device status word. */
#define CARAT_DEV_BAD_CONTEXT 0x1 /* context_length < 0, or key_count > capacity */
#define CARAT_DEV_BAD_CACHE_ID 0x2 /* ring/cache id outside [0, num_rings) */
#define CARAT_DEV_TIMEOUT 0x4      /* a kernel gave up waiting (bounded wait); results invalid */

/* Largest proposal_count the attention entry points accept. */
#define CARAT_MAX_PROPOSALS 16
/* Largest (q_heads / kv_heads) * proposal_count, the rows of one tile. */
#define CARAT_MAX_TILE_ROWS 128

/*
 * carat_ring_append -- write this step's new K and V rows into a ring.
 *
 * Source: "Announcing Carat ...", "Replacing page lookups with a ring
 * buffer" (slot = position mod window; a new token reuses the oldest slot
 * without shifting); "Improving Decode Throughput on Intel Gaudi 3", "Our
 * approach" (for each decoded token the new KV is written and the head moves
 * on by one; K and V in lockstep).
 *
 *   k_ring, v_ring   bf16 [num_rings][window][kv_heads][head_dim]; ring r
 *                    belongs to one request.  Slot s of ring r holds the
 *                    latest position t with t mod window == s.
 *   ring_ids         int32 [batch]: ring of request b; NULL = ring b
 *                    (then num_rings >= batch).
 *   k_new, v_new     bf16 [batch][proposal_count][kv_heads][head_dim]: rows
 *                    for positions context_lengths[b] + j.
 *   context_lengths  int32 [batch]: tokens in the ring before this append.
 *   displaced        bf16 [batch][proposal_count-1][2][kv_heads][head_dim]
 *                    (K then V) or NULL.  When proposal_count > 1 the new
 *                    tokens overwrite slots whose old rows the step's earlier
 *                    queries still attend to; if `displaced` is given, those
 *                    rows (positions context_length - window + 1 + i) are
 *                    copied there first, for carat_swa_attention.  Entries
 *                    whose position is negative are left untouched.
 *   window           ring slots (1024 for Gemma 4's sliding layers).  A
 *                    global-layer cache of `capacity` rows is a ring with
 *                    window = capacity whose positions never wrap.
 *
 * Limits: 1 <= proposal_count <= window; proposal_count <= 16 when
 * displaced != NULL; kv_heads * head_dim * 2 bytes must be a multiple of 16.
 * Appending proposal_count up to `window` rows with displaced == NULL is how a
 * prompt's last `window` tokens are written after prefill.
 */
carat_status carat_ring_append(void *k_ring, void *v_ring, int num_rings,
                               const int32_t *ring_ids,
                               const void *k_new, const void *v_new,
                               const int32_t *context_lengths, int proposal_count,
                               void *displaced,
                               int batch, int kv_heads, int head_dim, int window,
                               void *stream);

/*
 * carat_ring_rollback -- undo the rejected part of a speculative append.
 *
 * After a verify step appended proposal_count rows at positions
 * context_lengths[b] + j (carat_ring_append or carat_swa_append_attention
 * with a `displaced` buffer), the sampler keeps only the first accepted[b]
 * of them.  For every rejected row j >= max(accepted[b], 1) whose slot held a
 * token before the append (position context_lengths[b] + j - window >= 0),
 * the slot's old K and V rows are copied back from displaced[b][j-1].  The
 * ring then holds, for key count context_lengths[b] + accepted[b], the newest
 * token of every slot a later query can see.  (With accepted[b] == 0 the slot
 * of position context_lengths[b] - window is not restored: that position is
 * outside every later window, and the next append overwrites the slot.)
 * Rows of rejected proposals in slots that held no token stay where they are:
 * attention treats such slots as empty for the smaller key count.
 * The pages have no rollback step; the displaced rows are the reading
 * explained at carat_ring_append.  Global caches need no rollback: rows at or
 * past the key count are never read.
 *
 *   accepted   int32 [batch], device memory, 0 <= accepted[b] <=
 *              proposal_count (outside: the request is skipped and
 *              CARAT_DEV_BAD_CONTEXT is set).
 *   Other arguments as in carat_ring_append.  2 <= proposal_count <= 16.
 */
carat_status carat_ring_rollback(void *k_ring, void *v_ring, int num_rings,
                                 const int32_t *ring_ids, const void *displaced,
                                 const int32_t *context_lengths, const int32_t *accepted,
                                 int proposal_count, int batch, int kv_heads, int head_dim,
                                 int window, void *stream);

/*
 * carat_swa_attention -- sliding-window decode / verify attention read
 * straight from the rotated rings (no gather, no un-rotation).
 *
 * Source: "Improving Decode Throughput on Intel Gaudi 3", "Our approach"
 * (both ring buffers go straight into one fused attention kernel) and
 * "Patching sliding window KV allocation" (sliding layers attend to the most
 * recent 1024 tokens).  Query j at position p attends to positions
 * [max(0, p - window + 1), p], its own included.
 *
 *   out              fp32 [batch][proposal_count][q_heads][head_dim]
 *   queries          bf16 [batch][proposal_count][q_heads][head_dim], after
 *                    the positional embedding.
 *   k_ring, v_ring, num_rings, ring_ids   as in carat_ring_append, AFTER
 *                    this step's append.
 *   displaced        as written by carat_ring_append; required (non-NULL)
 *                    when proposal_count > 1, ignored when it is 1.
 *   context_lengths  int32 [batch]: tokens before this step.
 *   scale            softmax scale applied to q.k (e.g. 1/sqrt(head_dim)).
 *   workspace        device scratch of at least carat_swa_workspace_bytes(...)
 *                    bytes, owned by the caller; contents need no
 *                    initialisation and are overwritten.  Calls that overlap on
 *                    the GPU need separate workspaces.
 *
 * Supported: head_dim 256 or 512; (q_heads/kv_heads)*proposal_count <= 128;
 * q_heads/kv_heads <= 64; proposal_count <= 16 and <= window (other shapes:
 * CARAT_ERR_UNSUPPORTED, nothing launched).
 */
carat_status carat_swa_attention(float *out, const void *queries,
                                 const void *k_ring, const void *v_ring, int num_rings,
                                 const int32_t *ring_ids, const void *displaced,
                                 const int32_t *context_lengths, int proposal_count,
                                 int batch, int q_heads, int kv_heads, int head_dim,
                                 int window, float scale,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * carat_global_verify_attention -- grouped-head speculative-verify attention
 * over a full (global-layer) cache.
 *
 * Source: "Announcing Carat ...", "More FLOPs can be faster" (key_count =
 * context_length + proposal_count; QK^T, a causal softmax in which query j
 * ignores every key after its own position, then PV; the cache tail past key_count is
 * zero-initialised and masked, so padding the key dimension changes nothing)
 * and "Doing it all in one kernel can be slower" (the query heads sharing a
 * KV head and all proposal positions form one set of rows against the same
 * cached K and V).
 *
 *   out              fp32 [batch][proposal_count][q_heads][head_dim]
 *   queries          bf16 [batch][proposal_count][q_heads][head_dim]
 *   key_cache, value_cache  bf16 [num_caches][capacity][kv_heads][head_dim]:
 *                    row t of cache c holds position t.  This step's tokens
 *                    must already be appended (e.g. carat_ring_append with
 *                    window = capacity).  Rows past key_count are never read
 *                    into the result.
 *   cache_ids        int32 [batch] or NULL (= cache b; num_caches >= batch).
 *   context_lengths  int32 [batch]; key_count = context_length +
 *                    proposal_count must be <= capacity (checked on device).
 *   workspace        >= carat_global_workspace_bytes(...) bytes, as above.
 *
 * Supported: head_dim 256 or 512; (q_heads/kv_heads)*proposal_count <= 128;
 * q_heads/kv_heads <= 64; proposal_count <= 16 (other shapes:
 * CARAT_ERR_UNSUPPORTED, nothing launched).
 */
carat_status carat_global_verify_attention(float *out, const void *queries,
                                           const void *key_cache, const void *value_cache,
                                           int num_caches, const int32_t *cache_ids,
                                           const int32_t *context_lengths, int proposal_count,
                                           int batch, int q_heads, int kv_heads, int head_dim,
                                           int capacity, float scale,
                                           void *workspace, size_t workspace_bytes,
                                           void *stream);

/*
 * carat_swa_attention_noalloc -- carat_swa_attention without a workspace
 * argument, for callers that cannot allocate device memory: for example a
 * plugin running inside a host runtime that owns all GPU memory and gives its
 * plugins no allocator, or a latency-critical loop that must not call
 * cudaMalloc (which can synchronise the device).  The pages have no
 * counterpart to this entry point; it exists only for such callers.
 *
 * The split-K scratch lives in a fixed device array of
 * CARAT_NOALLOC_SCRATCH_BYTES (32 MiB) inside the library, which every GPU
 * that loads the library keeps reserved until the process exits.  Arguments,
 * layouts and results are those of carat_swa_attention.  Sizes whose
 * carat_swa_workspace_bytes(...) exceeds the array return
 * CARAT_ERR_WORKSPACE without launching anything (e.g. 12 requests with 4
 * proposals at head_dim 256 need about 4 MiB and fit; 8 requests with 16
 * proposals and 8 query heads per KV head at head_dim 512 need about 36 MiB
 * and do not).  Shapes whose workspace size is 0 use no scratch at all.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any
 * stream capture begins.  The cached address belongs to that device's
 * context as it was then: after cudaDeviceReset on a device, do not call this
 * library on that device again in the same process (the status word that
 * every entry point writes is cached the same way).  Every call uses the same array and nothing in it
 * needs to start at zero, but calls that can run at the same time on the GPU
 * (other streams or host threads without ordering between them) race on it:
 * order them on one stream.  No device memory is allocated or freed.
 */
#define CARAT_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
carat_status carat_swa_attention_noalloc(float *out, const void *queries,
                                         const void *k_ring, const void *v_ring,
                                         int num_rings, const int32_t *ring_ids,
                                         const void *displaced,
                                         const int32_t *context_lengths, int proposal_count,
                                         int batch, int q_heads, int kv_heads, int head_dim,
                                         int window, float scale, void *stream);

/* Size in bytes of the built-in scratch array used by
 * carat_swa_attention_noalloc (CARAT_NOALLOC_SCRATCH_BYTES). */
size_t carat_noalloc_scratch_bytes(void);

/*
 * carat_swa_append_attention -- carat_ring_append followed by
 * carat_swa_attention in one launch, without a displaced-row buffer.
 *
 * Same contract as the two calls in sequence (the pages' order: this step's
 * K/V rows are written into the ring, then attention reads the ring in place
 * -- "Improving Decode Throughput on Intel Gaudi 3", "Our approach"), except
 * that the rings are passed as they are BEFORE this step: the kernel reads the
 * old ring contents and this step's rows (k_new, v_new, layout as in
 * carat_ring_append) as keys, and each 128-slot tile of the ring that holds a
 * slot of a new row is overwritten only by the CTA that loads that tile,
 * after its own copy of the tile has landed.  On return (in stream order) the
 * rings hold exactly what carat_ring_append would have written.  When more
 * than 64 rows share a KV head the rows are split over several CTAs per tile;
 * then the new rows are written by a ring append launched right after the
 * attention.  displaced: NULL, or a buffer as in carat_ring_append that
 * receives the rows the new ones overwrite (for carat_ring_rollback).
 * workspace: carat_swa_workspace_bytes(...) bytes.
 * Supported: as carat_swa_attention.
 */
carat_status carat_swa_append_attention(float *out, const void *queries,
                                        void *k_ring, void *v_ring, int num_rings,
                                        const int32_t *ring_ids, void *displaced,
                                        const void *k_new, const void *v_new,
                                        const int32_t *context_lengths, int proposal_count,
                                        int batch, int q_heads, int kv_heads, int head_dim,
                                        int window, float scale,
                                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * carat_global_append_verify_attention -- appending this step's rows to the
 * global caches (rows context_length + j) followed by
 * carat_global_verify_attention, in one launch.  The caches are passed as
 * they are before this step; this step's rows are read from k_new / v_new and
 * written to the caches by the kernel.  context_length + proposal_count must
 * be <= capacity.  workspace: carat_global_workspace_bytes(...) bytes.
 */
carat_status carat_global_append_verify_attention(float *out, const void *queries,
                                                  void *key_cache, void *value_cache,
                                                  int num_caches, const int32_t *cache_ids,
                                                  const void *k_new, const void *v_new,
                                                  const int32_t *context_lengths,
                                                  int proposal_count, int batch, int q_heads,
                                                  int kv_heads, int head_dim, int capacity,
                                                  float scale, void *workspace,
                                                  size_t workspace_bytes, void *stream);

/*
 * Paged global caches in a shared pool.
 *
 * "Improving Decode Throughput on Intel Gaudi 3", "Our approach": the ring
 * buffers are allocated in the same HBM that backs the global-attention pages,
 * as one shared pool, so ring space and page space follow the requests' mix.
 * Here a pool is a bf16 array of num_pages pages; a global layer views it as
 * [num_pages][page_rows][kv_heads][head_dim] and a sliding layer with the same
 * page size in bytes views it as rings of window rows (a ring = an aligned run
 * of pages, ring id = first page / pages per ring), so rings and pages of all
 * layers can share one allocation (see carat_pool_*).  Position t of request
 * b lives in row t % page_rows of page page_table[b][t / page_rows].
 *
 *   page_table  int32 [batch][max_pages], device memory; entries of pages the
 *               request does not use are never read.  A page id outside
 *               [0, num_pages) reads as zeros and sets CARAT_DEV_BAD_CACHE_ID.
 *   page_rows   rows per page, a positive multiple of 128.
 *   Capacity per request: max_pages * page_rows rows.
 */

/* carat_global_append_verify_attention over paged caches (same contract; the
 * new rows are written through the page table).  workspace:
 * carat_global_workspace_bytes(batch, proposal_count, q_heads, kv_heads,
 * head_dim, max_pages * page_rows) bytes. */
carat_status carat_global_append_verify_attention_paged(
    float *out, const void *queries, void *key_pages, void *value_pages, int num_pages,
    const int32_t *page_table, int max_pages, int page_rows, const void *k_new, const void *v_new,
    const int32_t *context_lengths, int proposal_count, int batch, int q_heads, int kv_heads,
    int head_dim, float scale, void *workspace, size_t workspace_bytes, void *stream);

/* Write rows for positions context_lengths[b] + j (j < proposal_count, which
 * may be up to the capacity: e.g. a prompt after prefill) through the page
 * table.  k_new, v_new: bf16 [batch][proposal_count][kv_heads][head_dim]. */
carat_status carat_paged_append(void *key_pages, void *value_pages, int num_pages,
                                const int32_t *page_table, int max_pages, int page_rows,
                                const void *k_new, const void *v_new,
                                const int32_t *context_lengths, int proposal_count, int batch,
                                int kv_heads, int head_dim, void *stream);

/*
 * carat_pool_* -- host-side allocator of the page ids of one shared pool
 * (no device memory involved; the caller owns the pool's memory).
 *
 * A ring is an aligned run of pages_per_ring pages; carat_pool_alloc_ring
 * returns its ring id (first page / pages_per_ring), which is what the ring
 * entry points take in ring_ids when k_ring / v_ring point at the pool.  A
 * global-layer page is any single page.  Single pages come first from blocks
 * that single pages already use, so whole blocks stay free for rings.
 * Thread-safe.  Returns: alloc_ring -> ring id or -1 (no whole free block);
 * alloc_pages -> n, writing n page ids to out_pages, or -1 (fewer than n free:
 * nothing allocated); free_* -> 0, or -1 for an id that is not allocated (then
 * nothing is freed); stats -> out4 = {free pages, whole free blocks, rings in
 * use, single pages in use}.
 */
typedef struct carat_pool carat_pool;
carat_pool *carat_pool_create(int num_pages, int pages_per_ring);
void carat_pool_destroy(carat_pool *pool);
int carat_pool_alloc_ring(carat_pool *pool);
int carat_pool_free_ring(carat_pool *pool, int ring_id);
int carat_pool_alloc_pages(carat_pool *pool, int n, int32_t *out_pages);
int carat_pool_free_pages(carat_pool *pool, int n, const int32_t *pages);
int carat_pool_stats(carat_pool *pool, int32_t *out4);

/*
 * FP8 (e4m3) sliding-window rings -- "gemma-cuda-hybrid", "Features" /
 * "Server": the KV cache is stored as FP8 e4m3; "Limitations": FP8 KV is
 * lossy (outside the bit-exact comparison).  The pages give
 * no scaling scheme; here each ring tensor has one dequantisation scale:
 * the value of a stored byte is e4m3(byte) * k_scale (K) or * v_scale (V).
 *
 * carat_ring_append_fp8 -- carat_ring_append for e4m3 rings.  k_ring, v_ring
 *   are uint8 [num_rings][window][kv_heads][head_dim]; k_new, v_new stay bf16
 *   [batch][proposal_count][kv_heads][head_dim]; each element x is stored as
 *   e4m3_rn_satfinite(fp32(x * fp32(1 / scale))) (one binary32 product, then
 *   round to nearest even, magnitudes past 448 saturate).  displaced, when
 *   given, is uint8 [batch][proposal_count-1][2][kv_heads][head_dim] and
 *   receives the overwritten rows' bytes.  k_scale, v_scale: finite, > 0,
 *   with a finite reciprocal.  kv_heads * head_dim must be a multiple of 16.
 *
 * carat_ring_rollback_fp8 -- carat_ring_rollback for e4m3 rings and their
 *   uint8 displaced rows (the bytes are copied back unchanged).
 *
 * carat_swa_attention_fp8 -- carat_swa_attention over e4m3 rings: the
 *   attention of the dequantised K and V (bf16 queries, fp32 out).  Each e4m3
 *   value is widened exactly to f16 on chip; k_scale scales the scores and
 *   v_scale the output.  head_dim 256 only (CARAT_ERR_UNSUPPORTED else).  The
 *   workspace it needs is at most carat_swa_workspace_bytes for the same
 *   sizes.  When the call's units (request, KV head) outnumber the SMs, one
 *   CTA per SM takes whole units from a work counter in the workspace: each
 *   call tags the counter with a new epoch (so the workspace still needs no
 *   initialisation, whatever it held) and the call's last CTA clears it;
 *   concurrent calls on one workspace are as unsupported as for every other
 *   call.  Other arguments, limits and device-side error handling as in
 *   carat_swa_attention.
 */
carat_status carat_ring_append_fp8(void *k_ring, void *v_ring, int num_rings,
                                   const int32_t *ring_ids, const void *k_new,
                                   const void *v_new, const int32_t *context_lengths,
                                   int proposal_count, void *displaced, int batch,
                                   int kv_heads, int head_dim, int window, float k_scale,
                                   float v_scale, void *stream);
carat_status carat_ring_rollback_fp8(void *k_ring, void *v_ring, int num_rings,
                                     const int32_t *ring_ids, const void *displaced,
                                     const int32_t *context_lengths, const int32_t *accepted,
                                     int proposal_count, int batch, int kv_heads, int head_dim,
                                     int window, void *stream);
carat_status carat_swa_attention_fp8(float *out, const void *queries, const void *k_ring,
                                     const void *v_ring, int num_rings,
                                     const int32_t *ring_ids, const void *displaced,
                                     const int32_t *context_lengths, int proposal_count,
                                     int batch, int q_heads, int kv_heads, int head_dim,
                                     int window, float scale, float k_scale, float v_scale,
                                     void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes the attention calls need for these sizes (the same for the
 * plain and the fused-append entry points; 0 if the sizes are invalid, or if
 * the call needs no scratch).  Host arithmetic and a query of the current
 * device's SM count (a GB300's 152 when no device is visible); a launch on a
 * device with more SMs checks the size again and returns CARAT_ERR_WORKSPACE. */
size_t carat_swa_workspace_bytes(int batch, int proposal_count, int q_heads, int kv_heads,
                                 int head_dim, int window);
size_t carat_global_workspace_bytes(int batch, int proposal_count, int q_heads,
                                    int kv_heads, int head_dim, int capacity);

/*
 * Read (and, if clear != 0, reset) the current device's status word
 * (CARAT_DEV_* bits, 0 = nothing seen).  Enqueued on `stream` and
 * synchronised with it before returning.
 */
carat_status carat_get_device_status(int32_t *host_out, int clear, void *stream);

/*
 * Self-check of the bounded waits every kernel of this library uses: a
 * one-thread kernel waits on a barrier phase that nothing completes, gives up
 * after `limit_ns` nanoseconds (and a minimum number of polls), sets
 * CARAT_DEV_TIMEOUT in the current device's status word and returns; the
 * context stays usable.  limit_ns must lie in [1e6, 1e10] (1 ms .. 10 s), else
 * CARAT_ERR_INVALID_ARG.  Enqueued on `stream` (read the result with
 * carat_get_device_status); CARAT_ERR_CUDA if the launch fails.
 */
carat_status carat_check_bounded_wait(uint64_t limit_ns, void *stream);

/*
 * Launch floor, for measurement: one empty kernel, and with dependent != 0 a
 * second empty kernel launched after it with programmatic dependent launch
 * (it may start once the first has started and waits for it to finish) --
 * the two-launch pattern of a stream-K attention call and its merge launch.
 * Timing this call with CUDA events on `stream` gives the part of a call's
 * time that no kernel work can remove.  The pages have no counterpart.
 */
carat_status carat_launch_floor(int dependent, void *stream);

/* Static English text for a status code. */
const char *carat_status_string(carat_status status);

/* Number of CUDA kernels this library has launched in this process, on any
 * device (a host-side counter, incremented once per kernel launch). */
uint64_t carat_kernel_launches(void);

/* ABI version of this header (incremented on incompatible changes). */
#define CARAT_ABI_VERSION 1
int carat_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CARAT_H */
