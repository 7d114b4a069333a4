// carat_internal.cuh -- definitions shared by the CUDA translation units of
// libcarat.so (never installed, never seen by callers).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/carat.h"

namespace carat {

constexpr int kMaxProposals = CARAT_MAX_PROPOSALS;
constexpr int kMaxTileRows = CARAT_MAX_TILE_ROWS;

// Where the keys of one (request, KV head) come from.
enum class KeySource : int {
    kRing = 0,    // sliding layer: `window` ring slots + (proposal_count - 1) displaced rows
    kLinear = 1,  // global layer: cache row t holds position t, t < key_count
    kPaged = 2,   // global layer in pages: position t is row t % page_rows of page
                  // page_table[b][t / page_rows]
};

// Everything an attention launch needs; passed by value as a kernel argument.
struct AttnParams {
    const uint16_t *q;          // [B][k][Hq][D]
    const uint16_t *k_base;     // ring or cache, [num][rows][Hkv][D]
    const uint16_t *v_base;
    const int32_t *ids;         // ring/cache id per request, or nullptr
    const uint16_t *displaced;  // [B][k-1][2][Hkv][D] (ring source, k > 1)
    const int32_t *context_lengths;
    float *out;                 // [B][k][Hq][D]
    // Split partials (running max and sum in log2 units, unnormalised O):
    // two slots per CTA of a stream-K grid, [grid][2][rows per tile].
    float2 *part_ml;
    float *part_o;
    // Stream-K schedule: per (request, KV head, row group) unit, the range
    // holding its first tile (x), the ranges it spans (y; 0 when one CTA
    // covered it whole) and the partial slot of its first piece (z), for the
    // merge launch.
    int4 *units;
    // Unit mode: the work counter handing out units (word 0) and the count of
    // CTAs done (word 1), each tagged with the launch's epoch in its high 40
    // bits; the last CTA of a launch clears both.
    unsigned long long *sched;
    unsigned long long sched_epoch;
    int *dev_status;
    int num_ids;                // rings / caches available
    int batch, k, q_heads, kv_heads, head_dim, group, rows;
    int window;                 // ring slots (kRing) -- positions older than p-window+1 hidden
    int capacity;               // cache rows (kLinear)
    // Fused append: the caches hold the tokens before this
    // step and this step's rows come from k_new / v_new [B][k][Hkv][D]; when
    // fused_write is set the kernel also writes them into k_dst / v_dst.
    int fused;
    int fused_write;
    const uint16_t *k_new;
    const uint16_t *v_new;
    uint16_t *k_dst;
    uint16_t *v_dst;
    uint16_t *displaced_out;    // fused ring append: old rows saved here, or nullptr
    // Paged global caches (kPaged): page table [B][max_pages], page_rows rows per
    // page (a multiple of 128), num_pages pages in the pool.
    const int32_t *page_table;
    int max_pages;
    int page_rows;
    int num_pages;
    float scale_log2;           // softmax scale * log2(e) (FP8: times the K scale)
    float out_scale = 1.f;      // FP8: the V scale, applied to the output
    KeySource source;
};

struct AppendParams {
    uint16_t *k_ring, *v_ring;        // bf16 rows, or (elem_bytes 1) e4m3 bytes
    const int32_t *ids;
    const uint16_t *k_new, *v_new;
    const int32_t *context_lengths;
    uint16_t *displaced;
    int *dev_status;
    int num_ids, batch, k, kv_heads, head_dim, window;
    // Paged caches: rows go through the page table instead of a ring.
    const int32_t *page_table;
    int max_pages, page_rows, num_pages;
    // FP8 rings: 1-byte elements; new rows are quantised as
    // e4m3_rn(fp32(x * k_inv)) (k_inv = fp32(1 / k_scale)), likewise for V.
    int elem_bytes = 2;               // 2 (bf16) or 1 (e4m3)
    float k_inv = 1.f, v_inv = 1.f;
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// bf16 pair packed in a 32-bit word -> two fp32 values (exact: a bf16 is the
// upper half of an fp32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 2^x with the SFU instruction (about 2 ulp); inputs <= 0 here, -inf -> 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// L2 policy that marks lines for early eviction (K/V rows are read once).
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16-byte global load, no L1 allocation, with an L2 eviction-priority hint.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ void set_status(int *status, int bits) {
    if (status) atomicOr(status, bits);
}

// Whether a request's context length and cache/ring id are in range.
__device__ __forceinline__ bool request_valid(const AttnParams &p, int id, long long ctx) {
    if (ctx < 0 || (p.source != KeySource::kRing && ctx + p.k > p.capacity)) return false;
    return id >= 0 && id < p.num_ids;
}

// Resolve request b: its cache/ring id and context length; false when either
// is out of range (request_error_bits says which).
__device__ __forceinline__ bool request_ok(const AttnParams &p, int b, int *id_out,
                                           long long *ctx_out) {
    const long long ctx = p.context_lengths[b];
    const int id = p.ids ? p.ids[b] : b;
    *id_out = id;
    *ctx_out = ctx;
    return request_valid(p, id, ctx);
}

// CARAT_DEV_* bits describing why request_ok rejected a request.
__device__ __forceinline__ int request_error_bits(const AttnParams &p, int id, long long ctx) {
    int bits = 0;
    if (ctx < 0 || (p.source != KeySource::kRing && ctx + p.k > p.capacity))
        bits |= CARAT_DEV_BAD_CONTEXT;
    if (id < 0 || id >= p.num_ids) bits |= CARAT_DEV_BAD_CACHE_ID;
    return bits;
}

// Tensor-core path: 128-key tiles a request needs, and the index of its
// one special tile (or -1).
//  * Ring, append done before the call: the tiles covering the slots that hold
//    tokens (all `window` slots once the ring has wrapped), plus one tile of
//    displaced rows when some exist (key_count > window and k > 1).
//  * Ring, fused append: the tiles covering the slots that hold the tokens
//    before this step (min(context_length, window) slots), plus one tile of
//    this step's k new rows.
//  * Cache: ceil(key_count / 128); fused append: ceil(context_length / 128)
//    tiles of old rows plus the tile of new rows.
__host__ __device__ __forceinline__ int tc_request_tiles(KeySource src, int window, int k,
                                                         long long key_count, bool fused,
                                                         int *special_tile) {
    const long long ctx = key_count - k;
    if (src == KeySource::kRing) {
        const long long tokens = fused ? ctx : key_count;
        const long long held = tokens < window ? tokens : window;
        const int ring_tiles = (int)((held + 127) / 128);
        const bool extra = fused || (k > 1 && key_count > window);
        *special_tile = extra ? ring_tiles : -1;
        return ring_tiles + (extra ? 1 : 0);
    }
    if (fused) {
        const int old_tiles = (int)((ctx + 127) / 128);
        *special_tile = old_tiles;
        return old_tiles + 1;
    }
    *special_tile = -1;
    return (int)((key_count + 127) / 128);
}

// Row of the paged pool that holds position t of request b, or -1 when the
// page table entry is outside the pool.
__device__ __forceinline__ long long paged_row(const int32_t *page_table, int max_pages,
                                               int page_rows, int num_pages, int b, long long t) {
    const int page = page_table[(size_t)b * max_pages + (size_t)(t / page_rows)];
    if (page < 0 || page >= num_pages) return -1;
    return (long long)page * page_rows + t % page_rows;
}

// Host-side count of kernel launches (carat_kernel_launches).
void count_launches(int n);

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the .cu files)
// ---------------------------------------------------------------------------
cudaError_t launch_ring_append(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_ring_append_fp8(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_ring_rollback(const AppendParams &p, const int32_t *accepted,
                                 cudaStream_t stream);

// Tensor-core path (attention_tc.cu): rows per tile (16, 32 or 64) for a
// group size and proposal count, CTAs resident per SM, whether the shape is
// supported, (request, KV head, row group) units per request, and the launch
// over tiles of 128 keys on `grid` CTAs: whole units (unit_mode: one CTA per
// unit with bf16 caches, grid = units; persistent CTAs taking units from a
// work counter with FP8 caches, grid = resident slots) or the persistent
// stream-K schedule (grid = resident slots).
constexpr int kTcTileKeys = 128;
int tc_rows_per_tile(int group, int k);
int tc_ctas_per_sm(int head_dim, int rows_per_tile, bool fp8);
bool tc_supported(int head_dim, int group, int k);
bool tc_fp8_supported(int head_dim, int group, int k);   // FP8 e4m3 rings
int tc_units_per_request(int group, int k, int kv_heads);
cudaError_t launch_attention_tc(const AttnParams &p, int grid, bool unit_mode, bool fp8,
                                cudaStream_t stream, bool deep = false);
// Whether a one-CTA-per-SM kernel with a deep stage ring exists for this
// shape (used for calls with at most one tile per SM).
bool tc_has_deep_variant(int head_dim, int rows_per_tile);

}  // namespace carat
