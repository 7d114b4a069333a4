// api.cu -- the extern "C" entry points of libcarat.so.
//
// Host side only: argument checks (before any CUDA call), the split plan that
// sizes the caller's workspace, and the launches.  The kernels live in
// ring_append.cu and attention_*.cu.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "carat_internal.cuh"
#include "tc_common.cuh"

namespace carat {

// One status word per device, read back by carat_get_device_status.
__device__ int g_device_status;

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
int *g_status_ptr[kMaxDevices];

// Device address of this device's status word (looked up once per device).
int *device_status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mutex);
    if (!g_status_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(ptr);
    }
    return g_status_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_head_dim(int d) { return d == 256 || d == 512; }

struct SplitPlan {
    bool unit_mode = false;    // whole units from a work counter (else stream-K)
    bool fp8 = false;          // FP8 e4m3 rings
    bool deep = false;         // a call with at most one tile per SM: one CTA per SM, deep ring
    int grid = 0;              // CTAs launched
    size_t ml_bytes = 0;
    size_t o_bytes = 0;
    size_t unit_bytes = 0;
    size_t sched_bytes = 0;
    size_t total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// SMs of the current device (looked up once per device); 152, a GB300's
// count, when no device can be queried -- workspace sizes asked for without a
// GPU assume that GPU, and a launch re-checks against its own device.
int device_sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return 152;
    }
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
        cudaGetLastError();
        return 152;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Tensor-core path.  Units (request, KV head, row group) that fill every
// resident CTA slot and are all short (at most 16 tiles of 128 keys) are
// taken whole, one at a time, by one persistent CTA per resident slot from a
// work counter in the workspace (unit mode).  Otherwise one CTA per resident
// slot runs the stream-K schedule; each keeps two partial slots (the first
// and last segment of its range), and each unit a 16-byte entry for the merge
// launch.  The workspace holds both.
SplitPlan tc_plan(int batch, int group, int k, int kv_heads, int head_dim, long long max_tiles,
                  bool fp8 = false) {
    SplitPlan p;
    p.fp8 = fp8;
    const int n = tc_rows_per_tile(group, k);
    const int slots_total = tc_ctas_per_sm(head_dim, n, fp8) * device_sm_count();
    const long long units = (long long)batch * tc_units_per_request(group, k, kv_heads);
    // Whole units when there are enough of them and each is short.  With
    // bf16 caches one CTA per unit.  With FP8 caches (one CTA per SM, several
    // units each) one persistent CTA per SM: CTA g starts with unit g and then
    // takes the next unit the counter hands out as soon as it has issued its
    // current unit's loads, so the next unit's keys stream in while the
    // current one finishes.
    p.unit_mode = units >= slots_total && max_tiles <= 16 && units < (1ll << 24);
    p.grid = p.unit_mode && !fp8 ? (int)units : slots_total;
    // A stream-K call that cannot have more tiles than the GPU has SMs gives
    // each busy CTA about one tile: a kernel with a ring deep enough for a
    // whole tile's K and V loads them at once (one DRAM round trip, not two).
    const int sms = device_sm_count();
    if (!p.unit_mode && !fp8 && units * max_tiles <= sms && tc_has_deep_variant(head_dim, n)) {
        p.deep = true;
        p.grid = sms;
    }
    const size_t slots = (size_t)slots_total * 2 * n;
    p.ml_bytes = align256(slots * sizeof(float2));
    p.o_bytes = align256(slots * (size_t)head_dim * sizeof(float));
    p.unit_bytes = align256((size_t)batch * tc_units_per_request(group, k, kv_heads) * 16);
    p.sched_bytes = 256;
    p.total = p.ml_bytes + p.o_bytes + p.unit_bytes + p.sched_bytes;
    return p;
}

// Point the call's parameters at its workspace.
void set_split_fields(AttnParams &p, const SplitPlan &plan, void *workspace) {
    char *w = static_cast<char *>(workspace);
    p.part_ml = reinterpret_cast<float2 *>(w);
    p.part_o = w ? reinterpret_cast<float *>(w + plan.ml_bytes) : nullptr;
    p.units = w ? reinterpret_cast<int4 *>(w + plan.ml_bytes + plan.o_bytes) : nullptr;
    p.sched = w ? reinterpret_cast<unsigned long long *>(w + plan.ml_bytes + plan.o_bytes +
                                                          plan.unit_bytes)
                : nullptr;
}

int row_groups_for(int group, int k) {
    const int n = tc_rows_per_tile(group, k);
    int ppg = n / group;
    if (ppg > k) ppg = k;
    return (k + ppg - 1) / ppg;
}

bool attention_shape_ok(int batch, int proposal_count, int q_heads, int kv_heads, int head_dim) {
    return batch >= 0 && proposal_count >= 1 && proposal_count <= kMaxProposals && q_heads >= 1 &&
           kv_heads >= 1 && q_heads % kv_heads == 0 && head_dim >= 1;
}

// Shapes the tensor-core kernel takes: head_dim 256 or 512, at most
// kMaxTileRows rows per KV head, at most 64 query heads per KV head (one row
// group holds every head of a position).
carat_status attention_unsupported(int proposal_count, int q_heads, int kv_heads, int head_dim) {
    if (!supported_head_dim(head_dim)) return CARAT_ERR_UNSUPPORTED;
    if ((long long)(q_heads / kv_heads) * proposal_count > kMaxTileRows) return CARAT_ERR_UNSUPPORTED;
    if (!tc_supported(head_dim, q_heads / kv_heads, proposal_count)) return CARAT_ERR_UNSUPPORTED;
    return CARAT_OK;
}

SplitPlan swa_plan(int batch, int proposal_count, int q_heads, int kv_heads, int head_dim,
                   int window) {
    // ring tiles + one tile of displaced rows or (fused append) new rows
    return tc_plan(batch, q_heads / kv_heads, proposal_count, kv_heads, head_dim,
                   (window + kTcTileKeys - 1) / kTcTileKeys + 1);
}

SplitPlan global_plan(int batch, int proposal_count, int q_heads, int kv_heads, int head_dim,
                      int capacity) {
    // cache tiles + one tile of new rows (fused append)
    return tc_plan(batch, q_heads / kv_heads, proposal_count, kv_heads, head_dim,
                   ((long long)capacity + kTcTileKeys - 1) / kTcTileKeys + 1);
}

cudaError_t launch_attention(const AttnParams &p, const SplitPlan &plan, cudaStream_t stream) {
    return launch_attention_tc(p, plan.grid, plan.unit_mode, plan.fp8, stream, plan.deep);
}

carat_status launch_status(cudaError_t e) { return e == cudaSuccess ? CARAT_OK : CARAT_ERR_CUDA; }

}  // namespace
}  // namespace carat

using namespace carat;

extern "C" {

const char *carat_status_string(carat_status status) {
    switch (status) {
        case CARAT_OK: return "ok";
        case CARAT_ERR_INVALID_ARG: return "invalid argument";
        case CARAT_ERR_UNSUPPORTED: return "unsupported size";
        case CARAT_ERR_WORKSPACE: return "workspace missing or too small";
        case CARAT_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int carat_abi_version(void) { return CARAT_ABI_VERSION; }

uint64_t carat_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t carat_swa_workspace_bytes(int batch, int proposal_count, int q_heads, int kv_heads,
                                 int head_dim, int window) {
    if (!attention_shape_ok(batch, proposal_count, q_heads, kv_heads, head_dim) || window < 1 ||
        proposal_count > window)
        return 0;
    if (attention_unsupported(proposal_count, q_heads, kv_heads, head_dim) != CARAT_OK) return 0;
    if (batch == 0) return 0;
    return swa_plan(batch, proposal_count, q_heads, kv_heads, head_dim, window).total;
}

size_t carat_global_workspace_bytes(int batch, int proposal_count, int q_heads, int kv_heads,
                                    int head_dim, int capacity) {
    if (!attention_shape_ok(batch, proposal_count, q_heads, kv_heads, head_dim) ||
        capacity < proposal_count)
        return 0;
    if (attention_unsupported(proposal_count, q_heads, kv_heads, head_dim) != CARAT_OK) return 0;
    if (batch == 0) return 0;
    return global_plan(batch, proposal_count, q_heads, kv_heads, head_dim, capacity).total;
}

carat_status carat_ring_append(void *k_ring, void *v_ring, int num_rings, const int32_t *ring_ids,
                               const void *k_new, const void *v_new,
                               const int32_t *context_lengths, int proposal_count,
                               void *displaced, int batch, int kv_heads, int head_dim, int window,
                               void *stream) {
    if (batch < 0 || kv_heads < 1 || head_dim < 1 || window < 1 || proposal_count < 1 ||
        proposal_count > window || num_rings < 1)
        return CARAT_ERR_INVALID_ARG;
    if (((long long)kv_heads * head_dim * 2) % 16 != 0) return CARAT_ERR_INVALID_ARG;
    if (displaced && proposal_count > kMaxProposals) return CARAT_ERR_INVALID_ARG;
    if (!ring_ids && num_rings < batch) return CARAT_ERR_INVALID_ARG;
    if (batch == 0) return CARAT_OK;
    if (!k_ring || !v_ring || !k_new || !v_new || !context_lengths) return CARAT_ERR_INVALID_ARG;
    if (!aligned16(k_ring) || !aligned16(v_ring) || !aligned16(k_new) || !aligned16(v_new) ||
        (displaced && !aligned16(displaced)))
        return CARAT_ERR_INVALID_ARG;
    AppendParams p{};
    p.k_ring = static_cast<uint16_t *>(k_ring);
    p.v_ring = static_cast<uint16_t *>(v_ring);
    p.ids = ring_ids;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.context_lengths = context_lengths;
    p.displaced = (proposal_count > 1) ? static_cast<uint16_t *>(displaced) : nullptr;
    p.dev_status = device_status_ptr();
    p.num_ids = num_rings;
    p.batch = batch;
    p.k = proposal_count;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.window = window;
    return launch_status(launch_ring_append(p, static_cast<cudaStream_t>(stream)));
}

static carat_status check_attention_common(float *out, const void *queries, const void *k_base,
                                           const void *v_base, int num_ids, const int32_t *ids,
                                           const int32_t *context_lengths, int batch) {
    if (num_ids < 1 || (!ids && num_ids < batch)) return CARAT_ERR_INVALID_ARG;
    if (!out || !queries || !k_base || !v_base || !context_lengths) return CARAT_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(queries) || !aligned16(k_base) || !aligned16(v_base))
        return CARAT_ERR_INVALID_ARG;
    return CARAT_OK;
}

carat_status carat_swa_attention(float *out, const void *queries, const void *k_ring,
                                 const void *v_ring, int num_rings, const int32_t *ring_ids,
                                 const void *displaced, const int32_t *context_lengths,
                                 int proposal_count, int batch, int q_heads, int kv_heads,
                                 int head_dim, int window, float scale, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    if (!attention_shape_ok(batch, proposal_count, q_heads, kv_heads, head_dim) || window < 1 ||
        proposal_count > window || !std::isfinite(scale))
        return CARAT_ERR_INVALID_ARG;
    carat_status st = attention_unsupported(proposal_count, q_heads, kv_heads, head_dim);
    if (st != CARAT_OK) return st;
    if (batch == 0) return CARAT_OK;
    st = check_attention_common(out, queries, k_ring, v_ring, num_rings, ring_ids, context_lengths,
                                batch);
    if (st != CARAT_OK) return st;
    if (proposal_count > 1 && (!displaced || !aligned16(displaced))) return CARAT_ERR_INVALID_ARG;
    const SplitPlan plan = swa_plan(batch, proposal_count, q_heads, kv_heads, head_dim, window);
    if (plan.total > 0 && (!workspace || workspace_bytes < plan.total || !aligned16(workspace)))
        return CARAT_ERR_WORKSPACE;

    AttnParams p{};
    p.q = static_cast<const uint16_t *>(queries);
    p.k_base = static_cast<const uint16_t *>(k_ring);
    p.v_base = static_cast<const uint16_t *>(v_ring);
    p.ids = ring_ids;
    p.displaced = proposal_count > 1 ? static_cast<const uint16_t *>(displaced) : nullptr;
    p.context_lengths = context_lengths;
    p.out = out;
    set_split_fields(p, plan, workspace);
    p.dev_status = device_status_ptr();
    p.num_ids = num_rings;
    p.batch = batch;
    p.k = proposal_count;
    p.q_heads = q_heads;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.group = q_heads / kv_heads;
    p.rows = p.group * proposal_count;
    p.window = window;
    p.capacity = 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.source = KeySource::kRing;
    return launch_status(launch_attention(p, plan, static_cast<cudaStream_t>(stream)));
}

carat_status carat_global_verify_attention(float *out, const void *queries, const void *key_cache,
                                           const void *value_cache, int num_caches,
                                           const int32_t *cache_ids,
                                           const int32_t *context_lengths, int proposal_count,
                                           int batch, int q_heads, int kv_heads, int head_dim,
                                           int capacity, float scale, void *workspace,
                                           size_t workspace_bytes, void *stream) {
    if (!attention_shape_ok(batch, proposal_count, q_heads, kv_heads, head_dim) ||
        capacity < proposal_count || !std::isfinite(scale))
        return CARAT_ERR_INVALID_ARG;
    carat_status st = attention_unsupported(proposal_count, q_heads, kv_heads, head_dim);
    if (st != CARAT_OK) return st;
    if (batch == 0) return CARAT_OK;
    st = check_attention_common(out, queries, key_cache, value_cache, num_caches, cache_ids,
                                context_lengths, batch);
    if (st != CARAT_OK) return st;
    const SplitPlan plan = global_plan(batch, proposal_count, q_heads, kv_heads, head_dim, capacity);
    if (plan.total > 0 && (!workspace || workspace_bytes < plan.total || !aligned16(workspace)))
        return CARAT_ERR_WORKSPACE;

    AttnParams p{};
    p.q = static_cast<const uint16_t *>(queries);
    p.k_base = static_cast<const uint16_t *>(key_cache);
    p.v_base = static_cast<const uint16_t *>(value_cache);
    p.ids = cache_ids;
    p.displaced = nullptr;
    p.context_lengths = context_lengths;
    p.out = out;
    set_split_fields(p, plan, workspace);
    p.dev_status = device_status_ptr();
    p.num_ids = num_caches;
    p.batch = batch;
    p.k = proposal_count;
    p.q_heads = q_heads;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.group = q_heads / kv_heads;
    p.rows = p.group * proposal_count;
    p.window = 0;
    p.capacity = capacity;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.source = KeySource::kLinear;
    return launch_status(launch_attention(p, plan, static_cast<cudaStream_t>(stream)));
}

// Shared by the two fused entry points: attention over the caches as they are
// before this step plus this step's rows, which are then written into the
// caches (by the attention kernel itself, or by a ring append launched after
// it when several CTAs read each ring tile).
struct PagedArgs {
    const int32_t *page_table = nullptr;
    int max_pages = 0, page_rows = 0, num_pages = 0;
};

static carat_status append_attention(float *out, const void *queries, void *k_base, void *v_base,
                                     int num_ids, const int32_t *ids, void *displaced,
                                     const void *k_new,
                                     const void *v_new, const int32_t *context_lengths,
                                     int proposal_count, int batch, int q_heads, int kv_heads,
                                     int head_dim, int window, int capacity, float scale,
                                     void *workspace, size_t workspace_bytes, void *stream,
                                     KeySource source, PagedArgs pg = PagedArgs()) {
    const bool ring = source == KeySource::kRing;
    if (!attention_shape_ok(batch, proposal_count, q_heads, kv_heads, head_dim) ||
        !std::isfinite(scale))
        return CARAT_ERR_INVALID_ARG;
    if (ring ? (window < 1 || proposal_count > window) : capacity < proposal_count)
        return CARAT_ERR_INVALID_ARG;
    carat_status st = attention_unsupported(proposal_count, q_heads, kv_heads, head_dim);
    if (st != CARAT_OK) return st;
    const int group = q_heads / kv_heads;
    if (batch == 0) return CARAT_OK;
    st = check_attention_common(out, queries, k_base, v_base, num_ids, ids, context_lengths, batch);
    if (st != CARAT_OK) return st;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return CARAT_ERR_INVALID_ARG;
    if (displaced && !aligned16(displaced)) return CARAT_ERR_INVALID_ARG;
    const SplitPlan plan =
        ring ? swa_plan(batch, proposal_count, q_heads, kv_heads, head_dim, window)
             : global_plan(batch, proposal_count, q_heads, kv_heads, head_dim, capacity);
    if (plan.total > 0 && (!workspace || workspace_bytes < plan.total || !aligned16(workspace)))
        return CARAT_ERR_WORKSPACE;

    AttnParams p{};
    p.q = static_cast<const uint16_t *>(queries);
    p.k_base = static_cast<const uint16_t *>(k_base);
    p.v_base = static_cast<const uint16_t *>(v_base);
    p.ids = ids;
    p.displaced = nullptr;
    p.context_lengths = context_lengths;
    p.out = out;
    set_split_fields(p, plan, workspace);
    p.dev_status = device_status_ptr();
    p.num_ids = num_ids;
    p.batch = batch;
    p.k = proposal_count;
    p.q_heads = q_heads;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.group = group;
    p.rows = group * proposal_count;
    p.window = ring ? window : 0;
    p.capacity = ring ? 0 : capacity;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.source = source;
    p.fused = 1;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.k_dst = static_cast<uint16_t *>(k_base);
    p.v_dst = static_cast<uint16_t *>(v_base);
    p.displaced_out = (ring && proposal_count > 1) ? static_cast<uint16_t *>(displaced) : nullptr;
    p.page_table = pg.page_table;
    p.max_pages = pg.max_pages;
    p.page_rows = pg.page_rows;
    p.num_pages = pg.num_pages;
    // Several row groups read every ring tile: none of them may overwrite a
    // slot, so a ring append follows the attention instead.
    p.fused_write = (!ring || row_groups_for(group, proposal_count) == 1) ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_attention(p, plan, s);
    if (e == cudaSuccess && !p.fused_write) {
        AppendParams a{};
        a.k_ring = static_cast<uint16_t *>(k_base);
        a.v_ring = static_cast<uint16_t *>(v_base);
        a.ids = ids;
        a.k_new = p.k_new;
        a.v_new = p.v_new;
        a.context_lengths = context_lengths;
        a.displaced = p.displaced_out;
        a.dev_status = p.dev_status;
        a.num_ids = num_ids;
        a.batch = batch;
        a.k = proposal_count;
        a.kv_heads = kv_heads;
        a.head_dim = head_dim;
        a.window = window;
        e = launch_ring_append(a, s);
    }
    return launch_status(e);
}

carat_status carat_swa_append_attention(float *out, const void *queries, void *k_ring,
                                        void *v_ring, int num_rings, const int32_t *ring_ids,
                                        void *displaced, const void *k_new, const void *v_new,
                                        const int32_t *context_lengths, int proposal_count,
                                        int batch, int q_heads, int kv_heads, int head_dim,
                                        int window, float scale, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    return append_attention(out, queries, k_ring, v_ring, num_rings, ring_ids, displaced, k_new,
                            v_new,
                            context_lengths, proposal_count, batch, q_heads, kv_heads, head_dim,
                            window, 0, scale, workspace, workspace_bytes, stream,
                            KeySource::kRing);
}

carat_status carat_global_append_verify_attention(float *out, const void *queries,
                                                  void *key_cache, void *value_cache,
                                                  int num_caches, const int32_t *cache_ids,
                                                  const void *k_new, const void *v_new,
                                                  const int32_t *context_lengths,
                                                  int proposal_count, int batch, int q_heads,
                                                  int kv_heads, int head_dim, int capacity,
                                                  float scale, void *workspace,
                                                  size_t workspace_bytes, void *stream) {
    return append_attention(out, queries, key_cache, value_cache, num_caches, cache_ids, nullptr,
                            k_new, v_new, context_lengths, proposal_count, batch, q_heads, kv_heads,
                            head_dim, 0, capacity, scale, workspace, workspace_bytes, stream,
                            KeySource::kLinear);
}

static bool paged_args_ok(int num_pages, const int32_t *page_table, int max_pages,
                          int page_rows) {
    return num_pages >= 1 && page_table && max_pages >= 1 && page_rows >= kTcTileKeys &&
           page_rows % kTcTileKeys == 0 &&
           (long long)num_pages * page_rows < (1LL << 31) &&
           (long long)max_pages * page_rows < (1LL << 31);
}

carat_status carat_global_append_verify_attention_paged(
    float *out, const void *queries, void *key_pages, void *value_pages, int num_pages,
    const int32_t *page_table, int max_pages, int page_rows, const void *k_new, const void *v_new,
    const int32_t *context_lengths, int proposal_count, int batch, int q_heads, int kv_heads,
    int head_dim, float scale, void *workspace, size_t workspace_bytes, void *stream) {
    if (!paged_args_ok(num_pages, page_table, max_pages, page_rows)) return CARAT_ERR_INVALID_ARG;
    PagedArgs pg;
    pg.page_table = page_table;
    pg.max_pages = max_pages;
    pg.page_rows = page_rows;
    pg.num_pages = num_pages;
    // Requests address the pool only through the page table.
    return append_attention(out, queries, key_pages, value_pages, batch > 0 ? batch : 1, nullptr,
                            nullptr, k_new, v_new, context_lengths, proposal_count, batch,
                            q_heads, kv_heads, head_dim, 0, max_pages * page_rows, scale,
                            workspace, workspace_bytes, stream, KeySource::kPaged, pg);
}

carat_status carat_paged_append(void *key_pages, void *value_pages, int num_pages,
                                const int32_t *page_table, int max_pages, int page_rows,
                                const void *k_new, const void *v_new,
                                const int32_t *context_lengths, int proposal_count, int batch,
                                int kv_heads, int head_dim, void *stream) {
    if (!paged_args_ok(num_pages, page_table, max_pages, page_rows)) return CARAT_ERR_INVALID_ARG;
    if (batch < 0 || kv_heads < 1 || head_dim < 1 || proposal_count < 1 ||
        (long long)proposal_count > (long long)max_pages * page_rows)
        return CARAT_ERR_INVALID_ARG;
    if (((long long)kv_heads * head_dim * 2) % 16 != 0) return CARAT_ERR_INVALID_ARG;
    if (batch == 0) return CARAT_OK;
    if (!key_pages || !value_pages || !k_new || !v_new || !context_lengths)
        return CARAT_ERR_INVALID_ARG;
    if (!aligned16(key_pages) || !aligned16(value_pages) || !aligned16(k_new) || !aligned16(v_new))
        return CARAT_ERR_INVALID_ARG;
    AppendParams p{};
    p.k_ring = static_cast<uint16_t *>(key_pages);
    p.v_ring = static_cast<uint16_t *>(value_pages);
    p.ids = nullptr;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.context_lengths = context_lengths;
    p.displaced = nullptr;
    p.dev_status = device_status_ptr();
    p.num_ids = batch;
    p.batch = batch;
    p.k = proposal_count;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.window = max_pages * page_rows;
    p.page_table = page_table;
    p.max_pages = max_pages;
    p.page_rows = page_rows;
    p.num_pages = num_pages;
    return launch_status(launch_ring_append(p, static_cast<cudaStream_t>(stream)));
}

carat_status carat_ring_rollback(void *k_ring, void *v_ring, int num_rings,
                                 const int32_t *ring_ids, const void *displaced,
                                 const int32_t *context_lengths, const int32_t *accepted,
                                 int proposal_count, int batch, int kv_heads, int head_dim,
                                 int window, void *stream) {
    if (batch < 0 || kv_heads < 1 || head_dim < 1 || window < 1 || proposal_count < 2 ||
        proposal_count > kMaxProposals || proposal_count > window || num_rings < 1)
        return CARAT_ERR_INVALID_ARG;
    if (((long long)kv_heads * head_dim * 2) % 16 != 0) return CARAT_ERR_INVALID_ARG;
    if (!ring_ids && num_rings < batch) return CARAT_ERR_INVALID_ARG;
    if (batch == 0) return CARAT_OK;
    if (!k_ring || !v_ring || !displaced || !context_lengths || !accepted)
        return CARAT_ERR_INVALID_ARG;
    if (!aligned16(k_ring) || !aligned16(v_ring) || !aligned16(displaced))
        return CARAT_ERR_INVALID_ARG;
    AppendParams p{};
    p.k_ring = static_cast<uint16_t *>(k_ring);
    p.v_ring = static_cast<uint16_t *>(v_ring);
    p.ids = ring_ids;
    p.context_lengths = context_lengths;
    p.displaced = static_cast<uint16_t *>(const_cast<void *>(displaced));
    p.dev_status = device_status_ptr();
    p.num_ids = num_rings;
    p.batch = batch;
    p.k = proposal_count;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.window = window;
    return launch_status(launch_ring_rollback(p, accepted, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// FP8 (e4m3) rings: "gemma-cuda-hybrid", "Features" / "Server" (the KV cache
// is FP8 e4m3) and "Limitations" (lossy).  One dequantisation scale per
// tensor (K, V).
// ---------------------------------------------------------------------------

static bool fp8_scale_ok(float s) { return std::isfinite(s) && s > 0.f && std::isfinite(1.f / s); }

carat_status carat_ring_append_fp8(void *k_ring, void *v_ring, int num_rings,
                                   const int32_t *ring_ids, const void *k_new, const void *v_new,
                                   const int32_t *context_lengths, int proposal_count,
                                   void *displaced, int batch, int kv_heads, int head_dim,
                                   int window, float k_scale, float v_scale, void *stream) {
    if (batch < 0 || kv_heads < 1 || head_dim < 1 || window < 1 || proposal_count < 1 ||
        proposal_count > window || num_rings < 1 || !fp8_scale_ok(k_scale) ||
        !fp8_scale_ok(v_scale))
        return CARAT_ERR_INVALID_ARG;
    if (((long long)kv_heads * head_dim) % 16 != 0) return CARAT_ERR_INVALID_ARG;
    if (displaced && proposal_count > kMaxProposals) return CARAT_ERR_INVALID_ARG;
    if (!ring_ids && num_rings < batch) return CARAT_ERR_INVALID_ARG;
    if (batch == 0) return CARAT_OK;
    if (!k_ring || !v_ring || !k_new || !v_new || !context_lengths) return CARAT_ERR_INVALID_ARG;
    if (!aligned16(k_ring) || !aligned16(v_ring) || !aligned16(k_new) || !aligned16(v_new) ||
        (displaced && !aligned16(displaced)))
        return CARAT_ERR_INVALID_ARG;
    AppendParams p{};
    p.k_ring = static_cast<uint16_t *>(k_ring);
    p.v_ring = static_cast<uint16_t *>(v_ring);
    p.ids = ring_ids;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.context_lengths = context_lengths;
    p.displaced = (proposal_count > 1) ? static_cast<uint16_t *>(displaced) : nullptr;
    p.dev_status = device_status_ptr();
    p.num_ids = num_rings;
    p.batch = batch;
    p.k = proposal_count;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.window = window;
    p.elem_bytes = 1;
    p.k_inv = 1.f / k_scale;
    p.v_inv = 1.f / v_scale;
    return launch_status(launch_ring_append_fp8(p, static_cast<cudaStream_t>(stream)));
}

carat_status carat_ring_rollback_fp8(void *k_ring, void *v_ring, int num_rings,
                                     const int32_t *ring_ids, const void *displaced,
                                     const int32_t *context_lengths, const int32_t *accepted,
                                     int proposal_count, int batch, int kv_heads, int head_dim,
                                     int window, void *stream) {
    if (batch < 0 || kv_heads < 1 || head_dim < 1 || window < 1 || proposal_count < 2 ||
        proposal_count > kMaxProposals || proposal_count > window || num_rings < 1)
        return CARAT_ERR_INVALID_ARG;
    if (((long long)kv_heads * head_dim) % 16 != 0) return CARAT_ERR_INVALID_ARG;
    if (!ring_ids && num_rings < batch) return CARAT_ERR_INVALID_ARG;
    if (batch == 0) return CARAT_OK;
    if (!k_ring || !v_ring || !displaced || !context_lengths || !accepted)
        return CARAT_ERR_INVALID_ARG;
    if (!aligned16(k_ring) || !aligned16(v_ring) || !aligned16(displaced))
        return CARAT_ERR_INVALID_ARG;
    AppendParams p{};
    p.k_ring = static_cast<uint16_t *>(k_ring);
    p.v_ring = static_cast<uint16_t *>(v_ring);
    p.ids = ring_ids;
    p.context_lengths = context_lengths;
    p.displaced = static_cast<uint16_t *>(const_cast<void *>(displaced));
    p.dev_status = device_status_ptr();
    p.num_ids = num_rings;
    p.batch = batch;
    p.k = proposal_count;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.window = window;
    p.elem_bytes = 1;
    return launch_status(launch_ring_rollback(p, accepted, static_cast<cudaStream_t>(stream)));
}

carat_status carat_swa_attention_fp8(float *out, const void *queries, const void *k_ring,
                                     const void *v_ring, int num_rings, const int32_t *ring_ids,
                                     const void *displaced, const int32_t *context_lengths,
                                     int proposal_count, int batch, int q_heads, int kv_heads,
                                     int head_dim, int window, float scale, float k_scale,
                                     float v_scale, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    if (!attention_shape_ok(batch, proposal_count, q_heads, kv_heads, head_dim) || window < 1 ||
        proposal_count > window || !std::isfinite(scale) || !fp8_scale_ok(k_scale) ||
        !fp8_scale_ok(v_scale))
        return CARAT_ERR_INVALID_ARG;
    carat_status st = attention_unsupported(proposal_count, q_heads, kv_heads, head_dim);
    if (st != CARAT_OK) return st;
    const int group = q_heads / kv_heads;
    if (!tc_fp8_supported(head_dim, group, proposal_count)) return CARAT_ERR_UNSUPPORTED;
    if (batch == 0) return CARAT_OK;
    st = check_attention_common(out, queries, k_ring, v_ring, num_rings, ring_ids, context_lengths,
                                batch);
    if (st != CARAT_OK) return st;
    if (proposal_count > 1 && (!displaced || !aligned16(displaced))) return CARAT_ERR_INVALID_ARG;
    const SplitPlan plan = tc_plan(batch, group, proposal_count, kv_heads, head_dim,
                                   (window + kTcTileKeys - 1) / kTcTileKeys + 1, true);
    if (plan.total > 0 && (!workspace || workspace_bytes < plan.total || !aligned16(workspace)))
        return CARAT_ERR_WORKSPACE;

    AttnParams p{};
    p.q = static_cast<const uint16_t *>(queries);
    p.k_base = static_cast<const uint16_t *>(k_ring);
    p.v_base = static_cast<const uint16_t *>(v_ring);
    p.ids = ring_ids;
    p.displaced = proposal_count > 1 ? static_cast<const uint16_t *>(displaced) : nullptr;
    p.context_lengths = context_lengths;
    p.out = out;
    set_split_fields(p, plan, workspace);
    p.dev_status = device_status_ptr();
    p.num_ids = num_rings;
    p.batch = batch;
    p.k = proposal_count;
    p.q_heads = q_heads;
    p.kv_heads = kv_heads;
    p.head_dim = head_dim;
    p.group = group;
    p.rows = group * proposal_count;
    p.window = window;
    p.capacity = 0;
    // dequantised K = e4m3 * k_scale: the K scale joins the softmax scale;
    // dequantised V = e4m3 * v_scale: the V scale multiplies the output
    p.scale_log2 = scale * k_scale * 1.4426950408889634f;
    p.out_scale = v_scale;
    p.source = KeySource::kRing;
    return launch_status(launch_attention(p, plan, static_cast<cudaStream_t>(stream)));
}

namespace carat {
namespace {
// One bounded wait on a barrier phase that nothing completes: the wait the
// attention kernels use, given up after limit_ns.
__global__ void bounded_wait_check_kernel(int *dev_status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    if (!tc::mbar_wait(&bar, 0, limit_ns)) set_status(dev_status, CARAT_DEV_TIMEOUT);
}
}  // namespace
}  // namespace carat

namespace carat {
namespace {
// The launch floor: an empty kernel that lets a dependent launch start early
// (as the attention kernel does), and an empty dependent kernel that waits
// for it (as the merge launch does).
__global__ void floor_first_kernel() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__global__ void floor_dependent_kernel() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
}  // namespace
}  // namespace carat

carat_status carat_launch_floor(int dependent, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    carat::floor_first_kernel<<<1, 32, 0, s>>>();
    carat::count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !dependent) return launch_status(e);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, carat::floor_dependent_kernel);
    carat::count_launches(1);
    return launch_status(e);
}

carat_status carat_check_bounded_wait(uint64_t limit_ns, void *stream) {
    if (limit_ns < 1000000ull || limit_ns > 10000000000ull) return CARAT_ERR_INVALID_ARG;
    int *status = carat::device_status_ptr();
    if (!status) return CARAT_ERR_CUDA;
    carat::bounded_wait_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        status, (unsigned long long)limit_ns);
    carat::count_launches(1);
    return cudaGetLastError() == cudaSuccess ? CARAT_OK : CARAT_ERR_CUDA;
}

carat_status carat_get_device_status(int32_t *host_out, int clear, void *stream) {
    if (!host_out) return CARAT_ERR_INVALID_ARG;
    int *ptr = device_status_ptr();
    if (!ptr) return CARAT_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t value = 0;
    if (cudaMemcpyAsync(&value, ptr, sizeof(value), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return CARAT_ERR_CUDA;
    if (clear && cudaMemsetAsync(ptr, 0, sizeof(int), s) != cudaSuccess) return CARAT_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CARAT_ERR_CUDA;
    *host_out = value;
    return CARAT_OK;
}

}  // extern "C"
