// attention_tc.cu -- host side of the tensor-core attention path: shapes it
// takes, the grid and instantiation each call runs, and the tensor maps (the
// kernels themselves are in attention_tc.cuh).
#include "attention_tc.cuh"

namespace carat {

int tc_rows_per_tile(int group, int k) {
    const int rows = group * k;
    if (rows <= 16) return 16;
    if (rows <= 32) return 32;
    return 64;
}

int tc_ctas_per_sm(int head_dim, int rows_per_tile, bool fp8) {
    return (!fp8 && head_dim == 256 && rows_per_tile == 16) ? 2 : 1;
}

bool tc_fp8_supported(int head_dim, int group, int k) {
    return head_dim == 256 && tc_supported(head_dim, group, k);
}

bool tc_supported(int head_dim, int group, int k) {
    if (head_dim != 256 && head_dim != 512) return false;
    const int n = tc_rows_per_tile(group, k);
    return group <= n;
}

int tc_units_per_request(int group, int k, int kv_heads) {
    const int n = tc_rows_per_tile(group, k);
    int ppg = n / group;
    if (ppg > k) ppg = k;
    return kv_heads * ((k + ppg - 1) / ppg);
}

bool tc_has_deep_variant(int head_dim, int rows_per_tile) {
    return head_dim == 256 && rows_per_tile == 16;
}

// A new epoch (40 bits, never 0) per unit-mode launch: a launch's first
// increment of the work counter or the done count replaces a word tagged
// with another epoch, whatever the workspace held before.
static unsigned long long next_unit_epoch() {
    static std::atomic<unsigned long long> counter{0};
    unsigned long long e = 0;
    while (e == 0) e = (counter.fetch_add(1, std::memory_order_relaxed) + 1) & ((1ull << 40) - 1);
    return e;
}

cudaError_t launch_attention_tc(const AttnParams &p_call, int grid, bool unit_mode, bool fp8,
                                cudaStream_t stream, bool deep) {
    AttnParams p = p_call;
    if (unit_mode && fp8) {
        if (!p.sched) return cudaErrorInvalidValue;
        p.sched_epoch = next_unit_epoch();
    }
    const int n = tc_rows_per_tile(p.group, p.k);
    TcPlan plan{};
    plan.unit_mode = unit_mode ? 1 : 0;
    plan.pos_per_group = n / p.group;
    if (plan.pos_per_group > p.k) plan.pos_per_group = p.k;
    plan.row_groups = (p.k + plan.pos_per_group - 1) / plan.pos_per_group;
    plan.paired = (!unit_mode && plan.row_groups == 2 && grid >= 2) ? 1 : 0;

    TcMaps maps{};
    const uint64_t D = (uint64_t)p.head_dim;
    if (fp8) {
        // e4m3 rings: (128 d bytes, rows, 128-d block, head); a box is one raw
        // stage of 128 rows x 128 d, or 16 displaced rows x every block.
        if (p.head_dim != 256 || p.source != KeySource::kRing || p.fused)
            return cudaErrorNotSupported;
        const uint64_t row8 = (uint64_t)p.kv_heads * D;
        const uint64_t rows_total = (uint64_t)p.num_ids * (uint64_t)p.window;
        const uint64_t dims_kv[4] = {128, rows_total, D / 128, (uint64_t)p.kv_heads};
        const uint64_t strides_kv[3] = {row8, 128, D};
        const uint32_t box_kv[4] = {128, (uint32_t)kTileKeys, 1, 1};
        if (!make_u8_tensor_map(&maps.k, p.k_base, 4, dims_kv, strides_kv, box_kv, true) ||
            !make_u8_tensor_map(&maps.v, p.v_base, 4, dims_kv, strides_kv, box_kv, true))
            return cudaErrorInvalidValue;
        if (p.k > 1) {
            const uint64_t dims5[5] = {128, (uint64_t)p.batch * (p.k - 1), D / 128, 2,
                                       (uint64_t)p.kv_heads};
            const uint64_t strides5[4] = {2 * row8, 128, row8, D};
            const uint32_t box5[5] = {128, (uint32_t)kDispRows, (uint32_t)(D / 128), 1, 1};
            if (!make_u8_tensor_map(&maps.disp, p.displaced, 5, dims5, strides5, box5, true))
                return cudaErrorInvalidValue;
        } else {
            maps.disp = maps.k;
        }
        maps.knew = maps.k;
        maps.vnew = maps.v;
        const uint64_t dimsq[4] = {D, (uint64_t)p.q_heads, (uint64_t)p.k, (uint64_t)p.batch};
        const uint64_t stridesq[3] = {D * 2, (uint64_t)p.q_heads * D * 2,
                                      (uint64_t)p.k * p.q_heads * D * 2};
        const uint32_t boxq[4] = {64, (uint32_t)p.group, (uint32_t)plan.pos_per_group, 1};
        if (!make_bf16_tensor_map(&maps.q, p.q, 4, dimsq, stridesq, boxq, true))
            return cudaErrorInvalidValue;
        // one CTA per SM: f16 stages the widening warps fill and raw stages in
        // flight (16 rows: 5 and 3, the split measured best; else 3 and 6 or 4)
        if (n == 16 && unit_mode)
            return launch_tc_lane_sums(p, plan, maps, grid, n, true, stream);
        if (n == 16) return launch_tc<256, 16, 5, 1, 3>(p, plan, maps, grid, stream);
        if (n == 32) return launch_tc<256, 32, 3, 1, 6>(p, plan, maps, grid, stream);
        return launch_tc<256, 64, 3, 1, 4>(p, plan, maps, grid, stream);
    }
    const uint64_t row_bytes = (uint64_t)p.kv_heads * D * 2;
    const uint64_t slabs = D / 64;
    const uint64_t rows_total =
        p.source == KeySource::kPaged
            ? (uint64_t)p.num_pages * (uint64_t)p.page_rows
            : (uint64_t)p.num_ids * (uint64_t)(p.source == KeySource::kRing ? p.window : p.capacity);
    // (64 d, rows, slab, head): rows row_bytes apart, slabs 128 bytes, heads D * 2
    const uint64_t dims_kv[4] = {64, rows_total, slabs, (uint64_t)p.kv_heads};
    const uint64_t strides_kv[3] = {row_bytes, 128, D * 2};
    const uint32_t box_kv[4] = {64, (uint32_t)kTileKeys, 2, 1};
    if (!make_bf16_tensor_map(&maps.k, p.k_base, 4, dims_kv, strides_kv, box_kv, true) ||
        !make_bf16_tensor_map(&maps.v, p.v_base, 4, dims_kv, strides_kv, box_kv, true))
        return cudaErrorInvalidValue;
    if (p.source == KeySource::kRing && p.k > 1) {
        // displaced [B*(k-1)][2][Hkv][D]: (64 d, row, slab, K/V, head)
        const uint64_t dims5[5] = {64, (uint64_t)p.batch * (p.k - 1), slabs, 2,
                                   (uint64_t)p.kv_heads};
        const uint64_t strides5[4] = {2 * row_bytes, 128, row_bytes, D * 2};
        const uint32_t box5[5] = {64, (uint32_t)kDispRows, (uint32_t)slabs, 1, 1};
        if (!make_bf16_tensor_map(&maps.disp, p.displaced, 5, dims5, strides5, box5, true))
            return cudaErrorInvalidValue;
    } else {
        maps.disp = maps.k;
    }
    if (p.fused) {
        const uint64_t dimsn[4] = {64, (uint64_t)p.batch * p.k, slabs, (uint64_t)p.kv_heads};
        const uint32_t boxn[4] = {64, (uint32_t)kDispRows, (uint32_t)slabs, 1};
        if (!make_bf16_tensor_map(&maps.knew, p.k_new, 4, dimsn, strides_kv, boxn, true) ||
            !make_bf16_tensor_map(&maps.vnew, p.v_new, 4, dimsn, strides_kv, boxn, true))
            return cudaErrorInvalidValue;
    } else {
        maps.knew = maps.k;
        maps.vnew = maps.v;
    }
    {
        const uint64_t dimsq[4] = {D, (uint64_t)p.q_heads, (uint64_t)p.k, (uint64_t)p.batch};
        const uint64_t stridesq[3] = {D * 2, (uint64_t)p.q_heads * D * 2,
                                      (uint64_t)p.k * p.q_heads * D * 2};
        const uint32_t boxq[4] = {64, (uint32_t)p.group, (uint32_t)plan.pos_per_group, 1};
        if (!make_bf16_tensor_map(&maps.q, p.q, 4, dimsq, stridesq, boxq, true))
            return cudaErrorInvalidValue;
    }

    // 16-row tiles at head_dim 256 fit two CTAs per SM (registers and shared
    // memory), so one CTA's start-up and epilogue overlap the other's
    // streaming; the others run one CTA per SM with the stage ring taking the
    // rest of shared memory.
    if (p.head_dim == 256) {
        // a small call (at most one tile per SM): one CTA per SM with six
        // stages, so a tile's K and V stages all load at once
        if (n == 16 && deep) return launch_tc<256, 16, 6, 1>(p, plan, maps, grid, stream);
        // whole units of 16 rows: row sums kept by the softmax threads
        if (n == 16 && unit_mode)
            return launch_tc_lane_sums(p, plan, maps, grid, n, false, stream);
        if (n == 16) return launch_tc<256, 16, 3, 2>(p, plan, maps, grid, stream);
        if (n == 32) return launch_tc<256, 32, 6, 1>(p, plan, maps, grid, stream);
        return launch_tc<256, 64, 5, 1>(p, plan, maps, grid, stream);
    }
    if (n == 16) return launch_tc<512, 16, 4, 1>(p, plan, maps, grid, stream);
    if (n == 32) return launch_tc<512, 32, 5, 1>(p, plan, maps, grid, stream);
    return launch_tc<512, 64, 4, 1>(p, plan, maps, grid, stream);
}

}  // namespace carat
