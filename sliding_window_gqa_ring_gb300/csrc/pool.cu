// pool.cu -- host-side allocator of a shared HBM pool of KV pages.
//
// "Improving Decode Throughput on Intel Gaudi 3", "Our approach": the ring
// buffers of sliding-window layers are allocated in the same HBM that backs
// the global-attention KV pages, one shared pool, so that short requests can
// take more ring space and long requests more pages.  This allocator hands
// out page ids of one pool: a ring is an aligned run of `pages_per_ring`
// pages (its ring id is the first page / pages_per_ring, which is how the
// ring kernels address it), a global page is any single page.  Single pages
// are taken first from blocks that pages already broke up, then from the
// highest free block, so whole aligned blocks stay available for rings.
// Host code only; the device memory itself belongs to the caller.
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "carat_internal.cuh"

struct carat_pool {
    int num_pages = 0;
    int pages_per_ring = 0;
    int num_blocks = 0;
    std::vector<uint8_t> page_state;   // 0 free, 1 single page, 2 part of a ring
    std::vector<int> block_free;       // free pages per block
    std::vector<uint8_t> block_ring;   // block holds a ring
    int used_pages = 0;
    int used_rings = 0;
    std::mutex mutex;
};

namespace {

// Blocks: [b * ppr, (b + 1) * ppr) for b < num_blocks; pages past the last
// whole block can only be single pages.
int block_of(const carat_pool *p, int page) {
    const int b = page / p->pages_per_ring;
    return b < p->num_blocks ? b : -1;
}

}  // namespace

extern "C" {

carat_pool *carat_pool_create(int num_pages, int pages_per_ring) {
    if (num_pages < 1 || pages_per_ring < 1) return nullptr;
    carat_pool *p = new (std::nothrow) carat_pool;
    if (!p) return nullptr;
    p->num_pages = num_pages;
    p->pages_per_ring = pages_per_ring;
    p->num_blocks = num_pages / pages_per_ring;
    p->page_state.assign((size_t)num_pages, 0);
    p->block_free.assign((size_t)p->num_blocks, pages_per_ring);
    p->block_ring.assign((size_t)p->num_blocks, 0);
    return p;
}

void carat_pool_destroy(carat_pool *p) { delete p; }

int carat_pool_alloc_ring(carat_pool *p) {
    if (!p) return -1;
    std::lock_guard<std::mutex> lock(p->mutex);
    // lowest whole free block (single pages are taken from the top)
    for (int b = 0; b < p->num_blocks; ++b) {
        if (p->block_free[b] == p->pages_per_ring) {
            for (int i = 0; i < p->pages_per_ring; ++i) p->page_state[(size_t)b * p->pages_per_ring + i] = 2;
            p->block_free[b] = 0;
            p->block_ring[b] = 1;
            ++p->used_rings;
            return b;
        }
    }
    return -1;
}

int carat_pool_free_ring(carat_pool *p, int ring_id) {
    if (!p) return -1;
    std::lock_guard<std::mutex> lock(p->mutex);
    if (ring_id < 0 || ring_id >= p->num_blocks || !p->block_ring[ring_id]) return -1;
    for (int i = 0; i < p->pages_per_ring; ++i) p->page_state[(size_t)ring_id * p->pages_per_ring + i] = 0;
    p->block_free[ring_id] = p->pages_per_ring;
    p->block_ring[ring_id] = 0;
    --p->used_rings;
    return 0;
}

int carat_pool_alloc_pages(carat_pool *p, int n, int32_t *out_pages) {
    if (!p || n < 0 || (n > 0 && !out_pages)) return -1;
    std::lock_guard<std::mutex> lock(p->mutex);
    // all or nothing: count what single pages may use
    long long avail = 0;
    for (int b = 0; b < p->num_blocks; ++b)
        if (!p->block_ring[b]) avail += p->block_free[b];
    for (int pg = p->num_blocks * p->pages_per_ring; pg < p->num_pages; ++pg)
        avail += p->page_state[pg] == 0;
    if (avail < n) return -1;
    int got = 0;
    auto take = [&](int pg) {
        p->page_state[pg] = 1;
        const int b = block_of(p, pg);
        if (b >= 0) --p->block_free[b];
        out_pages[got++] = pg;
    };
    // 1. pages past the last whole block, 2. blocks already broken up by
    // single pages, 3. whole free blocks from the top
    for (int pg = p->num_blocks * p->pages_per_ring; pg < p->num_pages && got < n; ++pg)
        if (p->page_state[pg] == 0) take(pg);
    for (int b = p->num_blocks - 1; b >= 0 && got < n; --b) {
        if (p->block_ring[b] || p->block_free[b] == 0 || p->block_free[b] == p->pages_per_ring)
            continue;
        for (int i = 0; i < p->pages_per_ring && got < n; ++i) {
            const int pg = b * p->pages_per_ring + i;
            if (p->page_state[pg] == 0) take(pg);
        }
    }
    for (int b = p->num_blocks - 1; b >= 0 && got < n; --b) {
        if (p->block_ring[b] || p->block_free[b] != p->pages_per_ring) continue;
        for (int i = 0; i < p->pages_per_ring && got < n; ++i) take(b * p->pages_per_ring + i);
    }
    p->used_pages += got;
    return got;
}

int carat_pool_free_pages(carat_pool *p, int n, const int32_t *pages) {
    if (!p || n < 0 || (n > 0 && !pages)) return -1;
    std::lock_guard<std::mutex> lock(p->mutex);
    // all or nothing: every entry must be an allocated single page, listed once
    for (int i = 0; i < n; ++i) {
        const int pg = pages[i];
        if (pg < 0 || pg >= p->num_pages || p->page_state[pg] != 1) {
            for (int x = 0; x < i; ++x) p->page_state[pages[x]] = 1;
            return -1;
        }
        p->page_state[pg] = 3;  // marked for release
    }
    for (int i = 0; i < n; ++i) {
        const int pg = pages[i];
        p->page_state[pg] = 0;
        const int b = block_of(p, pg);
        if (b >= 0) ++p->block_free[b];
        --p->used_pages;
    }
    return 0;
}

int carat_pool_stats(carat_pool *p, int32_t *out4) {
    if (!p || !out4) return -1;
    std::lock_guard<std::mutex> lock(p->mutex);
    int whole = 0;
    for (int b = 0; b < p->num_blocks; ++b) whole += p->block_free[b] == p->pages_per_ring;
    out4[0] = p->num_pages - p->used_pages - p->used_rings * p->pages_per_ring;  // free pages
    out4[1] = whole;                                                             // whole free blocks
    out4[2] = p->used_rings;
    out4[3] = p->used_pages;
    return 0;
}

}  // extern "C"
