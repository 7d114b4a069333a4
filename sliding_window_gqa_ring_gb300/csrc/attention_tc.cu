// attention_tc.cu -- split-K grouped-query attention on the 5th-generation
// tensor cores (tcgen05 + TMEM) with TMA-staged K/V tiles.
//
// What it computes is what attention_simt.cu computes: for each request b and
// KV head c, the rows r = j*g + h' (the g query heads sharing KV head c times
// the proposal positions j; "Announcing Carat: An inference engine designed
// for Gemma 4", "Doing it all in one kernel can be slower") attend to the keys
// their position may see -- the last `window` positions for a sliding layer
// read in place from the rotated ring ("Improving Decode Throughput on Intel
// Gaudi 3", "Our approach"), every position up to their own for a global
// layer, with the tail past key_count masked ("More FLOPs can be faster").
//
// Tiles.  Keys come in tiles of 128 (ring slots 128i.., or cache rows 128i..,
// plus one tile of displaced rows for a sliding verify with k > 1).  Keys are
// the M dimension of both products, so any number of rows N in {16, 32, 64}
// fits one tile without padding the keys:
//     S^T [128 keys x N rows]  = K_tile [128 x D] . Q^T          (K-major A, B)
//     O^T [128 d   x N rows]  += V_tile^T [d x 128 keys] . P^T   (MN-major A)
// S^T and O^T live in tensor memory; P (bf16) is written to shared memory by
// the softmax threads.  Rows beyond 64 are split into row groups (separate
// CTAs).  The key-count tail is masked per key, never padded with work: a
// tile that holds no token in some rows has those V rows zeroed in shared
// memory so their contents (zero-initialised or not) cannot reach O.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K and V tiles in 32 KB stages
//               (128 keys x 128 d, two 64-d boxes with 128-byte swizzle)
//               through an NS-deep ring of shared-memory stages.
//   warp 1      allocates TMEM; one thread issues every tcgen05.mma and the
//               commits that free stages and signal the softmax warps.
//   warps 2-5   softmax: thread t owns key t of the tile (TMEM lane t): reads
//               its N scores, masks by position, finds each row's tile maximum
//               with a warp transpose-reduction and shared memory, updates the
//               running max / sum (log2 domain), writes P, rescales O^T in TMEM
//               when a row's maximum moved, and in the epilogue writes the
//               chunk's partial (max, sum, unnormalised O) for attn_combine.
//
// Every wait is bounded (mbar_wait): on a timeout the CTA records
// CARAT_DEV_TIMEOUT, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and returns.
#include <cfloat>

#include <cuda_bf16.h>

#include "carat_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace carat {

namespace {

constexpr int kTileKeys = 128;
constexpr int kBoxBytes = 128 * 128;        // [128 keys][64 bf16]
constexpr int kStageBytes = 2 * kBoxBytes;  // 128 keys x 128 d
constexpr int kDispRows = 16;               // displaced rows loaded per tile (>= k - 1)
constexpr int kMaxPagedTiles = 32;          // paged tiles whose rows a CTA resolves up front
constexpr int kDispBoxBytes = kDispRows * 128;
constexpr int kThreads = 192;
constexpr uint32_t kFull = 0xffffffffu;

template <int D, int N, int NS>
struct Layout {
    static constexpr int KS = D / 128;                 // stages per K (or V) tile
    static constexpr int kQBlock = N * 128;            // one 64-d block of Q rows
    static constexpr int kOffQ = NS * kStageBytes;
    static constexpr int kOffP = kOffQ + (D / 64) * kQBlock;
    static constexpr int kPBlock = N * 128;            // 64 keys of P rows
    static constexpr int kOffRed = kOffP + 2 * kPBlock;
    static constexpr int kRedFloats = 3 * 4 * N;       // 2 x max buffers + sum buffer
    static constexpr int kOffBar = kOffRed + kRedFloats * 4;
    static constexpr int kNumBars = 2 * NS + 6;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kOffRows = kOffMisc + 16;         // paged: rows of the CTA's tiles
    static constexpr int kBytes = kOffRows + kMaxPagedTiles * 8;
    static constexpr int kAlloc = kBytes + 1024;       // base alignment slack
    static constexpr int kTmemUsed = N * (2 + D / 128);   // two S^T buffers + O^T
    static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64
                                   : kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
    static_assert(kAlloc <= 232448, "more dynamic shared memory than one CTA may use");
    // The softmax warps zero masked V rows while all KS stages of a V tile are
    // resident, before the tile's PV product releases any of them.
    static_assert(NS >= KS, "the stage ring must hold a whole V tile");
    static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kPBlock % 1024 == 0 &&
                      kQBlock % 1024 == 0,
                  "operand blocks must be 1024-byte aligned for the 128-byte swizzle");
};

struct TcMaps {
    CUtensorMap k;     // (D, Hkv, rows)          ring slots or cache rows
    CUtensorMap v;
    CUtensorMap disp;  // (D, Hkv, 2, B*(k-1))    displaced rows, K (0) / V (1)
    CUtensorMap q;     // (D, Hq, k, B)           queries
    CUtensorMap knew;  // (D, Hkv, B*k)           this step's rows (fused append)
    CUtensorMap vnew;
};

struct TcPlan {
    int tiles_per_chunk;
    int row_groups;
    int pos_per_group;    // proposal positions per row group
};

// Barrier over the 128 softmax threads that also ORs a predicate across them,
// so every thread takes the same abort decision.
__device__ __forceinline__ bool named_bar_softmax_any(bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.or.pred pout, 1, 128, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)pred)
        : "memory");
    return out != 0;
}

// Wait for a barrier phase; false on timeout or when another thread aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int *dev_status) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (tc::globaltimer_ns() - t0 > 2000000000ull) {
            *abort_flag = 1;
            set_status(dev_status, CARAT_DEV_TIMEOUT);
            return false;
        }
    }
}

// Transpose-reduction across the 32 lanes of a warp: on entry v[i] is this
// lane's value for row i; on exit v[0 .. max(N/32,1)) hold the reduction over
// all 32 lanes for rows row_base + i.
template <int N, bool kMax>
__device__ __forceinline__ int warp_transpose_reduce(float (&v)[N], int lane) {
    int row_base = 0;
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int off = 16 >> s;
        const int cnt = (N >> s) > 1 ? (N >> s) : 1;
        const bool upper = (lane & off) != 0;
        if (cnt >= 2) {
            const int h = cnt / 2;
#pragma unroll
            for (int i = 0; i < h; ++i) {
                const float send = upper ? v[i] : v[i + h];
                const float keep = upper ? v[i + h] : v[i];
                const float recv = __shfl_xor_sync(kFull, send, off);
                v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
            }
            if (upper) row_base += h;
        } else {
            const float recv = __shfl_xor_sync(kFull, v[0], off);
            v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
        }
    }
    return row_base;
}

// Bits [0, n) set (n <= 64).
__device__ __forceinline__ uint64_t low_bits(int n) {
    return n >= 64 ? ~0ull : ((1ull << n) - 1ull);
}

// A row's running maximum is replaced only when a tile's maximum exceeds it by
// more than this (log2 units), so P <= 2^8 and O^T rescales are rare.
constexpr float kRescaleSlack = 8.0f;

struct KeyInfo {
    long long pos;  // absolute position of the token this key row holds
    bool data;      // the smem row holds a token of this request (else: zero it)
};

}  // namespace

template <int D, int N, int NS, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    attn_tc_kernel(const AttnParams p, const TcPlan plan, const __grid_constant__ TcMaps maps) {
    using L = Layout<D, N, NS>;
    constexpr int KS = L::KS;
    const int chunk = blockIdx.x;
    const int c = blockIdx.y / plan.row_groups;
    const int rg = blockIdx.y % plan.row_groups;
    const int b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    int id;
    long long ctx;
    const bool ok = request_ok(p, b, &id, &ctx);
    const long long key_count = ctx + p.k;
    const bool ring = p.source == KeySource::kRing;
    const bool paged = p.source == KeySource::kPaged;
    int special = -1;
    const int ntiles =
        ok ? tc_request_tiles(p.source, p.window, p.k, key_count, p.fused != 0, &special) : 0;
    const int disp_tile = p.fused ? -1 : special;   // displaced rows (append done before)
    const int new_tile = p.fused ? special : -1;    // this step's rows (fused append)
    // Tokens the caches hold for this call: all key_count of them, or with a
    // fused append only the context_length older ones.
    const long long held_tokens = p.fused ? ctx : key_count;
    const int t0 = chunk * plan.tiles_per_chunk;
    const int t1 = min(t0 + plan.tiles_per_chunk, ntiles);
    const int pos0 = rg * plan.pos_per_group;                       // first position of the group
    const int npos = min(plan.pos_per_group, p.k - pos0);
    const int row0 = pos0 * p.group;                                // first row of the group
    const int rows_here = npos * p.group;

    const size_t part = ((size_t)b * p.kv_heads + c) * p.nchunks + chunk;
    float2 *ml = p.part_ml + part * p.rows + row0;
    float *po = p.part_o + (part * p.rows + row0) * D;
    if (t0 >= t1) {
        if (p.direct) {
            // One split per request: no combine follows, so a request rejected
            // on the device gets its NaN outputs and status bit here.
            if (!ok && chunk == 0) {
                if (c == 0 && rg == 0 && threadIdx.x == 0)
                    set_status(p.dev_status, request_error_bits(p, id, ctx));
                for (int x = threadIdx.x; x < rows_here * D; x += blockDim.x) {
                    const int row = row0 + x / D, j = row / p.group, hp = row % p.group;
                    p.out[(((size_t)b * p.k + j) * p.q_heads + (size_t)c * p.group + hp) * D + x % D] =
                        __int_as_float(0x7fc00000);
                }
            }
        } else {
            for (int r = threadIdx.x; r < rows_here; r += blockDim.x)
                ml[r] = make_float2(-INFINITY, 0.f);
        }
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *full = bars;
    uint64_t *empty = bars + NS;
    uint64_t *s_full = bars + 2 * NS;   // [2]: one per S^T buffer
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = s_full + 3;
    uint64_t *q_full = s_full + 4;
    uint64_t *fin = s_full + 5;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
    float *red = reinterpret_cast<float *>(smem + L::kOffRed);
    uint8_t *s_q = smem + L::kOffQ;
    uint8_t *s_p = smem + L::kOffP;

    const int n = t1 - t0;                 // tiles of this CTA
    // Processing order of the CTA's tiles: the small tile of this step's rows
    // (fused append; always the request's last tile index) goes first, so its
    // work overlaps the first loads of the big tiles instead of ending the CTA.
    const bool new_first = new_tile >= t0 && new_tile < t1;
    auto tile_at = [t0, new_first, new_tile](int x) {
        return new_first ? (x == 0 ? new_tile : t0 + x - 1) : t0 + x;
    };
    // Load / consume order of the 128-key tiles' K and V parts: K(0), then
    // K(x+1) before V(x), then V(n-1), so the next tile's keys stream in and
    // its scores are computed while this tile's softmax runs.  Part index of
    // V(x) in that order (each part is KS stages):
    auto v_part = [n](int x) { return x == n - 1 ? 2 * n - 1 : 2 * x + 2; };

    // Paged caches: warp 0 resolves the pool rows of the CTA's tiles through
    // the page table in one parallel round trip, so the producer's issue path
    // never waits on a page-table read.
    long long *s_rows = reinterpret_cast<long long *>(smem + L::kOffRows);
    const bool rows_cached = paged && n <= kMaxPagedTiles;
    if (rows_cached && warp == 0) {
        if (lane < n) {
            const int i = t0 + lane;
            long long row = -1;
            if (i != new_tile) {
                row = paged_row(p.page_table, p.max_pages, p.page_rows, p.num_pages, b,
                                (long long)i * kTileKeys);
                if (row < 0) {
                    set_status(p.dev_status, CARAT_DEV_BAD_CACHE_ID);
                    row = (long long)p.num_pages * p.page_rows;
                }
            }
            s_rows[lane] = row;
        }
        __syncwarp();
    }

    // Producer state (thread 0): the next stage load to issue.
    uint32_t cnt = 0;
    int ppart = 0, pks = 0;
    bool alive_p = true;
    uint64_t pol = 0;
    // Issue stage loads in order until `limit` stages have been issued or the
    // tiles run out; a stage is reused only after the MMA released it.
    auto produce = [&](uint32_t limit) {
        while (alive_p && ppart < 2 * n && cnt < limit) {
            int x;
            bool is_v;
            if (ppart == 0) {
                x = 0;
                is_v = false;
            } else if (ppart == 2 * n - 1) {
                x = n - 1;
                is_v = true;
            } else {
                x = (ppart - 1) / 2 + ((ppart - 1) % 2 == 0 ? 1 : 0);
                is_v = (ppart - 1) % 2 == 1;
            }
            const int i = tile_at(x);
            const int s = cnt % NS;
            if (cnt >= NS &&
                !wait_or_abort(&empty[s], ((cnt / NS) & 1) ^ 1, abort_flag, p.dev_status)) {
                alive_p = false;
                break;
            }
            tc::mbar_arrive_expect_tx(&full[s], (i == disp_tile || i == new_tile)
                                                    ? 2 * kDispBoxBytes
                                                    : kStageBytes);
            const int d0 = pks * 128;
            uint8_t *dst = smem + s * kStageBytes;
#pragma unroll
            for (int box = 0; box < 2; ++box) {
                if (i == disp_tile) {
                    tc::tma_load_4d(dst + box * kBoxBytes, &maps.disp, d0 + box * 64, c,
                                    is_v ? 1 : 0, b * (p.k - 1), &full[s], pol);
                } else if (i == new_tile) {
                    tc::tma_load_3d(dst + box * kBoxBytes, is_v ? &maps.vnew : &maps.knew,
                                    d0 + box * 64, c, b * p.k, &full[s], pol);
                } else {
                    long long row;
                    if (ring) {
                        row = (long long)id * p.window + (long long)i * kTileKeys;
                    } else if (paged) {
                        // A tile never straddles pages (page_rows is a multiple of
                        // 128).  A page id outside the pool loads the zero fill
                        // past the tensor's end and is reported.
                        if (rows_cached) {
                            row = s_rows[i - t0];
                        } else {
                            row = paged_row(p.page_table, p.max_pages, p.page_rows, p.num_pages,
                                            b, (long long)i * kTileKeys);
                            if (row < 0) {
                                set_status(p.dev_status, CARAT_DEV_BAD_CACHE_ID);
                                row = (long long)p.num_pages * p.page_rows;
                            }
                        }
                    } else {
                        row = (long long)id * p.capacity + (long long)i * kTileKeys;
                    }
                    tc::tma_load_3d(dst + box * kBoxBytes, is_v ? &maps.v : &maps.k,
                                    d0 + box * 64, c, (int)row, &full[s], pol);
                }
            }
            ++cnt;
            if (++pks == KS) {
                pks = 0;
                ++ppart;
            }
        }
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], 1);
        }
        tc::mbar_init(&s_full[0], 1);
        tc::mbar_init(&s_full[1], 1);
        tc::mbar_init(p_full, 128);
        tc::mbar_init(o_done, 1);
        tc::mbar_init(q_full, 1);
        tc::mbar_init(fin, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        // Start streaming before the block-wide barrier: this thread made the
        // barriers, and the first NS stages need no release.
        pol = tc::l2_evict_first_policy();
        tc::tma_prefetch_map(&maps.k);
        tc::tma_prefetch_map(&maps.v);
        tc::tma_prefetch_map(&maps.q);
        tc::mbar_arrive_expect_tx(q_full, (D / 64) * 128 * p.group * plan.pos_per_group);
#pragma unroll
        for (int db = 0; db < D / 64; ++db)
            tc::tma_load_4d(s_q + db * L::kQBlock, &maps.q, db * 64, c * p.group, pos0, b,
                            q_full, pol);
        produce(NS);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tmem_o = tmem + 2 * N;  // O^T: KS blocks of N columns (S^T buffers: 0, N)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            produce(0xffffffffu);
            const bool alive = alive_p;
            if (!alive) {
                // Wait (bounded) for the copies already issued before leaving.
                for (uint32_t x = cnt > (uint32_t)NS ? cnt - NS : 0; x < cnt; ++x)
                    tc::mbar_wait(&full[x % NS], (x / NS) & 1, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, N, false, false);
            constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(128, N, true, false);
            const uint32_t q_base = tc::smem_u32(s_q);
            const uint32_t p_base = tc::smem_u32(s_p);
            bool alive = wait_or_abort(q_full, 0, abort_flag, p.dev_status);
            uint32_t cnt = 0;
            for (int step = 0; step <= n && alive; ++step) {
                if (step < n) {
                    // S^T[step & 1] = K_tile . Q^T over D in steps of 16
                    const uint32_t tmem_s = tmem + (step & 1) * N;
                    for (int ks = 0; ks < KS && alive; ++ks) {
                        const int s = cnt % NS;
                        if (!wait_or_abort(&full[s], (cnt / NS) & 1, abort_flag, p.dev_status)) {
                            alive = false;
                            break;
                        }
                        tc::tc_fence_after();
                        const uint32_t base = tc::smem_u32(smem + s * kStageBytes);
#pragma unroll
                        for (int box = 0; box < 2; ++box) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t a =
                                    tc::sdesc_sw128(base + box * kBoxBytes + kk * 32, 16, 1024);
                                const uint64_t q = tc::sdesc_sw128(
                                    q_base + (ks * 2 + box) * L::kQBlock + kk * 32, 16, 1024);
                                tc::mma_bf16_ss(tmem_s, a, q, idesc_qk, (ks | box | kk) != 0);
                            }
                        }
                        tc::mma_commit(&empty[s]);
                        ++cnt;
                    }
                    if (!alive) break;
                    tc::mma_commit(&s_full[step & 1]);
                }
                if (step >= 1) {
                    // O^T += V_tile^T . P^T over tile x's 128 keys in steps of 16
                    const int x = step - 1;
                    if (!wait_or_abort(p_full, x & 1, abort_flag, p.dev_status)) {
                        alive = false;
                        break;
                    }
                    tc::tc_fence_after();
                    for (int vs = 0; vs < KS && alive; ++vs) {
                        const int s = cnt % NS;
                        if (!wait_or_abort(&full[s], (cnt / NS) & 1, abort_flag, p.dev_status)) {
                            alive = false;
                            break;
                        }
                        tc::tc_fence_after();
                        const uint32_t base = tc::smem_u32(smem + s * kStageBytes);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint64_t a = tc::sdesc_sw128(base + kk * 2048, kBoxBytes, 1024);
                            const uint64_t pp = tc::sdesc_sw128(
                                p_base + (kk / 4) * L::kPBlock + (kk % 4) * 32, 16, 1024);
                            tc::mma_bf16_ss(tmem_o + vs * N, a, pp, idesc_pv, (x > 0 || kk > 0));
                        }
                        tc::mma_commit(&empty[s]);
                        ++cnt;
                    }
                    if (!alive) break;
                    tc::mma_commit(o_done);
                }
            }
            if (!alive) {
                // Make sure every MMA this thread issued has finished.
                tc::mma_commit(fin);
                tc::mbar_wait(fin, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int q4 = warp & 3;              // TMEM lane quadrant this warp may access
        const int t = q4 * 32 + lane;         // key of the tile / d within an O block
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        float m_run[N], l_part[N];
#pragma unroll
        for (int r = 0; r < N; ++r) {
            m_run[r] = -INFINITY;
            l_part[r] = 0.f;
        }
        bool alive = true;
        int idx = 0;
        // Slot that holds the newest token the caches hold (ring source).
        const long long newest = held_tokens - 1;
        const long long head_slot = (ring && newest >= 0) ? newest % p.window : 0;
        // Fused append: slot of this step's first row (ring source).
        const int base_slot = (ring && p.fused) ? (int)(ctx % p.window) : 0;
        for (; idx < n; ++idx) {
            const int i = tile_at(idx);
            // warp-uniform: the TMEM load below is warp-collective
            const bool w_ok = __all_sync(
                kFull, wait_or_abort(&s_full[idx & 1], (idx >> 1) & 1, abort_flag, p.dev_status));
            const uint32_t tmem_s = tmem + (idx & 1) * N;
            float x[N];
            if (w_ok) {
                tc::tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < N / 16; ++cb) {
                    uint32_t r16[16];
                    tc::tmem_ld16(tmem_s + lane_off + cb * 16, r16);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[cb * 16 + e] = __uint_as_float(r16[e]);
                }
            } else {
#pragma unroll
                for (int r = 0; r < N; ++r) x[r] = 0.f;
            }
            // Position of key t of tile i and which rows may see it.
            KeyInfo ki;
            if (i == new_tile) {
                ki.pos = t < p.k ? ctx + t : -1;
                ki.data = t < p.k;
            } else if (ring && i == disp_tile) {
                ki.pos = (t < p.k - 1) ? ctx - p.window + 1 + t : -1;
                ki.data = t < p.k - 1 && ki.pos >= 0;
            } else if (ring) {
                // Slot s holds the newest position congruent to s: head_slot - s
                // (mod window) positions before the newest token.
                const int slot = i * kTileKeys + t;
                long long delta = head_slot - slot;
                if (delta < 0) delta += p.window;
                ki.pos = (slot < p.window && newest >= 0) ? newest - delta : -1;
                ki.data = ki.pos >= 0;
            } else {
                const long long u = (long long)i * kTileKeys + t;
                ki.pos = u < held_tokens ? u : -1;
                ki.data = ki.pos >= 0;
            }
            // Query j of the group (position ctx + pos0 + j) sees the key iff
            // j >= d0 and, for a sliding window, j < d0 + window.
            uint64_t rowmask = 0;
            if (ki.data) {
                const long long d0 = ki.pos - (ctx + pos0);
                const long long jlo = d0 < 0 ? 0 : d0;
                long long jhi = ring ? d0 + p.window : npos;
                if (jhi > npos) jhi = npos;
                if (jlo < jhi) rowmask = low_bits((int)jhi * p.group) & ~low_bits((int)jlo * p.group);
            }
            float tmax[N];
#pragma unroll
            for (int r = 0; r < N; ++r) {
                x[r] = ((rowmask >> r) & 1ull) ? x[r] * p.scale_log2 : -INFINITY;
                tmax[r] = x[r];
            }
            const int rb = warp_transpose_reduce<N, true>(tmax, lane);
            float *red_max = red + (idx & 1) * 4 * N;
            constexpr int kHeld = N >= 32 ? N / 32 : 1;
#pragma unroll
            for (int e = 0; e < kHeld; ++e) red_max[q4 * N + rb + e] = tmax[e];
            if (named_bar_softmax_any(!w_ok || *abort_flag)) {
                alive = false;
                break;
            }
#pragma unroll
            for (int r = 0; r < N; r += 4) {
                float4 a0 = *reinterpret_cast<const float4 *>(red_max + 0 * N + r);
                float4 a1 = *reinterpret_cast<const float4 *>(red_max + 1 * N + r);
                float4 a2 = *reinterpret_cast<const float4 *>(red_max + 2 * N + r);
                float4 a3 = *reinterpret_cast<const float4 *>(red_max + 3 * N + r);
                tmax[r + 0] = fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x));
                tmax[r + 1] = fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y));
                tmax[r + 2] = fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z));
                tmax[r + 3] = fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w));
            }
            float alpha[N];
            bool rescale = false;
#pragma unroll
            for (int r = 0; r < N; ++r) {
                // Keep a stale running maximum unless the tile's maximum exceeds
                // it by more than kRescaleSlack (log2 units): P stays below
                // 2^kRescaleSlack and O^T is rescaled only when a row's maximum
                // really moves.
                const float mn = tmax[r] > m_run[r] + kRescaleSlack ? tmax[r] : m_run[r];
                const float ms = mn == -INFINITY ? 0.f : mn;
                alpha[r] = fast_exp2(m_run[r] - ms);
                const float pr = fast_exp2(x[r] - ms);
                l_part[r] = l_part[r] * alpha[r] + pr;
                x[r] = pr;
                rescale |= (mn != m_run[r]) && (m_run[r] != -INFINITY);
                m_run[r] = mn;
            }
            // PV of the previous tile must be done before P and O are touched.
            if (idx > 0) {
                alive = __all_sync(kFull, wait_or_abort(o_done, (idx - 1) & 1, abort_flag,
                                                        p.dev_status));
                tc::tc_fence_after();
            }
            if (alive) {
                // P^T as a K-major operand: row r, key t (two 64-key blocks).
                uint8_t *pblk = s_p + (t / 64) * L::kPBlock;
                const uint32_t col = t % 64;
#pragma unroll
                for (int r = 0; r < N; ++r) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(x[r]);
                    *reinterpret_cast<__nv_bfloat16 *>(pblk + tc::sw128_offset(r, col)) = h;
                }
                if (idx > 0 && rescale) {
#pragma unroll
                    for (int ob = 0; ob < KS; ++ob) {
#pragma unroll
                        for (int cb = 0; cb < N / 16; ++cb) {
                            uint32_t r16[16];
                            const uint32_t addr = tmem_o + ob * N + lane_off + cb * 16;
                            tc::tmem_ld16(addr, r16);
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                r16[e] = __float_as_uint(__uint_as_float(r16[e]) * alpha[cb * 16 + e]);
                            tc::tmem_st16(addr, r16);
                        }
                    }
                    tc::tmem_st_wait();
                }
                // Rows of the tile that hold no token of this request: zero their
                // V rows so their contents cannot reach O through P = 0.
                const bool tile_partial =
                    i == disp_tile || i == new_tile ||
                    (ring && ((long long)(i + 1) * kTileKeys > min((long long)p.window, held_tokens))) ||
                    (!ring && (long long)(i + 1) * kTileKeys > held_tokens);
                // Fused append into a ring: this CTA is the only one that loads
                // tile i, and it overwrites slots of the tile once its own
                // copies of the tile have landed.
                bool tile_writes = false;
                if (p.fused_write && ring && i != new_tile) {
                    for (int j = 0; j < p.k; ++j) {
                        int sj = base_slot + j;
                        if (sj >= p.window) sj -= p.window;
                        tile_writes |= sj / kTileKeys == i;
                    }
                }
                if (tile_partial || tile_writes) {
                    for (int vs = 0; vs < KS; ++vs) {
                        const uint32_t x_cnt = (uint32_t)v_part(idx) * KS + vs;
                        const int s = x_cnt % NS;
                        if (!wait_or_abort(&full[s], (x_cnt / NS) & 1, abort_flag, p.dev_status)) {
                            alive = false;
                            break;
                        }
                        if (!ki.data && tile_partial) {
                            uint8_t *row0p = smem + s * kStageBytes + t * 128;
#pragma unroll
                            for (int box = 0; box < 2; ++box)
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    *reinterpret_cast<uint4 *>(row0p + box * kBoxBytes + q * 16) =
                                        make_uint4(0, 0, 0, 0);
                        }
                    }
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            if (named_bar_softmax_any(!alive || *abort_flag)) {
                alive = false;
                break;
            }
            tc::mbar_arrive(p_full);
            if (p.fused_write && (ring || rg == 0)) {
                // Write this step's rows whose slot this tile covers (ring), or
                // that no loaded tile covers, or every row (cache), from the new
                // rows to the caches: warp q4 takes rows j = q4, q4 + 4, ...
                for (int j = q4; j < p.k; j += 4) {
                    long long dst_row;
                    int writer;
                    if (ring) {
                        int sj = base_slot + j;
                        if (sj >= p.window) sj -= p.window;
                        writer = sj / kTileKeys < new_tile ? sj / kTileKeys : new_tile;
                        dst_row = (long long)id * p.window + sj;
                    } else if (paged) {
                        writer = new_tile;
                        dst_row = paged_row(p.page_table, p.max_pages, p.page_rows, p.num_pages, b,
                                            ctx + j);
                        if (dst_row < 0) {
                            if (lane == 0) set_status(p.dev_status, CARAT_DEV_BAD_CACHE_ID);
                            continue;
                        }
                    } else {
                        writer = new_tile;
                        dst_row = (long long)id * p.capacity + ctx + j;
                    }
                    if (writer != i) continue;
                    const size_t src = (((size_t)b * p.k + j) * p.kv_heads + c) * D;
                    const size_t dst = ((size_t)dst_row * p.kv_heads + c) * D;
                    const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new + src);
                    const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new + src);
                    uint4 *kd = reinterpret_cast<uint4 *>(p.k_dst + dst);
                    uint4 *vd = reinterpret_cast<uint4 *>(p.v_dst + dst);
                    // Save the row this one displaces (position ctx + j - window),
                    // read by the same lane before it writes the same bytes.
                    const bool save = ring && p.displaced_out && j >= 1 && ctx + j - p.window >= 0;
                    uint4 *dk = nullptr, *dv = nullptr;
                    if (save) {
                        const size_t row = (size_t)p.kv_heads * D;
                        dk = reinterpret_cast<uint4 *>(p.displaced_out +
                                                       ((size_t)b * (p.k - 1) + (j - 1)) * 2 * row +
                                                       (size_t)c * D);
                        dv = dk + row / 8;
                    }
                    for (int e = lane; e < D / 8; e += 32) {
                        if (save) {
                            dk[e] = kd[e];
                            dv[e] = vd[e];
                        }
                        kd[e] = ks[e];
                        vd[e] = vs[e];
                    }
                }
            }
        }
        // ------------------------------------------------------------ epilogue
        if (alive) {
            if (!wait_or_abort(o_done, (idx - 1) & 1, abort_flag, p.dev_status)) alive = false;
            tc::tc_fence_after();
        }
        const int rbl = warp_transpose_reduce<N, false>(l_part, lane);
        float *red_sum = red + 2 * 4 * N;
        constexpr int kHeldL = N >= 32 ? N / 32 : 1;
#pragma unroll
        for (int e = 0; e < kHeldL; ++e) red_sum[q4 * N + rbl + e] = l_part[e];
        alive = !named_bar_softmax_any(!alive || *abort_flag);
        if (alive && p.direct) {
            // This CTA saw every key of its rows: normalise and write the output.
            float inv_l[N];
#pragma unroll
            for (int r = 0; r < N; ++r)
                inv_l[r] = 1.f / (red_sum[r] + red_sum[N + r] + red_sum[2 * N + r] + red_sum[3 * N + r]);
#pragma unroll
            for (int ob = 0; ob < KS; ++ob) {
#pragma unroll
                for (int cb = 0; cb < N / 16; ++cb) {
                    uint32_t r16[16];
                    tc::tmem_ld16(tmem_o + ob * N + lane_off + cb * 16, r16);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = cb * 16 + e;
                        if (r < rows_here) {
                            const int row = row0 + r, j = row / p.group, hp = row % p.group;
                            p.out[(((size_t)b * p.k + j) * p.q_heads + (size_t)c * p.group + hp) * D +
                                  ob * 128 + t] = __uint_as_float(r16[e]) * inv_l[r];
                        }
                    }
                }
            }
        } else if (alive) {
            if (t == 0) {
#pragma unroll
                for (int r = 0; r < N; ++r) {
                    if (r < rows_here) {
                        const float l = red_sum[r] + red_sum[N + r] + red_sum[2 * N + r] + red_sum[3 * N + r];
                        ml[r] = make_float2(m_run[r], l);
                    }
                }
            }
#pragma unroll
            for (int ob = 0; ob < KS; ++ob) {
#pragma unroll
                for (int cb = 0; cb < N / 16; ++cb) {
                    uint32_t r16[16];
                    tc::tmem_ld16(tmem_o + ob * N + lane_off + cb * 16, r16);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = cb * 16 + e;
                        if (r < rows_here) po[(size_t)r * D + ob * 128 + t] = __uint_as_float(r16[e]);
                    }
                }
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tc::tmem_dealloc(tmem, L::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace {

template <int D, int N, int NS, int MINB>
cudaError_t launch_tc(const AttnParams &p, const TcPlan &plan, const TcMaps &maps,
                      cudaStream_t stream) {
    using L = Layout<D, N, NS>;
    static_assert(MINB == 1 || 2 * (L::kAlloc + 1024) <= 233472, "two CTAs must fit one SM");
    auto kernel = attn_tc_kernel<D, N, NS, MINB>;
    static int configured_devices[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured_devices[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (e != cudaSuccess) return e;
        configured_devices[dev] = 1;
    }
    dim3 grid(p.nchunks, p.kv_heads * plan.row_groups, p.batch);
    kernel<<<grid, kThreads, L::kAlloc, stream>>>(p, plan, maps);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

int tc_rows_per_tile(int group, int k) {
    const int rows = group * k;
    if (rows <= 16) return 16;
    if (rows <= 32) return 32;
    return 64;
}

int tc_ctas_per_sm(int head_dim, int rows_per_tile) {
    return (head_dim == 256 && rows_per_tile == 16) ? 2 : 1;
}

bool tc_supported(int head_dim, int group, int k) {
    if (head_dim != 256 && head_dim != 512) return false;
    const int n = tc_rows_per_tile(group, k);
    return group <= n;
}

cudaError_t launch_attention_tc(const AttnParams &p, int tiles_per_chunk, cudaStream_t stream) {
    const int n = tc_rows_per_tile(p.group, p.k);
    TcPlan plan{};
    plan.tiles_per_chunk = tiles_per_chunk;
    plan.pos_per_group = n / p.group;
    if (plan.pos_per_group > p.k) plan.pos_per_group = p.k;
    plan.row_groups = (p.k + plan.pos_per_group - 1) / plan.pos_per_group;

    TcMaps maps{};
    const uint64_t D = (uint64_t)p.head_dim;
    const uint64_t row_bytes = (uint64_t)p.kv_heads * D * 2;
    const uint32_t box3[3] = {64, 1, (uint32_t)kTileKeys};
    const uint64_t rows_total =
        p.source == KeySource::kPaged
            ? (uint64_t)p.num_pages * (uint64_t)p.page_rows
            : (uint64_t)p.num_ids * (uint64_t)(p.source == KeySource::kRing ? p.window : p.capacity);
    const uint64_t dims3[3] = {D, (uint64_t)p.kv_heads, rows_total};
    const uint64_t strides3[2] = {D * 2, row_bytes};
    if (!make_bf16_tensor_map(&maps.k, p.k_base, 3, dims3, strides3, box3, true) ||
        !make_bf16_tensor_map(&maps.v, p.v_base, 3, dims3, strides3, box3, true))
        return cudaErrorInvalidValue;
    if (p.source == KeySource::kRing && p.k > 1) {
        const uint64_t dims4[4] = {D, (uint64_t)p.kv_heads, 2, (uint64_t)p.batch * (p.k - 1)};
        const uint64_t strides4[3] = {D * 2, row_bytes, 2 * row_bytes};
        const uint32_t box4[4] = {64, 1, 1, (uint32_t)kDispRows};
        if (!make_bf16_tensor_map(&maps.disp, p.displaced, 4, dims4, strides4, box4, true))
            return cudaErrorInvalidValue;
    } else {
        maps.disp = maps.k;
    }
    if (p.fused) {
        const uint64_t dimsn[3] = {D, (uint64_t)p.kv_heads, (uint64_t)p.batch * p.k};
        const uint32_t boxn[3] = {64, 1, (uint32_t)kDispRows};
        if (!make_bf16_tensor_map(&maps.knew, p.k_new, 3, dimsn, strides3, boxn, true) ||
            !make_bf16_tensor_map(&maps.vnew, p.v_new, 3, dimsn, strides3, boxn, true))
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
        if (n == 16) return launch_tc<256, 16, 3, 2>(p, plan, maps, stream);
        if (n == 32) return launch_tc<256, 32, 6, 1>(p, plan, maps, stream);
        return launch_tc<256, 64, 5, 1>(p, plan, maps, stream);
    }
    if (n == 16) return launch_tc<512, 16, 4, 1>(p, plan, maps, stream);
    if (n == 32) return launch_tc<512, 32, 5, 1>(p, plan, maps, stream);
    return launch_tc<512, 64, 4, 1>(p, plan, maps, stream);
}

}  // namespace carat
