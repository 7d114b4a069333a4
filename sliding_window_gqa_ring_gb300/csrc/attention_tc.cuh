// attention_tc.cuh -- grouped-query attention on the 5th-generation tensor
// cores (tcgen05 + TMEM) with TMA-staged K/V tiles, scheduled stream-K over a
// persistent grid.
//
// What it computes: for each request b and KV head c, the rows r = j*g + h'
// (the g query heads sharing KV head c times the proposal positions j;
// "Announcing Carat: An inference engine designed for Gemma 4", "Doing it all
// in one kernel can be slower") attend to the keys
// their position may see -- the last `window` positions for a sliding layer
// read in place from the rotated ring ("Improving Decode Throughput on Intel
// Gaudi 3", "Our approach"), every position up to their own for a global
// layer, with the tail past key_count masked ("More FLOPs can be faster").
//
// Tiles.  Keys come in tiles of 128 (ring slots 128i.., or cache rows 128i..,
// plus one tile of displaced rows for a sliding verify with k > 1, or of this
// step's rows for a fused append).  Keys are the M dimension of both
// products, so any number of rows N in {16, 32, 64} fits one tile without
// padding the keys:
//     S^T [128 keys x N rows]  = K_tile [128 x D] . Q^T          (K-major A, B)
//     O^T [128 d   x N rows]  += V_tile^T [d x 128 keys] . P^T   (MN-major A)
// S^T and O^T live in tensor memory; P (bf16; f16 with FP8 rings) is written
// to shared memory by the softmax threads.  Rows beyond 64 are split into row groups.  The
// key-count tail is masked per key, never padded with work: a tile that holds
// no token in some rows has those V rows zeroed in shared memory so their
// contents (zero-initialised or not) cannot reach O.
//
// Schedule.  A unit is one (request, KV head, row group).  When there are at
// least as many units as resident CTA slots and every unit is short (a
// sliding window), units are taken whole ("unit mode"): with bf16 caches CTA
// g simply takes unit g; with FP8 caches (one CTA per SM, several units each)
// the grid is one persistent CTA per SM, CTA g starts with unit g, and once
// its producer has issued a unit's loads it takes the next unit from a work
// counter in the workspace (so that unit's keys stream in while the last one
// finishes), publishing it to the other roles through a small queue in
// shared memory; the launch's last CTA clears the counter.  A whole unit's
// small special tile comes last when the stage ring holds a whole V tile
// besides it (see order_tile).  Otherwise (stream-K): a unit's tiles are
// taken in a fixed order (the small special tile first).  All units'
// tiles, request after request, form one flattened sequence of tiles, and
// the grid -- one CTA per resident slot, so every CTA starts at once -- cuts
// it into contiguous ranges of equal cost (stream-K), where a unit costs its
// tiles plus a fixed charge for the segment boundary it causes, so a range
// that touches more units gets fewer tiles.  A CTA walks its range as
// segments, one per unit it touches, streaming K/V through one stage ring
// without a break between segments.  A segment that covers a whole unit
// writes the normalised output; the at most two others (the range's first
// and last) write a partial (row max, row sum, unnormalised O) to the
// workspace, and the CTA holding a unit's first tile records in a unit table
// the range it starts in, how many ranges it spans and which partial slot
// its first piece uses.  A second launch (attn_fixup_kernel, one CTA per
// (unit, row), started early by programmatic dependent launch and waiting
// for this grid) merges the split units' pieces in parallel.  Ranges are
// long enough that no unit is cut into more than kMaxPieces pieces.  The CTAs
// never wait for one another (the unit queue's counter is an atomic add, never
// a wait).
//
// Warp roles (192 threads):
//   warp 0      computes the CTA's range (a scan over the requests' tile
//               counts), then as TMA producer loads each segment's Q and its
//               K and V tiles in 32 KB stages (128 keys x 128 d, two 64-d
//               boxes with 128-byte swizzle) through an NS-deep stage ring.
//   warp 1      allocates TMEM; one thread issues every tcgen05.mma and the
//               commits that free stages and signal the softmax warps.
//   warps 2-5   write NaN outputs for rejected requests, then run the
//               softmax: thread t owns key t of the tile (TMEM lane t) and
//               reads its N scores 16 rows at a time, masked by position; when
//               some score passes its row's running maximum (log2 domain, kept
//               in shared memory), the tile's row maxima are reduced (a warp
//               transpose-reduction, then across the warps) and O^T and the
//               row sums are rescaled in TMEM; then P is written.  Row sums
//               L^T in TMEM: the MMA thread adds ONES . P^T with the same P as
//               the PV product, which puts the whole sums in every lane; or
//               (LP kernels: unit-mode calls at head_dim 256) each thread adds
//               its key's rounded P of every row into its own lane and the
//               lanes are added up once per segment, which takes those 8
//               products per tile off the MMA thread.  Per segment they write
//               the output or the partial.
//   warps 6-9   (FP8 e4m3 caches only, 320 threads) widen each raw e4m3 stage
//               the producer lands into an f16 stage, in load order, and each
//               segment's Q into f16 with a power-of-two scale per row.
//
// Every wait is bounded (mbar_wait): on a timeout the CTA records
// CARAT_DEV_TIMEOUT, stops issuing work, waits (bounded) for its own copies
// and MMAs in flight, frees its TMEM and returns.
#pragma once

#include <atomic>
#include <cfloat>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "carat_internal.cuh"
#include "tc_common.cuh"
#include "tma_host.h"

namespace carat {

// K/V tensors are mapped with the head dimension cut into 64-element slabs
// as a dimension of its own, so one copy fills a whole stage (two slabs of
// 128 rows) or a whole special tile (every slab of 16 rows): in shared memory
// a box lands slab after slab, each slab its rows of 128 bytes.
struct TcMaps {
    CUtensorMap k;     // (64, rows, D/64, Hkv)            ring slots or cache rows
    CUtensorMap v;
    CUtensorMap disp;  // (64, B*(k-1), D/64, 2, Hkv)      displaced rows, K (0) / V (1)
    CUtensorMap q;     // (D, Hq, k, B)                    queries
    CUtensorMap knew;  // (64, B*k, D/64, Hkv)             this step's rows (fused append)
    CUtensorMap vnew;
};

struct TcPlan {
    int row_groups;
    int pos_per_group;    // proposal positions per row group
    int unit_mode;        // 1: whole units (bf16: CTA g takes unit g, grid = units;
                          // FP8: persistent CTAs and the unit queue); 0: stream-K
    // stream-K with two row groups: CTAs 2r and 2r + 1 walk the same range r
    // of the (request, KV head) order, one row group each, so each K/V tile is
    // read by both at about the same time and the second read comes from L2
    int paired;
};


namespace {

constexpr int kTileKeys = 128;
constexpr int kBoxBytes = 128 * 128;        // [128 keys][64 bf16]
constexpr int kStageBytes = 2 * kBoxBytes;  // 128 keys x 128 d
constexpr int kDispRows = 16;               // displaced rows loaded per tile (>= k - 1)
constexpr int kMaxPieces = 64;              // CTAs one unit may be split across
constexpr int kUnitQ = 4;                   // unit mode: queue slots of units taken
constexpr int kDispBoxBytes = kDispRows * 128;
constexpr int kThreads = 192;
constexpr int kConvThreads = 128;           // FP8 caches: four more warps widen the stages
constexpr uint32_t kFull = 0xffffffffu;

template <int D, int N, int NS, int NR = 0>
struct Layout {
    static constexpr int KS = D / 128;                 // stages per K (or V) tile
    static constexpr int kQBlock = N * 128;            // one 64-d block of Q rows
    // FP8 caches (NR > 0): NR raw stages of e4m3 bytes (128 keys x 128 d) in
    // front of the 16-bit stages the tensor core reads.
    static constexpr int kRawBytes = 128 * 128;
    static constexpr int kOffRaw = NS * kStageBytes;
    static constexpr int kOffQ = kOffRaw + NR * kRawBytes;
    static constexpr int kOffP = kOffQ + (D / 64) * kQBlock;
    static constexpr int kPBlock = N * 128;            // 64 keys of P rows
    // 8 rows of 128 bytes of ones (bf16, or f16 with FP8 caches): the A operand
    // of the row-sum product L^T += ONES . P^T, read for every 8-row group
    static constexpr int kOffOnes = kOffP + 2 * kPBlock;
    static constexpr int kOffRed = kOffOnes + 1024;
    // floats of the reduction area: the 4 softmax warps' tile maxima (4 x N),
    // the running row maxima, this tile's rescale factors, a finished
    // segment's row maxima, (lane-kept row sums) the 4 warps' row sums of a
    // finished segment (4 x N) and their totals, then (FP8) the row score
    // scales of two segments
    static constexpr int kRedMax = 0, kRedM = 4 * N, kRedAlpha = 5 * N, kRedMrow = 6 * N;
    static constexpr int kRedLsum = 7 * N, kRedL = 11 * N;
    static constexpr int kRedQscale = 12 * N;
    static constexpr int kRedFloats = 12 * N + (NR > 0 ? 2 : 0) * N;
    static constexpr int kOffBar = kOffRed + kRedFloats * 4;
    static constexpr int kNumBars = 2 * NS + 7 + 2 * NR + (NR > 0 ? 2 + 2 * kUnitQ : 0);
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;   // SkShared
    static constexpr int kBytes = kOffMisc + (NR > 0 ? 256 : 128);
    static constexpr int kAlloc = kBytes + 1024;       // base alignment slack
    // Two S^T buffers, then per segment an O^T buffer (KS blocks of N columns)
    // and a row-sum buffer L^T (N columns); two of each when they fit the 512
    // columns, so one segment's output is written while the next accumulates.
    static constexpr bool kDoubleO = N * (2 + 2 * (KS + 1)) <= 512;
    static constexpr int kTmemUsed = N * (2 + (kDoubleO ? 2 : 1) * (KS + 1));
    static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64
                                   : kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
    static_assert(kAlloc <= 232448, "more dynamic shared memory than one CTA may use");
    // The softmax warps zero masked V rows while all KS stages of a V tile are
    // resident, before the tile's PV product releases any of them.
    static_assert(NS >= KS, "the stage ring must hold a whole V tile");
    static_assert(kOffRaw % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0 &&
                      kPBlock % 1024 == 0 && kOffOnes % 1024 == 0 &&
                      kQBlock % 1024 == 0,
                  "operand blocks must be 1024-byte aligned for the 128-byte swizzle");
};

// Unit mode: a unit the producer took, as every role needs it (request,
// unit within it, ring or cache id, context length, tiles, special tile);
// u = -1: no unit left.
struct UnitDesc {
    int u, b, ur, id, ntiles, special;
    long long ctx;
};

// Per-CTA schedule, written by warp 0 before the block-wide barrier and read
// by every role.
struct SkShared {
    uint32_t tmem_slot;
    int abort_flag;
    int b0, ur0, off0;            // first segment: request, unit within it, order offset
    int id0, ntiles0, special0;   // first request's id, tiles and special tile
    long long ctx0;               // first request's context length
    long long s, e;               // tile range [s, e) of the flattened order
    long long len;                // stream-K: cost of one range (tiles plus unit charges)
    long long ucost0;             // cost position of the first segment's unit
    int segc;                     // cost charged per unit, in tiles
    int special_last;             // the units' special tiles come last (see order_tile)
    // FP8 unit mode: the units taken, in order (only FP8 kernels reserve the
    // space: the misc area is 128 bytes with bf16 caches, 256 with FP8)
    UnitDesc uq[kUnitQ];
};
static_assert(offsetof(SkShared, uq) <= 128 && sizeof(SkShared) <= 256,
              "SkShared must fit the misc area");

// Tiles of request b (0 when request_ok rejects it) and its special tile.
__device__ __forceinline__ int request_tiles(const AttnParams &p, int b, int *id, long long *ctx,
                                             int *special) {
    *special = -1;
    if (!request_ok(p, b, id, ctx)) return 0;
    return tc_request_tiles(p.source, p.window, p.k, *ctx + p.k, p.fused != 0, special);
}

// One unit's share of a CTA's range.
struct Segment {
    int b, id, c, rg, unit;
    long long ctx;
    int ntiles, special;       // tiles of the unit and its special tile (-1: none)
    int x0, x1;                // order indices [x0, x1) of the unit's tiles covered here
    bool special_last;         // the special tile comes last (else first)
    long long start;           // flattened index of the segment's first tile
    long long unit_start;      // flattened index of the unit's first tile
    long long unit_cost;       // cost position of the unit (see locate_range)
};

// Tile index of order index x: the special tile (this step's rows of a fused
// append, or the displaced rows of a sliding verify; always the last tile
// index) comes first, or, in unit mode with a ring deeper than one V tile,
// last (the natural order), so that a unit ends with its smallest PV product
// rather than a whole tile's.  It takes a single stage, held until its PV
// product.
__device__ __forceinline__ int order_tile(const Segment &sg, int x) {
    if (sg.special >= 0 && !sg.special_last) return x == 0 ? sg.special : x - 1;
    return x;
}

// Walks a CTA's range as segments.  Every role runs its own copy over the
// same inputs, so all of them see the same sequence.
struct SegIter {
    long long pos, end;
    int b, ur, off;
    int id, ntiles, special;
    long long ctx;
    long long ucost;   // cost position of the current unit
    int segc;          // cost charged per unit
    int rg_fixed;      // paired schedule: this CTA's row group (else -1)
    bool special_last; // the special tile comes last in each unit's order

    __device__ void init(const AttnParams &p, const SkShared *sk, int rg = -1) {
        rg_fixed = rg;
        ucost = sk->ucost0;
        segc = sk->segc;
        special_last = sk->special_last != 0;
        pos = sk->s;
        end = sk->e;
        b = sk->b0;
        ur = sk->ur0;
        off = sk->off0;
        id = sk->id0;
        ctx = sk->ctx0;
        ntiles = sk->ntiles0;
        special = sk->special0;
    }

    // Unit mode: unit u, whole, is the next segment.
    __device__ void set_unit(const AttnParams &p, int upr, int u) {
        b = u / upr;
        ur = u - b * upr;
        ntiles = request_tiles(p, b, &id, &ctx, &special);
        pos = 0;
        end = ntiles;
        off = 0;
    }
    // The same from the producer's description of it.
    __device__ void set_unit(const volatile UnitDesc &d) {
        b = d.b;
        ur = d.ur;
        id = d.id;
        ctx = d.ctx;
        ntiles = d.ntiles;
        special = d.special;
        pos = 0;
        end = ntiles;
        off = 0;
    }

    // upr: units per request in the flattened order (KV heads when paired).
    __device__ bool next(const AttnParams &p, int upr, int row_groups, Segment &sg) {
        if (pos >= end || ntiles <= off) return false;
        const long long left = end - pos;
        const int len = (long long)(ntiles - off) < left ? ntiles - off : (int)left;
        sg.b = b;
        sg.id = id;
        sg.ctx = ctx;
        sg.ntiles = ntiles;
        sg.special = special;
        sg.special_last = special_last;
        if (rg_fixed >= 0) {
            sg.c = ur;
            sg.rg = rg_fixed;
            sg.unit = (b * upr + ur) * row_groups + rg_fixed;
        } else {
            sg.c = ur / row_groups;
            sg.rg = ur % row_groups;
            sg.unit = b * upr + ur;
        }
        sg.x0 = off;
        sg.x1 = off + len;
        sg.start = pos;
        sg.unit_start = pos - off;
        sg.unit_cost = ucost;
        pos += len;
        off += len;
        if (off == ntiles && pos < end) {
            off = 0;
            ucost += ntiles + segc;
            if (++ur == upr) {
                ur = 0;
                ntiles = 0;
                while (ntiles == 0 && b + 1 < p.batch) {
                    ++b;
                    ntiles = request_tiles(p, b, &id, &ctx, &special);
                }
            }
        }
        return true;
    }
};

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Warp 0: this CTA's tile range of the flattened order and where it starts.
// Ranges have equal cost, not equal tile counts: each unit is charged segc
// tiles besides its own (a segment boundary writes an output or a partial,
// reloads Q and refills the stage ring), so a range that touches several units
// gets fewer tiles.  In cost positions, unit u (the u-th unit that has tiles)
// starts at U_u = P_u + segc * u, P_u being the flattened index of its first
// tile, and its tile o sits at U_u + segc + o; tile t belongs to range
// floor(cost(t) / T), T the cost of one range (the last range takes the rest).
// Runs once per CTA from a cold instruction cache, so it is kept to short
// loops (32 requests per pass, the later passes re-reading through L2) rather
// than unrolled code.
__device__ __noinline__ void locate_range(const AttnParams &p, int upr, int lane, SkShared *sk,
                                          int ranges, int rix, int seg_cost) {
    long long tiles = 0, units = 0;
    int nmax = 0;
#pragma unroll 1
    for (int base = 0; base < p.batch; base += 32) {
        const int b = base + lane;
        int v = 0;
        if (b < p.batch) {
            int id, sp;
            long long ctx;
            v = request_tiles(p, b, &id, &ctx, &sp);
        }
        tiles += v;
        units += v > 0 ? 1 : 0;
        nmax = max(nmax, v);
    }
    tiles = warp_sum_ll(tiles) * upr;
    units = warp_sum_ll(units) * upr;
    nmax = warp_max_int(nmax);
    // A call with fewer tiles than ranges gives every tile its own range.
    const int c = tiles >= ranges ? seg_cost : 0;
    const long long cost = tiles + (long long)c * units;
    long long T = (cost + ranges - 1) / ranges;
    // at most kMaxPieces ranges touch one unit; no range is empty but the last
    const long long min_T = (nmax + kMaxPieces - 3) / (kMaxPieces - 2);
    if (T < min_T) T = min_T;
    if (T < c + 1) T = c + 1;
    // First tile whose cost position is >= X: its flattened index, request,
    // unit within the request, offset in the unit and the unit's cost
    // position (index = tiles when there is none).
    struct Pos {
        long long tile, ucost;
        int b, ur, off, id, nt, sp;
        long long ctx;
    };
    auto find = [&](long long X, Pos &r) -> bool {
        long long cum_cost = 0, cum_tiles = 0;
#pragma unroll 1
        for (int base = 0; base < p.batch; base += 32) {
            const int b = base + lane;
            int v = 0, id = 0, sp = -1;
            long long ctx = 0;
            if (b < p.batch) v = request_tiles(p, b, &id, &ctx, &sp);
            const long long vc = v > 0 ? (long long)upr * (v + c) : 0;
            long long inc = vc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += y;
            }
            long long inct = (long long)upr * v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(kFull, inct, o);
                if (lane >= o) inct += y;
            }
            const unsigned hit = __ballot_sync(kFull, cum_cost + inc > X);
            if (hit) {
                const int src = __ffs(hit) - 1;
                if (lane == src) {
                    const long long rem = X - (cum_cost + inc - vc);   // cost into request b
                    const long long per = v + c;
                    const int j = (int)(rem / per);
                    const long long r2 = rem - (long long)j * per;
                    const int o = r2 <= c ? 0 : (int)(r2 - c);
                    r.tile = cum_tiles + inct - (long long)upr * v + (long long)j * v + o;
                    r.ucost = cum_cost + inc - vc + (long long)j * per;
                    r.b = b;
                    r.ur = j;
                    r.off = o;
                    r.id = id;
                    r.nt = v;
                    r.sp = sp;
                    r.ctx = ctx;
                }
                r.tile = __shfl_sync(kFull, r.tile, src);
                r.ucost = __shfl_sync(kFull, r.ucost, src);
                r.b = __shfl_sync(kFull, r.b, src);
                r.ur = __shfl_sync(kFull, r.ur, src);
                r.off = __shfl_sync(kFull, r.off, src);
                r.id = __shfl_sync(kFull, r.id, src);
                r.nt = __shfl_sync(kFull, r.nt, src);
                r.sp = __shfl_sync(kFull, r.sp, src);
                r.ctx = __shfl_sync(kFull, r.ctx, src);
                return true;
            }
            cum_cost += __shfl_sync(kFull, inc, 31);
            cum_tiles += __shfl_sync(kFull, inct, 31);
        }
        return false;
    };
    Pos st{}, en{};
    st.tile = en.tile = tiles;
    const long long X0 = (long long)rix * T;
    bool have = X0 < cost && find(X0, st);
    if (have && rix + 1 < ranges && (long long)(rix + 1) * T < cost) {
        // with no unit charge cost positions are tile indices: no second scan
        if (c == 0)
            en.tile = (long long)(rix + 1) * T;
        else
            find((long long)(rix + 1) * T, en);
    }
    if (!have) st.tile = tiles;
    if (lane == 0) {
        sk->s = st.tile;
        sk->e = en.tile;
        sk->len = T;
        sk->segc = c;
        sk->b0 = have ? st.b : 0;
        sk->ur0 = have ? st.ur : 0;
        sk->off0 = have ? st.off : 0;
        sk->ntiles0 = have ? st.nt : 0;
        sk->special0 = have ? st.sp : -1;
        sk->id0 = have ? st.id : 0;
        sk->ctx0 = have ? st.ctx : 0;
        sk->ucost0 = have ? st.ucost : 0;
    }
    __syncwarp();
}

// Warp 0, unit mode with bf16 caches: this CTA's range is unit blockIdx.x,
// whole (its own frame: tiles [0, n)); nothing is split, so no partials and
// no merges.
__device__ void locate_unit(const AttnParams &p, int upr, int lane, SkShared *sk) {
    if (lane == 0) {
        const int b = blockIdx.x / upr;
        int id = 0, sp = -1;
        long long ctx = 0;
        const int nt = b < p.batch ? request_tiles(p, b, &id, &ctx, &sp) : 0;
        sk->s = 0;
        sk->e = nt;
        sk->len = nt > 0 ? nt : 1;
        sk->ucost0 = 0;
        sk->segc = 0;
        sk->b0 = b;
        sk->ur0 = blockIdx.x % upr;
        sk->off0 = 0;
        sk->ntiles0 = nt;
        sk->special0 = sp;
        sk->id0 = id;
        sk->ctx0 = ctx;
    }
    __syncwarp();
}

// Warp 0, unit mode with FP8 caches: every role's iterator starts empty; each
// unit, whole, comes through the unit queue (unit blockIdx.x first, then the
// ones the work counter hands out).  Nothing is split, so no partials and no
// merges.
__device__ void locate_unit_queue(SkShared *sk, int lane) {
    if (lane == 0) {
        sk->s = 0;
        sk->e = 0;
        sk->len = 1;
        sk->ucost0 = 0;
        sk->segc = 0;
        sk->b0 = 0;
        sk->ur0 = 0;
        sk->off0 = 0;
        sk->ntiles0 = 0;
        sk->special0 = -1;
        sk->id0 = 0;
        sk->ctx0 = 0;
    }
    __syncwarp();
}

// Unit mode's work counter and count of finished CTAs: a 64-bit word whose
// high 40 bits hold the launch's epoch and low 24 bits the count; a word
// holding another epoch (left by an earlier launch, or never written) counts
// as 0.  Adds one and returns the count before the addition, or -1 if the
// word never settled.  One atomic add in the common case (a compare-and-swap
// loop would serialise the CTAs that finish a unit at about the same time,
// one round trip to L2 each).  A caller that finds the word stale replaces
// the stale value, whatever it has become, by (epoch, 1) and takes count 0,
// unless another caller installed the epoch first, in which case it adds
// again.  Each caller adds to a stale word at most once per installation, so
// the replacement loop ends; the epoch is installed once, so every count is
// returned once.
__device__ long long tagged_increment(unsigned long long *w, unsigned long long epoch) {
#pragma unroll 1
    for (int tries = 0; tries < 64; ++tries) {
        const unsigned long long old = atomicAdd(w, 1ull);
        if ((old >> 24) == epoch) return (long long)(old & 0xffffffull);
        unsigned long long cur = old + 1;
#pragma unroll 1
        for (int k = 0; k < 65536; ++k) {
            const unsigned long long seen = atomicCAS(w, cur, (epoch << 24) + 1);
            if (seen == cur) return 0;
            if ((seen >> 24) == epoch) break;
            cur = seen;
        }
    }
    return -1;
}

// Four e4m3 values (first in the low byte) -> four f16 values, two per word
// (first in the low half).  Exact: every e4m3 value, subnormals included, is
// an f16 value.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// One 128-byte row of e4m3 (a 128-d block, 128-byte swizzle at row `row`)
// -> its f16 image: 16-byte chunk c' of 64-d slab (c / 4) of the
// destination, each slab a 128-byte swizzled row; zero: write zeros.  All
// eight loads are issued before the first conversion (source and
// destination are both shared memory, so the compiler would not hoist a load
// above an earlier store by itself).
__device__ __forceinline__ void convert_row(const uint8_t *src, uint8_t *dst0, uint8_t *dst1,
                                            int row, bool zero) {
    const int sw = row & 7;
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        v[c] = zero ? make_uint4(0, 0, 0, 0)
                    : *reinterpret_cast<const uint4 *>(src + ((c ^ sw) << 4));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 o0, o1;
        e4m3x4_to_f16x4(v[c].x, o0.x, o0.y);
        e4m3x4_to_f16x4(v[c].y, o0.z, o0.w);
        e4m3x4_to_f16x4(v[c].z, o1.x, o1.y);
        e4m3x4_to_f16x4(v[c].w, o1.z, o1.w);
        uint8_t *d = (c < 4) ? dst0 : dst1;
        const int cc = 2 * (c & 3);
        *reinterpret_cast<uint4 *>(d + ((cc ^ sw) << 4)) = o0;
        *reinterpret_cast<uint4 *>(d + (((cc + 1) ^ sw) << 4)) = o1;
    }
}

// Two fp32 values -> an f16 pair (first in the low half), round to nearest.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// FP8 caches: the N query rows of a segment, loaded as bf16 (D/64 swizzled
// blocks of N rows x 128 bytes), rewritten in place as f16 for the f16
// tensor-core products.  Row r is multiplied by 2^s_r, s_r chosen so its
// largest |q| lands in [2^14, 2^15): every element down to 2^-28 of that
// maximum keeps its bf16 value exactly, and the row's scores come out
// multiplied by 2^s_r, which qscale[r] = scale_log2 * 2^-s_r takes back out
// (both factors powers of two, so nothing rounds).  128 threads, 128 / N per
// row, each over every (128 / N)-th 16-byte chunk of its row.
template <int D, int N, int QBlock>
__device__ __forceinline__ void convert_q_f16(uint8_t *s_q, float *qscale, float scale_log2,
                                              int t) {
    constexpr int kTpr = 128 / N;
    const int r = t / kTpr, j = t % kTpr;
    uint8_t *row = s_q + r * 128;
    const int sw = r & 7;
    uint32_t amax = 0;   // |q| bits; ordered like the values for non-NaN inputs
#pragma unroll
    for (int ch = j; ch < D / 8; ch += kTpr) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + (ch / 8) * QBlock +
                                                         (((ch % 8) ^ sw) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            amax = max(amax, max((w[e] << 16) & 0x7fffffffu, w[e] & 0x7fff0000u));
    }
#pragma unroll
    for (int o = 1; o < kTpr; o <<= 1) amax = max(amax, __shfl_xor_sync(kFull, amax, o));
    // floor(log2 amax) for a normal amax; zero or subnormal rows take s = 100
    int s = 14 - ((int)(amax >> 23) - 127);
    s = s < -100 ? -100 : (s > 100 ? 100 : s);
    const float up = __int_as_float((127 + s) << 23);
#pragma unroll
    for (int ch = j; ch < D / 8; ch += kTpr) {
        uint4 *a = reinterpret_cast<uint4 *>(row + (ch / 8) * QBlock + (((ch % 8) ^ sw) << 4));
        const uint4 v = *a;
        *a = make_uint4(f16x2_rn(bf16lo(v.x) * up, bf16hi(v.x) * up),
                        f16x2_rn(bf16lo(v.y) * up, bf16hi(v.y) * up),
                        f16x2_rn(bf16lo(v.z) * up, bf16hi(v.z) * up),
                        f16x2_rn(bf16lo(v.w) * up, bf16hi(v.w) * up));
    }
    if (j == 0) qscale[r] = scale_log2 * __int_as_float((127 - s) << 23);
}

// FP8 (ring, append done before the call): whether key t of ring tile i
// holds no token, so its V row is widened as zeros (its contents, zero or
// not, must not reach O through P = 0).  held: tokens the ring holds.
__device__ __forceinline__ bool ring_key_empty(int i, int t, int window, long long held) {
    if ((long long)(i + 1) * kTileKeys <= (held < window ? held : (long long)window)) return false;
    const long long newest = held - 1;
    const int slot = i * kTileKeys + t;
    if (newest < 0 || slot >= window) return true;
    long long delta = newest % window - slot;
    if (delta < 0) delta += window;
    return newest - delta < 0;
}

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
// The elapsed time is a signed difference, so a global timer that steps
// backwards cannot end the wait early.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int *dev_status) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (tc::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((long long)(tc::globaltimer_ns() - t0) > 2000000000ll) {
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

// LP: the row sums L^T are kept per lane by the softmax threads (each thread
// adds its key's P of every row into its own lane, the lanes are added up once
// per segment) instead of the MMA thread's ONES . P^T product.
template <int D, int N, int NS, int MINB, int NR = 0, bool LP = false>
__global__ void __launch_bounds__(NR > 0 ? kThreads + kConvThreads : kThreads, MINB)
    attn_tc_kernel(const AttnParams p, const TcPlan plan, const __grid_constant__ TcMaps maps) {
    using L = Layout<D, N, NS, NR>;
    constexpr int KS = L::KS;
    // FP8 caches: the producer fills raw e4m3 stages, the widening warps
    // convert each into an f16 stage (exactly: every e4m3 value is an f16
    // value, and one conversion instruction widens two of them) and rewrite
    // each segment's Q as f16 with a power-of-two scale per row, the softmax
    // warps write P as f16; the tensor core then runs the same products with
    // f16 operands.
    constexpr bool F8 = NR > 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int upr = p.kv_heads * plan.row_groups;   // units per request
    const bool paired = plan.paired != 0;
    const int upo = paired ? p.kv_heads : upr;      // units per request in the flattened order
    const int my_rg = paired ? (int)(blockIdx.x & 1) : -1;
    const bool ring = p.source == KeySource::kRing;
    const bool paged = p.source == KeySource::kPaged;

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
    uint64_t *q_empty = s_full + 5;
    uint64_t *fin = s_full + 6;
    uint64_t *raw_full = s_full + 7;     // [NR] FP8: e4m3 stage landed
    uint64_t *raw_empty = raw_full + NR; // [NR] FP8: e4m3 stage converted
    uint64_t *qs_ready = raw_empty + NR; // [2] FP8: a segment's Q rewritten (segments alternate)
    uint64_t *uq_full = qs_ready + (NR > 0 ? 2 : 0);   // [kUnitQ] unit mode: slot written
    uint64_t *uq_empty = uq_full + kUnitQ;             // [kUnitQ] unit mode: slot read by all
    uint8_t *s_raw = smem + L::kOffRaw;
    SkShared *sk = reinterpret_cast<SkShared *>(smem + L::kOffMisc);
    volatile int *abort_flag = &sk->abort_flag;
    volatile UnitDesc *unit_q = sk->uq;
    float *red = reinterpret_cast<float *>(smem + L::kOffRed);
    float *s_qscale = red + L::kRedQscale;   // FP8: row score scales of two segments (even, odd)
    uint8_t *s_q = smem + L::kOffQ;
    uint8_t *s_p = smem + L::kOffP;

    // Load / consume order of a segment's n tiles' K and V parts: K(0), then
    // K(x+1) before V(x), then V(n-1), so the next tile's keys stream in and
    // its scores are computed while this tile's softmax runs.  Part index of
    // V(x) in that order (each part is KS stages):
    auto v_part = [](int x, int n) { return x == n - 1 ? 2 * n - 1 : 2 * x + 2; };

    // ------------------------------------------------------------ producer state
    // (thread 0): the segment being loaded and the next stage load to issue.
    SegIter pit;
    Segment ps{};
    bool p_have = false, p_qdone = false, alive_p = true, p_units_done = false;
    int ppart = 0, pks = 0, psi = 0;
    uint32_t qcnt = 0;   // Q copies issued
    uint32_t cnt = 0;
    uint64_t pol = 0;
    // Paged caches: the page-table entries of the two pages last used and one
    // read ahead (the page after the newest), so a page-table read is in
    // flight while earlier stages stream instead of stalling the issue path.
    int pt_i0 = -1, pt_p0 = 0, pt_i1 = -1, pt_p1 = 0, pt_in = -1, pt_pn = 0;
    auto page_of = [&](int b, int pi) -> int {
        if (pi == pt_i0) return pt_p0;
        if (pi == pt_i1) return pt_p1;
        const int page = pi == pt_in ? pt_pn : p.page_table[(size_t)b * p.max_pages + pi];
        pt_i1 = pt_i0;
        pt_p1 = pt_p0;
        pt_i0 = pi;
        pt_p0 = page;
        pt_in = -1;
        if (pi + 1 < p.max_pages) {
            pt_in = pi + 1;
            pt_pn = p.page_table[(size_t)b * p.max_pages + pi + 1];
        }
        return page;
    };
    // Issue stage loads in order until `limit` stages have been issued or the
    // range runs out; a stage is reused only after the MMA released it.  With
    // first_only the producer stops at the end of the first segment (the
    // next segment's Q waits for MMAs that start after the block barrier).
    // Unit mode: the CTA's next unit with tiles -- unit blockIdx.x first, then
    // the ones the work counter hands out (gridDim.x + count) -- set as the
    // producer's next segment and published in the unit queue for the other
    // roles, or -1 (published too) when none is left.  Its slot is reused once
    // every role has read what it held kUnitQ units before.
    auto next_unit = [&]() -> bool {
        if (p_units_done) return false;
        const int total = p.batch * upr;
        const int slot = psi % kUnitQ;
        if (psi >= kUnitQ && !wait_or_abort(&uq_empty[slot], ((psi / kUnitQ) & 1) ^ 1,
                                            abort_flag, p.dev_status)) {
            alive_p = false;
            return false;
        }
        auto grab = [&]() -> int {
            const long long c = tagged_increment(&p.sched[0], p.sched_epoch);
            if (c < 0) {
                set_status(p.dev_status, CARAT_DEV_TIMEOUT);
                return total;
            }
            return (int)min((long long)gridDim.x + c, (long long)total);
        };
        int u = psi == 0 ? (int)blockIdx.x : grab();
        while (u < total) {
            pit.set_unit(p, upr, u);
            if (pit.ntiles > 0) break;
            u = grab();
        }
        volatile UnitDesc &d = unit_q[slot];
        if (u >= total) {
            u = -1;
            p_units_done = true;
        } else {
            d.b = pit.b;
            d.ur = pit.ur;
            d.id = pit.id;
            d.ctx = pit.ctx;
            d.ntiles = pit.ntiles;
            d.special = pit.special;
        }
        d.u = u;
        tc::mbar_arrive(&uq_full[slot]);
        return u >= 0;
    };
    auto produce = [&](uint32_t limit, bool first_only) {
        while (alive_p && cnt < limit) {
            if (!p_have) {
                if (first_only && psi > 0) return;
                if constexpr (F8) {
                    if (plan.unit_mode && !next_unit()) return;
                }
                if (!pit.next(p, upo, plan.row_groups, ps)) return;
                p_have = true;
                p_qdone = false;
                ppart = 0;
                pks = 0;
                pt_i0 = pt_i1 = pt_in = -1;
            }
            if (!p_qdone) {
                // This segment's Q: the buffer is free once the previous
                // segment's last QK product has finished.
                if (psi > 0 &&
                    !wait_or_abort(q_empty, (psi - 1) & 1, abort_flag, p.dev_status)) {
                    alive_p = false;
                    break;
                }
                tc::mbar_arrive_expect_tx(q_full, (D / 64) * 128 * p.group * plan.pos_per_group);
#pragma unroll
                for (int db = 0; db < D / 64; ++db)
                    tc::tma_load_4d(s_q + db * L::kQBlock, &maps.q, db * 64, ps.c * p.group,
                                    ps.rg * plan.pos_per_group, ps.b, q_full, pol);
                p_qdone = true;
                ++qcnt;
            }
            const int n = ps.x1 - ps.x0;
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
            const int i = order_tile(ps, ps.x0 + x);
            const bool special = i == ps.special;
            if (special && is_v) {
                // The special tile's V rows came in the stage of its K rows.
                if (++ppart == 2 * n) {
                    p_have = false;
                    ++psi;
                }
                continue;
            }
            if constexpr (F8) {
                // raw e4m3 stage; its slot is free once converted
                const int r = cnt % NR;
                if (cnt >= NR && !wait_or_abort(&raw_empty[r], ((cnt / NR) & 1) ^ 1, abort_flag,
                                                p.dev_status)) {
                    alive_p = false;
                    break;
                }
                uint8_t *rdst = s_raw + r * L::kRawBytes;
                if (special) {
                    // displaced rows: 16 rows x D bytes of K, then of V
                    tc::mbar_arrive_expect_tx(&raw_full[r], 2 * (D / 128) * kDispRows * 128);
                    tc::tma_load_5d(rdst, &maps.disp, 0, ps.b * (p.k - 1), 0, 0, ps.c, &raw_full[r],
                                    pol);
                    tc::tma_load_5d(rdst + (D / 128) * kDispRows * 128, &maps.disp, 0,
                                    ps.b * (p.k - 1), 0, 1, ps.c, &raw_full[r], pol);
                    ++cnt;
                    if (++ppart == 2 * n) {
                        p_have = false;
                        ++psi;
                    }
                    continue;
                }
                const long long row = ring ? (long long)ps.id * p.window + (long long)i * kTileKeys
                                           : (long long)ps.id * p.capacity + (long long)i * kTileKeys;
                tc::mbar_arrive_expect_tx(&raw_full[r], L::kRawBytes);
                tc::tma_load_4d(rdst, is_v ? &maps.v : &maps.k, 0, (int)row, pks, ps.c, &raw_full[r],
                                pol);
                ++cnt;
                if (++pks == KS) {
                    pks = 0;
                    if (++ppart == 2 * n) {
                        p_have = false;
                        ++psi;
                    }
                }
                continue;
            }
            const int s = cnt % NS;
            if (cnt >= NS &&
                !wait_or_abort(&empty[s], ((cnt / NS) & 1) ^ 1, abort_flag, p.dev_status)) {
                alive_p = false;
                break;
            }
            uint8_t *dst = smem + s * kStageBytes;
            if (special) {
                // One stage holds the whole special tile: D/64 boxes of 16 K
                // rows, then D/64 boxes of 16 V rows (displaced rows of a
                // sliding verify, or this step's rows of a fused append).
                tc::mbar_arrive_expect_tx(&full[s], 2 * (D / 64) * kDispBoxBytes);
                uint8_t *vdst = dst + (D / 64) * kDispBoxBytes;
                if (p.fused) {
                    tc::tma_load_4d(dst, &maps.knew, 0, ps.b * p.k, 0, ps.c, &full[s], pol);
                    tc::tma_load_4d(vdst, &maps.vnew, 0, ps.b * p.k, 0, ps.c, &full[s], pol);
                } else {
                    tc::tma_load_5d(dst, &maps.disp, 0, ps.b * (p.k - 1), 0, 0, ps.c, &full[s], pol);
                    tc::tma_load_5d(vdst, &maps.disp, 0, ps.b * (p.k - 1), 0, 1, ps.c, &full[s],
                                    pol);
                }
                ++cnt;
                if (++ppart == 2 * n) {
                    p_have = false;
                    ++psi;
                }
                continue;
            }
            long long row = 0;
            {
                if (ring) {
                    row = (long long)ps.id * p.window + (long long)i * kTileKeys;
                } else if (paged) {
                    // A tile never straddles pages (page_rows is a multiple of
                    // 128).  A page id outside the pool loads the zero fill
                    // past the tensor's end and is reported.
                    const long long t = (long long)i * kTileKeys;
                    const int page = page_of(ps.b, (int)(t / p.page_rows));
                    if (page < 0 || page >= p.num_pages) {
                        set_status(p.dev_status, CARAT_DEV_BAD_CACHE_ID);
                        row = (long long)p.num_pages * p.page_rows;
                    } else {
                        row = (long long)page * p.page_rows + t % p.page_rows;
                    }
                } else {
                    row = (long long)ps.id * p.capacity + (long long)i * kTileKeys;
                }
            }
            tc::mbar_arrive_expect_tx(&full[s], kStageBytes);
            // two 64-d slabs (d = 128 pks ..) of the tile's 128 rows
            tc::tma_load_4d(dst, is_v ? &maps.v : &maps.k, 0, (int)row, 2 * pks, ps.c, &full[s], pol);
            ++cnt;
            if (++pks == KS) {
                pks = 0;
                if (++ppart == 2 * n) {
                    p_have = false;
                    ++psi;
                }
            }
        }
    };

    // Unit mode, every role but the producer: the k-th unit this CTA takes
    // (the k-th the producer published), set as the iterator's next segment.
    // 1: a unit; 0: no unit left; -1: the wait gave up.
    auto take_unit = [&](SegIter &it, int k) -> int {
        const int slot = k % kUnitQ;
        if (!wait_or_abort(&uq_full[slot], (k / kUnitQ) & 1, abort_flag, p.dev_status)) return -1;
        const int u = unit_q[slot].u;
        if (u >= 0) it.set_unit(unit_q[slot]);
        tc::mbar_arrive(&uq_empty[slot]);
        return u >= 0 ? 1 : 0;
    };

    // ------------------------------------------------------------ prologue
    // The merge launch that follows a stream-K launch may start as soon as
    // every CTA of this grid is running; it waits for this grid to finish.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 0) {
        if (lane == 0) {
            // descriptors first: their fetch overlaps the range computation
            tc::tma_prefetch_map(&maps.q);
            tc::tma_prefetch_map(&maps.k);
            tc::tma_prefetch_map(&maps.v);
            tc::tma_prefetch_map(p.fused ? &maps.knew : &maps.disp);
            if (p.fused) tc::tma_prefetch_map(&maps.vnew);
            for (int i = 0; i < NS; ++i) {
                // bf16 stage filled by TMA (one arrival with its bytes), or
                // with FP8 caches by the 128 converting threads
                tc::mbar_init(&full[i], F8 ? kConvThreads : 1);
                tc::mbar_init(&empty[i], 1);
            }
            for (int i = 0; i < NR; ++i) {
                tc::mbar_init(&raw_full[i], 1);
                tc::mbar_init(&raw_empty[i], kConvThreads);
            }
            tc::mbar_init(&s_full[0], 1);
            tc::mbar_init(&s_full[1], 1);
            tc::mbar_init(p_full, 128);
            tc::mbar_init(o_done, 1);
            tc::mbar_init(q_full, 1);
            if (F8) {
                tc::mbar_init(&qs_ready[0], kConvThreads);
                tc::mbar_init(&qs_ready[1], kConvThreads);
            }
            tc::mbar_init(q_empty, 1);
            tc::mbar_init(fin, 1);
            for (int i = 0; i < (F8 ? kUnitQ : 0); ++i) {
                // read by the MMA thread, the 128 softmax threads and the 128
                // widening threads
                tc::mbar_init(&uq_full[i], 1);
                tc::mbar_init(&uq_empty[i], 1 + 128 + kConvThreads);
            }
            sk->abort_flag = 0;
            tc::fence_mbar_init();
            // K/V rows are read once, except by a pair, where the second read
            // should find them in L2
            pol = paired ? tc::l2_evict_normal_policy() : tc::l2_evict_first_policy();
            // Whole units whose ring holds a whole V tile besides the special
            // tile's stage end with the special tile (see order_tile).
            sk->special_last = (plan.unit_mode && NS > KS) ? 1 : 0;
        }
        if (plan.unit_mode) {
            if constexpr (F8)
                locate_unit_queue(sk, lane);
            else
                locate_unit(p, upr, lane, sk);
        }
        else
            locate_range(p, upo, lane, sk, paired ? gridDim.x / 2 : gridDim.x,
                         paired ? blockIdx.x / 2 : blockIdx.x, L::kDoubleO ? 1 : 2);
        if (lane == 0) {
            // Start streaming before the block-wide barrier: this thread made
            // the barriers, and the first NS stages need no release.
            pit.init(p, sk, my_rg);
            produce(F8 ? NR : NS, true);
        }
    } else if (warp == 1) {
        tc::tmem_alloc(&sk->tmem_slot, L::kTmemCols);
        tc::tmem_relinquish();
    } else if (warp < 6) {
        // The ones block of the row-sum product (64 16-byte pieces), made
        // visible to the tensor core before the block-wide barrier.
        const int t = threadIdx.x - 64;
        if (!LP && t < 64) {
            const uint32_t one2 = F8 ? 0x3C003C00u : 0x3F803F80u;   // two f16 / bf16 ones
            reinterpret_cast<uint4 *>(smem + L::kOffOnes)[t] = make_uint4(one2, one2, one2, one2);
            tc::fence_proxy_async_smem();
        }
        // Requests rejected on the device get NaN outputs and a status bit
        // (requests b = blockIdx.x, blockIdx.x + grid, ...); their units have
        // no tiles in the flattened order.
        for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
            int id;
            long long ctx;
            if (request_ok(p, b, &id, &ctx)) continue;
            if (t == 0) set_status(p.dev_status, request_error_bits(p, id, ctx));
            const size_t per = (size_t)p.k * p.q_heads * D;
            float *o = p.out + (size_t)b * per;
            for (size_t x = t; x < per; x += 128) o[x] = __int_as_float(0x7fc00000);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = sk->tmem_slot;
    // O^T buffer of segment si: KS blocks of N columns (S^T buffers: 0, N);
    // its row sums L^T: N columns after the O^T buffers
    auto tmem_o_of = [&](int si) -> uint32_t {
        return tmem + 2 * N + (L::kDoubleO ? (uint32_t)(si & 1) : 0u) * KS * N;
    };
    auto tmem_l_of = [&](int si) -> uint32_t {
        return tmem + 2 * N + (L::kDoubleO ? 2u : 1u) * KS * N +
               (L::kDoubleO ? (uint32_t)(si & 1) : 0u) * N;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            produce(0xffffffffu, false);
            if (!alive_p || *abort_flag) {
                // A role stopped early: wait (bounded) for the last copies
                // issued -- the Q copy and the stage ring, which holds every
                // copy still in flight -- so none lands in shared memory after
                // this CTA is gone.  (Not covered: a role that stops only after
                // the producer has finished; a wait at the kernel's end for
                // that case measured 0.5-1.5 us slower per call.)
                if (qcnt > 0) tc::mbar_wait(q_full, (qcnt - 1) & 1, 100000000ull);
                if constexpr (F8) {
                    for (uint32_t x = cnt > (uint32_t)NR ? cnt - NR : 0; x < cnt; ++x)
                        tc::mbar_wait(&raw_full[x % NR], (x / NR) & 1, 100000000ull);
                } else {
                    for (uint32_t x = cnt > (uint32_t)NS ? cnt - NS : 0; x < cnt; ++x)
                        tc::mbar_wait(&full[x % NS], (x / NS) & 1, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // FP8 caches compute with f16 operands (K, V, Q and P), else bf16.
            constexpr uint32_t idesc_qk = F8 ? tc::idesc_f16_f32(128, N, false, false)
                                             : tc::idesc_bf16_f32(128, N, false, false);
            constexpr uint32_t idesc_pv = F8 ? tc::idesc_f16_f32(128, N, true, false)
                                             : tc::idesc_bf16_f32(128, N, true, false);
            const uint32_t q_base = tc::smem_u32(s_q);
            const uint32_t p_base = tc::smem_u32(s_p);
            // ONES as a K-major operand whose every 8-row group reads the same
            // 8 rows of ones (stride 0), so the product is the column sums of
            // P^T, the same in every lane of L^T.
            const uint64_t ones_desc = tc::sdesc_sw128(tc::smem_u32(smem + L::kOffOnes), 16, 0);
            SegIter it;
            it.init(p, sk, my_rg);
            Segment sg;
            bool alive = true;
            uint32_t mcnt = 0, gt = 0;   // stages consumed, tiles before this segment
            int si = 0;
            // FP8 unit mode: the next unit the producer published, whole
            auto unit_next = [&]() -> bool {
                if (plan.unit_mode) {
                    const int tu = take_unit(it, si);
                    if (tu < 0) alive = false;
                    if (tu <= 0) return false;
                }
                return it.next(p, upo, plan.row_groups, sg);
            };
            while (alive && (F8 ? unit_next() : it.next(p, upo, plan.row_groups, sg))) {
                const int n = sg.x1 - sg.x0;
                if (!wait_or_abort(F8 ? &qs_ready[si & 1] : q_full, F8 ? (si >> 1) & 1 : si & 1,
                                   abort_flag, p.dev_status)) {
                    alive = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t tmem_o = tmem_o_of(si);
                const uint32_t tmem_l = tmem_l_of(si);
                int spec_stage = 0;   // stage holding the special tile's K and V rows
                const bool sp0 = order_tile(sg, sg.x0) == sg.special;   // segment leads with it
                for (int step = 0; step <= n && alive; ++step) {
                    if (step < n) {
                        // S^T[tile & 1] = K_tile . Q^T over D in steps of 16
                        const uint32_t tmem_s = tmem + ((gt + step) & 1) * N;
                        if (order_tile(sg, sg.x0 + step) == sg.special) {
                            // 16 K rows per 64-d box, 2 KB apart; key rows past
                            // 16 read other rows of the stage and are masked.
                            const int s = mcnt % NS;
                            if (!wait_or_abort(&full[s], (mcnt / NS) & 1, abort_flag,
                                               p.dev_status)) {
                                alive = false;
                                break;
                            }
                            tc::tc_fence_after();
                            const uint32_t base = tc::smem_u32(smem + s * kStageBytes);
#pragma unroll
                            for (int db = 0; db < D / 64; ++db) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t a = tc::sdesc_sw128(
                                        base + db * kDispBoxBytes + kk * 32, 16, 1024);
                                    const uint64_t q = tc::sdesc_sw128(
                                        q_base + db * L::kQBlock + kk * 32, 16, 1024);
                                    tc::mma_bf16_ss(tmem_s, a, q, idesc_qk, (db | kk) != 0);
                                }
                            }
                            spec_stage = s;   // released after the tile's PV product
                            ++mcnt;
                        }
                        for (int ks = 0; ks < KS && alive &&
                                         order_tile(sg, sg.x0 + step) != sg.special;
                             ++ks) {
                            const int s = mcnt % NS;
                            if (!wait_or_abort(&full[s], (mcnt / NS) & 1, abort_flag,
                                               p.dev_status)) {
                                alive = false;
                                break;
                            }
                            tc::tc_fence_after();
                            const uint32_t base = tc::smem_u32(smem + s * kStageBytes);
#pragma unroll
                            for (int box = 0; box < 2; ++box) {
#pragma unroll
                                for (int kk = 0; kk < 4; ++kk) {
                                    const uint64_t a = tc::sdesc_sw128(
                                        base + box * kBoxBytes + kk * 32, 16, 1024);
                                    const uint64_t q = tc::sdesc_sw128(
                                        q_base + (ks * 2 + box) * L::kQBlock + kk * 32, 16, 1024);
                                    tc::mma_bf16_ss(tmem_s, a, q, idesc_qk, (ks | box | kk) != 0);
                                }
                            }
                            tc::mma_commit(&empty[s]);
                            ++mcnt;
                        }
                        if (!alive) break;
                        tc::mma_commit(&s_full[(gt + step) & 1]);
                        // the segment's last QK product: Q may be replaced
                        if (step == n - 1) tc::mma_commit(q_empty);
                    }
                    // O^T += V_tile^T . P^T over tile x's keys: at step s >= 1
                    // that of tile s - 1.  When the ring holds only one K tile
                    // (NS == KS) the special tile's stage must be free before the
                    // next tile's K loads, so its product comes at step 0.
                    constexpr bool kEarlySpecialPV = NS == KS;
                    int x = -1;
                    if (step == 0)
                        x = (sp0 && kEarlySpecialPV) ? 0 : -1;
                    else if (!(step == 1 && sp0 && kEarlySpecialPV))
                        x = step - 1;
                    if (x >= 0) {
                        if (!wait_or_abort(p_full, (gt + x) & 1, abort_flag, p.dev_status)) {
                            alive = false;
                            break;
                        }
                        tc::tc_fence_after();
                        const bool special = order_tile(sg, sg.x0 + x) == sg.special;
                        if (special) {
                            // The 16 keys of the special tile: one K=16 product per
                            // 128-d block; V boxes of 16 rows follow the K boxes.
                            const uint32_t vbase = tc::smem_u32(smem + spec_stage * kStageBytes) +
                                                   (D / 64) * kDispBoxBytes;
#pragma unroll
                            for (int vs = 0; vs < KS; ++vs) {
                                const uint64_t a = tc::sdesc_sw128(
                                    vbase + vs * 2 * kDispBoxBytes, kDispBoxBytes, 1024);
                                const uint64_t pp = tc::sdesc_sw128(p_base, 16, 1024);
                                tc::mma_bf16_ss(tmem_o + vs * N, a, pp, idesc_pv, x > 0);
                            }
                            tc::mma_commit(&empty[spec_stage]);
                        }
                        for (int vs = 0; vs < KS && alive && !special; ++vs) {
                            const int s = mcnt % NS;
                            if (!wait_or_abort(&full[s], (mcnt / NS) & 1, abort_flag,
                                               p.dev_status)) {
                                alive = false;
                                break;
                            }
                            tc::tc_fence_after();
                            const uint32_t base = tc::smem_u32(smem + s * kStageBytes);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint64_t a =
                                    tc::sdesc_sw128(base + kk * 2048, kBoxBytes, 1024);
                                const uint64_t pp = tc::sdesc_sw128(
                                    p_base + (kk / 4) * L::kPBlock + (kk % 4) * 32, 16, 1024);
                                tc::mma_bf16_ss(tmem_o + vs * N, a, pp, idesc_pv,
                                                (x > 0 || kk > 0));
                            }
                            tc::mma_commit(&empty[s]);
                            ++mcnt;
                        }
                        if (!alive) break;
                        // Row sums of the same P: L^T += ONES . P^T over the tile's
                        // keys (LP: the softmax threads keep them).
                        if constexpr (!LP) {
                            if (special) {
                                tc::mma_bf16_ss(tmem_l, ones_desc,
                                                tc::sdesc_sw128(p_base, 16, 1024), idesc_qk, x > 0);
                            } else {
#pragma unroll
                                for (int kk = 0; kk < 8; ++kk) {
                                    const uint64_t pp = tc::sdesc_sw128(
                                        p_base + (kk / 4) * L::kPBlock + (kk % 4) * 32, 16, 1024);
                                    tc::mma_bf16_ss(tmem_l, ones_desc, pp, idesc_qk,
                                                    (x > 0 || kk > 0));
                                }
                            }
                        }
                        tc::mma_commit(o_done);
                    }
                }
                gt += n;
                ++si;
            }
            if (!alive) {
                // Make sure every MMA this thread issued has finished.
                tc::mma_commit(fin);
                tc::mbar_wait(fin, 0, 100000000ull);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax
        // Thread t owns key t of each tile (TMEM lane t).  Per-row state lives
        // in shared memory (running maxima) and tensor memory (row sums, L^T),
        // so a thread holds only 16 rows' scores at a time whatever N is.
        const int q4 = warp & 3;              // TMEM lane quadrant this warp may access
        const int t = q4 * 32 + lane;         // key of the tile / d within an O block
        const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
        SegIter it;
        it.init(p, sk, my_rg);
        Segment sg;
        bool alive = true;
        uint32_t gt = 0, cnt_base = 0;       // tiles and stages before this segment
        int si = 0;                          // segments before this one
        float *red_max = red + L::kRedMax;   // [4 warps][N] maxima of each warp's 32 keys
        float *s_m = red + L::kRedM;         // running row maxima of the current segment
        float *s_alpha = red + L::kRedAlpha; // this tile's rescale factor per row
        float *s_mrow = red + L::kRedMrow;   // a finished segment's row maxima
        // The epilogue of a finished segment, run once the next segment's first
        // tile is under way (or at once with a single O^T buffer).
        struct PendingEpi {
            bool on;
            bool whole;
            int si, b, c, pos0, row0, rows_here;
            long long start;
        } pend{};
        float *red_lsum = red + L::kRedLsum;  // LP: [4 warps][N] row sums over each warp's keys
        float *s_l = red + L::kRedL;          // LP: a finished segment's row sums
        float *s_inv = red_lsum;              // LP: out_scale / row sum (after the reduction)
        int *s_off = reinterpret_cast<int *>(red_lsum + N);   // LP: a row's output offset
        // LP: lane t of a finished segment's L^T holds the row sums over the
        // keys thread t owned; add them up over the 128 lanes (a warp
        // transpose-reduction per 16 rows, then across the four warps by one
        // thread per row), with each row's output factor and offset.  Run at
        // the segment's end, while its last PV product is still on the tensor
        // core: the softmax threads alone write L^T.
        auto reduce_row_sums = [&](int seg) {
            const uint32_t tml = tmem_l_of(seg);
#pragma unroll 1
            for (int cb = 0; cb < N / 16; ++cb) {
                uint32_t l16[16];
                tc::tmem_ld16(tml + lane_off + cb * 16, l16);
                tc::tmem_ld_wait();
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(l16[e]);
                const int rb = warp_transpose_reduce<16, false>(v, lane);
                red_lsum[q4 * N + cb * 16 + rb] = v[0];
            }
            named_bar_softmax_any(false);
            if (t < N) {
                s_l[t] = (red_lsum[t] + red_lsum[N + t]) +
                         (red_lsum[2 * N + t] + red_lsum[3 * N + t]);
                // the factor a whole segment's output row is scaled by, divided
                // once here rather than by every thread, and the row's offset in
                // the output (row t = j * group + h' goes to
                // out[b][pos0 + j][c * group + h'])
                s_inv[t] = p.out_scale / s_l[t];
                const int jr = t / p.group;
                s_off[t] = (jr * p.q_heads + (t - jr * p.group)) * D;
            }
            named_bar_softmax_any(false);
        };
        auto write_segment = [&](const PendingEpi &pe) {
            const uint32_t tmo = tmem_o_of(pe.si);
            const uint32_t tml = tmem_l_of(pe.si);
            // A piece of a split unit goes to this CTA's partial slot (0: the
            // range's first segment, 1: its last).
            const int slot = pe.start == sk->s ? 0 : 1;
            const size_t base = ((size_t)blockIdx.x * 2 + slot) * N;
#pragma unroll 1
            for (int cb = 0; cb < N / 16; ++cb) {
                // row sums of these 16 rows (without LP every lane of L^T
                // holds them)
                uint32_t l16[16];
                if constexpr (!LP) tc::tmem_ld16(tml + lane_off + cb * 16, l16);
                uint32_t o16[KS][16];
#pragma unroll
                for (int ob = 0; ob < KS; ++ob)
                    tc::tmem_ld16(tmo + ob * N + lane_off + cb * 16, o16[ob]);
                tc::tmem_ld_wait();
                if (LP && pe.whole) {
                    // The segment saw every key of its rows: normalise and write.
                    float *obase = p.out + (((size_t)pe.b * p.k + pe.pos0) * p.q_heads +
                                            (size_t)pe.c * p.group) * D + t;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = cb * 16 + e;
                        if (r < pe.rows_here) {
                            const float inv = s_inv[r];
                            float *o = obase + s_off[r];
#pragma unroll
                            for (int ob = 0; ob < KS; ++ob)
                                o[ob * 128] = __uint_as_float(o16[ob][e]) * inv;
                        }
                    }
                } else if (pe.whole) {
                    // The segment saw every key of its rows: normalise and write.
                    // Row r = j * group + h' goes to out[b][j][c * group + h'].
                    int jr = (cb * 16) / p.group, hp = (cb * 16) - jr * p.group;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = cb * 16 + e;
                        if (r < pe.rows_here) {
                            const float inv = p.out_scale / __uint_as_float(l16[e]);
                            float *o = p.out + (((size_t)pe.b * p.k + pe.pos0 + jr) * p.q_heads +
                                                (size_t)pe.c * p.group + hp) * D + t;
#pragma unroll
                            for (int ob = 0; ob < KS; ++ob)
                                o[ob * 128] = __uint_as_float(o16[ob][e]) * inv;
                        }
                        if (++hp == p.group) {
                            hp = 0;
                            ++jr;
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = cb * 16 + e;
                        if (r < pe.rows_here) {
                            if (t == 0)
                                p.part_ml[base + r] =
                                    make_float2(s_mrow[r], LP ? s_l[r] : __uint_as_float(l16[e]));
#pragma unroll
                            for (int ob = 0; ob < KS; ++ob)
                                p.part_o[(base + r) * D + ob * 128 + t] =
                                    __uint_as_float(o16[ob][e]) * p.out_scale;
                        }
                    }
                }
            }
        };
        // FP8 unit mode: the next unit the producer published, whole (every
        // thread took the same unit unless a wait gave up)
        auto unit_next = [&]() -> bool {
            if (plan.unit_mode) {
                const int tu = take_unit(it, si);
                if (named_bar_softmax_any(tu < 0)) {
                    alive = false;
                    return false;
                }
                if (tu == 0) return false;
            }
            return it.next(p, upo, plan.row_groups, sg);
        };
        while (alive && (F8 ? unit_next() : it.next(p, upo, plan.row_groups, sg))) {
            const uint32_t tmem_o = tmem_o_of(si);
            const uint32_t tmem_l = tmem_l_of(si);
            const int n = sg.x1 - sg.x0;
            if (t == 0 && sg.x0 == 0 && !plan.unit_mode) {
                // The unit's entry for the merge launch: the range holding its
                // first tile, the number of ranges it spans (0 when this
                // segment covers it whole) and the partial slot its first
                // piece uses (0: first segment of its range, 1: last); later
                // pieces each open their range (slot 0).
                const int ranges = paired ? (int)gridDim.x / 2 : (int)gridDim.x;
                const int rix = paired ? (int)blockIdx.x / 2 : (int)blockIdx.x;
                long long r_last = (sg.unit_cost + sk->segc + sg.ntiles - 1) / sk->len;
                if (r_last > ranges - 1) r_last = ranges - 1;
                const bool whole = sg.x1 == sg.ntiles;
                p.units[sg.unit] = make_int4(rix, whole ? 0 : (int)(r_last - rix + 1),
                                             sg.start == sk->s ? 0 : 1, 0);
            }
            const int b = sg.b, c = sg.c;
            const long long ctx = sg.ctx;
            const int disp_tile = p.fused ? -1 : sg.special;   // displaced rows (append done before)
            const int new_tile = p.fused ? sg.special : -1;    // this step's rows (fused append)
            // Tokens the caches hold for this call: all key_count of them, or
            // with a fused append only the context_length older ones.
            const long long held_tokens = p.fused ? ctx : ctx + p.k;
            const int pos0 = sg.rg * plan.pos_per_group;       // first position of the group
            const int npos = min(plan.pos_per_group, p.k - pos0);
            const int row0 = pos0 * p.group;                   // first row of the group
            const int rows_here = npos * p.group;
            // Slot that holds the newest token the caches hold (ring source).
            const long long newest = held_tokens - 1;
            const long long head_slot = (ring && newest >= 0) ? newest % p.window : 0;
            // Fused append: slot of this step's first row (ring source).
            const int base_slot = (ring && p.fused) ? (int)(ctx % p.window) : 0;
            // Segment-local index of the special tile (-1: not in this
            // segment): its K part takes one stage and its V part none.
            const int xs = sg.special < 0 ? -1
                           : sg.special_last ? (sg.x1 == sg.ntiles ? sg.ntiles - 1 - sg.x0 : -1)
                                             : (sg.x0 == 0 ? 0 : -1);
            // Stages the producer issued for the segment's parts before part P.
            auto stages_before = [&](int P) -> uint32_t {
                uint32_t st = (uint32_t)P * KS;
                if (xs >= 0) {
                    if ((xs == 0 ? 0 : 2 * xs - 1) < P) st -= KS - 1;
                    if (v_part(xs, n) < P) st -= KS;
                }
                return st;
            };
            // FP8: this segment's row score scales, written by the widening
            // warps with its f16 Q (segments alternate between two barriers
            // and two scale buffers: those warps run at most one segment ahead)
            const float *qsc = s_qscale + (si & 1) * N;
            if constexpr (F8) {
                const bool q_ok = wait_or_abort(&qs_ready[si & 1], (si >> 1) & 1, abort_flag,
                                                p.dev_status);
                if (named_bar_softmax_any(!q_ok || *abort_flag)) {
                    alive = false;
                    break;
                }
            }
            // 16-row tiles keep the segment's row maxima in registers; shared
            // memory serves only the reductions.
            constexpr bool kOneChunk = N == 16;
            float mreg[kOneChunk ? 16 : 1];
            if constexpr (kOneChunk) {
#pragma unroll
                for (int e = 0; e < 16; ++e) mreg[e] = -INFINITY;
            }
            int idx = 0;
            for (; idx < n; ++idx) {
                const uint32_t tile = gt + idx;
                const int i = order_tile(sg, sg.x0 + idx);
                // warp-uniform: the TMEM loads below are warp-collective
                const bool w_ok = __all_sync(kFull, alive && wait_or_abort(&s_full[tile & 1],
                                                                           (tile >> 1) & 1,
                                                                           abort_flag,
                                                                           p.dev_status));
                const uint32_t tmem_s = tmem + (tile & 1) * N;
                if (w_ok) tc::tc_fence_after();
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
                    if (jlo < jhi)
                        rowmask = low_bits((int)jhi * p.group) & ~low_bits((int)jlo * p.group);
                }
                // Scores of rows 16 cb .. 16 cb + 15 (log2 units), -inf where the
                // row may not see the key.  A 16-row tile is one chunk: its scores
                // and row maxima stay in registers across both passes below.
                auto load_chunk = [&](int cb, float (&v)[16]) {
                    uint32_t r16[16];
                    tc::tmem_ld16(tmem_s + lane_off + cb * 16, r16);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = cb * 16 + e;
                        const float sc = F8 ? qsc[r] : p.scale_log2;
                        v[e] = ((rowmask >> r) & 1ull) ? __uint_as_float(r16[e]) * sc : -INFINITY;
                    }
                };
                float x1[16];
                if (kOneChunk && w_ok) load_chunk(0, x1);
                // A row's running maximum is replaced only when a tile's maximum
                // exceeds it by more than kRescaleSlack (log2 units; P stays below
                // 2^kRescaleSlack and O^T is rescaled only when a maximum really
                // moves).  Pass 1 asks whether any score of this tile does (a
                // segment's first tile always sets the maxima); one predicated
                // barrier tells all 128 threads, and only then are the tile's row
                // maxima reduced (a warp transpose-reduction per 16 rows, then
                // across the 4 warps by one thread per row).
                bool need = idx == 0;
                if (!need && w_ok) {
#pragma unroll 1
                    for (int cb = 0; cb < N / 16; ++cb) {
                        float v[16];
                        if (kOneChunk) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = x1[e];
                        } else {
                            load_chunk(cb, v);
                        }
                        if constexpr (kOneChunk) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) need |= v[e] > mreg[e] + kRescaleSlack;
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const float4 m4 =
                                    *reinterpret_cast<const float4 *>(s_m + cb * 16 + e);
                                need |= (v[e] > m4.x + kRescaleSlack) |
                                        (v[e + 1] > m4.y + kRescaleSlack) |
                                        (v[e + 2] > m4.z + kRescaleSlack) |
                                        (v[e + 3] > m4.w + kRescaleSlack);
                            }
                        }
                    }
                }
                bool rescale = false;
                if (named_bar_softmax_any(need || !w_ok || *abort_flag)) {
#pragma unroll 1
                    for (int cb = 0; cb < N / 16; ++cb) {
                        float v[16];
                        if (w_ok && kOneChunk) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = x1[e];
                        } else if (w_ok) {
                            load_chunk(cb, v);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = -INFINITY;
                        }
                        const int rb = warp_transpose_reduce<16, true>(v, lane);
                        red_max[q4 * N + cb * 16 + rb] = v[0];
                    }
                    if (named_bar_softmax_any(!w_ok || *abort_flag)) {
                        alive = false;
                        break;
                    }
                    bool moved = false;
                    if (t < N) {
                        const float tmax = fmaxf(fmaxf(red_max[t], red_max[N + t]),
                                                 fmaxf(red_max[2 * N + t], red_max[3 * N + t]));
                        const float m_old = idx == 0 ? -INFINITY : s_m[t];
                        const float mn = tmax > m_old + kRescaleSlack ? tmax : m_old;
                        const float ms = mn == -INFINITY ? 0.f : mn;
                        s_alpha[t] = fast_exp2(m_old - ms);
                        s_m[t] = mn;
                        moved = mn != m_old && m_old != -INFINITY;
                    }
                    rescale = named_bar_softmax_any(moved);
                    if constexpr (kOneChunk) {
#pragma unroll
                        for (int e = 0; e < 16; e += 4)
                            *reinterpret_cast<float4 *>(mreg + e) =
                                *reinterpret_cast<const float4 *>(s_m + e);
                    }
                }
                // PV of the previous tile (of this segment or the one before)
                // must be done before P, O^T and L^T are touched.
                if (tile > 0) {
                    alive = __all_sync(kFull, wait_or_abort(o_done, (tile - 1) & 1, abort_flag,
                                                            p.dev_status));
                    tc::tc_fence_after();
                }
                if (alive) {
                    if (idx > 0 && rescale) {
                        // A row's maximum moved: scale its O^T column and row sum.
#pragma unroll 1
                        for (int cb = 0; cb < N / 16; ++cb) {
#pragma unroll 1
                            for (int ob = 0; ob <= KS; ++ob) {
                                uint32_t r16[16];
                                const uint32_t addr =
                                    (ob < KS ? tmem_o + ob * N : tmem_l) + lane_off + cb * 16;
                                tc::tmem_ld16(addr, r16);
                                tc::tmem_ld_wait();
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    r16[e] = __float_as_uint(__uint_as_float(r16[e]) *
                                                             s_alpha[cb * 16 + e]);
                                tc::tmem_st16(addr, r16);
                            }
                        }
                        tc::tmem_st_wait();
                    }
                    // Pass 2: P = 2^(score - row maximum), as the K-major operand
                    // P^T: row r, key t (two 64-key blocks).
                    uint8_t *pblk = s_p + (t / 64) * L::kPBlock;
                    const uint32_t col = t % 64;
#pragma unroll 1
                    for (int cb = 0; cb < N / 16; ++cb) {
                        // LP: lane t of L^T holds the row sums over the keys this
                        // thread owned so far in the segment (of the rounded P
                        // the PV product reads, so numerator and denominator use
                        // the same weights).
                        uint32_t ls[16];
                        if (LP && idx > 0) {
                            tc::tmem_ld16(tmem_l + lane_off + cb * 16, ls);
                            tc::tmem_ld_wait();
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) ls[e] = 0u;
                        }
                        float v[16], m[16];
                        if (kOneChunk) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = x1[e];
                        } else {
                            load_chunk(cb, v);
                        }
                        if constexpr (kOneChunk) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) m[e] = mreg[e];
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; e += 4)
                                *reinterpret_cast<float4 *>(m + e) =
                                    *reinterpret_cast<const float4 *>(s_m + cb * 16 + e);
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int r = cb * 16 + e;
                            const float pr =
                                fast_exp2(v[e] - (m[e] == -INFINITY ? 0.f : m[e]));
                            uint16_t h;
                            float pq;
                            if constexpr (F8) {
                                h = __half_as_ushort(__float2half_rn(pr));
                                pq = __half2float(__ushort_as_half(h));
                            } else {
                                h = __bfloat16_as_ushort(__float2bfloat16_rn(pr));
                                pq = __uint_as_float((uint32_t)h << 16);
                            }
                            *reinterpret_cast<uint16_t *>(pblk + tc::sw128_offset(r, col)) = h;
                            if constexpr (LP) ls[e] = __float_as_uint(__uint_as_float(ls[e]) + pq);
                        }
                        if constexpr (LP) tc::tmem_st16(tmem_l + lane_off + cb * 16, ls);
                    }
                    if constexpr (LP) tc::tmem_st_wait();
                    // Rows of the tile that hold no token of this request: zero their
                    // V rows so their contents cannot reach O through P = 0.
                    const bool tile_partial =
                        i == disp_tile || i == new_tile ||
                        (ring && ((long long)(i + 1) * kTileKeys >
                                  min((long long)p.window, held_tokens))) ||
                        (!ring && (long long)(i + 1) * kTileKeys > held_tokens);
                    // Fused append into a ring: the one CTA that loads tile i
                    // overwrites slots of the tile once its own copies of the
                    // tile have landed.
                    bool tile_writes = false;
                    if (p.fused_write && ring && i != new_tile) {
                        for (int j = 0; j < p.k; ++j) {
                            int sj = base_slot + j;
                            if (sj >= p.window) sj -= p.window;
                            tile_writes |= sj / kTileKeys == i;
                        }
                    }
                    if constexpr (F8) {
                        // (the widening warps write the V rows, zeros for keys
                        // that hold no token)
                    } else if (idx == xs) {
                        // The special tile's stage: zero its V rows that hold no
                        // token (only the 16 rows its PV product reads).
                        const uint32_t x_cnt =
                            cnt_base + stages_before(idx == 0 ? 0 : 2 * idx - 1);
                        const int s = x_cnt % NS;
                        if (!wait_or_abort(&full[s], (x_cnt / NS) & 1, abort_flag, p.dev_status)) {
                            alive = false;
                        } else if (!ki.data && t < kDispRows) {
                            uint8_t *vrow =
                                smem + s * kStageBytes + (D / 64) * kDispBoxBytes + t * 128;
#pragma unroll
                            for (int db = 0; db < D / 64; ++db)
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    *reinterpret_cast<uint4 *>(vrow + db * kDispBoxBytes +
                                                               q * 16) = make_uint4(0, 0, 0, 0);
                        }
                    } else if (tile_partial || tile_writes) {
                        for (int vs = 0; vs < KS; ++vs) {
                            const uint32_t x_cnt = cnt_base + stages_before(v_part(idx, n)) + vs;
                            const int s = x_cnt % NS;
                            if (!wait_or_abort(&full[s], (x_cnt / NS) & 1, abort_flag,
                                               p.dev_status)) {
                                alive = false;
                                break;
                            }
                            if (!ki.data && tile_partial) {
                                uint8_t *row0p = smem + s * kStageBytes + t * 128;
#pragma unroll
                                for (int box = 0; box < 2; ++box)
#pragma unroll
                                    for (int q = 0; q < 8; ++q)
                                        *reinterpret_cast<uint4 *>(row0p + box * kBoxBytes +
                                                                   q * 16) = make_uint4(0, 0, 0, 0);
                            }
                        }
                    }
                }
                // Each thread publishes its own P column (and zeroed V rows): the
                // MMA thread waits for all 128 arrivals.  A thread that gave up
                // a wait above goes on to the next barrier, where all 128 leave
                // together.
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                tc::mbar_arrive(p_full);
                if (p.fused_write && (ring || sg.rg == 0)) {
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
                            dst_row = (long long)sg.id * p.window + sj;
                        } else if (paged) {
                            writer = new_tile;
                            dst_row = paged_row(p.page_table, p.max_pages, p.page_rows,
                                                p.num_pages, b, ctx + j);
                            if (dst_row < 0) {
                                if (lane == 0 && writer == i)
                                    set_status(p.dev_status, CARAT_DEV_BAD_CACHE_ID);
                                continue;
                            }
                        } else {
                            writer = new_tile;
                            dst_row = (long long)sg.id * p.capacity + ctx + j;
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
                        const bool save =
                            ring && p.displaced_out && j >= 1 && ctx + j - p.window >= 0;
                        uint4 *dk = nullptr, *dv = nullptr;
                        if (save) {
                            const size_t rowe = (size_t)p.kv_heads * D;
                            dk = reinterpret_cast<uint4 *>(
                                p.displaced_out + ((size_t)b * (p.k - 1) + (j - 1)) * 2 * rowe +
                                (size_t)c * D);
                            dv = dk + rowe / 8;
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
                if (pend.on && (idx == 1 || n == 1)) {
                    // The previous segment's last PV finished before this
                    // segment's first P was written: its O^T buffer is final.
                    // Written after this segment's second tile, while the
                    // next tile's keys are still on their way.
                    write_segment(pend);
                    pend.on = false;
                }
            }
            if (!alive) break;
            // ------------------------------------------------ segment end
            // The row maxima go to s_mrow for the epilogue (the row sums stay in
            // this segment's L^T until then).
            alive = !named_bar_softmax_any(!alive || *abort_flag);
            if (!alive) break;
            if (t < N) s_mrow[t] = s_m[t];
            pend.on = true;
            pend.whole = sg.x0 == 0 && sg.x1 == sg.ntiles;
            pend.si = si;
            pend.b = b;
            pend.c = c;
            pend.pos0 = pos0;
            pend.row0 = row0;
            pend.rows_here = rows_here;
            pend.start = sg.start;
            if constexpr (LP) reduce_row_sums(si);
            gt += n;
            cnt_base += stages_before(2 * n);
            ++si;
            if (!L::kDoubleO) {
                // One O^T buffer: the next segment's first PV overwrites it, so
                // the output goes now.
                alive = __all_sync(kFull, wait_or_abort(o_done, (gt - 1) & 1, abort_flag,
                                                        p.dev_status));
                tc::tc_fence_after();
                if (named_bar_softmax_any(!alive || *abort_flag)) {
                    alive = false;
                    break;
                }
                write_segment(pend);
                pend.on = false;
            }
        }
        if (alive && pend.on) {
            // The range's last segment.
            alive = __all_sync(kFull, wait_or_abort(o_done, (gt - 1) & 1, abort_flag, p.dev_status));
            tc::tc_fence_after();
            if (!named_bar_softmax_any(!alive || *abort_flag)) write_segment(pend);
            else alive = false;
            pend.on = false;
        }

    } else {
        // ------------------------------------------------------------ widening
        // (warps 6-9, FP8 caches only) Thread t widens key row t of every raw
        // e4m3 stage, in load order, into the f16 stage ring the MMA thread
        // reads -- the part a TMA producer plays for a bf16 cache -- writing
        // zeros for V rows of keys that hold no token, and at the start of
        // each segment rewrites its Q as f16 with a power-of-two scale per row.
        if constexpr (F8) {
            const int t = threadIdx.x - kThreads;
            SegIter it;
            it.init(p, sk, my_rg);
            Segment sg;
            bool alive = true;
            uint32_t ccnt = 0;   // raw stages widened so far
            int si = 0;
            while (alive) {
                if (plan.unit_mode) {
                    const int tu = take_unit(it, si);
                    if (!__all_sync(kFull, tu >= 0)) {
                        alive = false;
                        break;
                    }
                    if (tu == 0) break;
                }
                if (!it.next(p, upo, plan.row_groups, sg)) break;
                const int n = sg.x1 - sg.x0;
                alive = __all_sync(kFull, wait_or_abort(q_full, si & 1, abort_flag, p.dev_status));
                if (!alive) break;
                convert_q_f16<D, N, L::kQBlock>(s_q, s_qscale + (si & 1) * N, p.scale_log2, t);
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&qs_ready[si & 1]);
                const long long held = sg.ctx + p.k;   // tokens the ring holds (append done)
                for (int part = 0; part < 2 * n && alive; ++part) {
                    int x;
                    bool is_v;
                    if (part == 0) {
                        x = 0;
                        is_v = false;
                    } else if (part == 2 * n - 1) {
                        x = n - 1;
                        is_v = true;
                    } else {
                        x = (part - 1) / 2 + ((part - 1) % 2 == 0 ? 1 : 0);
                        is_v = (part - 1) % 2 == 1;
                    }
                    const int i = order_tile(sg, sg.x0 + x);
                    const bool special = i == sg.special;
                    if (special && is_v) continue;   // its V rows came with its K rows
                    const bool zero_v = is_v && ring_key_empty(i, t, p.window, held);
                    for (int ks = 0; ks < (special ? 1 : KS); ++ks) {
                        const int sidx = ccnt % NS, r = ccnt % NR;
                        alive = __all_sync(
                            kFull, (ccnt < (uint32_t)NS ||
                                    wait_or_abort(&empty[sidx], ((ccnt / NS) & 1) ^ 1, abort_flag,
                                                  p.dev_status)) &&
                                       wait_or_abort(&raw_full[r], (ccnt / NR) & 1, abort_flag,
                                                     p.dev_status));
                        if (!alive) break;
                        const uint8_t *raw = s_raw + r * L::kRawBytes;
                        uint8_t *stg = smem + sidx * kStageBytes;
                        if (special) {
                            // 16 displaced rows: K slabs then V slabs (2 KB each)
                            if (t < kDispRows) {
                                const long long pos = sg.ctx - p.window + 1 + t;
                                const bool valid = t < p.k - 1 && pos >= 0;
#pragma unroll
                                for (int sl = 0; sl < D / 128; ++sl) {
                                    convert_row(raw + sl * 2048 + t * 128,
                                                stg + (2 * sl) * kDispBoxBytes + t * 128,
                                                stg + (2 * sl + 1) * kDispBoxBytes + t * 128, t,
                                                false);
                                    convert_row(raw + (D / 128 + sl) * 2048 + t * 128,
                                                stg + (D / 64 + 2 * sl) * kDispBoxBytes + t * 128,
                                                stg + (D / 64 + 2 * sl + 1) * kDispBoxBytes + t * 128,
                                                t, !valid);
                                }
                            }
                        } else {
                            convert_row(raw + t * 128, stg + t * 128, stg + kBoxBytes + t * 128, t,
                                        zero_v);
                        }
                        tc::fence_proxy_async_smem();
                        tc::mbar_arrive(&raw_empty[r]);
                        tc::mbar_arrive(&full[sidx]);
                        ++ccnt;
                    }
                }
                ++si;
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
    if (F8 && plan.unit_mode && threadIdx.x == 0) {
        // This CTA took its last unit; the launch's last CTA to get here
        // clears the work counter and this count for the next launch (its
        // epoch may be the same: a replayed graph).
        __threadfence();
        if (tagged_increment(&p.sched[1], p.sched_epoch) == (long long)gridDim.x - 1) {
            __threadfence();
            atomicExch(&p.sched[0], 0ull);
            atomicExch(&p.sched[1], 0ull);
        }
    }
}

// ---------------------------------------------------------------------------
// Merge of split units (stream-K launches)
// ---------------------------------------------------------------------------
//
// Each piece of a split unit left, per row, its running maximum m_s (log2
// units), its sum l_s and its unnormalised output O_s (already times the V
// scale); the softmax over the union of the pieces is
//     out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s,
// the rescaling an online softmax applies between key blocks; pieces with
// l_s = 0 saw no visible key.  One CTA per (unit, row), one thread per 16
// bytes of the row: the unit table says whether the unit was split and
// where it starts; piece q sits in slot 0 or 1 of the CTA holding range g =
// first range + q (with the paired schedule, CTA 2g + the unit's row group).  It starts before the attention grid
// ends (programmatic dependent launch) and waits for it with
// griddepcontrol.wait, which also makes the grid's writes visible.
template <int D>
__global__ void __launch_bounds__(D / 4) attn_fixup_kernel(const AttnParams p, int upr,
                                                            int row_groups, int pos_per_group,
                                                            int slot_rows, int slots, int paired) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int u = blockIdx.x, r = blockIdx.y;   // unit, row within its row group
    const int b = u / upr, ur = u % upr;
    const int c = ur / row_groups, rg = ur % row_groups;
    if (b >= p.batch) return;
    // the request's validity and the unit's entry, in one round trip
    const long long ctx = p.context_lengths[b];
    const int id = p.ids ? p.ids[b] : b;
    const int4 e = p.units[u];
    if (!request_valid(p, id, ctx)) return;     // NaN already written
    const int pos0 = rg * pos_per_group;
    const int npos = min(pos_per_group, p.k - pos0);
    if (r >= npos * p.group) return;
    const int np = e.y;
    if (np == 0) return;                          // whole: already written
    const int g_first = e.x, first_slot = e.z;
    // An entry the attention grid did not write this time (it stopped on a
    // timeout before reaching the unit) is not used: its pieces could lie
    // outside the workspace.
    if ((g_first < 0) | (np < 1) | (np > kMaxPieces) | (g_first > slots - np) |
        ((first_slot & ~1) != 0)) {
        if (threadIdx.x == 0) set_status(p.dev_status, CARAT_DEV_TIMEOUT);
        return;
    }
    auto piece_base = [&](int q) -> size_t {
        const int gq = g_first + q;                         // range holding piece q
        const int cta = paired ? 2 * gq + rg : gq;          // its CTA for this row group
        return ((size_t)cta * 2 + (q == 0 ? first_slot : 0)) * slot_rows;
    };
    // weights 2^(m_q - M) / L of the pieces, by warp 0 (each lane reads the
    // (max, sum) pairs of pieces lane and lane + 32 once)
    __shared__ float s_w[kMaxPieces];
    static_assert(kMaxPieces <= 64, "two pieces per lane");
    const int lane = threadIdx.x % 32;
    if (threadIdx.x < 32) {
        float2 v0 = make_float2(-INFINITY, 0.f), v1 = v0;
        if (lane < np) v0 = p.part_ml[piece_base(lane) + r];
        if (lane + 32 < np) v1 = p.part_ml[piece_base(lane + 32) + r];
        float M = fmaxf(v0.y > 0.f ? v0.x : -INFINITY, v1.y > 0.f ? v1.x : -INFINITY);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        const float w0 = v0.y > 0.f ? fast_exp2(v0.x - M) : 0.f;
        const float w1 = v1.y > 0.f ? fast_exp2(v1.x - M) : 0.f;
        float lsum = v0.y * w0 + v1.y * w1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(kFull, lsum, o);
        const float inv = 1.f / lsum;
        if (lane < np) s_w[lane] = w0 * inv;
        if (lane + 32 < np) s_w[lane + 32] = w1 * inv;
    }
    __syncthreads();
    // one 16-byte column per thread, eight pieces' loads in flight at a time
    const int d4 = threadIdx.x;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < np; q0 += 8) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (q0 + i < np)
                v[i] = reinterpret_cast<const float4 *>(p.part_o + (piece_base(q0 + i) + r) * D)[d4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (q0 + i < np) {
                const float w = s_w[q0 + i];
                if (w != 0.f) {
                    acc.x += v[i].x * w;
                    acc.y += v[i].y * w;
                    acc.z += v[i].z * w;
                    acc.w += v[i].w * w;
                }
            }
        }
    }
    const int row = pos0 * p.group + r, j = row / p.group, hp = row - j * p.group;
    reinterpret_cast<float4 *>(
        p.out + (((size_t)b * p.k + j) * p.q_heads + (size_t)c * p.group + hp) * D)[d4] = acc;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace {

template <int D, int N, int NS, int MINB, int NR = 0, bool LP = false>
cudaError_t launch_tc(const AttnParams &p, const TcPlan &plan, const TcMaps &maps, int grid,
                      cudaStream_t stream) {
    using L = Layout<D, N, NS, NR>;
    static_assert(MINB == 1 || 2 * (L::kAlloc + 1024) <= 233472, "two CTAs must fit one SM");
    auto kernel = attn_tc_kernel<D, N, NS, MINB, NR, LP>;
    static int configured_devices[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && !configured_devices[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
        if (e != cudaSuccess) return e;
        configured_devices[dev] = 1;
    }
    if (plan.paired) grid &= ~1;   // CTAs come in pairs, one per row group
    kernel<<<grid, NR > 0 ? kThreads + kConvThreads : kThreads, L::kAlloc, stream>>>(p, plan, maps);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess || plan.unit_mode) return e;
    // stream-K: merge the split units in a second launch that may start while
    // this one drains (it waits for this grid inside the kernel)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.batch * p.kv_heads * plan.row_groups, N);
    cfg.blockDim = dim3(D / 4);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int upr = p.kv_heads * plan.row_groups;
    e = cudaLaunchKernelEx(&cfg, attn_fixup_kernel<D>, p, upr, plan.row_groups,
                           plan.pos_per_group, N, plan.paired ? grid / 2 : grid, plan.paired);
    count_launches(1);
    return e;
}

}  // namespace

// Launches of the kernels that keep the row sums in the softmax threads'
// lanes (attention_tc_unit.cu): unit-mode calls at head_dim 256.
cudaError_t launch_tc_lane_sums(const AttnParams &p, const TcPlan &plan, const TcMaps &maps,
                                int grid, int rows_per_tile, bool fp8, cudaStream_t stream);

}  // namespace carat
