// attention_simt.cu -- split-K attention on CUDA cores, for any key source.
//
// Computes, for every (request b, KV head c), softmax(scale * Q K^T) V over
// the keys each query row may see: the last `window` positions up to its own
// for a sliding layer ("Improving Decode Throughput on Intel Gaudi 3",
// "Patching sliding window KV allocation"), every position up to its own for a
// global layer ("Announcing Carat: An inference engine designed for Gemma 4",
// "More FLOPs can be faster").  The rows of one tile are the query heads that
// share KV head c times the proposal positions ("Doing it all in one kernel
// can be slower"), so K and V are read once per tile, not once per head.
//
// Sliding-layer keys are read from the ring in slot order, i.e. rotated, and
// never un-rotated: each slot's position is derived from the slot index, and
// the mask is applied by position ("Our approach" on the Gaudi page).
//
// Work split: grid (key chunk, KV head, request).  Each CTA streams its chunk
// with 16-byte loads, keeps an online softmax per row (running max in log2
// units, running sum, unnormalised output), merges its warps through shared
// memory and writes one partial per row; attn_combine merges the chunks.
#include <cfloat>

#include "carat_internal.cuh"

namespace carat {

namespace {

constexpr int kWarps = 4;
constexpr int kUnroll = 2;

struct KeyRef {
    long long pos;  // absolute position, < 0 when the slot holds nothing
    const uint16_t *k;
    const uint16_t *v;
};

// Key index u of (request b, KV head c) -> its position and row pointers.
__device__ __forceinline__ KeyRef key_ref(const AttnParams &p, int b, int c, int id,
                                          long long ctx, long long u) {
    KeyRef r;
    const size_t row = (size_t)p.kv_heads * p.head_dim;
    if (p.source == KeySource::kLinear) {
        r.pos = u;
        size_t off = ((size_t)id * p.capacity + (size_t)u) * row + (size_t)c * p.head_dim;
        r.k = p.k_base + off;
        r.v = p.v_base + off;
        return r;
    }
    const long long key_count = ctx + p.k;
    if (u < p.window) {
        // Slot u holds the latest position <= key_count-1 congruent to u.
        const long long slot = u;
        r.pos = key_count - 1 - ((key_count - 1 - slot) % p.window + p.window) % p.window;
        size_t off = ((size_t)id * p.window + (size_t)slot) * row + (size_t)c * p.head_dim;
        r.k = p.k_base + off;
        r.v = p.v_base + off;
    } else {
        // Displaced row i: position ctx - window + 1 + i, saved by the append.
        const long long i = u - p.window;
        r.pos = ctx - p.window + 1 + i;
        size_t off = (((size_t)b * (p.k - 1) + (size_t)i) * 2) * row + (size_t)c * p.head_dim;
        r.k = p.displaced + off;
        r.v = p.displaced + off + row;
    }
    return r;
}

template <int EPL>
__device__ __forceinline__ void load_row(const uint16_t *src, int lane, uint64_t pol,
                                         float (&f)[EPL]) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src) + lane * (EPL / 8);
#pragma unroll
    for (int i = 0; i < EPL / 8; ++i) {
        uint4 w = ld_stream_v4(s + i, pol);
        f[i * 8 + 0] = bf16lo(w.x);
        f[i * 8 + 1] = bf16hi(w.x);
        f[i * 8 + 2] = bf16lo(w.y);
        f[i * 8 + 3] = bf16hi(w.y);
        f[i * 8 + 4] = bf16lo(w.z);
        f[i * 8 + 5] = bf16hi(w.z);
        f[i * 8 + 6] = bf16lo(w.w);
        f[i * 8 + 7] = bf16hi(w.w);
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace

template <int D, int RG>
__global__ void __launch_bounds__(kWarps * 32) attn_partial_simt(const AttnParams p) {
    constexpr int EPL = D / 32;
    const int chunk = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    int id;
    long long ctx;
    const bool ok = request_ok(p, b, &id, &ctx);
    const long long nkeys = ok ? keys_scanned(p.source, p.window, p.k, ctx + p.k) : 0;
    const long long u0 = (long long)chunk * p.chunk;
    const long long u1 = min(u0 + (long long)p.chunk, nkeys);

    const size_t part = ((size_t)b * p.kv_heads + c) * p.nchunks + chunk;
    float2 *ml = p.part_ml + part * p.rows;
    float *po = p.part_o + part * p.rows * D;

    if (u0 >= u1) {
        for (int r = threadIdx.x; r < p.rows; r += blockDim.x) ml[r] = make_float2(-INFINITY, 0.f);
        return;
    }

    const uint64_t pol = evict_first_policy();
    __shared__ float s_o[kWarps][RG][D];
    __shared__ float s_m[kWarps][RG];
    __shared__ float s_l[kWarps][RG];

    for (int r0 = 0; r0 < p.rows; r0 += RG) {
        float qf[RG][EPL];
        long long qpos[RG];
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
            const int r = r0 + rr;
            if (r < p.rows) {
                const int j = r / p.group, hp = r % p.group;
                const uint16_t *qrow =
                    p.q + (((size_t)b * p.k + j) * p.q_heads + (size_t)c * p.group + hp) * D;
                float t[EPL];
                const uint4 *s = reinterpret_cast<const uint4 *>(qrow) + lane * (EPL / 8);
#pragma unroll
                for (int i = 0; i < EPL / 8; ++i) {
                    uint4 w = s[i];
                    t[i * 8 + 0] = bf16lo(w.x);
                    t[i * 8 + 1] = bf16hi(w.x);
                    t[i * 8 + 2] = bf16lo(w.y);
                    t[i * 8 + 3] = bf16hi(w.y);
                    t[i * 8 + 4] = bf16lo(w.z);
                    t[i * 8 + 5] = bf16hi(w.z);
                    t[i * 8 + 6] = bf16lo(w.w);
                    t[i * 8 + 7] = bf16hi(w.w);
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) qf[rr][e] = t[e] * p.scale_log2;
                qpos[rr] = ctx + j;
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) qf[rr][e] = 0.f;
                qpos[rr] = -1;
            }
        }

        float m[RG], l[RG], o[RG][EPL];
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
            m[rr] = -INFINITY;
            l[rr] = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[rr][e] = 0.f;
        }

        for (long long ub = u0 + warp; ub < u1; ub += (long long)kWarps * kUnroll) {
            KeyRef kr[kUnroll];
            float kf[kUnroll][EPL], vf[kUnroll][EPL];
#pragma unroll
            for (int x = 0; x < kUnroll; ++x) {
                const long long u = ub + (long long)x * kWarps;
                kr[x].pos = -1;
                if (u < u1) kr[x] = key_ref(p, b, c, id, ctx, u);
                if (kr[x].pos >= 0) {
                    load_row<EPL>(kr[x].k, lane, pol, kf[x]);
                    load_row<EPL>(kr[x].v, lane, pol, vf[x]);
                }
            }
#pragma unroll
            for (int x = 0; x < kUnroll; ++x) {
                const long long pos = kr[x].pos;
                if (pos < 0) continue;  // warp-uniform
#pragma unroll
                for (int rr = 0; rr < RG; ++rr) {
                    float s = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) s = fmaf(qf[rr][e], kf[x][e], s);
                    s = warp_sum(s);
                    const long long qp = qpos[rr];
                    const bool visible = qp >= 0 && pos <= qp &&
                                         (p.source == KeySource::kLinear || pos > qp - p.window);
                    if (!visible) continue;  // warp-uniform
                    const float mn = fmaxf(m[rr], s);
                    const float alpha = fast_exp2(m[rr] - mn);
                    const float pe = fast_exp2(s - mn);
                    l[rr] = l[rr] * alpha + pe;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[rr][e] = fmaf(o[rr][e], alpha, pe * vf[x][e]);
                    m[rr] = mn;
                }
            }
        }

        // Merge the warps' states.
#pragma unroll
        for (int rr = 0; rr < RG; ++rr) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) s_o[warp][rr][lane * EPL + e] = o[rr][e];
            if (lane == 0) {
                s_m[warp][rr] = m[rr];
                s_l[warp][rr] = l[rr];
            }
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < RG * D; idx += blockDim.x) {
            const int rr = idx / D, d = idx % D;
            const int r = r0 + rr;
            if (r >= p.rows) continue;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][rr]);
            float acc = 0.f, L = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float f = fast_exp2(s_m[w][rr] - M);
                    acc += s_o[w][rr][d] * f;
                    L += s_l[w][rr] * f;
                }
            }
            po[(size_t)r * D + d] = acc;
            if (d == 0) ml[r] = make_float2(M, L);
        }
        __syncthreads();
    }
}

template <int D, int RG>
static cudaError_t launch_d(const AttnParams &p, cudaStream_t stream) {
    dim3 grid(p.nchunks, p.kv_heads, p.batch);
    attn_partial_simt<D, RG><<<grid, kWarps * 32, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_attention_simt(const AttnParams &p, cudaStream_t stream) {
    if (p.head_dim == 256) {
        if (p.rows <= 2) return launch_d<256, 2>(p, stream);
        if (p.rows <= 4) return launch_d<256, 4>(p, stream);
        return launch_d<256, 8>(p, stream);
    }
    if (p.head_dim == 512) {
        if (p.rows <= 2) return launch_d<512, 2>(p, stream);
        return launch_d<512, 4>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace carat
