// combine.cu -- merge the split-K partial results of a CUDA-core attention
// call (the tensor-core kernel merges its own).
//
// Each key chunk c of a (request, KV head) left, per row, its running maximum
// m_c (log2 units), its sum l_c = sum 2^(s - m_c) and its unnormalised output
// O_c = sum 2^(s - m_c) v.  The softmax over the union of the chunks is
//     out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,   M = max_c m_c,
// the same rescaling an online softmax applies between key blocks.  Chunks
// with l_c = 0 saw no visible key and are skipped.  A request rejected on
// the device gets NaN outputs (its status bit is set here).
//
// One CTA per (row, KV head, request): warp 0 turns the chunks' (m, l) into
// weights 2^(m_c - M) / L in shared memory once, then every thread streams
// 16-byte pieces of the chunks' partial rows.
#include "carat_internal.cuh"

namespace carat {

constexpr int kCombineThreads = 128;
constexpr int kMaxCombineChunks = 1024;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) attn_combine(const AttnParams p) {
    const int r = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
    const int j = r / p.group, hp = r % p.group;
    float *orow = p.out + (((size_t)b * p.k + j) * p.q_heads + (size_t)c * p.group + hp) * D;
    int id;
    long long ctx;
    if (!request_ok(p, b, &id, &ctx)) {
        if (r == 0 && c == 0 && threadIdx.x == 0) set_status(p.dev_status, request_error_bits(p, id, ctx));
        for (int d = threadIdx.x; d < D; d += blockDim.x) orow[d] = __int_as_float(0x7fc00000);
        return;
    }
    const int nch = min(p.nchunks, kMaxCombineChunks);

    __shared__ float s_w[kMaxCombineChunks];
    __shared__ int s_idx[kMaxCombineChunks];
    __shared__ int s_n;
    const size_t part0 = ((size_t)b * p.kv_heads + c) * p.nchunks;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        float m = -INFINITY;
        for (int ch = lane; ch < nch; ch += 32) {
            const float2 v = p.part_ml[(part0 + ch) * p.rows + r];
            if (v.y > 0.f) m = fmaxf(m, v.x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int ch = lane; ch < nch; ch += 32) {
            const float2 v = p.part_ml[(part0 + ch) * p.rows + r];
            const float w = v.y > 0.f ? fast_exp2(v.x - m) : 0.f;
            l += v.y * w;
            s_w[ch] = w;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        __syncwarp();
        if (lane == 0) {
            // compact the chunks with weight, scaled by 1/L
            int n = 0;
            const float inv = 1.f / l;
            for (int ch = 0; ch < nch; ++ch) {
                if (s_w[ch] > 0.f) {
                    s_w[n] = s_w[ch] * inv;
                    s_idx[n] = ch;
                    ++n;
                }
            }
            s_n = n;
        }
    }
    __syncthreads();
    const int n = s_n;
    for (int d4 = threadIdx.x; d4 < D / 4; d4 += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int x = 0;
        for (; x + 4 <= n; x += 4) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = reinterpret_cast<const float4 *>(
                    p.part_o + ((part0 + s_idx[x + u]) * p.rows + r) * D)[d4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float w = s_w[x + u];
                acc.x += v[u].x * w;
                acc.y += v[u].y * w;
                acc.z += v[u].z * w;
                acc.w += v[u].w * w;
            }
        }
        for (; x < n; ++x) {
            const float4 v = reinterpret_cast<const float4 *>(
                p.part_o + ((part0 + s_idx[x]) * p.rows + r) * D)[d4];
            const float w = s_w[x];
            acc.x += v.x * w;
            acc.y += v.y * w;
            acc.z += v.z * w;
            acc.w += v.w * w;
        }
        reinterpret_cast<float4 *>(orow)[d4] = acc;
    }
}

cudaError_t launch_combine(const AttnParams &p, cudaStream_t stream) {
    dim3 grid(p.rows, p.kv_heads, p.batch);
    if (p.head_dim == 256)
        attn_combine<256><<<grid, kCombineThreads, 0, stream>>>(p);
    else if (p.head_dim == 512)
        attn_combine<512><<<grid, kCombineThreads, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace carat
