// combine.cu -- merge the split-K partial results of an attention call.
//
// Each key chunk c of a (request, KV head) left, per row, its running maximum
// m_c (log2 units), its sum l_c = sum 2^(s - m_c) and its unnormalised output
// O_c = sum 2^(s - m_c) v.  The softmax over the union of the chunks is
//     out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,   M = max_c m_c,
// the same rescaling an online softmax applies between key blocks.  Chunks
// with l_c = 0 saw no visible key and are skipped.  A request rejected on
// the device gets NaN outputs (its status bit was set by the partial kernel
// or is set here).
#include "carat_internal.cuh"

namespace carat {

template <int D>
__global__ void __launch_bounds__(128) attn_combine(const AttnParams p) {
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
    const size_t part0 = ((size_t)b * p.kv_heads + c) * p.nchunks;
    float M = -INFINITY;
    for (int ch = 0; ch < p.nchunks; ++ch) {
        const float2 v = p.part_ml[(part0 + ch) * p.rows + r];
        if (v.y > 0.f) M = fmaxf(M, v.x);
    }
    float L = 0.f;
    for (int ch = 0; ch < p.nchunks; ++ch) {
        const float2 v = p.part_ml[(part0 + ch) * p.rows + r];
        if (v.y > 0.f) L += v.y * fast_exp2(v.x - M);
    }
    const float inv = 1.f / L;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float acc = 0.f;
        for (int ch = 0; ch < p.nchunks; ++ch) {
            const float2 v = p.part_ml[(part0 + ch) * p.rows + r];
            if (v.y > 0.f) acc += p.part_o[((part0 + ch) * p.rows + r) * D + d] * fast_exp2(v.x - M);
        }
        orow[d] = acc * inv;
    }
}

cudaError_t launch_combine(const AttnParams &p, cudaStream_t stream) {
    dim3 grid(p.rows, p.kv_heads, p.batch);
    if (p.head_dim == 256)
        attn_combine<256><<<grid, 128, 0, stream>>>(p);
    else if (p.head_dim == 512)
        attn_combine<512><<<grid, 128, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace carat
