// ring_append.cu -- write a step's new K/V rows into per-request rings.
//
// Slot of position t = t mod window ("Announcing Carat: An inference engine
// designed for Gemma 4", "Replacing page lookups with a ring buffer"); K and
// V rows are written by the same thread in the same order, so both rings
// keep one rotation ("Improving Decode Throughput on Intel Gaudi 3", "Our
// approach").
//
// One CTA per (new token j, request b).  Each thread moves 16-byte chunks of
// the token's [kv_heads][head_dim] row.  When `displaced` is given, the old
// row in the slot that token j >= 1 overwrites is copied out first by the
// same thread that then overwrites it, so the read precedes the write in
// program order and no other thread touches those bytes.
#include "carat_internal.cuh"

namespace carat {

__global__ void __launch_bounds__(256) ring_append_kernel(const AppendParams p) {
    const int j = blockIdx.x;
    const int b = blockIdx.y;
    const long long ctx = p.context_lengths[b];
    const int id = p.ids ? p.ids[b] : b;
    if (ctx < 0 || id < 0 || id >= p.num_ids) {
        if (threadIdx.x == 0 && j == 0)
            set_status(p.dev_status, ctx < 0 ? CARAT_DEV_BAD_CONTEXT : CARAT_DEV_BAD_CACHE_ID);
        return;
    }
    const long long t = ctx + j;                 // absolute position of new token j
    const size_t row_elems = (size_t)p.kv_heads * p.head_dim;
    const int chunks = (int)(row_elems * 2 / 16);
    long long dst_row;
    if (p.page_table) {
        // Paged cache: position t goes to its page's row; no ring, nothing displaced.
        if (t >= (long long)p.max_pages * p.page_rows) {
            if (threadIdx.x == 0) set_status(p.dev_status, CARAT_DEV_BAD_CONTEXT);
            return;
        }
        dst_row = paged_row(p.page_table, p.max_pages, p.page_rows, p.num_pages, b, t);
        if (dst_row < 0) {
            if (threadIdx.x == 0) set_status(p.dev_status, CARAT_DEV_BAD_CACHE_ID);
            return;
        }
    } else {
        dst_row = (long long)id * p.window + t % p.window;
    }

    uint4 *kdst = reinterpret_cast<uint4 *>(p.k_ring + (size_t)dst_row * row_elems);
    uint4 *vdst = reinterpret_cast<uint4 *>(p.v_ring + (size_t)dst_row * row_elems);
    const uint4 *ksrc =
        reinterpret_cast<const uint4 *>(p.k_new + ((size_t)b * p.k + j) * row_elems);
    const uint4 *vsrc =
        reinterpret_cast<const uint4 *>(p.v_new + ((size_t)b * p.k + j) * row_elems);

    // Old occupant of this slot: position t - window.  Token j >= 1 displaces a
    // row that query 0 .. j-1 of this step still needs, if it exists.
    const bool save = p.displaced != nullptr && !p.page_table && j >= 1 && t - p.window >= 0;
    uint4 *ddst = nullptr;
    if (save)
        ddst = reinterpret_cast<uint4 *>(p.displaced +
                                         (((size_t)b * (p.k - 1) + (j - 1)) * 2) * row_elems);

    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        uint4 kn = ksrc[c];
        uint4 vn = vsrc[c];
        if (save) {
            uint4 ko = kdst[c];
            uint4 vo = vdst[c];
            ddst[c] = ko;
            ddst[chunks + c] = vo;
        }
        kdst[c] = kn;
        vdst[c] = vn;
    }
}

// Rollback after a speculative append: one CTA per (rejected candidate row
// j >= 1, request b).  The old rows come back from the displaced buffer the
// append filled; rows of proposals that are kept, and slots that held no
// token before the append, are left alone.
__global__ void __launch_bounds__(256) ring_rollback_kernel(const AppendParams p,
                                                            const int32_t *accepted) {
    const int j = blockIdx.x + 1;
    const int b = blockIdx.y;
    const long long ctx = p.context_lengths[b];
    const int id = p.ids ? p.ids[b] : b;
    const int a = accepted[b];
    if (ctx < 0 || id < 0 || id >= p.num_ids || a < 0 || a > p.k) {
        if (threadIdx.x == 0 && j == 1)
            set_status(p.dev_status, (id < 0 || id >= p.num_ids) ? CARAT_DEV_BAD_CACHE_ID
                                                                   : CARAT_DEV_BAD_CONTEXT);
        return;
    }
    if (j < a || ctx + j - p.window < 0) return;
    const long long slot = (ctx + j) % p.window;
    // rows are moved as bytes, so bf16 and e4m3 rings share this kernel
    const size_t row_bytes = (size_t)p.kv_heads * p.head_dim * p.elem_bytes;
    const int chunks = (int)(row_bytes / 16);
    uint8_t *kr = reinterpret_cast<uint8_t *>(p.k_ring);
    uint8_t *vr = reinterpret_cast<uint8_t *>(p.v_ring);
    uint4 *kdst = reinterpret_cast<uint4 *>(kr + ((size_t)id * p.window + slot) * row_bytes);
    uint4 *vdst = reinterpret_cast<uint4 *>(vr + ((size_t)id * p.window + slot) * row_bytes);
    const uint4 *src = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const uint8_t *>(p.displaced) +
        (((size_t)b * (p.k - 1) + (j - 1)) * 2) * row_bytes);
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        kdst[c] = src[c];
        vdst[c] = src[chunks + c];
    }
}

cudaError_t launch_ring_rollback(const AppendParams &p, const int32_t *accepted,
                                 cudaStream_t stream) {
    const int chunks = p.kv_heads * p.head_dim * p.elem_bytes / 16;
    int threads = chunks < 256 ? ((chunks + 31) / 32) * 32 : 256;
    dim3 grid(p.k - 1, p.batch);
    ring_rollback_kernel<<<grid, threads, 0, stream>>>(p, accepted);
    count_launches(1);
    return cudaGetLastError();
}

// FP8 rings ("gemma-cuda-hybrid", "Features" / "Server": the KV cache is FP8
// e4m3): the same slot rule, with each new bf16 element stored as
// e4m3_rn(fp32(x * inv)) -- one binary32 product, then a saturating
// round-to-nearest-even conversion.  One CTA per (new token j, request b);
// each thread makes 16 output bytes from 32 input bytes.  A displaced row is
// saved as its e4m3 bytes, by the thread that then overwrites them.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    uint16_t lo, hi;
    // cvt packs its first source into the upper byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ uint4 quantize16(uint4 x0, uint4 x1, float inv) {
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = e4m3x4(__fmul_rn(bf16lo(w[2 * i]), inv), __fmul_rn(bf16hi(w[2 * i]), inv),
                      __fmul_rn(bf16lo(w[2 * i + 1]), inv), __fmul_rn(bf16hi(w[2 * i + 1]), inv));
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(256) ring_append_fp8_kernel(const AppendParams p) {
    const int j = blockIdx.x;
    const int b = blockIdx.y;
    const long long ctx = p.context_lengths[b];
    const int id = p.ids ? p.ids[b] : b;
    if (ctx < 0 || id < 0 || id >= p.num_ids) {
        if (threadIdx.x == 0 && j == 0)
            set_status(p.dev_status, ctx < 0 ? CARAT_DEV_BAD_CONTEXT : CARAT_DEV_BAD_CACHE_ID);
        return;
    }
    const long long t = ctx + j;
    const size_t row_elems = (size_t)p.kv_heads * p.head_dim;
    const int chunks = (int)(row_elems / 16);      // 16 e4m3 bytes per chunk
    const long long dst_row = (long long)id * p.window + t % p.window;
    uint8_t *kr = reinterpret_cast<uint8_t *>(p.k_ring);
    uint8_t *vr = reinterpret_cast<uint8_t *>(p.v_ring);
    uint4 *kdst = reinterpret_cast<uint4 *>(kr + (size_t)dst_row * row_elems);
    uint4 *vdst = reinterpret_cast<uint4 *>(vr + (size_t)dst_row * row_elems);
    const uint4 *ksrc =
        reinterpret_cast<const uint4 *>(p.k_new + ((size_t)b * p.k + j) * row_elems);
    const uint4 *vsrc =
        reinterpret_cast<const uint4 *>(p.v_new + ((size_t)b * p.k + j) * row_elems);
    const bool save = p.displaced != nullptr && j >= 1 && t - p.window >= 0;
    uint4 *ddst = nullptr;
    if (save)
        ddst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.displaced) +
                                         (((size_t)b * (p.k - 1) + (j - 1)) * 2) * row_elems);
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const uint4 kq = quantize16(ksrc[2 * c], ksrc[2 * c + 1], p.k_inv);
        const uint4 vq = quantize16(vsrc[2 * c], vsrc[2 * c + 1], p.v_inv);
        if (save) {
            const uint4 ko = kdst[c];
            const uint4 vo = vdst[c];
            ddst[c] = ko;
            ddst[chunks + c] = vo;
        }
        kdst[c] = kq;
        vdst[c] = vq;
    }
}

cudaError_t launch_ring_append_fp8(const AppendParams &p, cudaStream_t stream) {
    const int chunks = p.kv_heads * p.head_dim / 16;
    int threads = chunks < 256 ? ((chunks + 31) / 32) * 32 : 256;
    dim3 grid(p.k, p.batch);
    ring_append_fp8_kernel<<<grid, threads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_ring_append(const AppendParams &p, cudaStream_t stream) {
    const int chunks = p.kv_heads * p.head_dim * 2 / 16;
    int threads = chunks < 256 ? ((chunks + 31) / 32) * 32 : 256;
    dim3 grid(p.k, p.batch);
    ring_append_kernel<<<grid, threads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace carat
