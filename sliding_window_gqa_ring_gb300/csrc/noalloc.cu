// noalloc.cu -- sliding-window attention with built-in scratch memory.
//
// carat_swa_attention needs a caller-provided workspace for its split-K
// partial results.  Some callers cannot provide one: a plugin inside a host
// runtime that owns every byte of device memory and hands its plugins no
// allocator, or a latency-critical loop that must never call cudaMalloc
// (which can synchronise the whole device).  This file gives them one entry
// point that allocates nothing: the scratch is a fixed array in device global
// memory that exists as soon as the library is loaded on a GPU.
//
// Cost of that convenience: every GPU that loads the library keeps
// kNoAllocScratchBytes reserved until the process exits, and all calls share
// the one array, so calls that overlap on the GPU (different streams, or
// different host threads, without ordering between them) race on it.
#include <mutex>

#include "carat_internal.cuh"

namespace carat {
namespace {

constexpr size_t kNoAllocScratchBytes = CARAT_NOALLOC_SCRATCH_BYTES;

// The scratch array.  In host code this name is only a host-side stand-in
// for the device symbol; its device address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace carat

extern "C" {

size_t carat_noalloc_scratch_bytes(void) { return carat::kNoAllocScratchBytes; }

carat_status carat_swa_attention_noalloc(float *out, const void *queries, const void *k_ring,
                                         const void *v_ring, int num_rings,
                                         const int32_t *ring_ids, const void *displaced,
                                         const int32_t *context_lengths, int proposal_count,
                                         int batch, int q_heads, int kv_heads, int head_dim,
                                         int window, float scale, void *stream) {
    // Sizes first, on the host: the scratch cannot grow.
    const size_t need = carat_swa_workspace_bytes(batch, proposal_count, q_heads, kv_heads,
                                                  head_dim, window);
    if (need > carat::kNoAllocScratchBytes) return CARAT_ERR_WORKSPACE;
    if (batch == 0 || need == 0) {
        // Nothing to compute, or invalid sizes: let the regular entry point
        // report the same status it would for these arguments.
        return carat_swa_attention(out, queries, k_ring, v_ring, num_rings, ring_ids, displaced,
                                   context_lengths, proposal_count, batch, q_heads, kv_heads,
                                   head_dim, window, scale, nullptr, 0, stream);
    }
    void *scratch = nullptr;
    if (carat::scratch_address(&scratch) != cudaSuccess) return CARAT_ERR_CUDA;
    // Everything in the scratch (partials, the tensor-core path's unit table)
    // is written before it is read within a call, so the array needs no
    // clearing between calls.
    return carat_swa_attention(out, queries, k_ring, v_ring, num_rings, ring_ids, displaced,
                               context_lengths, proposal_count, batch, q_heads, kv_heads,
                               head_dim, window, scale, scratch, carat::kNoAllocScratchBytes,
                               stream);
}

}  // extern "C"
