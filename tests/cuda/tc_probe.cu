// tc_probe.cu -- GPU self-check of the tensor-core primitives in
// sliding_window_gqa_ring_gb300/csrc/tc_common.cuh (test infrastructure).
//
// One CTA computes a 128 x N tile with tcgen05.mma from operands staged the
// way the attention kernel stages them, and writes it out for comparison
// with a torch matmul:
//   mode 1: D[128][N] = A[128][128] . B[N][128]^T, A and B K-major, both
//           loaded by TMA with 128-byte swizzle (the QK^T product).
//   mode 2: D[128][N] = V^T . P^T with V[128 keys][128 d] loaded by TMA
//           (MN-major A operand) and P[N][128 keys] written into shared
//           memory by threads with the swizzle applied by hand (K-major B
//           operand) (the PV product).
// Both modes also scale D by 2 in tensor memory (tcgen05.st) and read it
// back, written to out[128*N ...].
// Every shared-memory address a descriptor can form lies inside the 200 KB
// dynamic allocation, whichever way its offsets are read.
#include <cstdint>

#include "../../sliding_window_gqa_ring_gb300/csrc/tc_common.cuh"
#include "../../sliding_window_gqa_ring_gb300/csrc/tma_host.h"

using namespace carat;

namespace {

constexpr int kSmemBytes = 200 * 1024;

__global__ void __launch_bounds__(128) probe_kernel(const __grid_constant__ CUtensorMap map_a,
                                                    const __grid_constant__ CUtensorMap map_b,
                                                    const uint16_t *p_global, float *out, int n,
                                                    int mode, int *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *s_a = smem;            // 2 x 16 KB
    uint8_t *s_b = smem + 32768;    // 2 x n x 128 B
    __shared__ uint64_t bar_load, bar_mma;
    __shared__ uint32_t tmem_base_s;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    if (tid == 0) {
        tc::mbar_init(&bar_load, 1);
        tc::mbar_init(&bar_mma, 1);
        tc::fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base_s, 64);
        tc::tmem_relinquish();
    }
    if (mode == 2) {
        // P[n][128] -> two K-major 128-byte-swizzled blocks of 64 keys.
        for (int idx = tid; idx < n * 16; idx += 128) {
            const int row = idx / 16, c = idx % 16, kb = c / 8, cc = c % 8;
            const uint4 v = reinterpret_cast<const uint4 *>(p_global + row * 128)[c];
            *reinterpret_cast<uint4 *>(s_b + kb * n * 128 + tc::sw128_offset(row, cc * 8)) = v;
        }
        tc::fence_proxy_async_smem();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (tid == 0) {
        const uint64_t pol = tc::l2_evict_first_policy();
        if (mode == 1) {
            tc::mbar_arrive_expect_tx(&bar_load, 32768 + n * 256);
            tc::tma_load_2d(s_a, &map_a, 0, 0, &bar_load, pol);
            tc::tma_load_2d(s_a + 16384, &map_a, 64, 0, &bar_load, pol);
            tc::tma_load_2d(s_b, &map_b, 0, 0, &bar_load, pol);
            tc::tma_load_2d(s_b + n * 128, &map_b, 64, 0, &bar_load, pol);
        } else {
            tc::mbar_arrive_expect_tx(&bar_load, 32768);
            tc::tma_load_2d(s_a, &map_a, 0, 0, &bar_load, pol);
            tc::tma_load_2d(s_a + 16384, &map_a, 64, 0, &bar_load, pol);
        }
        if (!tc::mbar_wait(&bar_load, 0)) {
            atomicExch(err, 1);
        } else {
            tc::tc_fence_after();
            const uint32_t base_a = tc::smem_u32(s_a), base_b = tc::smem_u32(s_b);
            for (int kk = 0; kk < 8; ++kk) {
                uint64_t da, db;
                uint32_t idesc;
                if (mode == 1) {
                    da = tc::sdesc_sw128(base_a + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024);
                    db = tc::sdesc_sw128(base_b + (kk / 4) * n * 128 + (kk % 4) * 32, 16, 1024);
                    idesc = tc::idesc_bf16_f32(128, n, false, false);
                } else {
                    da = tc::sdesc_sw128(base_a + kk * 2048, 16384, 1024);
                    db = tc::sdesc_sw128(base_b + (kk / 4) * n * 128 + (kk % 4) * 32, 16, 1024);
                    idesc = tc::idesc_bf16_f32(128, n, true, false);
                }
                tc::mma_bf16_ss(tmem, da, db, idesc, kk > 0 ? 1u : 0u);
            }
            tc::mma_commit(&bar_mma);
        }
    }
    __syncwarp();
    if (!tc::mbar_wait(&bar_mma, 0)) {
        atomicExch(err, 2);
    } else {
        tc::tc_fence_after();
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int row = warp * 32 + lane;
        for (int c = 0; c < n / 16; ++c) {
            uint32_t r[16];
            tc::tmem_ld16(tmem + lane_base + c * 16, r);
            tc::tmem_ld_wait();
            for (int i = 0; i < 16; ++i) out[row * n + c * 16 + i] = __uint_as_float(r[i]);
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * 2.0f);
            tc::tmem_st16(tmem + lane_base + c * 16, r);
            tc::tmem_st_wait();
            uint32_t s[16];
            tc::tmem_ld16(tmem + lane_base + c * 16, s);
            tc::tmem_ld_wait();
            for (int i = 0; i < 16; ++i)
                out[128 * n + row * n + c * 16 + i] = __uint_as_float(s[i]);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 64);
}

}  // namespace

// mode 1: a = A [128][128] bf16, b = B [n][128] bf16.
// mode 2: a = V [128][128] bf16 (keys x d), b = P [n][128] bf16.
// out: fp32 [2][128][n].  Returns 0, or a nonzero code on failure.
extern "C" int tc_probe_run(int mode, int n, const void *a, const void *b, float *out) {
    if (!(n == 16 || n == 32 || n == 64) || (mode != 1 && mode != 2)) return -1;
    CUtensorMap map_a{}, map_b{};
    const uint64_t dims_a[2] = {128, 128};
    const uint64_t strides_a[1] = {256};
    const uint32_t box_a[2] = {64, 128};
    if (!make_bf16_tensor_map(&map_a, a, 2, dims_a, strides_a, box_a, true)) return -2;
    if (mode == 1) {
        const uint64_t dims_b[2] = {128, (uint64_t)n};
        const uint32_t box_b[2] = {64, (uint32_t)n};
        if (!make_bf16_tensor_map(&map_b, b, 2, dims_b, strides_a, box_b, true)) return -3;
    } else {
        map_b = map_a;  // unused
    }
    int *err = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -4;
    cudaMemset(err, 0, sizeof(int));
    cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    probe_kernel<<<1, 128, kSmemBytes>>>(map_a, map_b, static_cast<const uint16_t *>(b), out, n,
                                         mode, err);
    cudaError_t e = cudaDeviceSynchronize();
    int h_err = 0;
    cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(err);
    if (e != cudaSuccess) return 100 + (int)e;
    return h_err;
}
