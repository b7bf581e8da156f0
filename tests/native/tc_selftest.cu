// Self-test of the tcgen05 helpers in gdn_tc.cuh (test code, not part of the
// library): one CTA stages A [128 x K] and B [N x K] (16-bit, row-major in global
// memory) into the canonical K-major layout, runs K/16 tcgen05.mma steps into
// TMEM and reads D back with tcgen05.ld.  mode bit 0: negate A; bit 1: run the
// K loop twice (D = 2 A B^T); bit 2: preload D0 into TMEM with tcgen05.st and
// accumulate onto it; bit 4: A from TMEM (fp16 / bf16 pairs packed two to a
// 32-bit column with tcgen05.st, K-step k0 at column k0 / 2); bit 5: A and B in
// the 128-byte swizzled K-major layout (64-element atoms along K), written by
// the threads element by element.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_device.cuh"
#include "gdn_tc.cuh"

using namespace gdn;

__global__ void __launch_bounds__(128, 1)
tc_selftest_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, const float *D0, float *D,
                   int K, int N, int mode, unsigned int *err)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // the swizzled layout wants 1024-byte aligned operands
    unsigned char *smem = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(8) uint64_t bar;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char *a_op = smem;
    unsigned char *b_op = smem + 128 * K * 2;

    if (warp == 0) tc::tmem_alloc(&tmem_slot, 512);
    if (tid == 0) {
        dev::mbar_init(&bar, 1);
        dev::fence_mbar_init();
    }
    const bool sw = (mode & 32) != 0;
    for (int i = tid; i < 128 * K; i += 128)
        *reinterpret_cast<__nv_bfloat16 *>(a_op + (sw ? tc::sw128_offset(i / K, i % K, 128)
                                                       : tc::op_offset(i / K, i % K, K))) = A[i];
    for (int i = tid; i < N * K; i += 128)
        *reinterpret_cast<__nv_bfloat16 *>(b_op + (sw ? tc::sw128_offset(i / K, i % K, N)
                                                       : tc::op_offset(i / K, i % K, K))) = B[i];
    dev::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tmem_slot;
    const int lb = 32 * (warp & 3);
    constexpr int TA = 256;  // TMEM column of the A operand (mode bit 4)
    if (mode & 16) {  // thread = row of A: K 16-bit values, two to a column
        for (int c = 0; c < K / 2; c += 16) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint16_t lo = reinterpret_cast<const uint16_t *>(A)[(lb + lane) * K + 2 * (c + i)];
                const uint16_t hi = reinterpret_cast<const uint16_t *>(A)[(lb + lane) * K + 2 * (c + i) + 1];
                w[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            tc::tmem_st16u(tc::taddr(tbase, lb, TA + c), w);
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    if (mode & 4) {
        for (int c = 0; c < N; c += 16) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = D0[(lb + lane) * N + c + i];
            tc::tmem_st16(tc::taddr(tbase, lb, c), v);
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    if (tid == 0) {
        const uint32_t idesc = tc::idesc_f16(128, N, (mode & 1) != 0, (mode & 8) == 0);
        const uint32_t a_addr = tc::smem_u32(a_op), b_addr = tc::smem_u32(b_op);
        const int passes = (mode & 2) ? 2 : 1;
        for (int p = 0; p < passes; ++p)
            for (int k0 = 0; k0 < K; k0 += 16) {
                const bool acc = (mode & 4) || p > 0 || k0 > 0;
                const uint64_t bd = sw ? tc::op_desc_sw128(b_addr + (k0 / 64) * N * 128, k0 % 64)
                                       : tc::op_desc(b_addr, k0, K);
                if (mode & 16)
                    tc::mma_f16_ta(tbase, tbase + TA + k0 / 2, bd, idesc, acc);
                else
                    tc::mma_f16(tbase, sw ? tc::op_desc_sw128(a_addr + (k0 / 64) * 128 * 128, k0 % 64)
                                          : tc::op_desc(a_addr, k0, K),
                                bd, idesc, acc);
            }
        tc::mma_commit(&bar);
    }
    if (!dev::mbar_wait_bounded(&bar, 0) && lane == 0) atomicOr(err, 1u);
    tc::fence_after_sync();
    for (int c = 0; c < N; c += 16) {
        float v[16];
        tc::tmem_ld16(tc::taddr(tbase, lb, c), v);
#pragma unroll
        for (int i = 0; i < 16; ++i) D[(lb + lane) * N + c + i] = v[i];
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

extern "C" __attribute__((visibility("default"))) int tc_selftest(const void *A, const void *B,
                                                                 const float *D0, float *D, int K,
                                                                 int N, int mode,
                                                                 unsigned int *err, void *stream)
{
    if (K < 16 || K > 128 || K % 16 || N < 16 || N > 128 || N % 16) return -1;
    if ((mode & 32) && K % 64) return -1;
    const int smem = (128 + N) * K * 2 + 1024;
    cudaError_t e = cudaFuncSetAttribute(tc_selftest_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return static_cast<int>(e);
    tc_selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(A), static_cast<const __nv_bfloat16 *>(B), D0, D, K, N,
        mode, err);
    return static_cast<int>(cudaGetLastError());
}
