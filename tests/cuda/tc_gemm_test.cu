// Unit test kernel for the tcgen05 building blocks of kda_tc.cuh:
// D[128][N] = 3 * A[128][K] * B[N][K]^T, computed as one MMA pass, a TMEM
// read-scale-write (x2) and a second MMA pass accumulating on top.
#include <cuda_bf16.h>

#include "../../linear_attention_mixer_gb300/csrc/kda_tc.cuh"

using namespace kda;

template <int N, int K>
__global__ void __launch_bounds__(128, 1) tc_gemm_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, float *D,
                                                         int *status)
{
    constexpr int kCols = N < 32 ? 32 : N;
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sA = sm;
    unsigned char *sB = sm + 128 * K * 2;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + N * K * 2);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    const int tid = threadIdx.x, w = tid >> 5;
    for (int e = tid; e < 128 * K; e += 128)
        *reinterpret_cast<__nv_bfloat16 *>(sA + tc::kmajor_off(e / K, e % K, K)) = A[e];
    for (int e = tid; e < N * K; e += 128)
        *reinterpret_cast<__nv_bfloat16 *>(sB + tc::kmajor_off(e / K, e % K, K)) = B[e];
    tc::fence_smem_to_async();
    if (w == 0) tc::tmem_alloc(tslot, kCols);
    if (tid == 0) { mbar_init(&bar[0], 1); mbar_init(&bar[1], 1); fence_mbar_init(); }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    constexpr uint32_t idesc = tc::idesc_bf16(128, N);
    if (tid == 0) {
        for (int kk = 0; kk < K / 16; ++kk)
            tc::mma_bf16(tbase, tc::kmajor_desc(sA, kk, K), tc::kmajor_desc(sB, kk, K), idesc, kk > 0);
        tc::mma_commit(&bar[0]);
    }
    bool ok = mbar_wait_bounded(&bar[0], 0, 1u << 24);
    tc::fence_after_sync();
    float v[16];
    for (int c = 0; c < N; c += 16) {  // scale the accumulator by 2 in place
        tc::tmem_ld16(tc::tmem_addr(tbase, 32 * w, c), v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= 2.f;
        tc::tmem_st16(tc::tmem_addr(tbase, 32 * w, c), v);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
        for (int kk = 0; kk < K / 16; ++kk)
            tc::mma_bf16(tbase, tc::kmajor_desc(sA, kk, K), tc::kmajor_desc(sB, kk, K), idesc, 1);
        tc::mma_commit(&bar[1]);
    }
    ok = mbar_wait_bounded(&bar[1], 0, 1u << 24) && ok;
    tc::fence_after_sync();
    for (int c = 0; c < N; c += 16) {
        tc::tmem_ld16(tc::tmem_addr(tbase, 32 * w, c), v);
#pragma unroll
        for (int i = 0; i < 16; ++i) D[tid * N + c + i] = v[i];
    }
    if (!ok) atomicExch(status, 1);
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(tbase, kCols);
}

template <int N, int K>
static int run(const void *A, const void *B, void *D, int *status, cudaStream_t s)
{
    const int smem = 128 * K * 2 + N * K * 2 + 64;
    cudaFuncSetAttribute(tc_gemm_kernel<N, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    tc_gemm_kernel<N, K><<<1, 128, smem, s>>>((const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B, (float *)D,
                                             status);
    return (int)cudaGetLastError();
}

extern "C" int tc_gemm_test(const void *A, const void *B, void *D, int N, int K, int *status, void *stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (N == 64 && K == 128) return run<64, 128>(A, B, D, status, s);
    if (N == 128 && K == 64) return run<128, 64>(A, B, D, status, s);
    if (N == 64 && K == 64) return run<64, 64>(A, B, D, status, s);
    if (N == 128 && K == 128) return run<128, 128>(A, B, D, status, s);
    return -1;
}
