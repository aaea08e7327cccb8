// Unit test kernels for the tcgen05 building blocks of kda_tc.cuh:
// D[128][N] = 3 * A[128][K] * B[N][K]^T, computed as one MMA pass, a TMEM
// read-scale-write (x2) and a second MMA pass accumulating on top; and
// D = A B^T with the A operand read from tensor memory.
#include <cuda_bf16.h>

#include "../../linear_attention_mixer_gb300/csrc/kda_tc.cuh"

using namespace kda;

template <int N, int K, bool PAD>
__global__ void __launch_bounds__(128, 1) tc_gemm_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, float *D,
                                                         int *status)
{
    constexpr int kCols = N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256));  // a power of two
    constexpr int kAB = PAD ? tc::kmajor_pad_bytes(128, K) : 128 * K * 2;
    constexpr int kBB = PAD ? tc::kmajor_pad_bytes(N, K) : N * K * 2;
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sA = sm;
    unsigned char *sB = sm + kAB;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + kBB);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    const int tid = threadIdx.x, w = tid >> 5;
    auto off = [](int r, int k) { return PAD ? tc::kmajor_off_pad(r, k, K) : tc::kmajor_off(r, k, K); };
    auto desc = [](const void *t, int kk) { return PAD ? tc::kmajor_desc_pad(t, kk, K) : tc::kmajor_desc(t, kk, K); };
    for (int e = tid; e < 128 * K; e += 128)
        *reinterpret_cast<__nv_bfloat16 *>(sA + off(e / K, e % K)) = A[e];
    for (int e = tid; e < N * K; e += 128)
        *reinterpret_cast<__nv_bfloat16 *>(sB + off(e / K, e % K)) = B[e];
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
            tc::mma_bf16(tbase, desc(sA, kk), desc(sB, kk), idesc, kk > 0);
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
            tc::mma_bf16(tbase, desc(sA, kk), desc(sB, kk), idesc, 1);
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

// D[128][N] = A[128][K] B[N][K]^T with A in tensor memory: row m of A in lane m, BF16 pairs per
// 32-bit column after the N accumulator columns; B in shared memory.
template <int N, int K>
__global__ void __launch_bounds__(128, 1) tc_gemm_ta_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, float *D,
                                                            int *status)
{
    constexpr int kCols = N + K / 2 <= 128 ? 128 : 256;
    static_assert(N + K / 2 <= 256, "TMEM columns");
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sB = sm;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + N * K * 2);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    const int tid = threadIdx.x, w = tid >> 5;
    for (int e = tid; e < N * K; e += 128)
        *reinterpret_cast<__nv_bfloat16 *>(sB + tc::kmajor_off(e / K, e % K, K)) = B[e];
    tc::fence_smem_to_async();
    if (w == 0) tc::tmem_alloc(tslot, kCols);
    if (tid == 0) { mbar_init(&bar[0], 1); fence_mbar_init(); }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    for (int c = 0; c < K / 2; c += 16) {  // row tid of A into lane tid
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 two;
            two.x = A[tid * K + 2 * (c + i)];
            two.y = A[tid * K + 2 * (c + i) + 1];
            p[i] = *reinterpret_cast<const uint32_t *>(&two);
        }
        tc::tmem_st16u_nowait(tc::tmem_addr(tbase, 32 * w, N + c), p);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) {
        for (int kk = 0; kk < K / 16; ++kk)
            tc::mma_bf16_ta(tbase, tbase + N + 8 * kk, tc::kmajor_desc(sB, kk, K), tc::idesc_bf16(128, N), kk > 0);
        tc::mma_commit(&bar[0]);
    }
    const bool ok = mbar_wait_bounded(&bar[0], 0, 1u << 24);
    tc::fence_after_sync();
    float v[16];
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
static int run_ta(const void *A, const void *B, void *D, int *status, cudaStream_t s)
{
    const int smem = N * K * 2 + 64;
    cudaFuncSetAttribute(tc_gemm_ta_kernel<N, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    tc_gemm_ta_kernel<N, K><<<1, 128, smem, s>>>((const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B, (float *)D,
                                                status);
    return (int)cudaGetLastError();
}

extern "C" int tc_gemm_ta_test(const void *A, const void *B, void *D, int N, int K, int *status, void *stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (N == 64 && K == 128) return run_ta<64, 128>(A, B, D, status, s);
    if (N == 128 && K == 128) return run_ta<128, 128>(A, B, D, status, s);
    if (N == 192 && K == 64) return run_ta<192, 64>(A, B, D, status, s);
    if (N == 128 && K == 64) return run_ta<128, 64>(A, B, D, status, s);
    return -1;
}

template <int N, int K, bool PAD>
static int run(const void *A, const void *B, void *D, int *status, cudaStream_t s)
{
    const int smem = (PAD ? tc::kmajor_pad_bytes(128, K) + tc::kmajor_pad_bytes(N, K) : 128 * K * 2 + N * K * 2) + 64;
    cudaFuncSetAttribute(tc_gemm_kernel<N, K, PAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    tc_gemm_kernel<N, K, PAD><<<1, 128, smem, s>>>((const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B,
                                                  (float *)D, status);
    return (int)cudaGetLastError();
}

extern "C" int tc_gemm_test(const void *A, const void *B, void *D, int N, int K, int pad, int *status, void *stream)
{
    cudaStream_t s = (cudaStream_t)stream;
    if (pad) {
        if (N == 128 && K == 128) return run<128, 128, true>(A, B, D, status, s);
        if (N == 64 && K == 128) return run<64, 128, true>(A, B, D, status, s);
        return -1;
    }
    if (N == 64 && K == 128) return run<64, 128, false>(A, B, D, status, s);
    if (N == 128 && K == 64) return run<128, 64, false>(A, B, D, status, s);
    if (N == 64 && K == 64) return run<64, 64, false>(A, B, D, status, s);
    if (N == 128 && K == 128) return run<128, 128, false>(A, B, D, status, s);
    if (N == 192 && K == 64) return run<192, 64, false>(A, B, D, status, s);
    return -1;
}
