// Test kernel for the FMA-pipe reciprocal of kda_ptx.cuh: y[i] = rcp_newton(x[i]).
#include <cuda_runtime.h>

#include "../../linear_attention_mixer_gb300/csrc/kda_ptx.cuh"

__global__ void rcp_kernel(const float *x, float *y, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = kda::rcp_newton(x[i]);
}

extern "C" int rcp_newton_test(const float *x, float *y, int n, void *stream)
{
    if (n <= 0) return 0;
    rcp_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
    return (int)cudaGetLastError();
}
