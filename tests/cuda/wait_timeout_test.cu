// Unit test kernel for the bounded mbarrier wait every kernel of the library uses
// (mbar_wait_bounded in kda_ptx.cuh). Thread 0 waits for a phase of a shared-memory
// mbarrier. With `arrive` = 0 nothing ever arrives, so the wait must give up after
// `limit` polls; the kernel then records KDA_ERR_TIMEOUT in *err, as the library's
// kernels do, and returns. With `arrive` = 1 the phase completes first and nothing is
// recorded. *polls receives the number of polls the wait took (limit when it gave up).
#include <stdint.h>

#include "../../include/kda.h"
#include "../../linear_attention_mixer_gb300/csrc/kda_ptx.cuh"

__global__ void wait_timeout_kernel(int32_t *err, uint32_t limit, int arrive, uint32_t *polls)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        kda::mbar_init(&bar, 1);
        kda::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (arrive) kda::mbar_arrive(&bar);
        uint32_t i = 0;
        bool ok = false;
        for (; i < limit && !ok; ++i) ok = kda::mbar_try_wait(&bar, 0);
        // the library's helper, on the same phase: it must agree
        const bool ok2 = kda::mbar_wait_bounded(&bar, 0, limit);
        *polls = i;
        if (!ok || !ok2) atomicExch(err, KDA_ERR_TIMEOUT);
    }
}

extern "C" int wait_timeout_test(int32_t *err, uint32_t limit, int arrive, uint32_t *polls, void *stream)
{
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit, arrive, polls);
    return (int)cudaGetLastError();
}
