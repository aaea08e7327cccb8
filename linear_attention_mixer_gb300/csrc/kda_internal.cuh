// kda_internal.cuh - shared device helpers and the state object of the KDA library.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/kda.h"

namespace kda {

constexpr int kD = 128;  // head dim (dk = dv)
constexpr int kK = 4;    // conv kernel
constexpr int kC = 64;   // prefill chunk

// The library-owned state object behind the opaque kda_state handle.
struct State {
    kda_config_t cfg;
    int32_t max_slots;
    int device;
    float *S;         // [max_slots][H][d][d] FP32
    void *tail;       // [max_slots][3][K-1][H*d] io dtype
    int32_t *err;     // device error word (0 = none)
    void *ws;         // prefill workspace
    size_t ws_bytes;
    int sms;          // SM count of the device, read once when the state is made (0: not read)
    // Kernels whose dynamic shared-memory limit has been raised on this state's device, one
    // bit each (kSmem* below). Raising it is a host driver call; doing it once per state keeps
    // it off the per-call path of the decode entry points. A state does not outlive its
    // device context, so the bits cannot go stale.
    mutable std::atomic<uint32_t> smem_raised;
};

enum : uint32_t {
    kSmemDecodeBf16 = 1u << 0, kSmemDecodeF32 = 1u << 1, kSmemPrepTc = 1u << 4, kSmemPrepF32 = 1u << 5,
    kSmemStateTc = 1u << 6, kSmemStateF32 = 1u << 7,
};
// the multi-token decode has one kernel per (I/O type, tokens per call n = 1 .. 8): bits 8 .. 23
constexpr uint32_t smem_bit_multi(bool f32, int n) { return 1u << (8 + 2 * (n - 1) + (f32 ? 1 : 0)); }

// Raise `kernel`'s dynamic shared-memory limit to `bytes` once per state.
template <typename Fn>
inline cudaError_t raise_smem_once(const State &st, uint32_t bit, Fn *kernel, size_t bytes)
{
    if (st.smem_raised.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) st.smem_raised.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// The SM count of the state's device (read at allocation; looked up if the state has none).
inline cudaError_t state_sms(const State &st, int *sms)
{
    if (st.sms > 0) {
        *sms = st.sms;
        return cudaSuccess;
    }
    return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, st.device);
}

// cuTensorMapEncodeTiled, looked up once from the driver through the runtime (the library does
// not link the driver library itself); null when the driver offers none.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }();
    return encode;
}

// Tensor map of a row-major [rows][cols] matrix of BF16 (elem_bytes 2) or FP32 (4) values, for
// 2-D boxes of box_cols x box_rows with no swizzle. The base must be 16-byte aligned and a row
// a multiple of 16 bytes.
inline cudaError_t encode_rows_box(CUtensorMap *m, const void *base, int elem_bytes, int64_t rows, int64_t cols,
                                   int box_cols, int box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * (cuuint64_t)elem_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r =
        encode(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ---------------------------------------------------------------- IO types
template <typename T> struct IO;
template <> struct IO<float> {
    static __device__ __forceinline__ float ld(const float *p) { return *p; }
    static __device__ __forceinline__ void st(float *p, float x) { *p = x; }
};
template <> struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void st(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Streaming (evict-first) 16-byte accesses for data touched once per launch.
__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }

// Error word codes (device side mirror of kda_status values).
constexpr int32_t kErrBadSlot = KDA_ERR_DEVICE;

// Launchers (host), defined in kda_decode.cu / kda_prefill.cu.
cudaError_t launch_decode(const State &st, const kda_layer_params &p, const int32_t *slots, int B,
                          const void *q, const void *k, const void *v, const void *z, const void *b,
                          const void *g, void *out, cudaStream_t stream);
cudaError_t launch_decode_multi(const State &st, const kda_layer_params &p, const int32_t *slots, int B, int n,
                                const void *q, const void *k, const void *v, const void *z, const void *b,
                                const void *g, void *out, cudaStream_t stream);

size_t prefill_workspace_bytes(const kda_config_t &cfg, int64_t total_chunks, int64_t total_T, int N);
// f and w_fb non-null: z is not read; it is formed in the prefill as W_fb f (BF16 I/O only)
cudaError_t launch_prefill(const State &st, const kda_layer_params &p, const int32_t *slots,
                           const int32_t *cu_seqlens, int N, int64_t total_T, int64_t total_chunks,
                           const void *q, const void *k, const void *v, const void *z, const void *b,
                           const void *g, void *out, void *ws, cudaStream_t stream, const void *f = nullptr,
                           const void *w_fb = nullptr);

// Error text and config checks shared by every entry point (kda_api.cu).
kda_status record_error(kda_status s, const char *msg);
// true when the per-token row tensors are 16-byte aligned (their rows move as bulk and
// tensor copies of whole 16-byte units; b is read element by element and needs no more
// than its own alignment)
inline bool io_aligned(const void *q, const void *k, const void *v, const void *z, const void *g, const void *out)
{
    const uintptr_t u = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(z) |
                        reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(out);
    return (u & 15u) == 0;
}
bool config_ok(const kda_config_t *c);

}  // namespace kda
