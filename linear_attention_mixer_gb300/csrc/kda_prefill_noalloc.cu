// kda_prefill_noalloc.cu - the prefill for callers that must not allocate
// device memory.
//
// Some callers cannot let a library call cudaMalloc: serving runtimes that hand
// out every byte of device memory from their own arena (so that memory is
// accounted exactly and no request can fail halfway on an allocation), and
// latency-critical loops that cannot accept the device-wide synchronisation
// that cudaMalloc / cudaFree may cause. kda_prefill keeps a per-state workspace
// that it grows with cudaMalloc; this entry point instead uses the file-scope
// array below, and takes the recurrent state as caller-owned buffers.
//
// The array is a __device__ variable: every GPU that loads the library holds
// it until the process exits. Every call on a device shares it and it keeps
// the previous call's contents, so calls whose work overlaps on the GPU race;
// callers order them (one stream, or events). The chunk list, the chunk factors
// and the o buffer are fully rewritten by each call; only the error word must
// start at zero, and it is cleared at the start of every call.
#include <cstdio>

#include "kda_internal.cuh"

namespace {

constexpr size_t kErrRegion = 256;  // first 256 bytes: the error word used when err == NULL

__device__ __align__(256) unsigned char g_noalloc_ws[KDA_NOALLOC_WORKSPACE_BYTES];

// The device address of the array in the current context. The array's host-side
// name is only a stand-in; kernels must get this address. It is looked up on
// every call (cudaGetSymbolAddress allocates nothing), so it stays right after a
// cudaDeviceReset and in whichever context is current; a cached address could
// point into a context that no longer exists. The first lookup in a context may
// load the library's module there.
kda_status workspace_address(unsigned char **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return kda::record_error(KDA_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                                : "cudaGetSymbolAddress gave a null address");
    }
    *out = static_cast<unsigned char *>(p);
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const kda_config_t *cfg, const kda_layer_params *params, float *S,
                                          void *tail, int32_t max_slots, int32_t *err, const int32_t *slots,
                                          const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int32_t N,
                                          const void *q, const void *k, const void *v, const void *z,
                                          const void *b, const void *g, void *out, void *stream)
{
    char msg[256];
    if (!kda::config_ok(cfg)) return KDA_ERR_INVALID;
    if (!params || !params->conv_w || !params->dt_bias || !params->A_log || !params->norm_w)
        return kda::record_error(KDA_ERR_INVALID, "layer params (or one of its pointers) is NULL");
    if (N < 0 || N > 65535) return kda::record_error(KDA_ERR_INVALID, "N must be in [0, 65535]");
    if (N == 0) return KDA_OK;
    if (!S || !tail || max_slots < 1) return kda::record_error(KDA_ERR_INVALID, "S / tail NULL or max_slots < 1");
    if (!slots || !cu_seqlens || !cu_seqlens_host)
        return kda::record_error(KDA_ERR_INVALID, "slots or cu_seqlens is NULL");
    if (cu_seqlens_host[0] != 0) return kda::record_error(KDA_ERR_INVALID, "cu_seqlens[0] must be 0");
    int64_t total_chunks = 0;
    for (int32_t i = 0; i < N; ++i) {
        const int64_t len = (int64_t)cu_seqlens_host[i + 1] - cu_seqlens_host[i];
        if (len < 0) return kda::record_error(KDA_ERR_INVALID, "cu_seqlens decreases");
        total_chunks += (len + kda::kC - 1) / kda::kC;
    }
    const int64_t total_T = cu_seqlens_host[N];
    if (total_T > 0 && (!q || !k || !v || !z || !b || !g || !out))
        return kda::record_error(KDA_ERR_INVALID, "a tensor pointer is NULL");
    if (total_T > 0 && !kda::io_aligned(q, k, v, z, g, out))
        return kda::record_error(KDA_ERR_INVALID, "q, k, v, z, g or out is not 16-byte aligned");
    const size_t need = kda::prefill_workspace_bytes(*cfg, total_chunks, total_T, N);
    if (need > KDA_NOALLOC_WORKSPACE_BYTES - kErrRegion) {
        snprintf(msg, sizeof(msg),
                 "this call needs %zu bytes of workspace; the static workspace holds %zu (split the call)",
                 need, (size_t)(KDA_NOALLOC_WORKSPACE_BYTES - kErrRegion));
        return kda::record_error(KDA_ERR_INVALID, msg);
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return kda::record_error(KDA_ERR_CUDA, cudaGetErrorString(e));
    unsigned char *base = nullptr;
    const kda_status s = workspace_address(&base);
    if (s != KDA_OK) return s;

    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    int32_t *errw = err;
    if (!errw) {  // the shared word keeps the last call's value: clear it
        errw = reinterpret_cast<int32_t *>(base);
        e = cudaMemsetAsync(errw, 0, sizeof(int32_t), strm);
        if (e != cudaSuccess) return kda::record_error(KDA_ERR_CUDA, cudaGetErrorString(e));
    }
    kda::State st{};
    st.cfg = *cfg;
    st.max_slots = max_slots;
    st.device = dev;
    st.S = S;
    st.tail = tail;
    st.err = errw;
    st.ws = base + kErrRegion;
    st.ws_bytes = KDA_NOALLOC_WORKSPACE_BYTES - kErrRegion;
    e = kda::launch_prefill(st, *params, slots, cu_seqlens, N, total_T, total_chunks, q, k, v, z, b, g, out,
                            st.ws, strm);
    if (e != cudaSuccess) return kda::record_error(KDA_ERR_CUDA, cudaGetErrorString(e));
    return KDA_OK;
}
