// kda_api.cu - host side of the C ABI declared in include/kda.h: argument
// checks, the state object (alloc / reset / snapshot / restore / free) and the
// dispatch to the decode and prefill kernels.
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "kda_internal.cuh"

using kda::State;

namespace {

thread_local char g_err[512] = "";

kda_status fail(kda_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

kda_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(e == cudaErrorMemoryAllocation ? KDA_ERR_OOM : KDA_ERR_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

size_t io_size(int32_t dt) { return dt == KDA_BF16 ? 2 : 4; }

bool cfg_check(const kda_config_t *c)
{
    if (!c) { fail(KDA_ERR_INVALID, "config is NULL"); return false; }
    if (c->num_heads < 1) { fail(KDA_ERR_INVALID, "num_heads must be >= 1 (got %d)", c->num_heads); return false; }
    if (c->head_dim != kda::kD) { fail(KDA_ERR_INVALID, "head_dim must be %d (got %d)", kda::kD, c->head_dim); return false; }
    if (c->conv_kernel != kda::kK) { fail(KDA_ERR_INVALID, "conv_kernel must be %d (got %d)", kda::kK, c->conv_kernel); return false; }
    if (c->chunk_size != kda::kC) { fail(KDA_ERR_INVALID, "chunk_size must be %d (got %d)", kda::kC, c->chunk_size); return false; }
    if (c->io_dtype != KDA_F32 && c->io_dtype != KDA_BF16) { fail(KDA_ERR_INVALID, "io_dtype must be KDA_F32 or KDA_BF16"); return false; }
    if (!(c->gate_lower_bound < 0.f) || !std::isfinite(c->gate_lower_bound)) { fail(KDA_ERR_INVALID, "gate_lower_bound must be finite and < 0"); return false; }
    if (!(c->l2_eps > 0.f) || !(c->rms_eps > 0.f) || !std::isfinite(c->q_scale)) { fail(KDA_ERR_INVALID, "eps must be > 0 and q_scale finite"); return false; }
    return true;
}

bool cfg_same(const kda_config_t &a, const kda_config_t &b)
{
    return a.num_heads == b.num_heads && a.head_dim == b.head_dim && a.conv_kernel == b.conv_kernel &&
           a.io_dtype == b.io_dtype && a.chunk_size == b.chunk_size && a.gate_lower_bound == b.gate_lower_bound &&
           a.l2_eps == b.l2_eps && a.rms_eps == b.rms_eps && a.q_scale == b.q_scale;
}

size_t state_bytes(const kda_config_t &c) { return (size_t)c.num_heads * c.head_dim * c.head_dim * sizeof(float); }
size_t tail_bytes(const kda_config_t &c)
{
    return (size_t)3 * (c.conv_kernel - 1) * c.num_heads * c.head_dim * io_size(c.io_dtype);
}

bool device_matches(const State *st)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != st->device) {
        fail(KDA_ERR_INVALID, "current device %d is not the state's device %d", dev, st->device);
        return false;
    }
    return true;
}

bool slots_check(const State *st, const int32_t *slots, int32_t n)
{
    if (n < 0) { fail(KDA_ERR_INVALID, "slot count must be >= 0 (got %d)", n); return false; }
    if (n > 0 && !slots) { fail(KDA_ERR_INVALID, "slots is NULL"); return false; }
    for (int32_t i = 0; i < n; ++i)
        if (slots[i] < 0 || slots[i] >= st->max_slots) {
            fail(KDA_ERR_INVALID, "slot id %d at position %d outside [0, %d)", slots[i], i, st->max_slots);
            return false;
        }
    return true;
}

bool params_check(const kda_layer_params *p)
{
    if (!p || !p->conv_w || !p->dt_bias || !p->A_log || !p->norm_w) {
        fail(KDA_ERR_INVALID, "layer params (or one of its pointers) is NULL");
        return false;
    }
    return true;
}

kda_blob_header make_header(const State *st, int32_t n)
{
    kda_blob_header h;
    memset(&h, 0, sizeof(h));
    h.magic = KDA_BLOB_MAGIC;
    h.version = KDA_BLOB_VERSION;
    h.num_heads = st->cfg.num_heads;
    h.head_dim = st->cfg.head_dim;
    h.conv_kernel = st->cfg.conv_kernel;
    h.io_dtype = st->cfg.io_dtype;
    h.n_slots = n;
    h.state_bytes_per_slot = state_bytes(st->cfg);
    h.tail_bytes_per_slot = tail_bytes(st->cfg);
    return h;
}

}  // namespace

static_assert(sizeof(kda_blob_header) == 64, "blob header must be 64 bytes");

namespace kda {
// For entry points defined in other translation units.
kda_status record_error(kda_status s, const char *msg) { return fail(s, "%s", msg); }
bool config_ok(const kda_config_t *c) { return cfg_check(c); }
}  // namespace kda

extern "C" {

const char *kda_last_error(void) { return g_err; }

kda_status kda_config(kda_config_t *cfg, int32_t num_heads, int32_t head_dim, int32_t io_dtype)
{
    if (!cfg) return fail(KDA_ERR_INVALID, "cfg is NULL");
    kda_config_t c;
    c.num_heads = num_heads;
    c.head_dim = head_dim;
    c.conv_kernel = kda::kK;
    c.io_dtype = io_dtype;
    c.chunk_size = kda::kC;
    c.gate_lower_bound = -5.0f;
    c.l2_eps = 1e-6f;
    c.rms_eps = 1e-6f;
    c.q_scale = head_dim > 0 ? 1.0f / sqrtf((float)head_dim) : 0.f;
    if (!cfg_check(&c)) return KDA_ERR_INVALID;
    *cfg = c;
    return KDA_OK;
}

kda_status kda_state_alloc(const kda_config_t *cfg, int32_t max_slots, kda_state **out)
{
    if (!out) return fail(KDA_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (!cfg_check(cfg)) return KDA_ERR_INVALID;
    if (max_slots < 1) return fail(KDA_ERR_INVALID, "max_slots must be >= 1 (got %d)", max_slots);
    State *st = new (std::nothrow) State();
    if (!st) return fail(KDA_ERR_OOM, "host allocation of the state object failed");
    st->cfg = *cfg;
    st->max_slots = max_slots;
    cudaError_t e = cudaGetDevice(&st->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&st->sms, cudaDevAttrMultiProcessorCount, st->device);
    const size_t sb = state_bytes(*cfg) * (size_t)max_slots, tb = tail_bytes(*cfg) * (size_t)max_slots;
    if (e == cudaSuccess) e = cudaMalloc(&st->S, sb);
    if (e == cudaSuccess) e = cudaMalloc(&st->tail, tb);
    if (e == cudaSuccess) e = cudaMalloc(&st->err, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemset(st->S, 0, sb);
    if (e == cudaSuccess) e = cudaMemset(st->tail, 0, tb);
    if (e == cudaSuccess) e = cudaMemset(st->err, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(st->S);
        cudaFree(st->tail);
        cudaFree(st->err);
        delete st;
        cudaGetLastError();
        return cuda_fail(e, "kda_state_alloc");
    }
    *out = reinterpret_cast<kda_state *>(st);
    return KDA_OK;
}

kda_status kda_state_free(kda_state *h)
{
    if (!h) return KDA_OK;
    State *st = reinterpret_cast<State *>(h);
    cudaError_t e = cudaDeviceSynchronize();
    cudaFree(st->S);
    cudaFree(st->tail);
    cudaFree(st->err);
    cudaFree(st->ws);
    delete st;
    if (e != cudaSuccess) return cuda_fail(e, "kda_state_free");
    return KDA_OK;
}

int32_t kda_state_max_slots(const kda_state *h)
{
    return h ? reinterpret_cast<const State *>(h)->max_slots : 0;
}

size_t kda_state_blob_bytes(const kda_state *h, int32_t n_slots)
{
    if (!h || n_slots < 0) return 0;
    const State *st = reinterpret_cast<const State *>(h);
    return sizeof(kda_blob_header) + (size_t)n_slots * (state_bytes(st->cfg) + tail_bytes(st->cfg));
}

kda_status kda_state_reset(kda_state *h, const int32_t *slots, int32_t n, void *stream)
{
    if (!h) return fail(KDA_ERR_INVALID, "state is NULL");
    State *st = reinterpret_cast<State *>(h);
    if (!slots_check(st, slots, n) || !device_matches(st)) return KDA_ERR_INVALID;
    const size_t sb = state_bytes(st->cfg), tb = tail_bytes(st->cfg);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int32_t i = 0; i < n; ++i) {
        cudaError_t e = cudaMemsetAsync(reinterpret_cast<char *>(st->S) + sb * slots[i], 0, sb, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(static_cast<char *>(st->tail) + tb * slots[i], 0, tb, s);
        if (e != cudaSuccess) return cuda_fail(e, "kda_state_reset");
    }
    return KDA_OK;
}

kda_status kda_state_snapshot(const kda_state *h, const int32_t *slots, int32_t n, void *dst,
                              int32_t dst_on_device, void *stream)
{
    if (!h) return fail(KDA_ERR_INVALID, "state is NULL");
    const State *st = reinterpret_cast<const State *>(h);
    if (!slots_check(st, slots, n) || !device_matches(st)) return KDA_ERR_INVALID;
    if (!dst) return fail(KDA_ERR_INVALID, "dst is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const kda_blob_header hdr = make_header(st, n);
    const size_t sb = state_bytes(st->cfg), tb = tail_bytes(st->cfg);
    char *d = static_cast<char *>(dst);
    const cudaMemcpyKind kind = dst_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost;
    cudaError_t e = cudaSuccess;
    if (dst_on_device)
        e = cudaMemcpyAsync(d, &hdr, sizeof(hdr), cudaMemcpyHostToDevice, s);  // pageable source: staged before return
    else
        memcpy(d, &hdr, sizeof(hdr));
    size_t off = sizeof(hdr);
    for (int32_t i = 0; i < n && e == cudaSuccess; ++i) {
        e = cudaMemcpyAsync(d + off, reinterpret_cast<const char *>(st->S) + sb * slots[i], sb, kind, s);
        off += sb;
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d + off, static_cast<const char *>(st->tail) + tb * slots[i], tb, kind, s);
        off += tb;
    }
    if (e != cudaSuccess) return cuda_fail(e, "kda_state_snapshot");
    return KDA_OK;
}

kda_status kda_state_restore(kda_state *h, const int32_t *slots, int32_t n, const void *src,
                             int32_t src_on_device, void *stream)
{
    if (!h) return fail(KDA_ERR_INVALID, "state is NULL");
    State *st = reinterpret_cast<State *>(h);
    if (!slots_check(st, slots, n) || !device_matches(st)) return KDA_ERR_INVALID;
    if (!src) return fail(KDA_ERR_INVALID, "src is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_blob_header hdr;
    if (src_on_device) {
        cudaError_t e = cudaStreamSynchronize(s);
        if (e == cudaSuccess) e = cudaMemcpy(&hdr, src, sizeof(hdr), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "kda_state_restore (header read)");
    } else {
        memcpy(&hdr, src, sizeof(hdr));
    }
    const kda_blob_header want = make_header(st, n);
    if (hdr.magic != want.magic) return fail(KDA_ERR_BLOB, "blob magic 0x%08x is not KDA1", hdr.magic);
    if (hdr.version != want.version) return fail(KDA_ERR_BLOB, "blob version %u, expected %u", hdr.version, want.version);
    if (hdr.num_heads != want.num_heads || hdr.head_dim != want.head_dim || hdr.conv_kernel != want.conv_kernel ||
        hdr.io_dtype != want.io_dtype)
        return fail(KDA_ERR_BLOB, "blob geometry H=%d d=%d K=%d dtype=%d does not match the state's H=%d d=%d K=%d dtype=%d",
                    hdr.num_heads, hdr.head_dim, hdr.conv_kernel, hdr.io_dtype, want.num_heads, want.head_dim,
                    want.conv_kernel, want.io_dtype);
    if (hdr.n_slots != n) return fail(KDA_ERR_BLOB, "blob holds %d slots, %d requested", hdr.n_slots, n);
    if (hdr.state_bytes_per_slot != want.state_bytes_per_slot || hdr.tail_bytes_per_slot != want.tail_bytes_per_slot)
        return fail(KDA_ERR_BLOB, "blob per-slot sizes do not match");
    const size_t sb = state_bytes(st->cfg), tb = tail_bytes(st->cfg);
    const char *p = static_cast<const char *>(src);
    const cudaMemcpyKind kind = src_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    size_t off = sizeof(hdr);
    cudaError_t e = cudaSuccess;
    for (int32_t i = 0; i < n && e == cudaSuccess; ++i) {
        e = cudaMemcpyAsync(reinterpret_cast<char *>(st->S) + sb * slots[i], p + off, sb, kind, s);
        off += sb;
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(st->tail) + tb * slots[i], p + off, tb, kind, s);
        off += tb;
    }
    if (e != cudaSuccess) return cuda_fail(e, "kda_state_restore");
    return KDA_OK;
}

kda_status kda_decode_token(const kda_config_t *cfg, const kda_layer_params *params, kda_state *h,
                            const int32_t *slots, int32_t B, const void *q, const void *k, const void *v,
                            const void *z, const void *b, const void *g, void *out, void *stream)
{
    if (!h) return fail(KDA_ERR_INVALID, "state is NULL");
    State *st = reinterpret_cast<State *>(h);
    if (!cfg_check(cfg)) return KDA_ERR_INVALID;
    if (!cfg_same(*cfg, st->cfg)) return fail(KDA_ERR_INVALID, "config differs from the state's config");
    if (!params_check(params)) return KDA_ERR_INVALID;
    if (B < 0) return fail(KDA_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (B == 0) return KDA_OK;
    if (!slots || !q || !k || !v || !z || !b || !g || !out) return fail(KDA_ERR_INVALID, "a tensor pointer is NULL");
    if (!kda::io_aligned(q, k, v, z, g, out)) return fail(KDA_ERR_INVALID, "q, k, v, z, g or out is not 16-byte aligned");
    if ((int64_t)B * cfg->num_heads > INT_MAX) return fail(KDA_ERR_INVALID, "B * num_heads exceeds the grid limit");
    if (!device_matches(st)) return KDA_ERR_INVALID;
    cudaError_t e = kda::launch_decode(*st, *params, slots, B, q, k, v, z, b, g, out,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_decode_token launch");
    return KDA_OK;
}

kda_status kda_decode_tokens(const kda_config_t *cfg, const kda_layer_params *params, kda_state *h,
                             const int32_t *slots, int32_t B, int32_t n, const void *q, const void *k,
                             const void *v, const void *z, const void *b, const void *g, void *out, void *stream)
{
    if (!h) return fail(KDA_ERR_INVALID, "state is NULL");
    State *st = reinterpret_cast<State *>(h);
    if (!cfg_check(cfg)) return KDA_ERR_INVALID;
    if (!cfg_same(*cfg, st->cfg)) return fail(KDA_ERR_INVALID, "config differs from the state's config");
    if (!params_check(params)) return KDA_ERR_INVALID;
    if (B < 0) return fail(KDA_ERR_INVALID, "B must be >= 0 (got %d)", B);
    if (n < 1 || n > KDA_DECODE_MAX_TOKENS)
        return fail(KDA_ERR_INVALID, "n must be in [1, %d] (got %d)", KDA_DECODE_MAX_TOKENS, n);
    if (B == 0) return KDA_OK;
    if (!slots || !q || !k || !v || !z || !b || !g || !out) return fail(KDA_ERR_INVALID, "a tensor pointer is NULL");
    if (!kda::io_aligned(q, k, v, z, g, out)) return fail(KDA_ERR_INVALID, "q, k, v, z, g or out is not 16-byte aligned");
    if ((int64_t)B * n * cfg->num_heads > INT_MAX) return fail(KDA_ERR_INVALID, "B * n * num_heads is too large");
    if (!device_matches(st)) return KDA_ERR_INVALID;
    cudaError_t e = kda::launch_decode_multi(*st, *params, slots, B, n, q, k, v, z, b, g, out,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kda_decode_tokens launch");
    return KDA_OK;
}

namespace {
// kda_prefill, or with f and w_fb (z NULL) the prefill that forms z = W_fb f itself
kda_status prefill_entry(const kda_config_t *cfg, const kda_layer_params *params, kda_state *h,
                         const int32_t *slots, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int32_t N,
                         const void *q, const void *k, const void *v, const void *z, const void *b, const void *g,
                         void *out, void *stream, bool fused, const void *f, const void *w_fb)
{
    if (!h) return fail(KDA_ERR_INVALID, "state is NULL");
    State *st = reinterpret_cast<State *>(h);
    if (!cfg_check(cfg)) return KDA_ERR_INVALID;
    if (!cfg_same(*cfg, st->cfg)) return fail(KDA_ERR_INVALID, "config differs from the state's config");
    if (!params_check(params)) return KDA_ERR_INVALID;
    if (N < 0) return fail(KDA_ERR_INVALID, "N must be >= 0 (got %d)", N);
    if (N == 0) return KDA_OK;
    if (N > 65535) return fail(KDA_ERR_INVALID, "N must be <= 65535 (got %d)", N);
    if (!slots || !cu_seqlens || !cu_seqlens_host) return fail(KDA_ERR_INVALID, "slots or cu_seqlens is NULL");
    if (cu_seqlens_host[0] != 0) return fail(KDA_ERR_INVALID, "cu_seqlens[0] must be 0");
    int64_t total_chunks = 0;
    for (int32_t i = 0; i < N; ++i) {
        const int64_t len = (int64_t)cu_seqlens_host[i + 1] - cu_seqlens_host[i];
        if (len < 0) return fail(KDA_ERR_INVALID, "cu_seqlens decreases at %d", i);
        total_chunks += (len + kda::kC - 1) / kda::kC;
    }
    const int64_t total_T = cu_seqlens_host[N];
    if (fused && cfg->io_dtype != KDA_BF16)
        return fail(KDA_ERR_INVALID, "the fused gate projection needs BF16 I/O");
    if (total_T > 0 && (!q || !k || !v || (fused ? (!f || !w_fb) : !z) || !b || !g || !out))
        return fail(KDA_ERR_INVALID, "a tensor pointer is NULL");
    if (total_T > 0 && !kda::io_aligned(q, k, v, fused ? f : z, g, out))
        return fail(KDA_ERR_INVALID, "q, k, v, %s, g or out is not 16-byte aligned", fused ? "f" : "z");
    if (fused && (reinterpret_cast<uintptr_t>(w_fb) & 15u)) return fail(KDA_ERR_INVALID, "w_fb is not 16-byte aligned");
    if (total_chunks * cfg->num_heads > INT_MAX || (total_T * cfg->num_heads + 7) / 8 > INT_MAX)
        return fail(KDA_ERR_INVALID, "too many tokens for one call");
    if (!device_matches(st)) return KDA_ERR_INVALID;
    const size_t need = kda::prefill_workspace_bytes(st->cfg, total_chunks, total_T, N);
    if (need > st->ws_bytes) {
        cudaFree(st->ws);  // synchronises: earlier calls may still use it
        st->ws = nullptr;
        st->ws_bytes = 0;
        cudaError_t e = cudaMalloc(&st->ws, need);
        if (e != cudaSuccess) {
            cudaGetLastError();
            st->ws = nullptr;
            return cuda_fail(e, "kda_prefill workspace");
        }
        st->ws_bytes = need;
    }
    cudaError_t e = kda::launch_prefill(*st, *params, slots, cu_seqlens, N, total_T, total_chunks, q, k, v, z, b,
                                        g, out, st->ws, static_cast<cudaStream_t>(stream), fused ? f : nullptr,
                                        fused ? w_fb : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "kda_prefill launch");
    return KDA_OK;
}
}  // namespace

kda_status kda_prefill(const kda_config_t *cfg, const kda_layer_params *params, kda_state *h,
                       const int32_t *slots, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int32_t N,
                       const void *q, const void *k, const void *v, const void *z, const void *b, const void *g,
                       void *out, void *stream)
{
    return prefill_entry(cfg, params, h, slots, cu_seqlens, cu_seqlens_host, N, q, k, v, z, b, g, out, stream,
                         false, nullptr, nullptr);
}

kda_status kda_prefill_gate_fused(const kda_config_t *cfg, const kda_layer_params *params, kda_state *h,
                                  const int32_t *slots, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                  int32_t N, const void *q, const void *k, const void *v, const void *f,
                                  const void *w_fb, const void *b, const void *g, void *out, void *stream)
{
    return prefill_entry(cfg, params, h, slots, cu_seqlens, cu_seqlens_host, N, q, k, v, nullptr, b, g, out, stream,
                         true, f, w_fb);
}

kda_status kda_state_poll_error(kda_state *h, int32_t *code)
{
    if (!h || !code) return fail(KDA_ERR_INVALID, "state or code is NULL");
    State *st = reinterpret_cast<State *>(h);
    if (!device_matches(st)) return KDA_ERR_INVALID;
    int32_t v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, st->err, sizeof(v), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(st->err, 0, sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(e, "kda_state_poll_error");
    *code = v;
    return KDA_OK;
}

}  // extern "C"
