// kda_photo.cu - recurrent-state photos (host side of include/kda.h's kda_photo_*): a
// bounded store of one slot's snapshots across a stack of KDA layers, keyed by the token
// prefix they were taken after, kept in pinned host memory or parked in files (kimi_k3.c
// header, the COLI_K3_CKPT and COLI_K3_CKPT_DIR serve options).
//
// The device side is kda_state_snapshot / kda_state_restore. The store adds the policy:
// exact prefix matching, least-recently-used eviction, and one spare buffer, so that a take
// never overwrites a photo before its own copy has succeeded.
#include <sys/stat.h>
#include <unistd.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "kda_internal.cuh"

namespace {

kda_status photo_fail(kda_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    return kda::record_error(s, buf);
}

struct Photo {
    int32_t id = -1;
    uint64_t stamp = 0;               // clock value of the last take or restore
    std::vector<int32_t> tokens;      // the prefix the photo was taken after
    std::vector<size_t> layer_bytes;  // snapshot blob bytes of each layer, back to back
    void *host = nullptr;             // pinned blob (memory mode)
    size_t host_bytes = 0;
    std::string path;                 // parked file (file mode)
};

size_t total_of(const std::vector<size_t> &v)
{
    size_t t = 0;
    for (size_t x : v) t += x;
    return t;
}

// pinned, portable host memory (usable whichever device the states live on)
cudaError_t pinned_alloc(void **p, size_t bytes) { return cudaHostAlloc(p, bytes, cudaHostAllocPortable); }

bool same_geometry(const kda::State *a, const kda::State *b)
{
    return a->cfg.num_heads == b->cfg.num_heads && a->cfg.head_dim == b->cfg.head_dim &&
           a->cfg.conv_kernel == b->cfg.conv_kernel && a->cfg.io_dtype == b->cfg.io_dtype;
}

bool write_file(const std::string &path, const void *p, size_t n)
{
    FILE *f = fopen(path.c_str(), "wb");
    if (!f) return false;
    const bool ok = fwrite(p, 1, n, f) == n;
    return (fclose(f) == 0) && ok;
}

bool read_file(const std::string &path, void *p, size_t n)
{
    FILE *f = fopen(path.c_str(), "rb");
    if (!f) return false;
    const bool ok = fread(p, 1, n, f) == n;
    fclose(f);
    return ok;
}

}  // namespace

struct kda_photo_store {
    int32_t capacity = 0;
    std::string dir;  // empty: photos in pinned host memory
    mutable std::mutex mu;
    std::vector<Photo> photos;
    int32_t next_id = 0;
    uint64_t clock = 0;
    // memory mode: the buffer the next take copies into; file mode: the staging buffer of
    // every file write and read
    void *spare = nullptr;
    size_t spare_bytes = 0;

    bool file_mode() const { return !dir.empty(); }

    // the spare buffer, at least `bytes` long
    kda_status reserve_spare(size_t bytes)
    {
        if (spare && spare_bytes >= bytes) return KDA_OK;
        if (spare) cudaFreeHost(spare);
        spare = nullptr;
        spare_bytes = 0;
        const cudaError_t e = pinned_alloc(&spare, bytes);
        if (e != cudaSuccess) {
            spare = nullptr;
            return photo_fail(e == cudaErrorMemoryAllocation ? KDA_ERR_OOM : KDA_ERR_CUDA,
                              "photo buffer of %zu bytes: %s", bytes, cudaGetErrorString(e));
        }
        spare_bytes = bytes;
        return KDA_OK;
    }

    // drop photo i: its pinned buffer becomes the spare when that is larger, its file goes
    void drop(size_t i)
    {
        Photo &p = photos[i];
        if (p.host) {
            if (!spare || p.host_bytes > spare_bytes) {
                if (spare) cudaFreeHost(spare);
                spare = p.host;
                spare_bytes = p.host_bytes;
            } else {
                cudaFreeHost(p.host);
            }
        }
        if (!p.path.empty()) unlink(p.path.c_str());
        photos.erase(photos.begin() + (long)i);
    }

    Photo *by_id(int32_t id)
    {
        for (Photo &p : photos)
            if (p.id == id) return &p;
        return nullptr;
    }
};

namespace {

// layers non-NULL, of one geometry, and slot valid in each
kda_status check_layers(kda_state *const *layers, int32_t n_layers, int32_t slot)
{
    if (!layers) return photo_fail(KDA_ERR_INVALID, "layers is NULL");
    if (n_layers < 1) return photo_fail(KDA_ERR_INVALID, "n_layers must be >= 1 (got %d)", n_layers);
    const kda::State *first = nullptr;
    for (int32_t i = 0; i < n_layers; ++i) {
        if (!layers[i]) return photo_fail(KDA_ERR_INVALID, "layer %d is NULL", i);
        const kda::State *st = reinterpret_cast<const kda::State *>(layers[i]);
        if (slot < 0 || slot >= st->max_slots)
            return photo_fail(KDA_ERR_INVALID, "slot %d outside [0, %d) of layer %d", slot, st->max_slots, i);
        if (!first) first = st;
        else if (!same_geometry(first, st))
            return photo_fail(KDA_ERR_INVALID, "layer %d has another geometry than layer 0", i);
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_photo_store_create(int32_t capacity, const char *dir, kda_photo_store **out)
{
    if (!out) return photo_fail(KDA_ERR_INVALID, "out is NULL");
    *out = nullptr;
    const bool has_dir = dir && dir[0];
    if (has_dir) {
        struct stat sb;
        if (stat(dir, &sb) != 0 || !S_ISDIR(sb.st_mode))
            return photo_fail(KDA_ERR_INVALID, "photo directory '%s' does not exist", dir);
    }
    kda_photo_store *ps = new (std::nothrow) kda_photo_store;
    if (!ps) return photo_fail(KDA_ERR_OOM, "photo store");
    // a directory alone implies 2 photos; a given capacity (0 included) always wins
    ps->capacity = capacity >= 0 ? capacity : (has_dir ? 2 : 0);
    if (has_dir) ps->dir = dir;
    *out = ps;
    return KDA_OK;
}

kda_status kda_photo_store_free(kda_photo_store *ps)
{
    if (!ps) return KDA_OK;
    {
        std::lock_guard<std::mutex> g(ps->mu);
        while (!ps->photos.empty()) ps->drop(ps->photos.size() - 1);
        if (ps->spare) cudaFreeHost(ps->spare);
        ps->spare = nullptr;
    }
    delete ps;
    return KDA_OK;
}

int32_t kda_photo_count(const kda_photo_store *ps)
{
    if (!ps) return 0;
    std::lock_guard<std::mutex> g(ps->mu);
    return (int32_t)ps->photos.size();
}

int32_t kda_photo_capacity(const kda_photo_store *ps) { return ps ? ps->capacity : 0; }

kda_status kda_photo_take(kda_photo_store *ps, kda_state *const *layers, int32_t n_layers, int32_t slot,
                          const int32_t *tokens, int64_t n_tokens, int32_t *photo_id, void *stream)
{
    if (photo_id) *photo_id = -1;
    if (!ps) return photo_fail(KDA_ERR_INVALID, "photo store is NULL");
    if (n_tokens < 0) return photo_fail(KDA_ERR_INVALID, "n_tokens must be >= 0");
    if (n_tokens > 0 && !tokens) return photo_fail(KDA_ERR_INVALID, "tokens is NULL");
    kda_status s = check_layers(layers, n_layers, slot);
    if (s != KDA_OK) return s;
    std::lock_guard<std::mutex> g(ps->mu);
    if (ps->capacity == 0) return KDA_OK;  // the store is off

    Photo p;
    p.layer_bytes.resize((size_t)n_layers);
    for (int32_t i = 0; i < n_layers; ++i) p.layer_bytes[(size_t)i] = kda_state_blob_bytes(layers[i], 1);
    const size_t bytes = total_of(p.layer_bytes);
    if ((s = ps->reserve_spare(bytes)) != KDA_OK) return s;

    // 1. the blobs into the spare buffer, complete before anything in the store changes
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *dst = static_cast<char *>(ps->spare);
    size_t off = 0;
    for (int32_t i = 0; i < n_layers; ++i) {
        if ((s = kda_state_snapshot(layers[i], &slot, 1, dst + off, 0, stream)) != KDA_OK) {
            cudaStreamSynchronize(st);
            return s;
        }
        off += p.layer_bytes[(size_t)i];
    }
    const cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return photo_fail(KDA_ERR_CUDA, "kda_photo_take: %s", cudaGetErrorString(e));

    // 2. park it: the spare becomes the photo's buffer, or it is written to a new file
    p.id = ps->next_id;
    if (ps->file_mode()) {
        char name[96];
        snprintf(name, sizeof(name), "/kda_photo_%ld_%p_%d.bin", (long)getpid(), (void *)ps, p.id);
        p.path = ps->dir + name;
        if (!write_file(p.path, ps->spare, bytes)) {
            unlink(p.path.c_str());
            return photo_fail(KDA_ERR_IO, "cannot write photo file %s", p.path.c_str());
        }
    } else {
        p.host = ps->spare;
        p.host_bytes = ps->spare_bytes;
        ps->spare = nullptr;
        ps->spare_bytes = 0;
    }
    p.tokens.assign(tokens, tokens + n_tokens);
    p.stamp = ++ps->clock;
    ++ps->next_id;

    // 3. the photo of the same prefix, else the least recently used one when full, goes
    for (size_t i = 0; i < ps->photos.size(); ++i)
        if (ps->photos[i].tokens == p.tokens) {
            ps->drop(i);
            break;
        }
    if ((int32_t)ps->photos.size() >= ps->capacity) {
        size_t lru = 0;
        for (size_t i = 1; i < ps->photos.size(); ++i)
            if (ps->photos[i].stamp < ps->photos[lru].stamp) lru = i;
        ps->drop(lru);
    }
    ps->photos.push_back(std::move(p));
    if (photo_id) *photo_id = ps->photos.back().id;
    return KDA_OK;
}

kda_status kda_photo_find(const kda_photo_store *ps, const int32_t *tokens, int64_t n_tokens,
                          int32_t *photo_id, int64_t *prefix_len)
{
    if (!ps || !photo_id || !prefix_len) return photo_fail(KDA_ERR_INVALID, "NULL store or output");
    *photo_id = -1;
    *prefix_len = 0;
    if (n_tokens < 0) return photo_fail(KDA_ERR_INVALID, "n_tokens must be >= 0");
    if (n_tokens > 0 && !tokens) return photo_fail(KDA_ERR_INVALID, "tokens is NULL");
    std::lock_guard<std::mutex> g(ps->mu);
    for (const Photo &p : ps->photos) {
        const int64_t len = (int64_t)p.tokens.size();
        if (len > n_tokens) continue;
        if (len > 0 && memcmp(p.tokens.data(), tokens, (size_t)len * sizeof(int32_t)) != 0) continue;
        if (*photo_id < 0 || len > *prefix_len || (len == *prefix_len && p.id > *photo_id)) {
            *photo_id = p.id;
            *prefix_len = len;
        }
    }
    return KDA_OK;
}

kda_status kda_photo_restore(kda_photo_store *ps, int32_t photo_id, kda_state *const *layers, int32_t n_layers,
                             int32_t slot, void *stream)
{
    if (!ps) return photo_fail(KDA_ERR_INVALID, "photo store is NULL");
    kda_status s = check_layers(layers, n_layers, slot);
    if (s != KDA_OK) return s;
    std::lock_guard<std::mutex> g(ps->mu);
    Photo *p = ps->by_id(photo_id);
    if (!p) return photo_fail(KDA_ERR_INVALID, "photo %d is not in the store (never taken, or evicted)", photo_id);
    if ((size_t)n_layers != p->layer_bytes.size())
        return photo_fail(KDA_ERR_INVALID, "photo %d holds %zu layers, %d given", photo_id, p->layer_bytes.size(),
                          n_layers);
    for (int32_t i = 0; i < n_layers; ++i)  // before any copy: no partial restore
        if (kda_state_blob_bytes(layers[i], 1) != p->layer_bytes[(size_t)i])
            return photo_fail(KDA_ERR_BLOB, "layer %d does not have the photo's geometry", i);
    const size_t bytes = total_of(p->layer_bytes);
    const char *src = static_cast<const char *>(p->host);
    if (ps->file_mode()) {
        if ((s = ps->reserve_spare(bytes)) != KDA_OK) return s;
        if (!read_file(p->path, ps->spare, bytes))
            return photo_fail(KDA_ERR_IO, "cannot read photo file %s", p->path.c_str());
        src = static_cast<const char *>(ps->spare);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    size_t off = 0;
    for (int32_t i = 0; i < n_layers; ++i) {
        if ((s = kda_state_restore(layers[i], &slot, 1, src + off, 0, stream)) != KDA_OK) {
            cudaStreamSynchronize(st);
            return s;
        }
        off += p->layer_bytes[(size_t)i];
    }
    const cudaError_t e = cudaStreamSynchronize(st);  // the source buffer may be reused after this
    if (e != cudaSuccess) return photo_fail(KDA_ERR_CUDA, "kda_photo_restore: %s", cudaGetErrorString(e));
    p->stamp = ++ps->clock;
    return KDA_OK;
}

}  // extern "C"
