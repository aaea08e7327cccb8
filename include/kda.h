/*
 * kda.h - C ABI of the KDA (Kimi Delta Attention) mixer core on GB300 (sm_103a).
 *
 * The library computes, for every token of every sequence and every head,
 * the KDA per-head recurrence stated in the kimi_k3.c header comment, block
 * "KDA per-head recurrence":
 *
 *   q,k,v = SiLU(ShortConv4(x))              depthwise, causal, taps oldest first
 *   q,k   = L2-normalised (eps 1e-6 inside the sqrt), q *= d^-1/2
 *   gk    = gmin * sigmoid(exp(A_log[h]) * (z + dt_bias)),  gmin = -5,  alpha = exp(gk)
 *   beta  = sigmoid(b)                        one scalar per head and token
 *   S     = (I - beta k k^T) Diag(alpha) S + beta k v^T      S[key][value], FP32
 *   o     = S^T q                             read after the update
 *   out   = sigmoid(g) * RMSNorm_head(o)      RMSNorm weight [d], shared by all heads
 *
 * The W_q/W_k/W_v/W_o/W_g projections stay outside: callers pass the
 * post-projection q, k, v, the gate pre-activation z (without dt_bias), the
 * beta logits b and the output-gate logits g. z and b can come from
 * kda_gate_proj below (the decay-gate and beta projections of the hidden state).
 *
 * Conventions for every entry point:
 *  - Status codes are returned; no call exits the process or traps on the GPU.
 *    The text of the last error of the calling thread is kda_last_error().
 *  - Argument checks happen on the host before anything is enqueued; a call
 *    that returns an error has enqueued nothing.
 *  - "stream" is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Work is enqueued on it and the call returns without waiting,
 *    except where a function says it synchronises.
 *  - The calling thread's current CUDA device must be the one the state was
 *    allocated on.
 *  - All tensors are dense, row-major, with the layouts given below. The caller
 *    owns every input, output and parameter buffer; the library owns the state.
 *  - The row tensors q, k, v, z, g and out must be 16-byte aligned (calls that
 *    get one that is not return KDA_ERR_INVALID); b needs only its element
 *    alignment. Other device pointers must be 16-byte aligned.
 *  - Calls that use the same kda_state must be ordered (same stream, or
 *    synchronised by the caller); the library keeps per-state workspace.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID = 1,  /* bad argument, shape or config: nothing was enqueued */
    KDA_ERR_OOM = 2,      /* a device or host allocation failed */
    KDA_ERR_CUDA = 3,     /* a CUDA runtime call failed (message holds cudaGetErrorString) */
    KDA_ERR_BLOB = 4,     /* a snapshot blob has the wrong magic, version, geometry or size */
    KDA_ERR_TIMEOUT = 5,  /* a bounded device-side wait gave up */
    KDA_ERR_DEVICE = 6,   /* a kernel recorded a bad index (see kda_state_poll_error) */
    KDA_ERR_IO = 7        /* a photo file could not be written or read back */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/*
 * Mixer geometry and constants (kimi_k3.c: config parsing of
 * "linear_attn_config" - num_heads, head_dim, short_conv_kernel_size,
 * gate_lower_bound; the header comment gives eps 1e-6 and the d^-1/2 q scale).
 * The RMSNorm eps is a field (default 1e-6).
 */
typedef struct {
    int32_t num_heads;       /* H >= 1 */
    int32_t head_dim;        /* d; this build supports 128 */
    int32_t conv_kernel;     /* K; this build supports 4 */
    int32_t io_dtype;        /* kda_dtype of q,k,v,z,b,g, out and the conv history */
    int32_t chunk_size;      /* prefill chunk length C; this build supports 64 */
    float gate_lower_bound;  /* gmin, default -5 */
    float l2_eps;            /* default 1e-6 */
    float rms_eps;           /* default 1e-6 */
    float q_scale;           /* default d^-1/2 */
} kda_config_t;

/*
 * Fill *cfg with the defaults above for the given geometry.
 * Returns KDA_ERR_INVALID (cfg untouched) for cfg == NULL, num_heads < 1,
 * head_dim != 128 or an io_dtype that is not KDA_F32/KDA_BF16.
 */
kda_status kda_config(kda_config_t *cfg, int32_t num_heads, int32_t head_dim, int32_t io_dtype);

/*
 * Per-layer parameters, device pointers, FP32, caller-owned (kimi_k3.c,
 * struct Kda: conv_q/conv_k/conv_v "[proj*4] depthwise taps, oldest first",
 * dt "dt_bias[proj]", A from A_log "[heads]", onw "o_norm[hd]").
 *   conv_w  [3][H*d][K]   taps for q, k, v in that order; tap 0 meets the oldest input
 *   dt_bias [H*d]
 *   A_log   [H]           the library takes exp(A_log) itself
 *   norm_w  [d]           RMSNorm weight shared by all heads
 */
typedef struct {
    const float *conv_w;
    const float *dt_bias;
    const float *A_log;
    const float *norm_w;
} kda_layer_params;

/* Opaque recurrent state for max_slots sequences. */
typedef struct kda_state kda_state;

/*
 * Allocate device state for max_slots sequences and zero it (synchronously)
 * (spark_model/kimi_k3/bound.rs, TransformerLayer::alloc_state ->
 * KdaState::new; kimi_k3.c, struct Model: kstate "[heads*hd*hd], S[k][v]" and
 * the conv windows cwq/cwk/cwv).
 * Per slot the library holds S [H][d][d] FP32 (row = key index) and the conv
 * history [3][K-1][H*d] in io_dtype: the last K-1 raw q, k, v inputs, oldest
 * first. The config is copied. *out receives the handle.
 * Errors: KDA_ERR_INVALID (NULL args, max_slots < 1, unsupported config),
 * KDA_ERR_OOM (cudaMalloc failed; nothing leaks), KDA_ERR_CUDA.
 */
kda_status kda_state_alloc(const kda_config_t *cfg, int32_t max_slots, kda_state **out);

/* Free the state and its workspace (spark_model/kimi_k3/bound.rs,
 * TransformerLayer::release_state). Synchronises the device first. NULL is a no-op. */
kda_status kda_state_free(kda_state *st);

/*
 * Zero S and the conv history of the n listed slots (host array of slot ids).
 * Errors: KDA_ERR_INVALID for a NULL state, n < 0, slots == NULL with n > 0,
 * or an id outside [0, max_slots).
 */
kda_status kda_state_reset(kda_state *st, const int32_t *slots, int32_t n, void *stream);

/* Geometry accessors. kda_state_blob_bytes returns 0 for a NULL state or n_slots < 0. */
int32_t kda_state_max_slots(const kda_state *st);
size_t kda_state_blob_bytes(const kda_state *st, int32_t n_slots);

/*
 * Snapshot / restore of the state of n slots (spark_model/kimi_k3/bound.rs,
 * TransformerLayer::snapshot_aux -> a byte blob, restore_aux(blob); the
 * "decode_rollback_unsupported" comment: a prefix snapshot and an explicit
 * restore are the only way back).
 * Blob = kda_blob_header (64 bytes) followed, for each listed slot in order,
 * by S [H][d][d] FP32 then the conv history [3][K-1][H*d] in io_dtype.
 * dst/src is host memory when *_on_device == 0, else device memory; its size
 * must be at least kda_state_blob_bytes(st, n). Copies are stream-ordered; a
 * host destination is complete once the stream is synchronised.
 * Restore checks magic, version, H, d, K, io_dtype and the slot count before
 * enqueuing any copy: a mismatch returns KDA_ERR_BLOB (for a device src the
 * header is read back synchronously).
 */
typedef struct {
    uint32_t magic;      /* KDA_BLOB_MAGIC */
    uint32_t version;    /* KDA_BLOB_VERSION */
    int32_t num_heads, head_dim, conv_kernel, io_dtype;
    int32_t n_slots;
    int32_t reserved0;
    uint64_t state_bytes_per_slot;
    uint64_t tail_bytes_per_slot;
    uint8_t reserved[16];
} kda_blob_header;
#define KDA_BLOB_MAGIC 0x3141444Bu  /* "KDA1" little-endian */
#define KDA_BLOB_VERSION 1u

kda_status kda_state_snapshot(const kda_state *st, const int32_t *slots, int32_t n,
                              void *dst, int32_t dst_on_device, void *stream);
kda_status kda_state_restore(kda_state *st, const int32_t *slots, int32_t n,
                             const void *src, int32_t src_on_device, void *stream);

/*
 * One decode token for a batch of B independent sequences (kimi_k3.c header,
 * "KDA per-head recurrence"; kimi_k3.c K3Seq/K3Row comment: a multiplexed
 * decode step reads each row's state from its own slot).
 *   slots   device int32 [B]: row r advances slot slots[r]; ids must be
 *           distinct within a call (duplicates race). An id outside
 *           [0, max_slots) skips that row and records KDA_ERR_DEVICE in the
 *           state's error word (read it with kda_state_poll_error).
 *   q,k,v,z,g  device [B][H*d] io_dtype;  b device [B][H] io_dtype
 *   out     device [B][H*d] io_dtype (must not alias an input)
 * B == 0 is a no-op. Errors: KDA_ERR_INVALID (NULL pointer, B < 0, config
 * different from the state's), KDA_ERR_CUDA (launch failure).
 */
kda_status kda_decode_token(const kda_config_t *cfg, const kda_layer_params *params, kda_state *st,
                            const int32_t *slots, int32_t B,
                            const void *q, const void *k, const void *v, const void *z,
                            const void *b, const void *g, void *out, void *stream);

/*
 * n consecutive decode tokens for each of B independent sequences in one call:
 * the per-head recurrence above applied n times in token order (kimi_k3.c
 * header, "KDA per-head recurrence"), identical in result to n calls of
 * kda_decode_token, but each sequence's state is read and written once. For
 * verifying n speculative draft tokens (kimi_k3.c K3Seq/K3Row multiplexed decode;
 * the state can only be taken back by restore, so take a kda_state_snapshot of
 * the rows first and, on a rejected draft, restore it and call again with the
 * accepted prefix).
 *   n        1 .. KDA_DECODE_MAX_TOKENS
 *   slots    device int32 [B], distinct; bad ids as in kda_decode_token
 *   q,k,v,z,g  device [B][n][H*d] io_dtype (token t of row r at r*n + t)
 *   b        device [B][n][H] io_dtype
 *   out      device [B][n][H*d] io_dtype (must not alias an input)
 * B == 0 is a no-op. Errors: KDA_ERR_INVALID (NULL pointer, B < 0, n out of
 * range, a row tensor not 16-byte aligned, config mismatch), KDA_ERR_CUDA.
 */
#define KDA_DECODE_MAX_TOKENS 8
kda_status kda_decode_tokens(const kda_config_t *cfg, const kda_layer_params *params, kda_state *st,
                             const int32_t *slots, int32_t B, int32_t n,
                             const void *q, const void *k, const void *v, const void *z,
                             const void *b, const void *g, void *out, void *stream);

/*
 * Prefill N variable-length sequences packed along the token axis
 * (kimi_k3.c ENV list, the K3_CHUNK entry; the per-token recurrence above
 * evaluated in chunks of C tokens with the WY/UT rewrite, which is exact in
 * real arithmetic). Each sequence continues from its slot's current state and
 * conv history and leaves its final state and history in the slot; nothing
 * crosses a sequence boundary.
 *   slots          device int32 [N], distinct (duplicates race); a bad id is
 *                  skipped and recorded as in kda_decode_token
 *   cu_seqlens     device int32 [N+1]; cu_seqlens_host: the same values on the host.
 *                  cu[0] = 0, non-decreasing; sequence i is tokens [cu[i], cu[i+1]).
 *                  Empty sequences are allowed and leave their slot unchanged.
 *   q,k,v,z,g      device [cu[N]][H*d] io_dtype;  b device [cu[N]][H] io_dtype
 *   out            device [cu[N]][H*d] io_dtype
 * The library grows a per-state device workspace as needed (cudaMalloc; this
 * call may then synchronise). Errors: KDA_ERR_INVALID (NULL pointer, N < 0,
 * bad cu_seqlens_host, config mismatch), KDA_ERR_OOM (workspace), KDA_ERR_CUDA.
 */
kda_status kda_prefill(const kda_config_t *cfg, const kda_layer_params *params, kda_state *st,
                       const int32_t *slots, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                       int32_t N,
                       const void *q, const void *k, const void *v, const void *z,
                       const void *b, const void *g, void *out, void *stream);

/*
 * kda_prefill_noalloc: the computation of kda_prefill for callers that must not
 * allocate device memory. The pages have no counterpart to this entry point; it
 * exists for callers such as serving runtimes that hand out every byte of device
 * memory from their own arena (exact accounting, no allocation failure halfway
 * through a request) or latency-critical loops that cannot accept the implicit
 * device-wide synchronisation of cudaMalloc/cudaFree. It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   S      device FP32 [max_slots][H][d][d], caller-owned (layout of a kda_state's S)
 *   tail   device io_dtype [max_slots][3][K-1][H*d], caller-owned conv history
 *   err    device int32 word that receives KDA_ERR_DEVICE for a bad slot id or a
 *          cu_seqlens that disagrees with cu_seqlens_host, or KDA_ERR_TIMEOUT if
 *          a bounded device-side wait gave up; never cleared by the library.
 *          NULL: a word inside the static workspace is used (and cleared at the
 *          start of each call), and such errors are not reported.
 *   slots .. out, stream: as for kda_prefill.
 * Its scratch is a file-scope __device__ array of KDA_NOALLOC_WORKSPACE_BYTES
 * (128 MiB; every GPU that loads the library holds it until the process exits).
 * A call whose workspace need exceeds it returns KDA_ERR_INVALID before
 * enqueuing anything; split such a call. The need is about 131.6 KB per (chunk
 * of 64 tokens, head) with BF16 I/O (at most 640 tokens, 10 chunks, of one
 * sequence at 96 heads), and 148 KB per (chunk, head) plus 512 B per (token,
 * head) with FP32 I/O. Every call looks up the array's device address in the
 * current context (cudaGetSymbolAddress, which allocates nothing), so the
 * address stays valid after cudaDeviceReset and in any context; the first
 * call in a context may load the library's module there, so make it before
 * any stream capture. All calls on a device share the array and it keeps the
 * previous call's contents: calls whose work overlaps on the GPU race, so
 * order them (one stream, or events).
 */
#define KDA_NOALLOC_WORKSPACE_BYTES ((size_t)128 << 20)
kda_status kda_prefill_noalloc(const kda_config_t *cfg, const kda_layer_params *params, float *S, void *tail,
                               int32_t max_slots, int32_t *err, const int32_t *slots, const int32_t *cu_seqlens,
                               const int32_t *cu_seqlens_host, int32_t N,
                               const void *q, const void *k, const void *v, const void *z,
                               const void *b, const void *g, void *out, void *stream);

/*
 * The decay-gate and beta input projections of a KDA layer (kimi_k3.c header
 * comment, block "KDA per-head recurrence": the gate pre-activation is the
 * low-rank product W_fb (W_fa x) and the beta logit is W_b x; struct Kda:
 * fa [hd][hidden], fb [proj][hd], bp [heads][hidden]). Per token:
 *   f = W_fa x  (d values),  z = W_fb f  (H*d values),  b = W_b x  (H values)
 * z and b are what kda_prefill / kda_decode_token take (dt_bias and the
 * sigmoids are applied there).
 *   hidden     width of x; a positive multiple of 64 (7168 for Kimi K3)
 *   T          tokens (rows of x); 0 is a no-op
 *   x          device io_dtype [T][hidden]
 *   w_fa       device io_dtype [d][hidden]
 *   w_fb       device io_dtype [H*d][d]
 *   w_b        device io_dtype [H][hidden]
 *   z          device io_dtype [T][H*d]     out
 *   b          device io_dtype [T][H]       out (aligned to its element size)
 *   workspace  device scratch of at least kda_gate_proj_workspace_bytes(cfg,
 *              hidden, T) bytes, 16-byte aligned, owned by the caller. Its
 *              first int32 is an error word: the call clears it and a kernel
 *              writes KDA_ERR_TIMEOUT there if a bounded wait gave up (read it
 *              after synchronising if needed). Calls that share a workspace
 *              must be ordered.
 * With BF16 I/O the products run on the tensor cores and accumulate in FP32; f
 * is rounded to BF16 once before the second product, and z, b are rounded to
 * BF16 (nearest even). With FP32 I/O they run on CUDA cores in FP32 throughout
 * (the correctness path). Needs num_heads <= 128. Errors:
 * KDA_ERR_INVALID (bad shape, dtype, alignment, NULL pointer, workspace too
 * small), KDA_ERR_CUDA. The workspace need is 256 bytes plus T * (d + 16
 * ceil(H / 16)) FP32 values (the sums W_fa x and W_b x); the query returns 0
 * for invalid arguments and does not touch the device.
 */
size_t kda_gate_proj_workspace_bytes(const kda_config_t *cfg, int32_t hidden, int64_t T);
kda_status kda_gate_proj(const kda_config_t *cfg, int32_t hidden, int64_t T, const void *x, const void *w_fa,
                         const void *w_fb, const void *w_b, void *z, void *b, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * The gate/beta input projections folded into the prefill (kimi_k3.c header comment, block
 * "KDA per-head recurrence": z = W_fb (W_fa x), beta = sigmoid(W_b x); struct Kda: fa
 * [hd][hidden], fb [proj][hd], bp [heads][hidden]). z, H*d values per token, is never
 * written to memory: kda_gate_proj_in produces the first product f = W_fa x (d values per
 * token) and b = W_b x, and kda_prefill_gate_fused forms z = W_fb f inside the prefill, on
 * the tensor cores, in FP32 (f is rounded to BF16 once, as in kda_gate_proj).
 * kda_gate_proj_in:
 *   hidden, T, x, w_fa, w_b, workspace: as for kda_gate_proj (the same workspace size)
 *   f     device BF16 [T][d]    out
 *   b     device BF16 [T][H]    out (aligned to its element size)
 * kda_prefill_gate_fused: kda_prefill with z replaced by
 *   f     device BF16 [total_T][d], 16-byte aligned: f = W_fa x of every token
 *   w_fb  device BF16 [H*d][d], 16-byte aligned
 * Both need BF16 I/O (KDA_ERR_INVALID otherwise). Errors as for kda_gate_proj / kda_prefill.
 */
kda_status kda_gate_proj_in(const kda_config_t *cfg, int32_t hidden, int64_t T, const void *x, const void *w_fa,
                            const void *w_b, void *f, void *b, void *workspace, size_t workspace_bytes, void *stream);
kda_status kda_prefill_gate_fused(const kda_config_t *cfg, const kda_layer_params *params, kda_state *state,
                                  const int32_t *slots, const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                  int32_t N, const void *q, const void *k, const void *v, const void *f,
                                  const void *w_fb, const void *b, const void *g, void *out, void *stream);

/*
 * The dense projections around the mixer: y = x W^T (+ r) in BF16 with FP32
 * accumulation on the tensor cores. A KDA layer takes q, k, v and the output-gate
 * logits g from W_q, W_k, W_v, W_g applied to the hidden state x, and applies W_o to
 * the mixer's gated output (kimi_k3.c header comment, block "KDA per-head
 * recurrence": q,k,v = SiLU(ShortConv4(W{q,k,v} x)), out = W_o [sigmoid(W_g x) *
 * RMSNorm_head(o)]; struct Kda: W q, k, v, o, g). They carry no KDA arithmetic; the
 * library provides them so that a whole layer runs on its own kernels.
 *   M, N, K    rows of x and y, rows of W (output columns), columns of x and W;
 *              N a multiple of 128, K a multiple of 64, M >= 0 (0 is a no-op)
 *   x          device BF16 [M][K]
 *   w          device BF16 [N][K]
 *   r          device BF16 [M][N] added to the product before rounding, or NULL;
 *              only with ysplit == 0 or ysplit == N
 *   y          device BF16, out. ysplit == 0 (or N): [M][N]. Otherwise the columns
 *              are split into N / ysplit consecutive matrices [M][ysplit] (column
 *              n goes to matrix n / ysplit), e.g. q, k, v and g from one product
 *              with the four weight matrices stacked; ysplit a multiple of 128
 *              that divides N
 *   workspace  device scratch of at least kda_linear_workspace_bytes(M, N, K)
 *              bytes (query with the call's device current), 16-byte aligned; its
 *              first int32 is an error word the call clears and a kernel sets to
 *              KDA_ERR_TIMEOUT if a bounded wait gave up. Calls sharing a
 *              workspace must be ordered.
 * All pointers 16-byte aligned. When the tile grid is too small to fill the GPU the
 * K dimension is split; the partial sums are added in split order, so results do
 * not depend on timing. Errors: KDA_ERR_INVALID (shape, alignment, NULL pointer,
 * workspace too small), KDA_ERR_CUDA.
 */
size_t kda_linear_workspace_bytes(int32_t M, int32_t N, int32_t K);
kda_status kda_linear(int32_t M, int32_t N, int32_t K, const void *x, const void *w, const void *r, void *y,
                      int32_t ysplit, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Recurrent-state photos (kimi_k3.c header, the COLI_K3_CKPT and
 * COLI_K3_CKPT_DIR serve options). A store keeps up to `capacity` photos of
 * one sequence slot across a stack of KDA layers (one kda_state per layer),
 * each taken after a token prefix, normally at a turn boundary. When a later
 * prompt diverges from an earlier one (an edit), kda_photo_find names the
 * deepest photo whose prefix is still a prefix of the new prompt: restoring it
 * and prefilling only the tokens after it replaces a prefill from token 0.
 *   capacity  photos kept. 0 turns the store off (kda_photo_take stores
 *             nothing). A negative value means "not given": 2 when dir is
 *             set, else 0. A given value always wins.
 *   dir       NULL keeps photos in pinned host memory. Otherwise each photo is
 *             parked in a file under dir (an existing directory). Files are
 *             removed when their photo is evicted and when the store is freed,
 *             so no photo outlives its store.
 * A photo holds, per layer, the kda_state_snapshot blob of the slot, and a
 * copy of the prefix's token ids, which kda_photo_find compares exactly.
 * All calls on one store are serialised by a lock inside it.
 */
typedef struct kda_photo_store kda_photo_store;

/* Errors: KDA_ERR_INVALID (out == NULL, dir not a directory), KDA_ERR_OOM. */
kda_status kda_photo_store_create(int32_t capacity, const char *dir, kda_photo_store **out);

/* Free the store, its host memory and its files. NULL is a no-op. */
kda_status kda_photo_store_free(kda_photo_store *ps);

/* Photos held now, and the capacity the store resolved (0 for NULL). */
int32_t kda_photo_count(const kda_photo_store *ps);
int32_t kda_photo_capacity(const kda_photo_store *ps);

/*
 * Photo of slot `slot` of each of the n_layers states layers[0..n_layers) (all
 * of one geometry) after the prefix tokens[0..n_tokens) (host int32 ids). The
 * states must hold that prefix's result. The copies are enqueued on `stream`
 * and the call synchronises it before returning, so the photo is complete and
 * the states may move on. A photo of the same prefix is replaced. When the
 * store is full, the least recently used photo (by take or restore) is
 * evicted. A store of capacity 0 returns KDA_OK and *photo_id = -1.
 *   photo_id  optional out: the new photo's id (ids are never reused).
 * Errors: KDA_ERR_INVALID (NULL store or layers, tokens == NULL with
 * n_tokens > 0, n_layers < 1, n_tokens < 0, slot out of range for a layer,
 * layers of different geometry), KDA_ERR_OOM, KDA_ERR_CUDA, KDA_ERR_IO. On an
 * error the store keeps the photos it had.
 */
kda_status kda_photo_take(kda_photo_store *ps, kda_state *const *layers, int32_t n_layers, int32_t slot,
                          const int32_t *tokens, int64_t n_tokens, int32_t *photo_id, void *stream);

/*
 * The deepest photo whose prefix equals tokens[0..len) for some len <=
 * n_tokens (the most recently taken one on a tie): *photo_id and *prefix_len,
 * or -1 and 0 when there is none. Host only; nothing is copied.
 * Errors: KDA_ERR_INVALID (NULL store or outputs, tokens == NULL with
 * n_tokens > 0, n_tokens < 0).
 */
kda_status kda_photo_find(const kda_photo_store *ps, const int32_t *tokens, int64_t n_tokens,
                          int32_t *photo_id, int64_t *prefix_len);

/*
 * Put photo photo_id back into slot `slot` of the n_layers states, which must
 * match the photo's layer count and each layer's geometry. The copies are
 * enqueued on `stream` and the call synchronises it before returning.
 * Errors: KDA_ERR_INVALID (unknown or evicted id, NULL arguments, a layer
 * count other than the photo's, slot out of range), KDA_ERR_BLOB (a layer of
 * another geometry), KDA_ERR_IO, KDA_ERR_CUDA.
 */
kda_status kda_photo_restore(kda_photo_store *ps, int32_t photo_id, kda_state *const *layers, int32_t n_layers,
                             int32_t slot, void *stream);

/*
 * Synchronise the device, read and clear the state's device error word.
 * *code receives 0 or a kda_status recorded by a kernel (KDA_ERR_DEVICE for a
 * bad slot id). Returns KDA_OK unless the read itself failed.
 */
kda_status kda_state_poll_error(kda_state *st, int32_t *code);

/* Message of the last failed call on this thread ("" if none). Never NULL. */
const char *kda_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H */
