// kda_decode_multi.cu - n consecutive decode tokens per sequence in one pass over
// the state (verification of speculative drafts, or any short run of known tokens).
//
// Each (sequence, head) unit is the per-head recurrence of the kimi_k3.c header
// comment ("KDA per-head recurrence") applied n times in order. The unit's 64 KB
// FP32 state is read once, stays in registers across the n tokens and is written
// once, so n tokens cost one state round trip instead of n. Per token the
// arithmetic is the single-token decode's (conv + SiLU, L2 norms, gates, the
// delta-rule update in the expanded form S' = Diag(a) S + k u^T with
// u = beta (v - (Diag(a) S)^T k), the readout o = S'^T q and the gated RMSNorm);
// the conv history slides through the run in registers.
//
// One CTA per SM walks a contiguous range of units (head-major); the state (one bulk
// copy), the n input rows of each of q,k,v,z,g (one 2-D TMA box per stream: the rows of
// one sequence are consecutive) and the history (one box of its 9 rows) of the next unit
// arrive in a shared-memory stage while the current unit is computed. The per-token state step is the single-token decode's
// (kda_decode_common.cuh): warp w owns state rows 16w .. 16w+15, lane l columns 4l..4l+3.
#include "kda_decode_common.cuh"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

template <typename T>
struct MultiStage {
    static constexpr int kS = kD * kD * 4;                             // state
    static constexpr int kRow = kD * (int)sizeof(T);                   // one row of one head
    static constexpr int kIn = 5 * KDA_DECODE_MAX_TOKENS * kRow;       // [5][n][d] q,k,v,z,g
    static constexpr int kTail = 9 * kRow;                             // [3][3][d] history
    static constexpr int kBytes = kS + kIn + kTail;
};

constexpr uint32_t kMultiWaitLimit = 1u << 26;

// NST stage buffers per CTA. NST = 1 fits two CTAs (two units) on an SM, so that one unit's
// serial token chain overlaps the other's, and requests the next unit's copy as soon as the
// prologue has read the stage (the copy then lands under the token chain); NST = 2 keeps one
// CTA per SM and prefetches its next unit a whole unit ahead. n, the tokens per sequence, is a
// template parameter so that the prologue's token loop unrolls.
template <typename T, int NST, int n>
__global__ void __launch_bounds__(256, 3 - NST)
decode_multi_kernel(const float *__restrict__ conv_w, const float *__restrict__ dt_bias,
                    const float *__restrict__ A_log, const float *__restrict__ norm_w,
                    float *__restrict__ S_all, T *__restrict__ tail_all, int32_t *__restrict__ err,
                    const int32_t *__restrict__ slots, int B, int H, int max_slots,
                    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    const T *__restrict__ z, const T *__restrict__ bl, const T *__restrict__ g,
                    T *__restrict__ out, float gmin, float l2_eps, float rms_eps, float q_scale,
                    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_tail)
{
    using L = MultiStage<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int kNT = KDA_DECODE_MAX_TOKENS;
    float *sh_k = reinterpret_cast<float *>(smem + NST * L::kBytes);  // [token][d] k^ of every token
    float *sh_q = sh_k + kNT * kD, *sh_a = sh_q + kNT * kD, *sh_v = sh_a + kNT * kD, *sh_gw = sh_v + kNT * kD;
    // alpha k^ per row; alpha q^ per row is sh_q (q^ itself is not needed past the prologue)
    float *sh_ak = sh_gw + kNT * kD, *sh_aq = sh_q;
    float *su = sh_ak + kNT * kD, *so = su + kD;  // [d] u, o of the current token
    float *red = so + kD;                          // warp partials of p and r (kRedFloats)
    float *part = red + kRedFloats;                // [token][3][4] quarter sums of squares
    float *sbeta = part + kNT * 12;                                  // [token] beta
    float *skq = sbeta + kNT;                                        // [token] k^ . q^
    uint64_t *bar = reinterpret_cast<uint64_t *>(skq + kNT);         // [2]

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int n_units = B * H;
    const int per = (n_units + gridDim.x - 1) / gridDim.x;
    const int u_begin = blockIdx.x * per;
    const int u_end = min(n_units, u_begin + per);
    if (u_begin >= u_end) return;
    const size_t D = (size_t)H * kD;
    const CUtensorMap *tm5[5] = {&tm_q, &tm_k, &tm_v, &tm_z, &tm_g};

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&bar[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    auto issue = [&](int stage, int u) {  // thread 0 only
        const int h = u / B, r = u - (u / B) * B;
        const int slot = slots[r];
        unsigned char *st = smem + stage * L::kBytes;
        if (slot < 0 || slot >= max_slots) {
            mbar_arrive(&bar[stage]);  // completes the phase with no data
            return;
        }
        mbar_arrive_expect_tx(&bar[stage], (uint32_t)(L::kS + (5 * n + 9) * L::kRow));
        bulk_g2s_hint(st, S_all + ((size_t)slot * H + h) * kD * kD, L::kS, &bar[stage], pol);
        for (int x = 0; x < 5; ++x)  // rows r n .. r n + n - 1, channels of head h
            tma_load_2d(st + L::kS + x * KDA_DECODE_MAX_TOKENS * L::kRow, tm5[x], h * kD, r * n, &bar[stage]);
        tma_load_2d(st + L::kS + L::kIn, &tm_tail, h * kD, slot * 9, &bar[stage]);
    };

    if (tid == 0) issue(0, u_begin);
    bool timed_out = false;
    int it = 0;
    for (int u = u_begin; u < u_end; ++u, ++it) {
        const int stage = NST == 2 ? (it & 1) : 0;
        if (NST == 2 && tid == 0 && u + 1 < u_end) issue(stage ^ 1, u + 1);  // the other stage is free
        const int h = u / B, r = u - (u / B) * B;
        const int slot = slots[r];
        const bool bad = slot < 0 || slot >= max_slots;
        // per-unit scalars and parameters are loaded before the wait, so their latency hides
        // behind the copies (the beta logit of each token, and channel tid & 127's taps)
        T braw = T(0.f);
        if (tid < n) braw = bl[((size_t)r * n + tid) * H + h];
        const int pi = tid & (kD - 1);
        const size_t pc = (size_t)h * kD + pi;
        float4 wt[3];
#pragma unroll
        for (int x = 0; x < 3; ++x) wt[x] = __ldg(reinterpret_cast<const float4 *>(conv_w + ((size_t)x * D + pc) * kK));
        const float dti = __ldg(dt_bias + pc), nwi = __ldg(norm_w + pi);
        const float eA = expf(__ldg(A_log + h));
        const bool ok = mbar_wait_bounded(&bar[stage], (uint32_t)((NST == 2 ? it >> 1 : it) & 1), kMultiWaitLimit);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        if (bad) {
            if (tid == 0) atomicExch(err, kErrBadSlot);
            __syncthreads();
            if (NST == 1 && tid == 0 && u + 1 < u_end) issue(0, u + 1);
            continue;
        }
        const unsigned char *st = smem + stage * L::kBytes;
        const T *in = reinterpret_cast<const T *>(st + L::kS);          // [5][8][d]
        const T *tl = reinterpret_cast<const T *>(st + L::kS + L::kIn);  // [3][3][d]

        // the unit's state tile in registers for the whole run
        float4 s[16];
        const float4 *S4s = reinterpret_cast<const float4 *>(st);
#pragma unroll
        for (int m = 0; m < 16; ++m) s[m] = S4s[(16 * w + m) * 32 + l];

        // prologue of every token at once (it does not depend on the state): thread (channel
        // i, token parity tg) takes tokens tg, tg + 2, ...; the conv window of token t is raw
        // rows t-3 .. t, the first ones from the history
        {
            const int i = pi, tg = tid >> 7;
            if (tid < n) sbeta[tid] = sigmoid_ftz(IO<T>::ld(&braw));
            auto raw = [&](int x, int j) -> float {  // raw input of stream x at token j (j >= -3)
                return j >= 0 ? IO<T>::ld(in + (x * KDA_DECODE_MAX_TOKENS + j) * kD + i)
                              : IO<T>::ld(tl + (x * 3 + (j + 3)) * kD + i);
            };
            // the new history (the last three raw inputs) leaves now, so that the stage is free
            // once the prologue is done
            if (tid < kD) {
                T *tg_out = tail_all + (size_t)slot * 9 * D + (size_t)h * kD + tid;
#pragma unroll
                for (int x = 0; x < 3; ++x)
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        const int tok = n - 3 + j;
                        tg_out[(size_t)(x * 3 + j) * D] = tok >= 0 ? in[(x * KDA_DECODE_MAX_TOKENS + tok) * kD + tid]
                                                                   : tl[(x * 3 + (tok + 3)) * kD + tid];
                    }
            }
#pragma unroll
            for (int jt = 0; jt < (n + 1) / 2; ++jt) {
                const int t = tg + 2 * jt;
                if (t < n) {  // uniform per warp
                    float y[3];
#pragma unroll
                    for (int x = 0; x < 3; ++x)
                        y[x] = silu_ftz(fmaf(wt[x].x, raw(x, t - 3), fmaf(wt[x].y, raw(x, t - 2),
                                      fmaf(wt[x].z, raw(x, t - 1), wt[x].w * raw(x, t)))));
                    sh_q[t * kD + i] = y[0];
                    sh_k[t * kD + i] = y[1];
                    sh_v[t * kD + i] = y[2];
                    sh_a[t * kD + i] = exp_ftz(gmin * sigmoid_ftz(eA * (IO<T>::ld(in + (3 * KDA_DECODE_MAX_TOKENS + t) * kD + i) + dti)));
                    sh_gw[t * kD + i] = sigmoid_ftz(IO<T>::ld(in + (4 * KDA_DECODE_MAX_TOKENS + t) * kD + i)) * nwi;
                    const float a0 = warp_sum(y[0] * y[0]), a1 = warp_sum(y[1] * y[1]), a2 = warp_sum(y[0] * y[1]);
                    if (l == 0) { part[t * 12 + (w & 3)] = a0; part[t * 12 + 4 + (w & 3)] = a1; part[t * 12 + 8 + (w & 3)] = a2; }
                }
            }
            __syncthreads();
            if (tid < n) {  // k^ . q^ of token tid, from the quarter sums
                const float *pt = part + tid * 12;
                const float sqq = pt[0] + pt[1] + pt[2] + pt[3];
                const float skk = pt[4] + pt[5] + pt[6] + pt[7];
                const float sqk = pt[8] + pt[9] + pt[10] + pt[11];
                skq[tid] = sqk * (q_scale * rsqrt_ftz(sqq + l2_eps)) * (rsqrt_ftz(skk + l2_eps));
            }
#pragma unroll
            for (int jt = 0; jt < (n + 1) / 2; ++jt) {
                const int t = tg + 2 * jt;
                if (t < n) {
                    const float *pt = part + t * 12;
                    const float rq = q_scale * rsqrt_ftz((pt[0] + pt[1] + pt[2] + pt[3]) + l2_eps);
                    const float rk = rsqrt_ftz((pt[4] + pt[5] + pt[6] + pt[7]) + l2_eps);
                    const float kn = sh_k[t * kD + i] * rk, qn = sh_q[t * kD + i] * rq, a = sh_a[t * kD + i];
                    sh_k[t * kD + i] = kn;
                    sh_ak[t * kD + i] = a * kn;
                    sh_aq[t * kD + i] = a * qn;  // over q^ (sh_aq is sh_q): this thread's own element
                }
            }
            __syncthreads();
        }
        // the stage has been read (state, inputs and history): the next unit's copy may land in it
        if (NST == 1 && tid == 0 && u + 1 < u_end) issue(0, u + 1);

        if constexpr (n > 4) {
            // the tokens in order
#pragma unroll 1
            for (int t = 0; t < n; ++t) {
                const size_t row = (size_t)r * n + t;
                decode_token_step<T>(s, sh_ak + t * kD, sh_aq + t * kD, sh_a + t * kD, sh_k + t * kD, sh_v + t * kD,
                                     sh_gw + t * kD, sbeta[t], skq[t], red, su, so, out + row * D + (size_t)h * kD,
                                     rms_eps, w, l);
            }
            // the state after the run
            float4 *S4 = reinterpret_cast<float4 *>(S_all + ((size_t)slot * H + h) * kD * kD);
#pragma unroll
            for (int m = 0; m < 16; ++m) st_stream(S4 + (16 * w + m) * 32 + l, s[m]);
        } else {
            // (n <= 4) the last token's step is written out here, so that each updated state row is
            // stored as soon as it is final: the same operations in the same order as
            // decode_token_step, so the results stay those of n single-token calls. (Measured faster at
            // n = 4 and slower at n = 8, where the plain form is kept.)
#pragma unroll 1
            for (int t = 0; t < n - 1; ++t) {
                const size_t row = (size_t)r * n + t;
                decode_token_step<T>(s, sh_ak + t * kD, sh_aq + t * kD, sh_a + t * kD, sh_k + t * kD, sh_v + t * kD,
                                     sh_gw + t * kD, sbeta[t], skq[t], red, su, so, out + row * D + (size_t)h * kD,
                                     rms_eps, w, l);
            }
            float4 *S4 = reinterpret_cast<float4 *>(S_all + ((size_t)slot * H + h) * kD * kD);
            {
                const int t = n - 1;
                const float *a = sh_a + t * kD, *kk = sh_k + t * kD, *v = sh_v + t * kD;
                float4 p, rr;
                dc_partials(s, sh_ak + t * kD, sh_aq + t * kD, w, p, rr);
                reinterpret_cast<float4 *>(red)[w * 32 + l] = p;
                reinterpret_cast<float4 *>(red + kRedR)[w * 32 + l] = rr;
                __syncthreads();
                {
                    const int c = 16 * w + (l & 15), which = l >> 4;
                    const float *col = red + which * kRedR + c;
                    float acc = col[0];
#pragma unroll
                    for (int ww = 1; ww < 8; ++ww) acc += col[ww * kD];
                    const float r_c = __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
                    if (l < 16) {
                        const float u = dc_u(sbeta[t], v[c], acc);
                        su[c] = u;
                        so[c] = dc_o(skq[t], u, r_c);
                    }
                }
                __syncthreads();
                const float4 uu = reinterpret_cast<const float4 *>(su)[l];
                const float4 oo = reinterpret_cast<const float4 *>(so)[l];
                const float4 *a4 = reinterpret_cast<const float4 *>(a + 16 * w);
                const float4 *k4 = reinterpret_cast<const float4 *>(kk + 16 * w);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 av = a4[j], kv = k4[j];
                    const float aa[4] = {av.x, av.y, av.z, av.w}, kq[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float4 &sv = s[4 * j + e];
                        sv = make_float4(fmaf(aa[e], sv.x, kq[e] * uu.x), fmaf(aa[e], sv.y, kq[e] * uu.y),
                                         fmaf(aa[e], sv.z, kq[e] * uu.z), fmaf(aa[e], sv.w, kq[e] * uu.w));
                        st_stream(S4 + (16 * w + 4 * j + e) * 32 + l, sv);  // the state after the run
                    }
                }
                dc_norm_store(oo, sh_gw + t * kD, out + ((size_t)r * n + t) * D + (size_t)h * kD, rms_eps, w, l);
            }
        }
        __syncthreads();  // the prologue arrays and the partials are free (and, NST = 2, the stage)
    }
    if (timed_out) {
        if (tid == 0) {
            atomicExch(err, KDA_ERR_TIMEOUT);
            // copies that may still be in flight: the next unit's (NST = 2) or the one waited on
            if (NST == 2 && u_begin + it + 1 < u_end)
                mbar_wait_bounded(&bar[(it + 1) & 1], (uint32_t)(((it + 1) >> 1) & 1), kMultiWaitLimit);
            if (NST == 1) mbar_wait_bounded(&bar[0], (uint32_t)(it & 1), kMultiWaitLimit);  // the copy that timed out
        }
        __syncthreads();
    }
}

template <typename T, int NST, int n>
cudaError_t launch_multi_typed(const State &st, const kda_layer_params &p, const int32_t *slots, int B,
                               const void *q, const void *k, const void *v, const void *z, const void *b,
                               const void *g, void *out, cudaStream_t stream)
{
    using L = MultiStage<T>;
    const kda_config_t &c = st.cfg;
    const int H = c.num_heads;
    const size_t smem = NST * (size_t)L::kBytes + 6 * KDA_DECODE_MAX_TOKENS * kD * 4 + 2 * kD * 4 + kRedFloats * 4 +
                        KDA_DECODE_MAX_TOKENS * 14 * 4 + 2 * 8;
    cudaError_t e = raise_smem_once(st, smem_bit_multi(sizeof(T) == 4, n), decode_multi_kernel<T, NST, n>, smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = state_sms(st, &sms)) != cudaSuccess) return e;
    // one map per input stream ([B n][H d] rows, boxes of n rows x one head) and one for the
    // conv history ([slots 9][H d] rows, boxes of 9 rows x one head)
    const int64_t D = (int64_t)H * kD;
    CUtensorMap tm[6];
    const void *src[5] = {q, k, v, z, g};
    for (int x = 0; x < 5; ++x)
        if ((e = encode_rows_box(&tm[x], src[x], (int)sizeof(T), (int64_t)B * n, D, kD, n)) != cudaSuccess) return e;
    if ((e = encode_rows_box(&tm[5], st.tail, (int)sizeof(T), (int64_t)st.max_slots * 9, D, kD, 9)) != cudaSuccess)
        return e;
    const int n_units = B * H;
    const int ctas = (3 - NST) * sms;  // CTAs resident at once
    const int grid = n_units < ctas ? n_units : ctas;
    decode_multi_kernel<T, NST, n><<<grid, 256, smem, stream>>>(
        p.conv_w, p.dt_bias, p.A_log, p.norm_w, st.S, (T *)st.tail, st.err, slots, B, H, st.max_slots,
        (const T *)q, (const T *)k, (const T *)v, (const T *)z, (const T *)b, (const T *)g, (T *)out,
        c.gate_lower_bound, c.l2_eps, c.rms_eps, c.q_scale, tm[0], tm[1], tm[2], tm[3], tm[4], tm[5]);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multi(const State &st, const kda_layer_params &p, const int32_t *slots, int B, int n,
                                const void *q, const void *k, const void *v, const void *z, const void *b,
                                const void *g, void *out, cudaStream_t stream)
{
#define KDA_MULTI_CASE(N)                                                                                   \
    case N:                                                                                                 \
        return st.cfg.io_dtype == KDA_BF16                                                                  \
                   ? launch_multi_typed<__nv_bfloat16, 1, N>(st, p, slots, B, q, k, v, z, b, g, out, stream) \
                   : launch_multi_typed<float, 2, N>(st, p, slots, B, q, k, v, z, b, g, out, stream);
    switch (n) {
        KDA_MULTI_CASE(1)
        KDA_MULTI_CASE(2)
        KDA_MULTI_CASE(3)
        KDA_MULTI_CASE(4)
        KDA_MULTI_CASE(5)
        KDA_MULTI_CASE(6)
        KDA_MULTI_CASE(7)
        KDA_MULTI_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef KDA_MULTI_CASE
}

}  // namespace kda
