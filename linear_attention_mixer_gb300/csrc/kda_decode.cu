// kda_decode.cu - fused one-token KDA decode for a batch of sequences.
//
// Every step of the per-head recurrence (kimi_k3.c header comment, "KDA per-head
// recurrence") is fused around one read and one write of the unit's 64 KB FP32
// state: ShortConv4 + SiLU on q,k,v (history shifted in place), L2 norms with the
// q scale, the decay gate alpha and beta, the delta-rule update with its readout,
// and the gated per-head RMSNorm.
//
// The update is evaluated in the form
//   S^ = Diag(alpha) S,  p = S^T k,  r = S^T q   (column reductions of S^)
//   u  = beta (v - p),   S' = S^ + k u^T,   o = S'^T q = r + u (k . q)
// which is (I - beta k k^T) Diag(alpha) S + beta k v^T expanded, so the state
// stays in registers between the reductions and the write-back.
//
// Thread layout (256 threads, 8 warps): warp w owns state rows 16w .. 16w+15
// and lane l owns columns 4l..4l+3 of each of them, so every warp load/store
// instruction moves one full 512-byte row. The per-token step (column
// reductions, update, RMSNorm) is shared with the multi-token decode
// (kda_decode_common.cuh).
#include "kda_decode_common.cuh"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

// ---------------------------------------------------------------------------
// One CTA per SM walks a contiguous range of units in
// head-major order (unit = h * B + r, so the per-head conv taps and dt_bias
// change rarely and stay in shared memory). Each unit's 64 KB state, its
// q,k,v,z,g rows and its conv history arrive by bulk async copies into a ring
// of NS shared-memory stages; the copies for the next NS-1 units are always in
// flight while the current unit is computed, so the state stream never pauses.
// The state is written back from registers with streaming stores.
template <typename T>
struct StageLayout {
    static constexpr int kS = kD * kD * 4;            // state bytes
    static constexpr int kIn = 5 * kD * (int)sizeof(T);   // q,k,v,z,g rows
    static constexpr int kTail = 9 * kD * (int)sizeof(T); // conv history [3][3][d]
    static constexpr int kBytes = kS + kIn + kTail;
};

constexpr uint32_t kWaitLimit = 1u << 26;  // bounded spin on an mbarrier phase

template <typename T, int NS>
__global__ void __launch_bounds__(256, 1)
decode_persistent_kernel(const float *__restrict__ conv_w, const float *__restrict__ dt_bias,
                         const float *__restrict__ A_log, const float *__restrict__ norm_w,
                         float *__restrict__ S_all, T *__restrict__ tail_all, int32_t *__restrict__ err,
                         const int32_t *__restrict__ slots, int B, int H, int max_slots,
                         const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                         const T *__restrict__ z, const T *__restrict__ bl, const T *__restrict__ g,
                         T *__restrict__ out, float gmin, float l2_eps, float rms_eps, float q_scale)
{
    using L = StageLayout<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    float4 *cw = reinterpret_cast<float4 *>(smem + NS * L::kBytes);   // [3][d] conv taps of the current head
    float *sdt = reinterpret_cast<float *>(cw + 3 * kD);               // [d]
    float *snw = sdt + kD;                                             // [d]
    float *sh_k = snw + kD, *sh_a = sh_k + kD, *sh_v = sh_a + kD, *sh_gw = sh_v + kD;
    float *sh_ak = sh_gw + kD, *sh_aq = sh_ak + kD, *su = sh_aq + kD, *so = su + kD;  // [d] each
    float *red = so + kD;                                              // warp partials of p and r (kRedFloats)
    float *part = red + kRedFloats;                                    // [3][4]
    uint64_t *bar = reinterpret_cast<uint64_t *>(part + 16);           // [NS]

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int n_units = B * H;
    const int per = (n_units + gridDim.x - 1) / gridDim.x;
    const int u_begin = blockIdx.x * per;
    const int u_end = min(n_units, u_begin + per);
    if (u_begin >= u_end) return;
    const size_t D = (size_t)H * kD;
    const T *src5[5] = {q, k, v, z, g};

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    if (tid < kD) snw[tid] = __ldg(norm_w + tid);
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
        mbar_arrive_expect_tx(&bar[stage], L::kBytes);
        bulk_g2s_hint(st, S_all + ((size_t)slot * H + h) * kD * kD, L::kS, &bar[stage], pol);
#pragma unroll
        for (int x = 0; x < 5; ++x)
            bulk_g2s(st + L::kS + x * kD * sizeof(T), src5[x] + (size_t)r * D + (size_t)h * kD, kD * sizeof(T),
                     &bar[stage]);
#pragma unroll
        for (int e = 0; e < 9; ++e)
            bulk_g2s(st + L::kS + L::kIn + e * kD * sizeof(T), tail_all + ((size_t)slot * 9 + e) * D + (size_t)h * kD,
                     kD * sizeof(T), &bar[stage]);
    };

    if (tid == 0)
        for (int s = 0; s < NS - 1; ++s)
            if (u_begin + s < u_end) issue(s, u_begin + s);

    int cur_h = -1;
    float eA = 0.f;
    bool timed_out = false;
    int it = 0;
    for (int u = u_begin; u < u_end; ++u, ++it) {
        const int stage = it % NS;
        const uint32_t parity = (uint32_t)((it / NS) & 1);
        if (tid == 0 && u + NS - 1 < u_end) issue((it + NS - 1) % NS, u + NS - 1);
        const int h = u / B, r = u - (u / B) * B;
        const int slot = slots[r];
        const bool bad = slot < 0 || slot >= max_slots;
        const float beta = sigmoid_ftz(IO<T>::ld(bl + (size_t)r * H + h));
        if (h != cur_h) {  // new head: its conv taps and dt_bias into shared memory
            if (tid < kD) {
                const size_t c = (size_t)h * kD + tid;
#pragma unroll
                for (int x = 0; x < 3; ++x) cw[x * kD + tid] = __ldg(reinterpret_cast<const float4 *>(conv_w + ((size_t)x * D + c) * kK));
                sdt[tid] = __ldg(dt_bias + c);
            }
            eA = expf(__ldg(A_log + h));
            cur_h = h;
        }
        const bool ok = mbar_wait_bounded(&bar[stage], parity, kWaitLimit);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        if (bad) {
            if (tid == 0) atomicExch(err, kErrBadSlot);
            __syncthreads();
            continue;
        }
        const unsigned char *st = smem + stage * L::kBytes;
        const T *in = reinterpret_cast<const T *>(st + L::kS);
        const T *tl = reinterpret_cast<const T *>(st + L::kS + L::kIn);
        T *tl_g = tail_all + (size_t)slot * 9 * D + (size_t)h * kD;

        float yq = 0.f, yk = 0.f;
        if (tid < kD) {
            const int i = tid;
            float y[3];
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                const float4 wt = cw[x * kD + i];
                const T h0 = tl[(x * 3 + 0) * kD + i], h1 = tl[(x * 3 + 1) * kD + i], h2 = tl[(x * 3 + 2) * kD + i];
                const T raw = in[x * kD + i];
                y[x] = silu_ftz(fmaf(wt.x, IO<T>::ld(&h0), fmaf(wt.y, IO<T>::ld(&h1),
                              fmaf(wt.z, IO<T>::ld(&h2), wt.w * IO<T>::ld(&raw)))));
                tl_g[(size_t)(x * 3 + 0) * D + i] = h1;
                tl_g[(size_t)(x * 3 + 1) * D + i] = h2;
                tl_g[(size_t)(x * 3 + 2) * D + i] = raw;
            }
            yq = y[0]; yk = y[1];
            sh_v[i] = y[2];
            sh_a[i] = exp_ftz(gmin * sigmoid_ftz(eA * (IO<T>::ld(in + 3 * kD + i) + sdt[i])));
            sh_gw[i] = sigmoid_ftz(IO<T>::ld(in + 4 * kD + i)) * snw[i];
            const float a0 = warp_sum(yq * yq), a1 = warp_sum(yk * yk), a2 = warp_sum(yq * yk);
            if (l == 0) { part[w] = a0; part[4 + w] = a1; part[8 + w] = a2; }
        }
        // the state tile of this unit, row i = w + 8m, columns 4l..4l+3
        float4 s[16];
        const float4 *S4s = reinterpret_cast<const float4 *>(st);
#pragma unroll
        for (int m = 0; m < 16; ++m) s[m] = S4s[(16 * w + m) * 32 + l];
        __syncthreads();
        const float sqq = part[0] + part[1] + part[2] + part[3];
        const float skk = part[4] + part[5] + part[6] + part[7];
        const float sqk = part[8] + part[9] + part[10] + part[11];
        const float rq = q_scale * rsqrt_ftz(sqq + l2_eps);
        const float rk = rsqrt_ftz(skk + l2_eps);
        const float kq = sqk * rq * rk;
        if (tid < kD) {
            const float kn = yk * rk, a = sh_a[tid];
            sh_k[tid] = kn;
            sh_ak[tid] = a * kn;
            sh_aq[tid] = a * (yq * rq);
        }
        __syncthreads();
        decode_token_step<T>(s, sh_ak, sh_aq, sh_a, sh_k, sh_v, sh_gw, beta, kq, red, su, so,
                             out + (size_t)r * D + (size_t)h * kD, rms_eps, w, l);
        float4 *S4 = reinterpret_cast<float4 *>(S_all + ((size_t)slot * H + h) * kD * kD);
#pragma unroll
        for (int m = 0; m < 16; ++m) st_stream(S4 + (16 * w + m) * 32 + l, s[m]);
        __syncthreads();  // the stage, sh_* and red are free for the next unit
    }
    if (timed_out) {
        if (tid == 0) {
            atomicExch(err, KDA_ERR_TIMEOUT);
            // let copies already issued land before the CTA's shared memory goes away
            for (int j = 0; j < NS; ++j) {
                const int it2 = it + j;
                if (u_begin + it2 < u_end) mbar_wait_bounded(&bar[it2 % NS], (uint32_t)((it2 / NS) & 1), kWaitLimit);
            }
        }
        __syncthreads();
    }
}

template <typename T, int NS>
cudaError_t launch_persistent(const State &st, const kda_layer_params &p, const int32_t *slots, int B,
                              const void *q, const void *k, const void *v, const void *z, const void *b,
                              const void *g, void *out, cudaStream_t stream)
{
    const kda_config_t &c = st.cfg;
    const int H = c.num_heads;
    const size_t smem = (size_t)NS * StageLayout<T>::kBytes + 3 * kD * 16 + 2 * kD * 4 + 8 * kD * 4 +
                        kRedFloats * 4 + 16 * 4 + NS * 8;
    cudaError_t e = raise_smem_once(st, sizeof(T) == 2 ? kSmemDecodeBf16 : kSmemDecodeF32,
                                    decode_persistent_kernel<T, NS>, smem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = state_sms(st, &sms)) != cudaSuccess) return e;
    const int n_units = B * H;
    const int grid = n_units < sms ? n_units : sms;
    decode_persistent_kernel<T, NS><<<grid, 256, smem, stream>>>(
        p.conv_w, p.dt_bias, p.A_log, p.norm_w, st.S, (T *)st.tail, st.err, slots, B, H, st.max_slots,
        (const T *)q, (const T *)k, (const T *)v, (const T *)z, (const T *)b, (const T *)g, (T *)out,
        c.gate_lower_bound, c.l2_eps, c.rms_eps, c.q_scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const State &st, const kda_layer_params &p, const int32_t *slots, int B,
                          const void *q, const void *k, const void *v, const void *z, const void *b,
                          const void *g, void *out, cudaStream_t stream)
{
    if (st.cfg.io_dtype == KDA_BF16)
        return launch_persistent<__nv_bfloat16, 3>(st, p, slots, B, q, k, v, z, b, g, out, stream);
    return launch_persistent<float, 2>(st, p, slots, B, q, k, v, z, b, g, out, stream);
}

}  // namespace kda
