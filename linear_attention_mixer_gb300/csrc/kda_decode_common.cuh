// kda_decode_common.cuh - the per-token state step shared by the single-token and the
// multi-token decode kernels (so that n tokens in one call equal n calls bit for bit).
//
// For one (sequence, head) unit and one token, with the state in registers (256 threads:
// warp w owns rows 16w .. 16w+15, lane l columns 4l .. 4l+3, s[m] = row 16w + m):
//   p = (Diag(a) S)^T k,  r = (Diag(a) S)^T q       column reductions
//   u = beta (v - p),     o = r + (k . q) u         (o = S'^T q)
//   S' = Diag(a) S + k u^T
//   out = gw * o / sqrt(mean(o^2) + eps)            gated RMSNorm, gw = sigmoid(g) * norm_w
// which is the kimi_k3.c header's per-head recurrence ("KDA per-head recurrence") expanded.
#pragma once

#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {

// The warp partials of p sit at red[0 .. 8 kD) and those of r at red[kRedR .. kRedR + 8 kD).
// The 16-float gap keeps the two apart by a bank offset: in the column finish, lanes 0..15 read
// p and lanes 16..31 read r of the same columns, and without it every such load would be a
// two-way bank conflict.
constexpr int kRedR = 8 * kD + 16;
constexpr int kRedFloats = kRedR + 8 * kD;

__device__ __forceinline__ float4 dc_fma4(float a, float4 x, float4 y)
{
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

// Pieces of the per-token step for the 16 state rows 16w .. 16w+15 held as s[0..15] (lane l:
// columns 4l .. 4l+3). Every kernel that runs the step is built from these, so results agree
// bit for bit across them.

// 1. this row group's partial column sums p = sum_i ak[i] S[i][.], r = sum_i aq[i] S[i][.]
__device__ __forceinline__ void dc_partials(const float4 (&s)[16], const float *ak, const float *aq, int w,
                                            float4 &p, float4 &rr)
{
    p = make_float4(0.f, 0.f, 0.f, 0.f);
    rr = p;
    const float4 *ak4 = reinterpret_cast<const float4 *>(ak + 16 * w);
    const float4 *aq4 = reinterpret_cast<const float4 *>(aq + 16 * w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 x = ak4[j], y = aq4[j];
        p = dc_fma4(x.x, s[4 * j + 0], p);  rr = dc_fma4(y.x, s[4 * j + 0], rr);
        p = dc_fma4(x.y, s[4 * j + 1], p);  rr = dc_fma4(y.y, s[4 * j + 1], rr);
        p = dc_fma4(x.z, s[4 * j + 2], p);  rr = dc_fma4(y.z, s[4 * j + 2], rr);
        p = dc_fma4(x.w, s[4 * j + 3], p);  rr = dc_fma4(y.w, s[4 * j + 3], rr);
    }
}

// 2. (per column, once its 8 row-group partials are added in group order) u and o
__device__ __forceinline__ float dc_u(float beta, float v, float p_sum) { return beta * (v - p_sum); }
__device__ __forceinline__ float dc_o(float kq, float u, float r_sum) { return fmaf(kq, u, r_sum); }

// 3a. the rank-1 update of this row group: S' = Diag(a) S + k u^T
__device__ __forceinline__ void dc_update(float4 (&s)[16], const float *a, const float *k, float4 uu, int w)
{
    const float4 *a4 = reinterpret_cast<const float4 *>(a + 16 * w);
    const float4 *k4 = reinterpret_cast<const float4 *>(k + 16 * w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 av = a4[j], kv = k4[j];
        const float aa[4] = {av.x, av.y, av.z, av.w}, kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float4 &sv = s[4 * j + e];
            sv = make_float4(fmaf(aa[e], sv.x, kk[e] * uu.x), fmaf(aa[e], sv.y, kk[e] * uu.y),
                             fmaf(aa[e], sv.z, kk[e] * uu.z), fmaf(aa[e], sv.w, kk[e] * uu.w));
        }
    }
}

// 3b. the gated RMSNorm of o (this lane's 4 values oo; the warp holds all 128): lanes 4w ..
//     4w+3 write columns 16w .. 16w+15 of out_row
template <typename T>
__device__ __forceinline__ void dc_norm_store(float4 oo, const float *gw, T *out_row, float rms_eps, int w, int l)
{
    const float ss = warp_sum(oo.x * oo.x + oo.y * oo.y + oo.z * oo.z + oo.w * oo.w);
    if ((l >> 2) == w) {
        const float rinv = rsqrt_ftz(ss * (1.0f / kD) + rms_eps);
        const float4 g4 = reinterpret_cast<const float4 *>(gw)[l];
        T *dst = out_row + 4 * l;
        IO<T>::st(dst + 0, g4.x * (oo.x * rinv));
        IO<T>::st(dst + 1, g4.y * (oo.y * rinv));
        IO<T>::st(dst + 2, g4.z * (oo.z * rinv));
        IO<T>::st(dst + 3, g4.w * (oo.w * rinv));
    }
}

// ak[i] = a_i k^_i, aq[i] = a_i q^_i, a[i], k[i] (k^), v[c], gw[c]: shared-memory vectors of 128
// red: kRedFloats floats (warp partials of p and of r, see kRedR), su, so: [128] floats (u and o).
// kq = k^ . q^. out_row: this unit's 128 output values. Contains two __syncthreads.
template <typename T>
__device__ __forceinline__ void decode_token_step(float4 (&s)[16], const float *ak, const float *aq,
                                                  const float *a, const float *k, const float *v,
                                                  const float *gw, float beta, float kq, float *red, float *su,
                                                  float *so, T *out_row, float rms_eps, int w, int l)
{
    // 1. partial column sums over this warp's 16 rows
    float4 p, rr;
    dc_partials(s, ak, aq, w, p, rr);
    reinterpret_cast<float4 *>(red)[w * 32 + l] = p;
    reinterpret_cast<float4 *>(red + kRedR)[w * 32 + l] = rr;
    __syncthreads();
    // 2. warp w finishes columns 16w .. 16w+15: lanes 0..15 sum p, lanes 16..31 sum r
    {
        const int c = 16 * w + (l & 15), which = l >> 4;
        const float *col = red + which * kRedR + c;
        float acc = col[0];
#pragma unroll
        for (int ww = 1; ww < 8; ++ww) acc += col[ww * kD];
        const float r_c = __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
        if (l < 16) {
            const float u = dc_u(beta, v[c], acc);
            su[c] = u;
            so[c] = dc_o(kq, u, r_c);
        }
    }
    __syncthreads();
    // 3. the rank-1 update of this warp's rows, and the gated RMSNorm (every warp holds all
    //    128 values of o; warp w writes columns 16w .. 16w+15)
    const float4 uu = reinterpret_cast<const float4 *>(su)[l];
    const float4 oo = reinterpret_cast<const float4 *>(so)[l];
    dc_update(s, a, k, uu, w);
    dc_norm_store(oo, gw, out_row, rms_eps, w, l);
}

}  // namespace kda
