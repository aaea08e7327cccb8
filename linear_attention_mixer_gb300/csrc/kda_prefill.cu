// kda_prefill.cu - chunked (WY / UT-transform) KDA prefill over packed
// variable-length sequences.
//
// The per-token recurrence of the kimi_k3.c header comment ("KDA per-head
// recurrence") is evaluated in chunks of C = 64 tokens. For a chunk starting
// from state S0, with G_r the cumulative log decay (sum of gk over the chunk's
// tokens up to r, a vector over the key dim), the exact rewrite is
//   A[r][i] = beta_r sum_c k_r[c] k_i[c] exp(G_r[c] - G_i[c])   (i < r)
//   W  = (I + A)^-1 Diag(beta) (K o exp(G)),  U' = (I + A)^-1 Diag(beta) V
//   U  = U' - W S0
//   O  = (Q o exp(G)) S0 + (P o M) U,  P[r][i] = sum_c q_r[c] k_i[c] exp(G_r[c] - G_i[c])
//   S  = Diag(exp(G_last)) S0 + (K o exp(G_last - G))^T U
// exp(G_r - G_i) is formed as a product of two factors that are both finite in
// FP32: for each 16-row block with first row n, exp(G_r - G_n) (<= 1) times
// exp(G_n - G_i) (<= 1 for i <= n, <= e^75 inside the block).
//
// Kernels, in stream order:
//   chunk_table_kernel  chunk list (sequence, first token, length) from cu_seqlens
//   prep_kernel         per (chunk, head): conv+SiLU, L2, gates, G, A, P,
//                       the triangular solve, W, U', Q o exp(G), K o exp(G_last - G)
//   state_kernel        per (sequence, head, 32-column block of v): the serial
//                       pass over the chunks carrying S; writes o and the final
//                       state, and the new conv history
//   epilogue_kernel     gated per-head RMSNorm of o
// With BF16 I/O, prep_tc_kernel (A and P on tensor cores) and state_tc_kernel (one CTA
// per (sequence, head), the chunk products on tensor cores, the RMSNorm fused) replace
// prep_kernel, state_kernel and epilogue_kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kBlk = 16;                  // sub-block rows for the decay reference
constexpr int kVB = 32;                   // v columns per state_kernel CTA
constexpr int kChunkFloats = 4 * kC * kD + kC * kC + kD;  // W, U', QG, KD, P, gC
constexpr int kKRS = kC + 1;  // padded row of the transposed right factor (no bank conflicts)
constexpr int kPrepSmemFloats = 4 * kC * kD + 2 * kC * kC + kD * kKRS + 2 * kBlk * kD + kC;
constexpr int kStateSmemFloats = kD * kVB + 3 * kC * kD + 2 * kC * kVB + kC * kC + kD;

// Tensor-core path (BF16 I/O): per (chunk, head) the prep kernel writes one block that the
// state kernel reads as two bulk copies (tile A with exp(G_last), then tile B) plus U' read
// by its threads. Operand tiles are BF16 in the K-major interleaved layout of kda_tc.cuh.
// The factors that carry the state (W, K o exp(G_last - G), and P for the output's U term)
// are stored as a BF16 high part and a low part (x - high): with single BF16 operands the
// state drifts by up to a few percent when the decay is near 1, beta near 1 and the keys
// strongly correlated (the products then cancel), so each product is formed as
// hi*hi + lo*hi + hi*lo, about 16 bits of mantissa.
//   tile A [192 rows][128 k]: rows 0..63 W_hi [r][k], 64..127 QG [r][k], 128..191 W_lo
//          B operands of S^T [W_hi | QG]^T (N = 128), S^T W_hi^T and S^T W_lo^T (N = 64)
//   gamma  [128] FP32 exp(G_last), right after tile A (it travels with tile A's copy)
//   tile B [384 rows][64 r]: rows 0..63 P_hi [r][i], 64..191 KDT_hi [k][r], 192..255 P_lo,
//          256..383 KDT_lo; B operands of U^T [P | KDT] (N = 192, hi rows or lo rows)
//   U'     [64 r][128 v] FP32, read by the state pass's threads
constexpr int kOffTA = 0, kOffGam = 49152, kOffTB = 49664, kOffUp = 98816;
constexpr int kTcChunkBytes = 131584;
constexpr int kStageABytes = kOffTB;   // tile A + gamma
constexpr int kStageBBytes = kOffUp - kOffTB;
static_assert(kStageBBytes == 49152 && kOffUp + kC * kD * 4 == kTcChunkBytes, "chunk block layout");
// state_tc_kernel shared memory: stage A | stage B | g/out rows | sums | barriers (the A
// operands are in tensor memory)
constexpr int kSmA = 0, kSmB = kSmA + kStageABytes, kSmGY = kSmB + kStageBBytes;
constexpr int kSmRed = kSmGY + kC * kD * 2, kSmGam = kSmRed + 4 * kC * 4, kSmBar = kSmGam + 2 * kD * 4;
constexpr int kStateTcSmem = kSmBar + 12 * 8 + 16;
static_assert(kSmB % 128 == 0 && kSmGY % 128 == 0, "TMA and bulk destinations");
static_assert(kStateTcSmem <= 232448, "state_tc_kernel shared memory");
constexpr uint32_t kTcWaitLimit = 1u << 26;

struct ChunkEntry { int seq, t0, n, pos0; };

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t table, seq_first, chunks, obuf, total;
};

// tc: BF16 tensor-core layout (no o buffer: the RMSNorm is fused into the state pass)
WsLayout ws_layout(int H, int64_t total_chunks, int64_t total_T, int N, bool tc) {
    WsLayout L;
    size_t off = 0;
    L.table = off;     off = align_up(off + sizeof(ChunkEntry) * (size_t)total_chunks, 256);
    L.seq_first = off; off = align_up(off + sizeof(int32_t) * (size_t)(N + 1), 256);
    L.chunks = off;
    off = align_up(off + (tc ? (size_t)kTcChunkBytes : sizeof(float) * (size_t)kChunkFloats) * total_chunks * H, 256);
    L.obuf = off;
    if (!tc) off = align_up(off + sizeof(float) * (size_t)total_T * H * kD, 256);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------- chunk table
// One thread builds the chunk list. The device copy of cu_seqlens is checked
// against what the host sized the launch for (N + 1 entries, starting at 0,
// non-decreasing, ending at total_T, at most max_chunks chunks); on a mismatch
// the list is left empty (every sequence gets no chunk) and the error word is set.
__global__ void chunk_table_kernel(const int32_t *__restrict__ cu, int N, int64_t total_T, int64_t max_chunks,
                                   ChunkEntry *__restrict__ table, int32_t *__restrict__ seq_first,
                                   int32_t *__restrict__ err)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    bool ok = cu[0] == 0 && (int64_t)cu[N] == total_T;
    int64_t count = 0;
    for (int s = 0; s < N && ok; ++s) {
        const int len = cu[s + 1] - cu[s];
        if (len < 0) ok = false;
        else count += (len + kC - 1) / kC;
    }
    if (count > max_chunks) ok = false;
    if (!ok) {
        atomicExch(err, kErrBadSlot);
        for (int s = 0; s <= N; ++s) seq_first[s] = 0;
        for (int64_t i = 0; i < max_chunks; ++i) table[i] = ChunkEntry{0, 0, 0, 0};
        return;
    }
    int idx = 0;
    for (int s = 0; s < N; ++s) {
        seq_first[s] = idx;
        const int start = cu[s], len = cu[s + 1] - cu[s];
        for (int p = 0; p < len; p += kC) {
            ChunkEntry e;
            e.seq = s; e.t0 = start + p; e.n = min(kC, len - p); e.pos0 = p;
            table[idx++] = e;
        }
    }
    seq_first[N] = idx;
    for (int64_t i = idx; i < max_chunks; ++i) table[i] = ChunkEntry{0, 0, 0, 0};
}

// ---------------------------------------------------------------- prep
// FP32 I/O: writes the FP32 chunk block (kChunkFloats per (chunk, head)).
template <typename T>
__global__ void __launch_bounds__(256, 1)
prep_kernel(const float *__restrict__ conv_w, const float *__restrict__ dt_bias,
            const float *__restrict__ A_log, const T *__restrict__ tail_all,
            const int32_t *__restrict__ slots, int H, int max_slots,
            const ChunkEntry *__restrict__ table,
            const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
            const T *__restrict__ z, const T *__restrict__ bl,
            unsigned char *__restrict__ chunks, float gmin, float l2_eps, float q_scale)
{
    extern __shared__ __align__(16) float sm[];
    float *Yq = sm;                 // [C][d]   q^ after L2 and scale
    float *Yk = Yq + kC * kD;       // [C][d]   k^
    float *Yv = Yk + kC * kD;       // [C][d]   v
    float *G = Yv + kC * kD;        // [C][d]   cumulative log decay
    float *Am = G + kC * kD;        // [C][C]   A (strict lower, beta folded)
    float *Pm = Am + kC * kC;       // [C][C]   P (inclusive lower)
    float *KRT = Pm + kC * kC;      // [d][C+1] k_i o exp(G_n - G_i), transposed, padded rows
    float *KL = KRT + kD * kKRS;    // [16][d]  k_r o exp(G_r - G_n)
    float *QL = KL + kBlk * kD;     // [16][d]  q_r o exp(G_r - G_n)
    float *sbeta = QL + kBlk * kD;  // [C]

    const int chunk = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
    const ChunkEntry e = table[chunk];
    if (e.n <= 0) return;  // empty entry: the chunk list was rejected
    const int slot = slots[e.seq];
    if (slot < 0 || slot >= max_slots) return;  // recorded by state_kernel
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = e.n;
    const size_t D = (size_t)H * kD;

    // 0. (BF16 inputs) the chunk's raw q, k, v rows with their 3 rows of history, and z,
    //    staged in shared memory with 16-byte loads; the region is reused from step 4 on.
    constexpr int kRows = kC + 3;  // staged row j holds position j - 3 of the chunk
    T *raw = reinterpret_cast<T *>(Am);
    constexpr bool kStage = sizeof(T) == 2;
    static_assert(!kStage || 4 * kRows * kD * sizeof(T) <= (2 * kC * kC + kD * kKRS + 2 * kBlk * kD) * sizeof(float),
                  "raw staging must fit in the A/P/KRT/KL/QL region");
    if constexpr (kStage) {
        const T *srcs[4] = {q, k, v, z};
        const T *tl0 = tail_all + (size_t)slot * 3 * (kK - 1) * D + (size_t)h * kD;
        for (int e2 = tid; e2 < 4 * kRows * 16; e2 += 256) {
            const int x = e2 / (kRows * 16), rem = e2 - x * (kRows * 16);
            const int j = rem >> 4, vec = rem & 15;
            const int p = j - 3;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (p < n && !(x == 3 && p < 0)) {
                const int pos = e.pos0 + p;  // position within the sequence
                const T *srcp = pos >= 0 ? srcs[x] + (size_t)(e.t0 + p) * D + (size_t)h * kD
                                         : tl0 + (size_t)(x * 3 + (pos + 3)) * D;
                val = __ldg(reinterpret_cast<const uint4 *>(srcp) + vec);
            }
            reinterpret_cast<uint4 *>(raw + ((size_t)x * kRows + j) * kD)[vec] = val;
        }
        __syncthreads();
    }

    // 1. conv + SiLU. Thread (i, half): channel i, rows [32 half, 32 half + 32).
    {
        const int i = tid & (kD - 1), half = tid >> 7;
        const size_t c = (size_t)h * kD + i;
        const T *src[3] = {q, k, v};
        float *dst[3] = {Yq, Yk, Yv};
        const T *tl = tail_all + (size_t)slot * 3 * (kK - 1) * D + c;
        const int r0 = 32 * half;
#pragma unroll
        for (int x = 0; x < 3; ++x) {
            const float4 wt = __ldg(reinterpret_cast<const float4 *>(conv_w + ((size_t)x * D + c) * kK));
            if constexpr (kStage) {
                const T *col = raw + (size_t)x * kRows * kD + i;
                for (int rr = 0; rr < 32; ++rr) {
                    const int r = r0 + rr;
                    float y = 0.f;
                    if (r < n)
                        y = siluf_(fmaf(wt.x, IO<T>::ld(col + r * kD), fmaf(wt.y, IO<T>::ld(col + (r + 1) * kD),
                                   fmaf(wt.z, IO<T>::ld(col + (r + 2) * kD), wt.w * IO<T>::ld(col + (r + 3) * kD)))));
                    dst[x][r * kD + i] = y;
                }
            } else {
                float hst[3] = {0.f, 0.f, 0.f};
                if (r0 < n) {  // rows of this half exist; their history lies inside the sequence or the tail
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        const int pos = e.pos0 + r0 - 3 + j;  // position within the sequence
                        hst[j] = pos >= 0 ? IO<T>::ld(src[x] + (size_t)(e.t0 + r0 - 3 + j) * D + c)
                                          : IO<T>::ld(tl + (size_t)(x * 3 + (pos + 3)) * D);
                    }
                }
                for (int rr = 0; rr < 32; ++rr) {
                    const int r = r0 + rr;
                    float y = 0.f;
                    if (r < n) {
                        const float xin = IO<T>::ld(src[x] + (size_t)(e.t0 + r) * D + c);
                        y = siluf_(fmaf(wt.x, hst[0], fmaf(wt.y, hst[1], fmaf(wt.z, hst[2], wt.w * xin))));
                        hst[0] = hst[1]; hst[1] = hst[2]; hst[2] = xin;
                    }
                    dst[x][r * kD + i] = y;
                }
            }
        }
        // 2. gates: gk = gmin * sigmoid(exp(A_log) (z + dt)), cumulative over rows
        const float eA = expf(__ldg(A_log + h));
        const float dt = __ldg(dt_bias + c);
        float acc = 0.f;
        for (int rr = 0; rr < 32; ++rr) {
            const int r = r0 + rr;
            float gk = 0.f;
            if (r < n) {
                const float zz = kStage ? IO<T>::ld(raw + ((size_t)3 * kRows + r + 3) * kD + i)
                                        : IO<T>::ld(z + (size_t)(e.t0 + r) * D + c);
                gk = gmin * sigmoidf_(eA * (zz + dt));
            }
            acc += gk;
            G[r * kD + i] = acc;
        }
    }
    __syncthreads();
    if (tid >= kD) {  // second half adds the first half's total
        const int i = tid - kD;
        const float base = G[31 * kD + i];
        for (int r = 32; r < kC; ++r) G[r * kD + i] += base;
    }
    // 3. L2 norms and beta: warp w handles rows w + 8m.
    for (int m = 0; m < kC / 8; ++m) {
        const int r = warp + 8 * m;
        float4 a = reinterpret_cast<float4 *>(Yq + r * kD)[lane];
        float4 b = reinterpret_cast<float4 *>(Yk + r * kD)[lane];
        const float sq = warp_sum(a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w);
        const float sk = warp_sum(b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w);
        const float rq = q_scale / sqrtf(sq + l2_eps), rk = 1.0f / sqrtf(sk + l2_eps);
        a.x *= rq; a.y *= rq; a.z *= rq; a.w *= rq;
        b.x *= rk; b.y *= rk; b.z *= rk; b.w *= rk;
        reinterpret_cast<float4 *>(Yq + r * kD)[lane] = a;
        reinterpret_cast<float4 *>(Yk + r * kD)[lane] = b;
        if (lane == 0) sbeta[r] = r < n ? sigmoidf_(IO<T>::ld(bl + (size_t)(e.t0 + r) * H + h)) : 0.f;
    }
    __syncthreads();

    // 4. A and P, one 16-row block at a time, reference row nR = 16 R.
    for (int R = 0; R < kC / kBlk; ++R) {
        const int nR = R * kBlk, m = nR + kBlk;
        {
            // thread (c, half): consecutive threads walk consecutive c, so the row reads of
            // Yk / G and the padded transposed writes are both free of bank conflicts
            const int c = tid & (kD - 1), ih = tid >> 7;
            const float gn = G[nR * kD + c];
            for (int i = 32 * ih; i < min(m, 32 * ih + 32); ++i)
                KRT[c * kKRS + i] = Yk[i * kD + c] * expf(gn - G[i * kD + c]);
        }
        {
            for (int e2 = tid; e2 < kBlk * kD; e2 += 256) {
                const int rr = e2 / kD, c = e2 - rr * kD;
                const float f = expf(G[(nR + rr) * kD + c] - G[nR * kD + c]);
                KL[e2] = Yk[(nR + rr) * kD + c] * f;
                QL[e2] = Yq[(nR + rr) * kD + c] * f;
            }
        }
        __syncthreads();
        {
            const int i = tid & (kC - 1), rg = tid >> 6;
            float a[4] = {0.f, 0.f, 0.f, 0.f}, p[4] = {0.f, 0.f, 0.f, 0.f};
            if (i < m) {
                for (int c = 0; c < kD; ++c) {
                    const float kr = KRT[c * kKRS + i];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        a[qq] = fmaf(KL[(4 * rg + qq) * kD + c], kr, a[qq]);
                        p[qq] = fmaf(QL[(4 * rg + qq) * kD + c], kr, p[qq]);
                    }
                }
            }
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int r = nR + 4 * rg + qq;
                Am[r * kC + i] = (i < r) ? sbeta[r] * a[qq] : 0.f;
                Pm[r * kC + i] = (i <= r) ? p[qq] : 0.f;
            }
        }
        __syncthreads();
    }

    float *out = reinterpret_cast<float *>(chunks) + (size_t)blockIdx.x * kChunkFloats;
    float *W = out, *Up = W + kC * kD, *QG = Up + kC * kD, *KD = QG + kC * kD, *P = KD + kC * kD,
          *GC = P + kC * kC;
    // 5. Forward substitution (I + A) X = Diag(beta) B, one column per thread:
    //    columns 0..127 of B are k o exp(G), 128..255 are v.
    {
        const int j = tid;
        const bool isk = j < kD;
        const int cj = isk ? j : j - kD;
        float X[kC];
#pragma unroll
        for (int r = 0; r < kC; ++r) {
            const float bb = isk ? Yk[r * kD + cj] * expf(G[r * kD + cj]) : Yv[r * kD + cj];
            // four independent partial sums over i, A read 4 at a time
            float x0 = sbeta[r] * bb, x1 = 0.f, x2 = 0.f, x3 = 0.f;
#pragma unroll
            for (int i = 0; i + 4 <= r; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(Am + r * kC + i);
                x0 = fmaf(-a4.x, X[i], x0);
                x1 = fmaf(-a4.y, X[i + 1], x1);
                x2 = fmaf(-a4.z, X[i + 2], x2);
                x3 = fmaf(-a4.w, X[i + 3], x3);
            }
#pragma unroll
            for (int i = r & ~3; i < r; ++i) x0 = fmaf(-Am[r * kC + i], X[i], x0);
            X[r] = (x0 + x1) + (x2 + x3);
        }
        float *dstc = isk ? W : Up;
#pragma unroll
        for (int r = 0; r < kC; ++r) dstc[r * kD + cj] = X[r];
    }
    // 6. The remaining chunk factors.
    for (int e2 = tid; e2 < kC * kD; e2 += 256) {
        const int r = e2 / kD, c = e2 - r * kD;
        const float g = G[r * kD + c];
        QG[e2] = Yq[e2] * expf(g);
        KD[e2] = Yk[e2] * expf(G[(n - 1) * kD + c] - g);
    }
    for (int e2 = tid; e2 < kC * kC; e2 += 256) P[e2] = Pm[e2];
    if (tid < kD) GC[tid] = expf(G[(n - 1) * kD + tid]);
}

// ---------------------------------------------------------------- prep on tensor cores
// BF16 path, one CTA (512 threads) per (chunk, head). Differences from prep_kernel:
//  * the chunk's raw rows arrive by bulk copies on one mbarrier, and the CTA that will most
//    likely run next on this SM has its q, k, v, z rows prefetched to L2;
//  * every decay factor is the exp of a difference of the cumulative log decay G (one scan per
//    channel), so threads form factor elements independently, 8 channels at a time:
//      exp(G_r - G_n) <= 1 (left), exp(G_n - G_i) <= 1 for i <= n (right), <= e^75 on a block
//      diagonal; exp(G_r), exp(G_last - G_r) <= 1; all finite in FP32;
//  * A and P come from tcgen05 in one accumulator: left rows are k_r o exp(G_r - G_n) (rows
//    0..63) and q_r o exp(G_r - G_n) (rows 64..127), n = 16 (r / 16) the first row of r's
//    16-row block; right rows are, for each block R, k_i o exp(G_n - G_i) for i < n + 16
//    (160 rows in all). Row r of block R reads the columns of R's own right rows. Every factor
//    is split into a BF16 hi part and a lo part (x - hi) and three MMA chains accumulate
//    hi*hi + lo*hi + hi*lo, so A and P carry about FP32-level error instead of BF16's 2^-9.
//    The tiles are built one half of the channels at a time (24 MMAs in all: an MMA has a
//    fixed issue cost, so few wide ones beat many narrow ones);
//  * the solve is explicit: T = (I + A)^-1 by blocked inversion (16 x 16 diagonal blocks by
//    forward substitution, then one block row at a time), then W = T Diag(beta) (K o exp(G))
//    and U'^T = (Diag(beta) V)^T T^T on the tensor core, again split hi/lo;
//  * Q o exp(G), (K o exp(G_last - G))^T and exp(G_last) are written while the A/P MMAs run.
// Shared memory: FP32 [64][132] arrays (rows padded against bank conflicts) for q^, k^, v and
// G, then one reused region (raw inputs -> A/P tiles -> B_lo, T tile, A matrix); after the A/P
// phase the q^ array holds B_hi, and after the B build the v and G arrays hold T and scratch.
// c[i][j] += sum_{k < 4 G} a[i pa + k] b[k pb + j] (i < 2, j < 4): a 2 x 4 register tile of a
// product of two FP32 matrices in shared memory, a read 4 k at a time as float4 along its rows
template <int G>
__device__ __forceinline__ void tile24(float (&c)[2][4], const float *a, int pa, const float *b, int pb)
{
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float4 a0 = *reinterpret_cast<const float4 *>(a + 4 * g);
        const float4 a1 = *reinterpret_cast<const float4 *>(a + pa + 4 * g);
        float4 bv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = *reinterpret_cast<const float4 *>(b + (4 * g + j) * pb);
        const float x0[4] = {a0.x, a0.y, a0.z, a0.w}, x1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c[0][0] = fmaf(x0[j], bv[j].x, c[0][0]); c[0][1] = fmaf(x0[j], bv[j].y, c[0][1]);
            c[0][2] = fmaf(x0[j], bv[j].z, c[0][2]); c[0][3] = fmaf(x0[j], bv[j].w, c[0][3]);
            c[1][0] = fmaf(x1[j], bv[j].x, c[1][0]); c[1][1] = fmaf(x1[j], bv[j].y, c[1][1]);
            c[1][2] = fmaf(x1[j], bv[j].z, c[1][2]); c[1][3] = fmaf(x1[j], bv[j].w, c[1][3]);
        }
    }
}

// 2 x 4 tile rows r, r + 1, columns c .. c + 3, times sg, to the BF16 T tile: hi parts in rows
// r, r + 1 and lo parts in rows 64 + r, 64 + r + 1 (8 bytes per row)
__device__ __forceinline__ void put24_split(unsigned char *tile, int r, int c, const float (&v)[2][4], float sg)
{
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h[2], l[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float x0 = sg * v[i][2 * e], x1 = sg * v[i][2 * e + 1];
            const __nv_bfloat162 p = __floats2bfloat162_rn(x0, x1);
            const uint32_t u = *reinterpret_cast<const uint32_t *>(&p);
            h[e] = u;
            const __nv_bfloat162 q = __floats2bfloat162_rn(x0 - __uint_as_float(u << 16), x1 - __uint_as_float(u & 0xFFFF0000u));
            l[e] = *reinterpret_cast<const uint32_t *>(&q);
        }
        *reinterpret_cast<uint2 *>(tile + tc::kmajor_off(r + i, c, kC)) = make_uint2(h[0], h[1]);
        *reinterpret_cast<uint2 *>(tile + tc::kmajor_off(kC + r + i, c, kC)) = make_uint2(l[0], l[1]);
    }
}

// a 2 x 4 tile times sg to dst (row pitch pd), one float4 per row
__device__ __forceinline__ void put24(float *dst, int pd, const float (&c)[2][4], float sg)
{
#pragma unroll
    for (int i = 0; i < 2; ++i)
        *reinterpret_cast<float4 *>(dst + i * pd) = make_float4(sg * c[i][0], sg * c[i][1], sg * c[i][2], sg * c[i][3]);
}

constexpr int kYS = kD + 4;   // padded FP32 row
constexpr int kMS = kC + 4;   // row pitch of the FP32 A / T matrices (16-byte aligned rows)
constexpr int kPtY = 73728;   // reused region
// A/P phase, one half of the channels at a time: left tiles hi and lo [128 rows: k rows 0..63,
// q rows 64..127][64 channels], right tiles hi and lo [160 rows][64], block R's segment of
// right rows (i < 16 (R + 1), reference row 16 R) starting at row 8 R (R + 1).
constexpr int kApN = 160;
constexpr int kApLh = 0, kApLl = 16384, kApRh = 32768, kApRl = 32768 + kApN * 128;
// solve phase: B_lo [256][64], T tile [hi rows 0..63, lo rows 64..127][64] (a descriptor
// starting at row 64 covers rows 64..191, ending 24 KB into the tile) and the FP32 A matrix.
// The diagonal blocks T_RR of the inverse follow M, as [4][16][kTD] FP32.
constexpr int kPtBl = 0, kPtT = 32768, kPtM = 49152, kTD = 20, kPtD = kPtM + kC * kMS * 4;
static_assert(kApRl + kApN * 128 <= kPtY, "A/P tiles");
static_assert(kPtT + 24576 <= kPtY && kPtD + 4 * 16 * kTD * 4 <= kPtY, "solve tiles");
static_assert(256 * kC * 2 <= kC * kYS * 4, "B_hi must fit in the q^ array");
constexpr int kPrepTcSmem = 4 * kC * kYS * 4 + kPtY + kC * 4 + 64;

// 8 FP32 values -> BF16 hi parts (nearest) and lo parts (x - hi, nearest), 16 bytes each
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        const uint32_t u = *reinterpret_cast<const uint32_t *>(&p);
        h[i] = u;
        const __nv_bfloat162 q = __floats2bfloat162_rn(x[2 * i] - __uint_as_float(u << 16),
                                                       x[2 * i + 1] - __uint_as_float(u & 0xFFFF0000u));
        l[i] = *reinterpret_cast<const uint32_t *>(&q);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ uint4 pack8_bf16(const float *x)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void ld8f(const float *p, float *x)
{
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void st16(unsigned char *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

// Three MMA chains hi*hi + lo*hi + hi*lo into one accumulator. The descriptors are those of
// K-step 0; step kk starts 256 bytes (16 descriptor units) later.
__device__ __forceinline__ void mma_split3(uint32_t d, uint64_t a_hi, uint64_t a_lo, uint64_t b_hi, uint64_t b_lo,
                                           uint32_t idesc, int ksteps, bool acc0)
{
    for (int kk = 0; kk < ksteps; ++kk)
        tc::mma_bf16(d, a_hi + 16u * kk, b_hi + 16u * kk, idesc, (acc0 || kk > 0) ? 1u : 0u);
    for (int kk = 0; kk < ksteps; ++kk) tc::mma_bf16(d, a_lo + 16u * kk, b_hi + 16u * kk, idesc, 1u);
    for (int kk = 0; kk < ksteps; ++kk) tc::mma_bf16(d, a_hi + 16u * kk, b_lo + 16u * kk, idesc, 1u);
}

// 2^x by the special-function unit (about 2 ulp); results below the smallest normal number flush
// to zero. prep_tc keeps the cumulative log decay in base 2 (G log2(e)), so that each of its
// exponentials of G, or of a difference of G values, is this one instruction.
__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// conv + SiLU of two adjacent channels over 32 output rows: col points at the staged raw row
// of the first output's oldest tap (staged row j holds position j - 3), w0 and w1 are the two
// channels' taps (oldest first), dst at the first output row (row pitch kYS). Rows at or past
// n_valid are written as zero (only checked when kFull is false).
template <bool kFull>
__device__ __forceinline__ void conv_silu_pair32(const __nv_bfloat16 *col, float4 w0, float4 w1, float *dst,
                                                 int n_valid)
{
    auto ld2 = [&](int j) { return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(col + j * kD)); };
    float2 h0 = ld2(0), h1 = ld2(1), h2 = ld2(2);
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += 8) {
        float2 cv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float2 xin = ld2(r0 + u + 3);
            cv[u].x = fmaf(w0.x, h0.x, fmaf(w0.y, h1.x, fmaf(w0.z, h2.x, w0.w * xin.x)));
            cv[u].y = fmaf(w1.x, h0.y, fmaf(w1.y, h1.y, fmaf(w1.z, h2.y, w1.w * xin.y)));
            h0 = h1; h1 = h2; h2 = xin;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            // sigmoid(x) = (1 + tanh(x/2)) / 2: one SFU operation instead of two; the hardware
            // tanh's error (about 2^-11 relative) is far below BF16's rounding
            const float sx = fmaf(0.5f, tanh_approx(0.5f * cv[u].x), 0.5f);
            const float sy = fmaf(0.5f, tanh_approx(0.5f * cv[u].y), 0.5f);
            float2 y = make_float2(cv[u].x * sx, cv[u].y * sy);
            if (!kFull && r0 + u >= n_valid) y = make_float2(0.f, 0.f);
            *reinterpret_cast<float2 *>(dst + (r0 + u) * kYS) = y;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(512, 1)
prep_tc_kernel(const float *__restrict__ conv_w, const float *__restrict__ dt_bias,
               const float *__restrict__ A_log, const T *__restrict__ tail_all,
               const int32_t *__restrict__ slots, int H, int max_slots,
               const ChunkEntry *__restrict__ table,
               const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
               const T *__restrict__ z, const T *__restrict__ bl,
               unsigned char *__restrict__ chunks, int32_t *__restrict__ err,
               float gmin, float l2_eps, float q_scale, int n_items, int box_rows, int f_rows, int fused,
               const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_z,
               const __grid_constant__ CUtensorMap tm_f, const __grid_constant__ CUtensorMap tm_fb)
{
    extern __shared__ __align__(1024) float smf[];
    float *Yq = smf;                                  // [64][132] q^
    float *Yk = Yq + kC * kYS;                        // [64][132] k^
    float *Yv = Yk + kC * kYS;                        // [64][132] v
    float *GL = Yv + kC * kYS;                        // [64][132] G log2(e), G the cumulative log decay
    unsigned char *Y = reinterpret_cast<unsigned char *>(GL + kC * kYS);
    float *sbeta = reinterpret_cast<float *>(Y + kPtY);
    // [0] z operands (fused), [1..2] A/P buffers, [3] solve, [4] z product (fused)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbeta + kC);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 5);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t D = (size_t)H * kD;
    // staged row j of stream x holds position j - 3 of the chunk; 3 spare rows at the end take
    // the overhang of a box that starts at the chunk's first row
    constexpr int kRows = kC + 6;
    T *raw = reinterpret_cast<T *>(Y);
    static_assert(4 * kRows * kD * sizeof(T) <= kPtY, "raw staging must fit in the reused region");
    static_assert((kRows * kD * sizeof(T)) % 128 == 0, "TMA destinations must be 128-byte aligned");

    // One CTA per SM takes the items (chunk, head) = blockIdx.x + i gridDim.x, chunk-major. An
    // item is skipped when its chunk entry is empty (the chunk list was rejected) or its slot is
    // out of range (recorded by the state pass); every thread decides alike.
    auto item_ok = [&](int it) {
        const ChunkEntry ei = table[it / H];
        if (ei.n <= 0) return false;
        const int si = slots[ei.seq];
        return si >= 0 && si < max_slots;
    };
    auto next_item = [&](int it) {
        while (it < n_items && !item_ok(it)) it += (int)gridDim.x;
        return it;
    };
    // With the gate projection fused (fused != 0) an item's z = W_fb,h f is one tcgen05 product at
    // the item's start, in place of the z rows: the head's W_fb rows (128 x 128) arrive in the
    // gate array (only the gate threads write it, after the product) and the chunk's f rows
    // (64 x 128) past the q, k, v rows of the staging region, both as 128-byte-swizzled TMA boxes
    // with the item's other inputs; the product (lane = channel, column = row) lands in TMEM
    // columns 160..223, where the gate threads read it in FP32.
    unsigned char *sFb = reinterpret_cast<unsigned char *>(GL);        // [2 k halves][128 rows][128 B]
    unsigned char *sF = Y + 54272;                                      // [2 k halves][64 rows][128 B]
    constexpr uint32_t kZCol = 160;
    static_assert(2 * kD * 128 <= kC * kYS * 4 && 54272 >= 3 * (kC + 6) * kD * 2 && 54272 % 1024 == 0 &&
                  54272 + 2 * kC * 128 <= kPtY && (4 * kC * kYS * 4 - kC * kYS * 4) % 1024 == 0,
                  "z operands fit and are 1024-byte aligned");

    // 0. (one thread) an item's inputs, counted on bars[0]: one 2-D box of box_rows rows (x = the
    //    head's 128 channels) per stream, from 3 rows before the chunk, or, for a sequence's
    //    first chunk (and for z), from its first row, with the 3 history rows then taken from
    //    the conv tail. Rows past the chunk are whatever follows in the tensor (or zero past its
    //    end): every value computed from them is masked.
    auto stage = [&](int it) {
        const int ci = it / H, hi = it - ci * H;
        const ChunkEntry ei = table[ci];
        const bool first = ei.pos0 == 0;
        mbar_arrive_expect_tx(bars, (uint32_t)(((fused ? 3 : 4) * box_rows + (first ? 9 : 0)) * kD * sizeof(T)) +
                                        (fused ? (uint32_t)(2 * (kD + f_rows) * 128) : 0u));
        const int hx = hi * kD;
        const int ylo = first ? ei.t0 : ei.t0 - 3, jlo = first ? 3 : 0;
        tma_load_2d(raw + (size_t)(0 * kRows + jlo) * kD, &tm_q, hx, ylo, bars);
        tma_load_2d(raw + (size_t)(1 * kRows + jlo) * kD, &tm_k, hx, ylo, bars);
        tma_load_2d(raw + (size_t)(2 * kRows + jlo) * kD, &tm_v, hx, ylo, bars);
        if (fused) {  // the z operands instead of the z rows
            tma_load_2d(sFb, &tm_fb, 0, hi * kD, bars);
            tma_load_2d(sFb + kD * 128, &tm_fb, 64, hi * kD, bars);
            tma_load_2d(sF, &tm_f, 0, ei.t0, bars);
            tma_load_2d(sF + kC * 128, &tm_f, 64, ei.t0, bars);
        } else {
            tma_load_2d(raw + (size_t)(3 * kRows + 3) * kD, &tm_z, hx, ei.t0, bars);
        }
        if (first) {
            const T *tl0 = tail_all + (size_t)slots[ei.seq] * 3 * (kK - 1) * D + (size_t)hi * kD;
            for (int x = 0; x < 3; ++x)
                for (int j = 0; j < 3; ++j)
                    bulk_g2s(raw + (size_t)(x * kRows + j) * kD, tl0 + (size_t)(x * 3 + j) * D, kD * sizeof(T), bars);
        }
    };

    if (warp == 0) tc::tmem_alloc(tslot, 512);
    int it = next_item((int)blockIdx.x);
    bool staged = false;    // (thread 32) z operand copies in flight, completing phase staged_ph
    uint32_t staged_ph = 0;
    bool zmma_out = false;  // (thread 32) a z product in flight, completing phase zmma_ph
    uint32_t zmma_ph = 0;
    if (tid == 32) {
        for (int i = 0; i < 5; ++i) mbar_init(bars + i, 1);
        fence_mbar_init();
        if (it < n_items) {
            stage(it);
            staged = true;
        }
    }
    tc::fence_before_sync();
    __syncthreads();  // barrier init and TMEM base visible
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    // 8. an item's W and U' from TMEM to its chunk block, by ng groups of four warps (gi = this
    //    warp's group): W (lanes 0..63, columns 256..383) as BF16 16-byte chunks by the warps on
    //    lane quarters 0 and 1, U' (lanes 0..127, columns 384..447) as coalesced FP32 stores.
    //    They stay in TMEM until the next item's W/U' MMAs, so each item's are written while the
    //    next item solves for T, by warps that the solve leaves idle.
    auto write_wu = [&](unsigned char *b, int gi, int ng) {
        const int qd = warp & 3;
        if (qd < 2) {
            const int r = 32 * qd + lane;
            for (int c32 = 0; c32 < 4 / ng; ++c32) {
                const int col = (kD / ng) * gi + 32 * c32;
                uint32_t wv[32];
                tc::tmem_ld32_nowait(tb + ((uint32_t)(32 * qd) << 16) + 256 + col, wv);
                tc::tmem_wait_ld();
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float o[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) o[t] = __uint_as_float(wv[8 * g8 + t]);
                    uint4 hi, lo;
                    split8(o, hi, lo);
                    st16(b + kOffTA + tc::kmajor_off(r, col + 8 * g8, kD), hi);
                    st16(b + kOffTA + tc::kmajor_off(2 * kC + r, col + 8 * g8, kD), lo);
                }
            }
        }
        for (int c16 = 0; c16 < 4 / ng; ++c16) {
            const int col = (kC / ng) * gi + 16 * c16;
            float uv[16];
            tc::tmem_ld16(tb + ((uint32_t)(32 * qd) << 16) + 384 + col, uv);
            float *Up = reinterpret_cast<float *>(b + kOffUp) + 32 * qd + lane;
#pragma unroll
            for (int t = 0; t < 16; ++t) Up[(col + t) * kD] = uv[t];
        }
    };
    // 8b. an item's P (inclusive mask) from the A/P accumulator (lanes 64..127, the q rows) to its
    //     chunk block as BF16 hi and lo parts, by the write-out warps on lane quarters 2 and 3:
    //     warp w reads block R = 2 (w % 2) + (w / 4) % 2's segment, used by lanes 16 ((w / 4) % 2) .. +15
    auto write_p = [&](unsigned char *b) {
        const int qd = warp & 3, half = (warp >> 2) & 1, R = 2 * (qd & 1) + half, oR = 8 * R * (R + 1);
        uint32_t a0[32], a1[32];
        const uint32_t ta = tb + ((uint32_t)(32 * qd) << 16) + oR;
        tc::tmem_ld32_nowait(ta, a0);
        tc::tmem_ld32_nowait(ta + 32, a1);
        tc::tmem_wait_ld();
        if ((lane >> 4) == half) {
            const int r = 32 * (qd - 2) + lane;
#pragma unroll
            for (int g8 = 0; g8 < kC / 8; ++g8) {
                float o[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const int i = 8 * g8 + t;
                    const float pv = __uint_as_float(i < 32 ? a0[i] : a1[i - 32]);
                    o[t] = i <= r ? pv : 0.f;
                }
                uint4 hi, lo;
                split8(o, hi, lo);
                st16(b + kOffTB + tc::kmajor_off(r, 8 * g8, kC), hi);
                st16(b + kOffTB + tc::kmajor_off(3 * kC + r, 8 * g8, kC), lo);
            }
        }
    };
    bool good = true;
    bool aborted = false;
    unsigned char *blk_prev = nullptr;  // the previous item's block: its W and U' are still in TMEM
    uint32_t done = 0;    // items processed: the phase parity of bars[0] and bars[3]
    for (; it < n_items; ++done) {
        const int chunk = it / H, h = it - chunk * H;
        const int n = table[chunk].n;
        const int nxt = next_item(it + (int)gridDim.x);
        // the next item's boxes go to L2 now; its copies start once this item's operand tiles
        // have been consumed
        if (tid == 256 && nxt < n_items) {
            const int c2 = nxt / H, h2 = nxt - c2 * H;
            const ChunkEntry e2 = table[c2];
            const int y2 = e2.pos0 == 0 ? e2.t0 : e2.t0 - 3;
            tma_prefetch_2d(&tm_q, h2 * kD, y2);
            tma_prefetch_2d(&tm_k, h2 * kD, y2);
            tma_prefetch_2d(&tm_v, h2 * kD, y2);
            if (fused) {
                tma_prefetch_2d(&tm_f, 0, e2.t0);
                tma_prefetch_2d(&tm_f, 64, e2.t0);
                tma_prefetch_2d(&tm_fb, 0, h2 * kD);
                tma_prefetch_2d(&tm_fb, 64, h2 * kD);
            } else {
                tma_prefetch_2d(&tm_z, h2 * kD, e2.t0);
            }
        }
        const int t0 = table[chunk].t0;
        unsigned short braw = 0;
        if (tid < kC && tid < n) braw = ld_nc_u16(bl + (size_t)(t0 + tid) * H + h);
        // this thread's per-channel parameters
        const int pc = tid & (kD - 1), px = tid >> 7;  // channel, stream (q, k, v, or the gate)
        // (conv threads, px < 3: channels 2 cp, 2 cp + 1 of stream px, output rows 32 rh .. +31)
        const int cp = tid & 63, rh = (tid >> 6) & 1;
        float4 p_w0 = make_float4(0.f, 0.f, 0.f, 0.f), p_w1 = p_w0;
        if (px < 3) {
            const float4 *wb = reinterpret_cast<const float4 *>(conv_w + ((size_t)px * D + (size_t)h * kD + 2 * cp) * kK);
            p_w0 = __ldg(wb);
            p_w1 = __ldg(wb + 1);
        }
        const float p_dt = __ldg(dt_bias + (size_t)h * kD + pc);
        const float p_eA = expf(__ldg(A_log + h));
        // the gate in base 2: exp(-eA (z + dt)) = 2^(p_eA2 (z + dt)) (the cap 115 ~ 80 log2(e):
        // the sigmoid is then below 2e-35), and G log2(e) accumulates gk log2(e) = gmin2 sg
        const float p_eA2 = -p_eA * 1.4426950408889634f, gmin2 = gmin * 1.4426950408889634f;
        {
            const bool ok = mbar_wait_bounded(bars, done & 1u, kTcWaitLimit);
            good &= ok;
            if (ok && tid == 32) staged = false;
        }
        if (fused && tid == 32 && good) {  // z = W_fb,h f for this item's rows (8 K steps of 16)
            {
                tc::fence_after_sync();
                const uint32_t idz = tc::idesc_bf16(128, kC);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ko = (uint32_t)(kk & 3) * 32;
                    tc::mma_bf16(tb + kZCol, tc::sw128_desc(smem_u32(sFb + (kk >> 2) * kD * 128) + ko),
                                 tc::sw128_desc(smem_u32(sF + (kk >> 2) * kC * 128) + ko), idz, kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(bars + 4);
                zmma_out = true;
                zmma_ph = done & 1u;
            }
        }
        if (tid < kC) sbeta[tid] = tid < n ? sigmoidf_(__bfloat162float(__ushort_as_bfloat16(braw))) : 0.f;

        // 1. conv + SiLU (sliding window in registers) for stream px < 3, two channels and 32 rows a
        //    thread, 2. the gates for px == 3, one channel and all 64 rows a thread. The gate's
        //    exponent is capped at 80 (the sigmoid is then below 2e-35).
        if (px < 3) {
            // Yq, Yk, Yv are consecutive: the stores stay shared
            float *dst = Yq + px * (kC * kYS) + (32 * rh) * kYS + 2 * cp;
            const __nv_bfloat16 *col = reinterpret_cast<const __nv_bfloat16 *>(raw) + (size_t)(px * kRows + 32 * rh) * kD + 2 * cp;
            if (n == kC) conv_silu_pair32<true>(col, p_w0, p_w1, dst, kC);
            else conv_silu_pair32<false>(col, p_w0, p_w1, dst, n - 32 * rh);
        } else {
            // the gate thread of channel pc also carries G_r = sum_{t<=r} gk_t down the rows (gk = 0,
            // no decay, past the chunk, so G stays at G_last there); z from TMEM (fused) or the
            // staged rows
            if (fused) {
                good &= mbar_wait_bounded(bars + 4, done & 1u, kTcWaitLimit);
                tc::fence_after_sync();
            }
            const T *col = raw + ((size_t)3 * kRows + 3) * kD + pc;
            float acc = 0.f;
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {  // 32 rows at a time
                float zz[32];
                if (fused) {
                    uint32_t zr[32];
                    tc::tmem_ld32_nowait(tb + ((uint32_t)(32 * (warp & 3)) << 16) + kZCol + 32 * hb, zr);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) zz[j] = __uint_as_float(zr[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) zz[j] = IO<T>::ld(col + (32 * hb + j) * kD);
                }
                // (fused: the product has completed, so the array that held W_fb takes G)
                if (n == kC) {  // a full chunk: no row mask
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float sg = rcp_ftz(1.0f + ex2_ftz(fminf(p_eA2 * (zz[j] + p_dt), 115.f)));
                        acc += gmin2 * sg;
                        GL[(32 * hb + j) * kYS + pc] = acc;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int r = 32 * hb + j;
                        const float sg = rcp_ftz(1.0f + ex2_ftz(fminf(p_eA2 * (zz[j] + p_dt), 115.f)));
                        acc += r < n ? gmin2 * sg : 0.f;
                        GL[r * kYS + pc] = acc;
                    }
                }
            }
        }
        __syncthreads();
        // 2b. the L2 norms of q and k: warp w takes rows 4 w .. 4 w + 3, 8 lanes a row, lane j of a
        //     row the channels 4 j + 32 i (i < 4), so each quarter warp reads 128 contiguous bytes
        {
            const int r = 4 * warp + (lane >> 3), j = lane & 7;
            float4 *qr = reinterpret_cast<float4 *>(Yq + r * kYS) + j, *kr = reinterpret_cast<float4 *>(Yk + r * kYS) + j;
            float4 a[4], b[4];
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = qr[8 * i];
                b[i] = kr[8 * i];
                sq += a[i].x * a[i].x + a[i].y * a[i].y + a[i].z * a[i].z + a[i].w * a[i].w;
                sk += b[i].x * b[i].x + b[i].y * b[i].y + b[i].z * b[i].z + b[i].w * b[i].w;
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
                sk += __shfl_xor_sync(0xFFFFFFFFu, sk, o);
            }
            const float rq = q_scale * rsqrt_ftz(sq + l2_eps), rk = rsqrt_ftz(sk + l2_eps);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                qr[8 * i] = make_float4(a[i].x * rq, a[i].y * rq, a[i].z * rq, a[i].w * rq);
                kr[8 * i] = make_float4(b[i].x * rk, b[i].y * rk, b[i].z * rk, b[i].w * rk);
            }
        }
        __syncthreads();

        // blocks are head-major (block of chunk c, head h at h * total_chunks + c), so one head's
        // consecutive chunks are adjacent for the state pass
        unsigned char *blk = chunks + ((size_t)h * (unsigned)(n_items / H) + chunk) * kTcChunkBytes;
        // 3. A and P on the tensor core: the four 16-row blocks share one accumulator of 160 TMEM
        //    columns (lane = left row, column = right row; only each block's own segment is used),
        //    built and multiplied one half of the channels at a time by all 16 warps. While the
        //    MMAs of half 0 run, the CTA writes Q o exp(G) to the chunk block; while those of half 1
        //    run, (K o exp(G_last - G))^T and exp(G_last) (G is constant past the chunk, so row 63
        //    holds G_last).
        unsigned char *tLh = Y + kApLh, *tLl = Y + kApLl, *tRh = Y + kApRh, *tRl = Y + kApRl;
        for (int half = 0; half < 2; ++half) {
            const int c_h = half * (kD / 2);
            if (half) {
                good &= mbar_wait_bounded(bars + 1, 0u, kTcWaitLimit);  // half 0 has read the tiles
                tc::fence_after_sync();
            }
            // item (row r, 8-channel group): k_r, q_r and G_r are read once; the item writes the left
            // rows r (k) and 64 + r (q) with factor exp(G_r - G_n), n = 16 (r / 16), and row r of every
            // right segment R >= r / 16: k_r o exp(G_16R - G_r) (<= 1 for R > r / 16, <= e^75 on the
            // diagonal block)
            {
                const int u = tid;  // 512 items, one per thread
                const int r = (u & 7) | ((u >> 6) << 3), cl = 8 * ((u >> 3) & 7), c0 = c_h + cl;
                const int b = r >> 4;
                float kv[8], qv[8], gr[8], gn[8], kl[8], ql[8];
                ld8f(Yk + r * kYS + c0, kv);
                ld8f(Yq + r * kYS + c0, qv);
                ld8f(GL + r * kYS + c0, gr);
                ld8f(GL + kBlk * b * kYS + c0, gn);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float f = ex2_ftz(gr[j] - gn[j]);
                    kl[j] = kv[j] * f;
                    ql[j] = qv[j] * f;
                }
                uint4 hi, lo;
                split8(kl, hi, lo);
                st16(tLh + tc::kmajor_off(r, cl, kD / 2), hi);
                st16(tLl + tc::kmajor_off(r, cl, kD / 2), lo);
                split8(ql, hi, lo);
                st16(tLh + tc::kmajor_off(kC + r, cl, kD / 2), hi);
                st16(tLl + tc::kmajor_off(kC + r, cl, kD / 2), lo);
                // block 0's rows have four segments and block 3's one: block 0's last segment (R = 3)
                // is built by the block-3 threads, each for the block-0 row 48 rows above its own
                const int R_end = b == 0 ? kC / kBlk - 1 : kC / kBlk;
                for (int R = b; R < R_end; ++R) {  // warp-uniform: a warp's 8 rows share a block
                    if (R != b) ld8f(GL + kBlk * R * kYS + c0, gn);
                    float kx[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) kx[j] = kv[j] * ex2_ftz(gn[j] - gr[j]);
                    split8(kx, hi, lo);
                    const int row = 8 * R * (R + 1) + r;
                    st16(tRh + tc::kmajor_off(row, cl, kD / 2), hi);
                    st16(tRl + tc::kmajor_off(row, cl, kD / 2), lo);
                }
                if (b == kC / kBlk - 1) {  // gn holds G_48 here
                    const int r0 = r - kBlk * (kC / kBlk - 1);
                    float k0[8], g0[8], kx[8];
                    ld8f(Yk + r0 * kYS + c0, k0);
                    ld8f(GL + r0 * kYS + c0, g0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) kx[j] = k0[j] * ex2_ftz(gn[j] - g0[j]);
                    split8(kx, hi, lo);
                    const int row = 8 * (kC / kBlk - 1) * (kC / kBlk) + r0;
                    st16(tRh + tc::kmajor_off(row, cl, kD / 2), hi);
                    st16(tRl + tc::kmajor_off(row, cl, kD / 2), lo);
                }
            }
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            // (issued by a thread of warp 12, whose rows have the fewest right segments, so that the
            // issue time does not lengthen the most loaded warps' shadow work)
            if (tid == 384) {
                mma_split3(tb, tc::kmajor_desc(tLh, 0, kD / 2), tc::kmajor_desc(tLl, 0, kD / 2),
                           tc::kmajor_desc(tRh, 0, kD / 2), tc::kmajor_desc(tRl, 0, kD / 2), tc::idesc_bf16(128, kApN),
                           kD / 2 / 16, half != 0);
                tc::mma_commit(bars + 1);
            }
            {
                // (K o exp(G_last - G))^T hi and lo: items u in [u0, u1) (channel c, rows 8 rb .. +7)
                auto kdt = [&](int u0, int u1) {
                    for (int u = u0 + tid; u < u1; u += 512) {
                        const int c = u & (kD - 1), rb = u >> 7;
                        const float gl = GL[(kC - 1) * kYS + c];
                        float o[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int r = 8 * rb + j;
                            o[j] = Yk[r * kYS + c] * ex2_ftz(gl - GL[r * kYS + c]);
                        }
                        uint4 hi, lo;
                        split8(o, hi, lo);
                        st16(blk + kOffTB + tc::kmajor_off(kC + c, 8 * rb, kC), hi);
                        st16(blk + kOffTB + tc::kmajor_off(4 * kC + c, 8 * rb, kC), lo);
                    }
                };
                if (half == 0) {
                for (int u = tid; u < kC * (kD / 8); u += 512) {
                    const int r = (u & 7) | ((u >> 7) << 3), c0 = 8 * ((u >> 3) & 15);
                    float qv[8], gr[8], o[8];
                    ld8f(Yq + r * kYS + c0, qv);
                    ld8f(GL + r * kYS + c0, gr);
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = qv[j] * ex2_ftz(gr[j]);
                    st16(blk + kOffTA + tc::kmajor_off(kC + r, c0, kD), pack8_bf16(o));
                }
                    kdt(0, 512);
                } else {
                    kdt(512, 1024);
                    if (tid < kD) reinterpret_cast<float *>(blk + kOffGam)[tid] = ex2_ftz(GL[(kC - 1) * kYS + tid]);
                }
            }
        }
        good &= mbar_wait_bounded(bars + 1, 1u, kTcWaitLimit);  // second completion: half 1
        tc::fence_before_sync();
        if (__syncthreads_or(!good) && tid == 0) atomicExch(err, KDA_ERR_TIMEOUT);
        tc::fence_after_sync();

        // 5. warps 0, 1, 4 and 5 read A back (beta and the strict mask applied) to the FP32 matrix M
        //    (P stays in TMEM until the write-out warps take it, step 8b). Then warps 2, 3 and 6..15
        //    build the solve operands: rows 0..127 (beta K o exp(G))^T, rows 128..255 (beta V)^T,
        //    K = the 64 chunk rows, hi parts in the q^ array (free now), lo parts in the region.
        float *Mm = reinterpret_cast<float *>(Y + kPtM), *TD = reinterpret_cast<float *>(Y + kPtD);
        unsigned char *tBh = reinterpret_cast<unsigned char *>(Yq), *tBl = Y + kPtBl, *tT = Y + kPtT;
        if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {
            // lane quarter qd < 2 holds the k rows 32 qd .. +31; this warp reads block R's
            // segment, used by lanes 16 half .. +15 (P, on lane quarters 2 and 3, is written out
            // later by the write-out warps, step 8b)
            const int qd = warp & 3, half = warp >> 2, R = 2 * (qd & 1) + half, oR = 8 * R * (R + 1);
            uint32_t a0[32], a1[32];
            const uint32_t ta = tb + ((uint32_t)(32 * qd) << 16) + oR;
            tc::tmem_ld32_nowait(ta, a0);
            tc::tmem_ld32_nowait(ta + 32, a1);
            tc::tmem_wait_ld();
            // columns past the segment belong to other blocks; the mask (i < r) drops them
            if ((lane >> 4) == half) {
                const int r = 32 * qd + lane;
                const float bt = sbeta[r];
#pragma unroll
                for (int i4 = 0; i4 < kC / 4; ++i4) {
                    float o[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int i = 4 * i4 + t;
                        const float a = __uint_as_float(i < 32 ? a0[i] : a1[i - 32]);
                        o[t] = i < r ? bt * a : 0.f;
                    }
                    reinterpret_cast<float4 *>(Mm + r * kMS)[i4] = make_float4(o[0], o[1], o[2], o[3]);
                }
            }
        }
        // 6a. The diagonal blocks TD of T = (I + A)^-1, T_RR = (I + A_RR)^-1, by forward substitution
        //     (threads 0..63, one column each) as soon as the A rows are in M (warps 0, 1, 4 and 5
        //     read A back: a named barrier over those four), while the other warps write the zero
        //     blocks of the T tile above the diagonal (columns c >= 16 (r / 16 + 1)) and build the B
        //     operand.
        if (warp == 0 || warp == 1 || warp == 4 || warp == 5) named_bar_sync(3, 128);
        if (tid < kC) {
            const int R = tid >> 4, j = tid & (kBlk - 1), nR = kBlk * R;
            float x[kBlk];
#pragma unroll
            for (int r = 0; r < kBlk; ++r) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i) {
                    if (i & 1) s1 = fmaf(-Mm[(nR + r) * kMS + nR + i], x[i], s1);
                    else s0 = fmaf(-Mm[(nR + r) * kMS + nR + i], x[i], s0);
                }
                x[r] = r == j ? 1.f : (r < j ? 0.f : s0 + s1);
            }
            // stored after the loop, so that no shared store sits between the loads of the rows
#pragma unroll
            for (int r = 0; r < kBlk; ++r) TD[(nR + r) * kTD + j] = x[r];
        } else if (tid < 256) {
            const int u = tid - kC;  // 192 groups of 8 columns, hi and lo parts
            const int r = u < 96 ? u / 6 : (u < 160 ? kBlk + (u - 96) / 4 : 2 * kBlk + (u - 160) / 2);
            const int g = u < 96 ? 2 + u % 6 : (u < 160 ? 4 + (u - 96) % 4 : 6 + (u - 160) % 2);
            st16(tT + tc::kmajor_off(r, 8 * g, kC), make_uint4(0u, 0u, 0u, 0u));
            st16(tT + tc::kmajor_off(kC + r, 8 * g, kC), make_uint4(0u, 0u, 0u, 0u));
        }
        if (tid >= kC && (warp < 4 || warp >= 6)) {  // warps 2, 3 (after the zero blocks) and 6..15 build B
            for (int u = warp < 4 ? tid - kC : tid - 2 * kC; u < 256 * (kC / 8); u += 512 - 2 * kC) {
                const int nn = u & 255, i0 = 8 * (u >> 8);
                float o[8], bt[8];
                ld8f(sbeta + i0, bt);
                if (nn < kD) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        o[j] = bt[j] * (Yk[(i0 + j) * kYS + nn] * ex2_ftz(GL[(i0 + j) * kYS + nn]));
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = bt[j] * Yv[(i0 + j) * kYS + nn - kD];
                }
                uint4 hi, lo;
                split8(o, hi, lo);
                st16(tBh + tc::kmajor_off(nn, i0, kC), hi);
                st16(tBl + tc::kmajor_off(nn, i0, kC), lo);
            }
        }
        __syncthreads();
        if (warp >= 8) {
            tc::fence_after_sync();
            __nanosleep(300);  // let the merge's first shared-memory loads go ahead of the write-out's stores
            if (blk_prev) write_wu(blk_prev, (warp >> 2) - 2, 2);
            if ((warp & 3) >= 2) write_p(blk);  // this item's P
        } else {
            // 6b. T = (I + A)^-1 as BF16 hi and lo parts in the T tile, by blocks of 16 and a two-level
            //    merge, by warps 0..7 (a 256-thread named barrier between phases), from the diagonal
            //    blocks TD of 6a. With X = rows/columns 0..31 and Y = 32..63,
            //    T_YX = -T_YY A_YX T_XX, and inside each half T_10 = -T_11 A_10 T_00,
            //    T_32 = -T_33 A_32 T_22. Three phases:
            //      1. Y1_p = A_(2p+1)(2p) T_(2p)(2p) (p = 0, 1), Z0 = A_Y0 T_00, Z1 = A_Y1 T_11;
            //      2. T_10 = -T_11 Y1_0, T_32 = -T_33 Y1_1 (also kept in FP32), and Y2 = A_YX T_XX,
            //         whose left half is Z0 + A_Y1 T_10 = Z0 - Z1 Y1_0 and whose right half is Z1;
            //         and the diagonal blocks to the tile;
            //      3. T_YX = -T_YY Y2.
            //    Each product is tiled 2 x 4 per thread (rows 2 rp, 2 rp + 1; columns 4 ct .. 4 ct + 3);
            //    the 8 lanes of a quarter warp share their rows and take consecutive column tiles.
            float *T32 = Yv, *Y1 = GL, *Y2 = GL + 2 * kBlk * kBlk;  // T32: [16][kMS], Y1: [2][16][16], Y2: [32][kY2]
            constexpr int kY2 = 36;
            // (phase 0, the diagonal blocks, ran before the barrier)
            // phase 1 (threads 0..191)
            if (tid < 64) {
                const int p = tid >> 5, rp = (tid >> 2) & 7, ct = tid & 3, o = 2 * kBlk * p;
                float c[2][4] = {};
                tile24<kBlk / 4>(c, Mm + (o + kBlk + 2 * rp) * kMS + o, kMS, TD + o * kTD + 4 * ct, kTD);
                put24(Y1 + p * kBlk * kBlk + 2 * rp * kBlk + 4 * ct, kBlk, c, 1.f);
            } else if (tid < 192) {
                const int t = tid - 64, rp = t >> 3, ct = t & 7, o = kBlk * (ct >> 2);
                float c[2][4] = {};
                tile24<kBlk / 4>(c, Mm + (2 * kBlk + 2 * rp) * kMS + o, kMS, TD + o * kTD + 4 * (ct & 3), kTD);
                put24(Y2 + 2 * rp * kY2 + 4 * ct, kY2, c, 1.f);
            }
            named_bar_sync(1, 256);
            // phase 2; each thread overwrites only its own tile of Z0
            if (tid < 64) {
                const int p = tid >> 5, rp = (tid >> 2) & 7, ct = tid & 3, o = 2 * kBlk * p;
                float c[2][4] = {};
                tile24<kBlk / 4>(c, TD + (o + kBlk + 2 * rp) * kTD, kTD, Y1 + p * kBlk * kBlk + 4 * ct, kBlk);
                put24_split(tT, o + kBlk + 2 * rp, o + 4 * ct, c, -1.f);
                if (p) put24(T32 + 2 * rp * kMS + 4 * ct, kMS, c, -1.f);
            } else if (tid < 128) {
                const int t = tid - 64, rp = t >> 2, ct = t & 3;
                float c[2][4];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float4 z = *reinterpret_cast<const float4 *>(Y2 + (2 * rp + i) * kY2 + 4 * ct);
                    c[i][0] = -z.x; c[i][1] = -z.y; c[i][2] = -z.z; c[i][3] = -z.w;
                }
                tile24<kBlk / 4>(c, Y2 + 2 * rp * kY2 + kBlk, kY2, Y1 + 4 * ct, kBlk);
                put24(Y2 + 2 * rp * kY2 + 4 * ct, kY2, c, -1.f);
            } else {
                const int t = tid - 128, R = t >> 5, r = kBlk * R + ((t >> 1) & (kBlk - 1)), g = t & 1;
                float tv[8];
                ld8f(TD + r * kTD + 8 * g, tv);
                uint4 hi, lo;
                split8(tv, hi, lo);
                st16(tT + tc::kmajor_off(r, kBlk * R + 8 * g, kC), hi);
                st16(tT + tc::kmajor_off(kC + r, kBlk * R + 8 * g, kC), lo);
            }
            named_bar_sync(1, 256);
            // phase 3 (threads 0..127): rows 32 + 2 rp (+1); T_YY's rows are [T_22 0] for warps 0, 1
            // and [T_32 T_33] for warps 2, 3
            if (tid < 128) {
                const int rp = tid >> 3, ct = tid & 7;
                float c[2][4] = {};
                if (warp < 2) {
                    tile24<kBlk / 4>(c, TD + (2 * kBlk + 2 * rp) * kTD, kTD, Y2 + 4 * ct, kY2);
                } else {
                    tile24<kBlk / 4>(c, T32 + (2 * rp - kBlk) * kMS, kMS, Y2 + 4 * ct, kY2);
                    tile24<kBlk / 4>(c, TD + (2 * kBlk + 2 * rp) * kTD, kTD, Y2 + kBlk * kY2 + 4 * ct, kY2);
                }
                put24_split(tT, 2 * kBlk + 2 * rp, 4 * ct, c, -1.f);
            }
        }
        tc::fence_smem_to_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // 7. W (rows r = lanes 0..63, 128 channel columns at TMEM 256..383) = T B_K^T, and
        //    U'^T (rows v = lanes 0..127, 64 row columns at TMEM 384..447) = B_V T^T
        if (tid == 0) {
            const uint64_t dT = tc::kmajor_desc(tT, 0, kC), dTlo = dT + ((kC / 8) * kC * 16 >> 4);
            const uint64_t dBh = tc::kmajor_desc(tBh, 0, kC), dBl = tc::kmajor_desc(tBl, 0, kC);
            const uint64_t vOff = (uint64_t)((kD / 8) * kC * 16 >> 4);  // B rows 128.. = (beta V)^T
            mma_split3(tb + 256, dT, dTlo, dBh, dBl, tc::idesc_bf16(128, kD), kC / 16, false);
            mma_split3(tb + 384, dBh + vOff, dBl + vOff, dT, dTlo, tc::idesc_bf16(128, kC), kC / 16, false);
            tc::mma_commit(bars + 3);
        }
        good = __all_sync(0xFFFFFFFFu, good && mbar_wait_bounded(bars + 3, done & 1u, kTcWaitLimit));  // warp-uniform
        tc::fence_after_sync();
        blk_prev = blk;
        tc::fence_before_sync();
        const bool bad = __syncthreads_or(!good);
        tc::fence_after_sync();
        if (bad) {
            if (tid == 0) atomicExch(err, KDA_ERR_TIMEOUT);
            aborted = true;
            break;
        }
        // the operand tiles are consumed: the next item's inputs may land in the reused region
        // (issued past the barrier, so that no other thread waits for the copies' issue)
        if (tid == 32 && nxt < n_items) {
            tc::fence_smem_to_async();
            stage(nxt);
            staged = true;
            staged_ph = (done + 1) & 1u;
        }
        it = nxt;
    }
    // after an abort a z operand copy or product may still be in flight: wait for it (bounded)
    if (staged) mbar_wait_bounded(bars, staged_ph, kTcWaitLimit);
    if (zmma_out && !aborted) zmma_out = false;
    if (zmma_out) mbar_wait_bounded(bars + 4, zmma_ph, kTcWaitLimit);
    if (!aborted && blk_prev) write_wu(blk_prev, warp >> 2, 4);  // the last item's W and U'
    if (warp == 0) tc::tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- state pass
template <typename T>
__global__ void __launch_bounds__(256, 1)
state_kernel(float *__restrict__ S_all, T *__restrict__ tail_all, int32_t *__restrict__ err,
             const int32_t *__restrict__ slots, int H, int max_slots,
             const ChunkEntry *__restrict__ table, const int32_t *__restrict__ seq_first,
             const float *__restrict__ chunks, float *__restrict__ obuf,
             const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v)
{
    extern __shared__ __align__(16) float sm[];
    float *Ss = sm;                 // [d][32]  state columns of this block
    float *Wc = Ss + kD * kVB;      // [C][d]
    float *QGc = Wc + kC * kD;      // [C][d]
    float *KDc = QGc + kC * kD;     // [C][d]
    float *Upc = KDc + kC * kD;     // [C][32]
    float *Uc = Upc + kC * kVB;     // [C][32]
    float *Pc = Uc + kC * kVB;      // [C][C]
    float *GCc = Pc + kC * kC;      // [d]

    const int vb = blockIdx.x, h = blockIdx.y, seq = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = slots[seq];
    if (slot < 0 || slot >= max_slots) {
        if (tid == 0) atomicExch(err, kErrBadSlot);
        return;
    }
    const size_t D = (size_t)H * kD;
    float *Sg = S_all + ((size_t)slot * H + h) * kD * kD + vb * kVB;

    const int c_first = seq_first[seq], c_last = seq_first[seq + 1];

    // new conv history (the last K-1 raw inputs), written by the vb == 0 CTA;
    // the sequence's extent comes from its (validated) chunk list
    if (vb == 0 && tid < kD && c_last > c_first) {
        const int start = table[c_first].t0;
        const int len = table[c_last - 1].t0 + table[c_last - 1].n - start;
        T *tl = tail_all + (size_t)slot * 3 * (kK - 1) * D + (size_t)h * kD + tid;
        const T *src[3] = {q, k, v};
#pragma unroll
        for (int x = 0; x < 3; ++x) {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int pos = len - 3 + j;
                const T val = pos >= 0 ? src[x][(size_t)(start + pos) * D + (size_t)h * kD + tid]
                                       : tl[(size_t)(x * 3 + (pos + 3)) * D];
                tl[(size_t)(x * 3 + j) * D] = val;
            }
        }
    }

    for (int e2 = tid; e2 < kD * kVB; e2 += 256) {
        const int c = e2 / kVB, j = e2 - c * kVB;
        Ss[e2] = Sg[(size_t)c * kD + j];
    }

    for (int ci = c_first; ci < c_last; ++ci) {
        const ChunkEntry e = table[ci];
        const float *src = chunks + ((size_t)ci * H + h) * kChunkFloats;
        __syncthreads();
        {
            const float4 *s4 = reinterpret_cast<const float4 *>(src);
            float4 *w4 = reinterpret_cast<float4 *>(Wc);
            float4 *qg4 = reinterpret_cast<float4 *>(QGc);
            float4 *kd4 = reinterpret_cast<float4 *>(KDc);
            for (int e2 = tid; e2 < kC * kD / 4; e2 += 256) {
                w4[e2] = s4[e2];
                qg4[e2] = s4[2 * kC * kD / 4 + e2];
                kd4[e2] = s4[3 * kC * kD / 4 + e2];
            }
            for (int e2 = tid; e2 < kC * kVB / 4; e2 += 256) {
                const int r = e2 / (kVB / 4), j4 = e2 - r * (kVB / 4);
                reinterpret_cast<float4 *>(Upc)[e2] = s4[kC * kD / 4 + r * (kD / 4) + vb * (kVB / 4) + j4];
            }
            for (int e2 = tid; e2 < kC * kC / 4; e2 += 256)
                reinterpret_cast<float4 *>(Pc)[e2] = s4[4 * kC * kD / 4 + e2];
            if (tid < kD / 4)
                reinterpret_cast<float4 *>(GCc)[tid] = s4[(4 * kC * kD + kC * kC) / 4 + tid];
        }
        __syncthreads();
        // U = U' - W S and the inter-chunk part of O = (Q o exp G) S; warp w owns rows 8w..8w+7.
        float accu[8], acco[8];
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) { accu[mm] = 0.f; acco[mm] = 0.f; }
        for (int c = 0; c < kD; c += 4) {
            const float s0 = Ss[(c + 0) * kVB + lane], s1 = Ss[(c + 1) * kVB + lane];
            const float s2 = Ss[(c + 2) * kVB + lane], s3 = Ss[(c + 3) * kVB + lane];
#pragma unroll
            for (int mm = 0; mm < 8; ++mm) {
                const int r = 8 * warp + mm;
                const float4 wv = *reinterpret_cast<const float4 *>(Wc + r * kD + c);
                const float4 qv = *reinterpret_cast<const float4 *>(QGc + r * kD + c);
                accu[mm] = fmaf(wv.x, s0, fmaf(wv.y, s1, fmaf(wv.z, s2, fmaf(wv.w, s3, accu[mm]))));
                acco[mm] = fmaf(qv.x, s0, fmaf(qv.y, s1, fmaf(qv.z, s2, fmaf(qv.w, s3, acco[mm]))));
            }
        }
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            const int r = 8 * warp + mm;
            Uc[r * kVB + lane] = Upc[r * kVB + lane] - accu[mm];
        }
        __syncthreads();
        // O += (P o M) U, written for the chunk's real rows
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            const int r = 8 * warp + mm;
            float o = acco[mm];
            for (int i = 0; i <= r; ++i) o = fmaf(Pc[r * kC + i], Uc[i * kVB + lane], o);
            if (r < e.n) obuf[((size_t)(e.t0 + r) * H + h) * kD + vb * kVB + lane] = o;
        }
        // S = Diag(gC) S + KD^T U; warp w owns state rows 16w..16w+15.
        float accs[16];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
            const int c = 16 * warp + cc;
            accs[cc] = GCc[c] * Ss[c * kVB + lane];
        }
        for (int r = 0; r < kC; ++r) {
            const float u = Uc[r * kVB + lane];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const float4 kd = *reinterpret_cast<const float4 *>(KDc + r * kD + 16 * warp + 4 * c4);
                accs[4 * c4 + 0] = fmaf(kd.x, u, accs[4 * c4 + 0]);
                accs[4 * c4 + 1] = fmaf(kd.y, u, accs[4 * c4 + 1]);
                accs[4 * c4 + 2] = fmaf(kd.z, u, accs[4 * c4 + 2]);
                accs[4 * c4 + 3] = fmaf(kd.w, u, accs[4 * c4 + 3]);
            }
        }
        __syncthreads();  // everyone is done reading Ss for this chunk
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) Ss[(16 * warp + cc) * kVB + lane] = accs[cc];
    }
    __syncthreads();
    for (int e2 = tid; e2 < kD * kVB; e2 += 256) {
        const int c = e2 / kVB, j = e2 - c * kVB;
        Sg[(size_t)c * kD + j] = Ss[e2];
    }
}

// ---------------------------------------------------------------- state pass on tensor cores
// One CTA per (sequence, head), warp-specialised, 416 threads. All A operands live in tensor
// memory (512 columns; lane v = value index v):
//   D1  = S^T W^T       [v][r]  columns   0.. 63  (S_hi W_hi + S_lo W_hi)
//   D2  = S^T QG^T      [v][r]  columns  64..127, then += U^T P^T  -> O^T
//   D1b = S_hi^T W_lo^T [v][r]  columns 128..191
//   S^T hi / lo parts   [v][k]  columns 192..255 / 256..319 (BF16 pairs, K = 128)
//   D3  = S^T           [v][k]  columns 320..447, the FP32 state (scaled by the chunk's decay
//                               before MMA2, += U^T KD)
//   U^T hi / lo parts   [v][r]  columns 448..479 / 480..511 (BF16 pairs, K = 64)
// The products that carry the state, and the output's U term (whose terms cancel when the
// keys are strongly correlated), are formed as hi*hi + lo*hi + hi*lo (about 16 bits of
// mantissa); the output's S term takes one BF16 pass:
//   MMA1: [D1 | D2 | D1b] = S_hi^T [W_hi | QG | W_lo]^T (N = 192), D1 += S_lo^T W_hi^T
//   MMA2: D3 += U_hi^T KDT_hi + U_lo^T KDT_hi + U_hi^T KDT_lo (committed: the state may be
//         read), then D2 += U_hi^T P_hi + U_lo^T P_hi + U_hi^T P_lo
// Roles (each hand-off is an mbarrier; every wait is bounded):
//   warps 0-7  (state): per chunk, U^T = U' - D1 - D1b as hi/lo parts (after MMA1), then after
//              the state products of MMA2 the S^T parts from D3 and the next chunk's decay put
//              on D3. Warps w and w + 4 share lane quarter w % 4 and split the columns in halves.
//   warp 8     (issuer, one lane): MMA1 once S^T is ready and D2 has been read out, MMA2 once
//              U^T is ready; the chunk-block copies (stage A after MMA1, stage B after MMA2),
//              the gate-row boxes and the L2 prefetches.
//   warps 9-12 (epilogue): O^T from D2 right after MMA2 (so MMA1 of the next chunk may start),
//              then the gated RMSNorm and the output box, under the next chunk's products.
// The serial chain per chunk is MMA1 -> U -> MMA2 (state part) -> refresh; the output product,
// the epilogue and the copies run beside it.
constexpr int kStThreads = 416;
constexpr uint32_t kTD1 = 0, kTD2 = 64, kTD1b = 128, kTSh = 192, kTSl = 256, kTD3 = 320, kTUh = 448, kTUl = 480;

// AND of pred over the `count` threads of named barrier `id` (also a barrier), so that every
// thread of a group takes the same branch after a bounded wait.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// 32 FP32 values of this thread's lane -> BF16 high parts (nearest) and low parts (x - high,
// nearest), two per 32-bit word (value 2c in the low half of word c), stored to 16 + 16
// tensor-memory columns starting at t_hi and t_lo (no wait).
__device__ __forceinline__ void tmem_put_split32(uint32_t t_hi, uint32_t t_lo, const float *x)
{
    uint32_t h[16], l[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(x[2 * c], x[2 * c + 1]);
        const uint32_t u = *reinterpret_cast<const uint32_t *>(&p);
        h[c] = u;
        const __nv_bfloat162 q = __floats2bfloat162_rn(x[2 * c] - __uint_as_float(u << 16),
                                                       x[2 * c + 1] - __uint_as_float(u & 0xFFFF0000u));
        l[c] = *reinterpret_cast<const uint32_t *>(&q);
    }
    tc::tmem_st16u_nowait(t_hi, h);
    tc::tmem_st16u_nowait(t_lo, l);
}

template <typename T>
__global__ void __launch_bounds__(kStThreads, 1)
state_tc_kernel(float *__restrict__ S_all, T *__restrict__ tail_all, int32_t *__restrict__ err,
                const int32_t *__restrict__ slots, int H, int max_slots,
                const ChunkEntry *__restrict__ table, const int32_t *__restrict__ seq_first,
                const unsigned char *__restrict__ chunks, int total_chunks,
                const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                const float *__restrict__ norm_w, T *__restrict__ out, float rms_eps, int box_rows,
                const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_out)
{
    static_assert(sizeof(T) == 2, "the tensor-core path reads BF16 gate logits");
    extern __shared__ __align__(1024) float smf[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(smf);
    unsigned char *sA = sm + kSmA, *sB = sm + kSmB;
    // exp(G_last) of chunk it in slot it % 2 (its own copy, so that stage A can be refilled
    // before the decay has been put on the state)
    const float *sgam2 = reinterpret_cast<const float *>(sm + kSmGam);
    __nv_bfloat16 *sGY = reinterpret_cast<__nv_bfloat16 *>(sm + kSmGY);  // gate rows, then output rows
    // [64 tokens][4 value quarters] partial sums of squares, added in a fixed order (so that the
    // outputs do not depend on the order the warps finish in)
    float *red = reinterpret_cast<float *>(sm + kSmRed);
    // [0] stage A landed, [1] stage B landed, [2] MMA1 done, [3] state products of MMA2 done,
    // [4] gate rows landed, [5] U^T ready (8 warps), [6] S^T ready (8 warps), [7] D2 read out
    // (4 warps), [8] output box read out of the gate/output buffer (1 thread), [9] MMA2 done
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kSmBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 12);

    const int h = blockIdx.x, seq = blockIdx.y;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int slot = slots[seq];
    if (slot < 0 || slot >= max_slots) {
        if (tid == 0) atomicExch(err, kErrBadSlot);
        return;
    }
    const size_t D = (size_t)H * kD;
    const int c_first = seq_first[seq], c_last = seq_first[seq + 1];
    const int n_chunks = c_last - c_first;
    float *Sg = S_all + ((size_t)slot * H + h) * kD * kD;
    auto block_of = [&](int ci) { return chunks + ((size_t)h * total_chunks + ci) * kTcChunkBytes; };

    if (w == 0) tc::tmem_alloc(tslot, 512);
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
        mbar_init(&bar[5], 8);
        mbar_init(&bar[6], 8);
        mbar_init(&bar[7], 4);
        mbar_init(&bar[8], 1);
        mbar_init(&bar[9], 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tb = *tslot;
    bool good = true;

    if (w < 8) {
        // ------------------------------------------------------------ state warps
        const int qtr = w & 3, grp = w >> 2;
        const int vi = 32 * qtr + lane;
        const uint32_t tl = tb + ((uint32_t)(32 * qtr) << 16);   // this warp's lane quarter
        const int k0 = 64 * grp, r0 = 32 * grp;
        float vals[32];
        // initial state: S[k][v] -> the S^T parts of row v and D3 row v (FP32, with the first
        // chunk's decay; stage A brings its gamma)
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            const int kb = k0 + 32 * half;
#pragma unroll
            for (int j = 0; j < 32; ++j) vals[j] = Sg[(size_t)(kb + j) * kD + vi];
            tmem_put_split32(tl + kTSh + kb / 2, tl + kTSl + kb / 2, vals);
            if (n_chunks > 0) {
                if (half == 0) good &= mbar_wait_bounded(&bar[0], 0, kTcWaitLimit);
#pragma unroll
                for (int j = 0; j < 32; ++j) vals[j] *= sgam2[kb + j];
            }
            tc::tmem_st32(tl + kTD3 + kb, vals);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[6]);  // S^T of the first chunk is ready
        for (int it = 0; it < n_chunks && good; ++it) {
            const int ci = c_first + it;
            const uint32_t par = (uint32_t)(it & 1);
            // U' of this thread's tokens (a warp reads 128 contiguous bytes per token)
            float up[32];
            {
                const float *Up = reinterpret_cast<const float *>(block_of(ci) + kOffUp) + vi;
#pragma unroll
                for (int j = 0; j < 32; ++j) up[j] = __ldcs(Up + (size_t)(r0 + j) * kD);
            }
            if (!(good = mbar_wait_bounded(&bar[2], par, kTcWaitLimit))) break;
            tc::fence_after_sync();
            {   // U^T = U'^T - (W S)^T on this thread's tokens, as BF16 high and low parts
                uint32_t a[32];
                tc::tmem_ld32_nowait(tl + kTD1 + r0, a);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) vals[j] = up[j] - __uint_as_float(a[j]);
                tc::tmem_ld32_nowait(tl + kTD1b + r0, a);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) vals[j] -= __uint_as_float(a[j]);
                tmem_put_split32(tl + kTUh + r0 / 2, tl + kTUl + r0 / 2, vals);
            }
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[5]);
            if (!(good = mbar_wait_bounded(&bar[3], par, kTcWaitLimit))) break;
            tc::fence_after_sync();
            // the S^T parts from the updated FP32 state, handed over first; then the next chunk's
            // decay put on D3 (MMA2 of the next chunk follows this warp's U^T hand-off, after its
            // wait on these stores); after the last chunk, the final state back to HBM
            const bool last = it + 1 == n_chunks;
            float v0[32], v1[32];
            {
                uint32_t raw[32];
                tc::tmem_ld32_nowait(tl + kTD3 + k0, raw);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) v0[j] = __uint_as_float(raw[j]);
                tc::tmem_ld32_nowait(tl + kTD3 + k0 + 32, raw);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) v1[j] = __uint_as_float(raw[j]);
            }
            if (last) {
#pragma unroll
                for (int j = 0; j < 32; ++j) Sg[(size_t)(k0 + j) * kD + vi] = v0[j];
#pragma unroll
                for (int j = 0; j < 32; ++j) Sg[(size_t)(k0 + 32 + j) * kD + vi] = v1[j];
                break;
            }
            tmem_put_split32(tl + kTSh + k0 / 2, tl + kTSl + k0 / 2, v0);
            tmem_put_split32(tl + kTSh + k0 / 2 + 16, tl + kTSl + k0 / 2 + 16, v1);
            // the next chunk's stage A (and its gamma) has landed: waited on before the hand-off,
            // since the issuer may refill stage A once the next MMA1 has run
            if (!(good = mbar_wait_bounded(&bar[0], (uint32_t)((it + 1) & 1), kTcWaitLimit))) break;
            tc::tmem_wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[6]);
            {
                const float *gam = sgam2 + ((it + 1) & 1) * kD + k0;
#pragma unroll
                for (int j = 0; j < 32; ++j) v0[j] *= gam[j];
#pragma unroll
                for (int j = 0; j < 32; ++j) v1[j] *= gam[32 + j];
                tc::tmem_st32(tl + kTD3 + k0, v0);
                tc::tmem_st32(tl + kTD3 + k0 + 32, v1);
            }
        }
        if (!good) atomicExch(err, KDA_ERR_TIMEOUT);
        // new conv history (the last K-1 raw inputs of the sequence)
        if (good && n_chunks > 0 && tid < kD) {
            const int start = table[c_first].t0;
            const int len = table[c_last - 1].t0 + table[c_last - 1].n - start;
            T *tlh = tail_all + (size_t)slot * 3 * (kK - 1) * D + (size_t)h * kD + tid;
            const T *src[3] = {q, k, v};
#pragma unroll
            for (int x = 0; x < 3; ++x) {
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    const int pos = len - 3 + j;
                    const T val = pos >= 0 ? src[x][(size_t)(start + pos) * D + (size_t)h * kD + tid]
                                           : tlh[(size_t)(x * 3 + (pos + 3)) * D];
                    tlh[(size_t)(x * 3 + j) * D] = val;
                }
            }
        }
    } else if (w == 8) {
        // ------------------------------------------------------------ issuer
        if (lane == 0 && n_chunks > 0) {
            auto issue_a = [&](int ci) {
                mbar_arrive_expect_tx(&bar[0], kStageABytes);
                bulk_g2s(sA, block_of(ci) + kOffTA, kOffGam - kOffTA, &bar[0]);
                bulk_g2s(sm + kSmGam + ((ci - c_first) & 1) * kD * 4, block_of(ci) + kOffGam, kD * 4, &bar[0]);
            };
            auto issue_b = [&](int ci) {
                mbar_arrive_expect_tx(&bar[1], kStageBBytes);
                bulk_g2s(sB, block_of(ci) + kOffTB, kStageBBytes, &bar[1]);
            };
            auto prefetch_block = [&](int ci) {  // into L2 ahead of its copies, one request
                prefetch_l2_bulk(block_of(ci), (uint32_t)kTcChunkBytes);
            };
            constexpr uint32_t id64 = tc::idesc_bf16(128, 64), id128 = tc::idesc_bf16(128, 128);
            constexpr uint32_t id192 = tc::idesc_bf16(128, 192);
            const uint64_t dA = tc::kmajor_desc(sA, 0, kD);                               // W_hi | QG | W_lo
            const uint64_t dP = tc::kmajor_desc(sB, 0, kC);                               // P_hi
            const uint64_t dPl = tc::kmajor_desc(sB + tc::kmajor_off(3 * kC, 0, kC), 0, kC);  // P_lo
            const uint64_t dKh = tc::kmajor_desc(sB + tc::kmajor_off(kC, 0, kC), 0, kC);      // KDT_hi
            const uint64_t dKl = tc::kmajor_desc(sB + tc::kmajor_off(4 * kC, 0, kC), 0, kC);  // KDT_lo
            issue_a(c_first);
            issue_b(c_first);
            if (n_chunks > 1) prefetch_block(c_first + 1);
            if (n_chunks > 2) prefetch_block(c_first + 2);
            tma_prefetch_2d(&tm_g, h * kD, table[c_first].t0);
            // copies and products in flight when a wait gives up
            int a_out = 1, b_out = 1, m1_out = 0, m2_out = 0;
            for (int it = 0; it < n_chunks && good; ++it) {
                const int ci = c_first + it;
                const uint32_t par = (uint32_t)(it & 1);
                if (it + 1 < n_chunks) tma_prefetch_2d(&tm_g, h * kD, table[ci + 1].t0);
                if (it + 2 < n_chunks) prefetch_block(ci + 2);
                // MMA1: S^T ready, D2 read out by the epilogue of the previous chunk, stage A landed
                good = mbar_wait_bounded(&bar[6], par, kTcWaitLimit) && mbar_wait_bounded(&bar[7], par, kTcWaitLimit) &&
                       mbar_wait_bounded(&bar[0], par, kTcWaitLimit);
                if (!good) break;
                a_out = 0;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ta(tb + kTD1, tb + kTSh + 8 * kk, dA + 16u * kk, id192, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ta(tb + kTD1, tb + kTSl + 8 * kk, dA + 16u * kk, id64, 1);
                tc::mma_commit(&bar[2]);
                m1_out = 1;
                if (!(good = mbar_wait_bounded(&bar[2], par, kTcWaitLimit))) break;
                m1_out = 0;
                // stage A is free (MMA1 read its tiles; its gamma was used by the previous refresh)
                if (it + 1 < n_chunks) {
                    issue_a(ci + 1);
                    a_out = 1;
                }
                // MMA2: U^T ready, stage B landed; the state products first
                good = mbar_wait_bounded(&bar[5], par, kTcWaitLimit) && mbar_wait_bounded(&bar[1], par, kTcWaitLimit);
                if (!good) break;
                b_out = 0;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tb + kTD3, tb + kTUh + 8 * kk, dKh + 16u * kk, id128, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tb + kTD3, tb + kTUl + 8 * kk, dKh + 16u * kk, id128, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tb + kTD3, tb + kTUh + 8 * kk, dKl + 16u * kk, id128, 1);
                tc::mma_commit(&bar[3]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tb + kTD2, tb + kTUh + 8 * kk, dP + 16u * kk, id64, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tb + kTD2, tb + kTUl + 8 * kk, dP + 16u * kk, id64, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc::mma_bf16_ta(tb + kTD2, tb + kTUh + 8 * kk, dPl + 16u * kk, id64, 1);
                tc::mma_commit(&bar[9]);
                m2_out = 1;
                if (!(good = mbar_wait_bounded(&bar[9], par, kTcWaitLimit))) break;
                m2_out = 0;
                if (it + 1 < n_chunks) {
                    issue_b(ci + 1);
                    b_out = 1;
                }
                // this chunk's gate rows, once the previous output box has left the buffer
                if (!(good = mbar_wait_bounded(&bar[8], par, kTcWaitLimit))) break;
                mbar_arrive_expect_tx(&bar[4], (uint32_t)(box_rows * kD * sizeof(T)));
                tma_load_2d(sGY, &tm_g, h * kD, table[ci].t0, &bar[4]);
            }
            if (!good) {
                atomicExch(err, KDA_ERR_TIMEOUT);
                // let what this CTA issued land before its memory goes away (bounded; the phases
                // of a copy that never completed are not waited on twice)
                if (a_out) mbar_wait_bounded(&bar[0], 0, kTcWaitLimit);
                if (b_out) mbar_wait_bounded(&bar[1], 0, kTcWaitLimit);
                if (m1_out) mbar_wait_bounded(&bar[2], 0, kTcWaitLimit);
                if (m2_out) mbar_wait_bounded(&bar[9], 0, kTcWaitLimit);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue warps
        const int qe = w & 3;                     // TMEM lane quarter of this warp
        const int vi = 32 * qe + lane;            // value index
        const int et = tid - 9 * 32;              // 0 .. 127 within the epilogue group
        const uint32_t tD2 = tb + ((uint32_t)(32 * qe) << 16) + 64;
        const float nw = __ldg(norm_w + vi);
        if (et == 0) mbar_arrive(&bar[8]);        // the gate/output buffer starts free
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[7]);      // D2 may be written by the first MMA1
        for (int it = 0; it < n_chunks; ++it) {
            const int ci = c_first + it;
            const uint32_t par = (uint32_t)(it & 1);
            const ChunkEntry e = table[ci];
            if (!bar_and(2, 128, mbar_wait_bounded(&bar[9], par, kTcWaitLimit))) { good = false; break; }
            tc::fence_after_sync();
            float o[64];
            {
                uint32_t raw[64];
                tc::tmem_ld32_nowait(tD2, raw);
                tc::tmem_ld32_nowait(tD2 + 32, raw + 32);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 64; ++j) o[j] = __uint_as_float(raw[j]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[7]);  // D2 is free for the next chunk's MMA1
            // sums of squares over this warp's 32 v for each token: a reduce-scatter butterfly per
            // 32 tokens (31 shuffles) leaves the sum of token 32 hf + lane in lane `lane`; values
            // 2j and 2j + 1 travel as a pair while they move together (offsets 16 .. 2)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float2 sq[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 x = make_float2(o[32 * hf + 2 * j], o[32 * hf + 2 * j + 1]);
                    sq[j] = f2_mul(x, x);
                }
#pragma unroll
                for (int off = 16; off >= 2; off >>= 1) {
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int j = 0; j < off / 2; ++j) {
                        const float2 keep = upper ? sq[j + off / 2] : sq[j];
                        const float2 send = upper ? sq[j] : sq[j + off / 2];
                        const float2 recv = make_float2(__shfl_xor_sync(0xffffffffu, send.x, off),
                                                        __shfl_xor_sync(0xffffffffu, send.y, off));
                        sq[j] = f2_add(keep, recv);
                    }
                }
                const bool upper = (lane & 1) != 0;
                const float keep = upper ? sq[0].y : sq[0].x, send = upper ? sq[0].x : sq[0].y;
                red[(32 * hf + lane) * 4 + qe] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
            }
            // (the AND is also the barrier after every warp's sums are in red)
            if (!bar_and(2, 128, mbar_wait_bounded(&bar[4], par, kTcWaitLimit))) { good = false; break; }
            // gated RMSNorm; the BF16 results overwrite the gate logits in place
            float rinv_l[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const float4 pl = reinterpret_cast<const float4 *>(red)[32 * hf + lane];
                rinv_l[hf] = rsqrt_ftz(((pl.x + pl.y) + (pl.z + pl.w)) * (1.0f / kD) + rms_eps);
            }
            __nv_bfloat16 y[64];
            const float2 half2 = make_float2(0.5f, 0.5f), nw2 = make_float2(nw, nw);
#pragma unroll
            for (int r = 0; r < 64; r += 2) {  // tokens r and r + 1 as a pair
                const float2 rinv = make_float2(__shfl_sync(0xFFFFFFFFu, rinv_l[r >> 5], r & 31),
                                                __shfl_sync(0xFFFFFFFFu, rinv_l[r >> 5], (r + 1) & 31));
                const float2 gv = make_float2(__bfloat162float(sGY[r * kD + vi]), __bfloat162float(sGY[(r + 1) * kD + vi]));
                // sigmoid(g) = (1 + tanh(g/2)) / 2; the hardware tanh's error is below the BF16
                // rounding of the output it multiplies
                const float2 hg = f2_mul(half2, gv);
                const float2 sg = f2_fma(half2, make_float2(tanh_approx(hg.x), tanh_approx(hg.y)), half2);
                const float2 yy = f2_mul(f2_mul(sg, nw2), f2_mul(make_float2(o[r], o[r + 1]), rinv));
                const __nv_bfloat162 yb = __floats2bfloat162_rn(yy.x, yy.y);
                y[r] = yb.x;
                y[r + 1] = yb.y;
            }
            if (e.n == kC) {  // each thread overwrites only the gate values it has read
#pragma unroll
                for (int r = 0; r < 64; ++r) sGY[r * kD + vi] = y[r];
                tc::fence_smem_to_async();
                named_bar_sync(2, 128);
                if (et == 0) {
                    tma_store_2d(&tm_out, h * kD, e.t0, sGY);
                    bulk_commit_group();
                    bulk_wait_read_all();
                    mbar_arrive(&bar[8]);
                }
            } else {
                T *obase = out + (size_t)e.t0 * D + (size_t)h * kD + vi;
#pragma unroll
                for (int r = 0; r < 64; ++r)
                    if (r < e.n) obase[(size_t)r * D] = y[r];
                named_bar_sync(2, 128);
                if (et == 0) mbar_arrive(&bar[8]);
            }
        }
        if (!good) atomicExch(err, KDA_ERR_TIMEOUT);
        if (et == 0) bulk_wait_all();  // committed output boxes are written before the CTA exits
    }
    tc::fence_before_sync();
    __syncthreads();
    if (w == 0) tc::tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------- epilogue
template <typename T>
__global__ void __launch_bounds__(256)
epilogue_kernel(const float *__restrict__ obuf, const float *__restrict__ norm_w, const T *__restrict__ g,
                T *__restrict__ out, int64_t n_rows, float rms_eps)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // (token, head) pair
    if (row >= n_rows) return;
    const float4 o = reinterpret_cast<const float4 *>(obuf + row * kD)[lane];
    const float ss = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
    const float rinv = 1.0f / sqrtf(ss * (1.0f / kD) + rms_eps);
    const float4 w = __ldg(reinterpret_cast<const float4 *>(norm_w) + lane);
    const T *gp = g + row * kD + 4 * lane;
    T *op = out + row * kD + 4 * lane;
    IO<T>::st(op + 0, sigmoidf_(IO<T>::ld(gp + 0)) * w.x * (o.x * rinv));
    IO<T>::st(op + 1, sigmoidf_(IO<T>::ld(gp + 1)) * w.y * (o.y * rinv));
    IO<T>::st(op + 2, sigmoidf_(IO<T>::ld(gp + 2)) * w.z * (o.z * rinv));
    IO<T>::st(op + 3, sigmoidf_(IO<T>::ld(gp + 3)) * w.w * (o.w * rinv));
}

// Tensor map of a packed [rows][D] BF16 input for 2-D box copies of box_rows rows x 128
// channels (one head).
cudaError_t encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t D, int box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of a packed [rows][cols] BF16 matrix for 2-D boxes of 64 columns x box_rows rows
// with 128-byte swizzle (MMA operands).
cudaError_t encode_sw128_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_typed(const State &st, const kda_layer_params &p, const int32_t *slots,
                         const int32_t *cu, int N, int64_t total_T, int64_t total_chunks,
                         const void *q, const void *k, const void *v, const void *z, const void *b,
                         const void *g, void *out, void *ws, cudaStream_t stream, const void *f,
                         const void *w_fb)
{
    // BF16 I/O runs the tensor-core state pass; FP32 I/O keeps every contraction in FP32.
    constexpr bool kTC = sizeof(T) == 2;
    const kda_config_t &c = st.cfg;
    const int H = c.num_heads;
    const WsLayout L = ws_layout(H, total_chunks, total_T, N, kTC);
    char *base = static_cast<char *>(ws);
    ChunkEntry *table = reinterpret_cast<ChunkEntry *>(base + L.table);
    int32_t *seq_first = reinterpret_cast<int32_t *>(base + L.seq_first);
    unsigned char *chunks = reinterpret_cast<unsigned char *>(base + L.chunks);
    float *obuf = reinterpret_cast<float *>(base + L.obuf);

    chunk_table_kernel<<<1, 32, 0, stream>>>(cu, N, total_T, total_chunks, table, seq_first, st.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (total_chunks > 0) {
        if constexpr (kTC) {
            int sms = 0;
            if ((e = state_sms(st, &sms)) != cudaSuccess) return e;
            // boxes of 67 rows (3 history rows + a chunk); never taller than the tensor
            const int box_rows = (int)(total_T < kC + 3 ? total_T : kC + 3);
            const int64_t Dm = (int64_t)H * kD;
            CUtensorMap tmq, tmk, tmv, tmz, tmf, tmfb;
            const bool fused = f != nullptr;
            const int f_rows = (int)(total_T < kC ? total_T : kC);
            if ((e = encode_rows_map(&tmq, q, total_T, Dm, box_rows)) != cudaSuccess ||
                (e = encode_rows_map(&tmk, k, total_T, Dm, box_rows)) != cudaSuccess ||
                (e = encode_rows_map(&tmv, v, total_T, Dm, box_rows)) != cudaSuccess)
                return e;
            if (fused) {
                // z is formed in prep from f = W_fa x ([T][d]) and the head's rows of W_fb ([H d][d])
                if ((e = encode_sw128_map(&tmf, f, total_T, kD, f_rows)) != cudaSuccess ||
                    (e = encode_sw128_map(&tmfb, w_fb, Dm, kD, kD)) != cudaSuccess)
                    return e;
                memcpy(&tmz, &tmq, sizeof(tmz));
            } else {
                if ((e = encode_rows_map(&tmz, z, total_T, Dm, box_rows)) != cudaSuccess) return e;
                memcpy(&tmf, &tmq, sizeof(tmf));
                memcpy(&tmfb, &tmq, sizeof(tmfb));
            }
            e = raise_smem_once(st, kSmemPrepTc, prep_tc_kernel<T>, kPrepTcSmem);
            if (e != cudaSuccess) return e;
            // persistent: one CTA per SM strides over the (chunk, head) items
            const int n_items = total_chunks * H;
            prep_tc_kernel<T><<<(unsigned)(n_items < sms ? n_items : sms), 512, kPrepTcSmem, stream>>>(
                p.conv_w, p.dt_bias, p.A_log, (const T *)st.tail, slots, H, st.max_slots, table,
                (const T *)q, (const T *)k, (const T *)v, (const T *)z, (const T *)b, chunks, st.err,
                c.gate_lower_bound, c.l2_eps, c.q_scale, n_items, box_rows, f_rows, fused ? 1 : 0, tmq, tmk, tmv,
                tmz, tmf, tmfb);
        } else {
            const int prep_smem = kPrepSmemFloats * (int)sizeof(float);
            e = raise_smem_once(st, kSmemPrepF32, prep_kernel<T>, prep_smem);
            if (e != cudaSuccess) return e;
            prep_kernel<T><<<(unsigned)(total_chunks * H), 256, prep_smem, stream>>>(
                p.conv_w, p.dt_bias, p.A_log, (const T *)st.tail, slots, H, st.max_slots, table,
                (const T *)q, (const T *)k, (const T *)v, (const T *)z, (const T *)b, chunks,
                c.gate_lower_bound, c.l2_eps, c.q_scale);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if constexpr (kTC) {
        e = raise_smem_once(st, kSmemStateTc, state_tc_kernel<T>, kStateTcSmem);
        if (e != cudaSuccess) return e;
        // gate logits in and output rows out as 64-row boxes (never taller than the tensor)
        const int box_g = (int)(total_T < kC ? total_T : kC);
        CUtensorMap tmg, tmo;
        if (total_T > 0) {
            if ((e = encode_rows_map(&tmg, g, total_T, (int64_t)H * kD, box_g)) != cudaSuccess ||
                (e = encode_rows_map(&tmo, out, total_T, (int64_t)H * kD, box_g)) != cudaSuccess)
                return e;
        } else {
            memset(&tmg, 0, sizeof(tmg));
            memset(&tmo, 0, sizeof(tmo));
        }
        state_tc_kernel<T><<<dim3(H, N), kStThreads, kStateTcSmem, stream>>>(
            st.S, (T *)st.tail, st.err, slots, H, st.max_slots, table, seq_first, chunks, (int)total_chunks,
            (const T *)q, (const T *)k, (const T *)v, p.norm_w, (T *)out, c.rms_eps, box_g, tmg, tmo);
        return cudaGetLastError();
    } else {
        const int state_smem = kStateSmemFloats * (int)sizeof(float);
        e = raise_smem_once(st, kSmemStateF32, state_kernel<T>, state_smem);
        if (e != cudaSuccess) return e;
        state_kernel<T><<<dim3(kD / kVB, H, N), 256, state_smem, stream>>>(
            st.S, (T *)st.tail, st.err, slots, H, st.max_slots, table, seq_first,
            reinterpret_cast<const float *>(chunks), obuf, (const T *)q, (const T *)k, (const T *)v);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (total_T > 0) {
            const int64_t rows = total_T * H;
            epilogue_kernel<T><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(obuf, p.norm_w, (const T *)g,
                                                                             (T *)out, rows, c.rms_eps);
            e = cudaGetLastError();
        }
        return e;
    }
}

}  // namespace

size_t prefill_workspace_bytes(const kda_config_t &cfg, int64_t total_chunks, int64_t total_T, int N)
{
    return ws_layout(cfg.num_heads, total_chunks, total_T, N, cfg.io_dtype == KDA_BF16).total;
}

cudaError_t launch_prefill(const State &st, const kda_layer_params &p, const int32_t *slots,
                           const int32_t *cu_seqlens, int N, int64_t total_T, int64_t total_chunks,
                           const void *q, const void *k, const void *v, const void *z, const void *b,
                           const void *g, void *out, void *ws, cudaStream_t stream, const void *f,
                           const void *w_fb)
{
    if (st.cfg.io_dtype == KDA_BF16)
        return launch_typed<__nv_bfloat16>(st, p, slots, cu_seqlens, N, total_T, total_chunks, q, k, v, z, b,
                                           g, out, ws, stream, f, w_fb);
    if (f) return cudaErrorInvalidValue;  // the fused gate projection runs on the tensor-core path
    return launch_typed<float>(st, p, slots, cu_seqlens, N, total_T, total_chunks, q, k, v, z, b, g, out, ws,
                               stream, nullptr, nullptr);
}

}  // namespace kda
