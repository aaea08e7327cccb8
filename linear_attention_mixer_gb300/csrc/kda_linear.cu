// kda_linear.cu - y = x W^T (+ r): the dense BF16 projections around the KDA mixer
// (kimi_k3.c header comment, block "KDA per-head recurrence": q,k,v =
// SiLU(ShortConv4(W{q,k,v} x)) and out = W_o [sigmoid(W_g x) * RMSNorm_head(o)];
// struct Kda holds W q, k, v, o, g). They are plain dense products with no KDA
// arithmetic; the layer harness chains them with the mixer calls.
//
// A persistent tcgen05 GEMM. A work unit is (m block of 256 rows, n block of 128
// columns, k split). Its two 128-row halves accumulate in two TMEM accumulators
// that share every weight box, so each weight tile is read once per m block; for a
// decode batch of up to 256 rows the weights stream from HBM exactly once. Units
// are ordered m block fastest, then split, then n block, and CTA c takes units
// c, c + grid, ... so CTAs working at the same time read the same weight tiles.
//   warp 4 lane 0: TMA producer, a ring of kLnStages stages (A: two 128 x 64 boxes,
//                  B: one 128 x 64 box, 128-byte swizzled)
//   warp 5 lane 0: MMA issuer; two TMEM buffers of 256 columns, so one unit's
//                  epilogue runs under the next unit's MMAs
//   warps 0-3:     epilogue, warp q on TMEM lanes 32q .. 32q + 31: FP32 -> BF16
//                  (+ the residual) -> a swizzled staging box -> TMA store; with a
//                  k split, FP32 partials go to the workspace instead and a second
//                  kernel adds the splits in split order (+ the residual), so the
//                  result does not depend on timing.
// Every wait is bounded; a wait that gives up writes KDA_ERR_TIMEOUT to the
// workspace's error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "kda_internal.cuh"
#include "kda_ptx.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kLnBM = 128;                          // rows per accumulator (MMA M)
constexpr int kLnMT = 2;                            // accumulators per unit along M
constexpr int kLnBN = 128;                          // columns per unit (MMA N)
constexpr int kLnBK = 64;                           // K per stage (one 128-byte row)
constexpr int kLnStages = 4;
constexpr int kLnAtom = 128;                        // bytes per swizzled row
constexpr int kLnABytes = kLnBM * kLnAtom;          // one A box (16 KB)
constexpr int kLnStage = kLnMT * kLnABytes + kLnBN * kLnAtom;
constexpr int kLnStg = 32 * kLnAtom;                // one staging box: 32 rows x 128 bytes
constexpr int kLnEpiWarps = 4;
constexpr int kLnThreads = 32 * (kLnEpiWarps + 2);
constexpr int kLnAlign = 1024;
constexpr int kLnSmem = kLnStages * kLnStage + kLnEpiWarps * 2 * kLnStg + 256 + kLnAlign;
constexpr uint32_t kLnSpin = 1u << 26;
constexpr int kLnMaxSplit = 8;
static_assert(kLnSmem <= 232448, "kda_linear shared memory");

__device__ __forceinline__ unsigned char *ln_align(unsigned char *p)
{
    const uint32_t a = smem_u32(p);
    return p + (((a + kLnAlign - 1) & ~(uint32_t)(kLnAlign - 1)) - a);
}

// K-major descriptor of a 128-byte-swizzled tile (rows of 128 bytes, 8-row groups 1024 bytes
// apart); a K step of 16 moves the start by 32 bytes.
__device__ __forceinline__ uint64_t ln_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ uint32_t ln_pack(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void tma_store_3d(const void *tmap, int x, int y, int z, const void *src)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
                 "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
                 : "memory");
}

struct LnShape {
    int M, N, K;
    int n_mblk, n_nblk, split, kb_per_split, n_units;
    int ysplit;  // columns per output matrix
};

__global__ void __launch_bounds__(kLnThreads, 1)
ln_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
          const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_p,
          const __nv_bfloat16 *__restrict__ res, const LnShape sh, int a_rows, int32_t *err)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = ln_align(smem_raw);
    unsigned char *stages = smem;
    unsigned char *stg = stages + kLnStages * kLnStage;  // [4 warps][2 buffers][32 rows][128 bytes]
    uint64_t *bars = reinterpret_cast<uint64_t *>(stg + kLnEpiWarps * 2 * kLnStg);
    uint64_t *full = bars, *empty = bars + kLnStages, *accfull = bars + 2 * kLnStages;
    uint64_t *accempty = accfull + 2, *fin = accempty + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(fin + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kLnStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accfull[a], 1);
            mbar_init(&accempty[a], kLnEpiWarps);
        }
        mbar_init(fin, 1);
        fence_mbar_init();
    }
    if (warp == kLnEpiWarps + 1) tc::tmem_alloc(tslot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    auto unit_coords = [&](int u, int &mb, int &ks, int &nb) {
        mb = u % sh.n_mblk;
        const int r = u / sh.n_mblk;
        ks = r % sh.split;
        nb = r / sh.split;
    };
    auto kb_range = [&](int ks, int &k0, int &k1) {
        k0 = ks * sh.kb_per_split;
        k1 = min(sh.K / kLnBK, k0 + sh.kb_per_split);
    };

    if (warp == kLnEpiWarps) {
        if (lane == 0) {  // producer
            bool ok = true;
            int step = 0;
            for (int u = blockIdx.x; u < sh.n_units && ok; u += gridDim.x) {
                int mb, ks, nb, k0, k1;
                unit_coords(u, mb, ks, nb);
                kb_range(ks, k0, k1);
                const int m0 = mb * kLnMT * kLnBM;
                const int n_a = min(kLnMT, (sh.M - m0 + kLnBM - 1) / kLnBM);  // A boxes with rows
                const uint32_t bytes = (uint32_t)(n_a * a_rows + kLnBN) * kLnAtom;
                for (int kb = k0; kb < k1; ++kb, ++step) {
                    const int s = step % kLnStages;
                    if (step >= kLnStages && !mbar_wait_bounded(&empty[s], ((step / kLnStages) - 1) & 1, kLnSpin)) {
                        ok = false;
                        break;
                    }
                    unsigned char *st = stages + s * kLnStage;
                    mbar_arrive_expect_tx(&full[s], bytes);
                    for (int mt = 0; mt < n_a; ++mt)
                        tma_load_2d(st + mt * kLnABytes, &tm_x, kb * kLnBK, m0 + mt * kLnBM, &full[s]);
                    tma_load_2d(st + kLnMT * kLnABytes, &tm_w, kb * kLnBK, nb * kLnBN, &full[s]);
                }
            }
            if (!ok) atomicExch(err, KDA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kLnEpiWarps + 1) {
        if (lane == 0) {  // MMA issuer
            bool ok = true;
            int step = 0, it = 0;
            const uint32_t idesc = tc::idesc_bf16(kLnBM, kLnBN);
            for (int u = blockIdx.x; u < sh.n_units && ok; u += gridDim.x, ++it) {
                int mb, ks, nb, k0, k1;
                unit_coords(u, mb, ks, nb);
                kb_range(ks, k0, k1);
                const int n_a = min(kLnMT, (sh.M - mb * kLnMT * kLnBM + kLnBM - 1) / kLnBM);
                const int a = it & 1;
                if (it >= 2 && !mbar_wait_bounded(&accempty[a], ((it >> 1) - 1) & 1, kLnSpin)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                for (int kb = k0; kb < k1; ++kb, ++step) {
                    const int s = step % kLnStages;
                    if (!mbar_wait_bounded(&full[s], (step / kLnStages) & 1, kLnSpin)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t sa = smem_u32(stages + s * kLnStage);
                    const uint32_t sb = sa + kLnMT * kLnABytes;
                    for (int mt = 0; mt < n_a; ++mt)
#pragma unroll
                        for (int kk = 0; kk < kLnBK / 16; ++kk)
                            tc::mma_bf16(tmem + (uint32_t)(a * kLnMT * kLnBN + mt * kLnBN),
                                         ln_desc(sa + mt * kLnABytes + kk * 32), ln_desc(sb + kk * 32), idesc,
                                         (kb > k0 || kk > 0) ? 1u : 0u);
                    tc::mma_commit(&empty[s]);
                }
                if (ok) tc::mma_commit(&accfull[a]);
            }
            tc::mma_commit(fin);
            if (!mbar_wait_bounded(fin, 0, kLnSpin)) ok = false;
            if (!ok) atomicExch(err, KDA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {  // epilogue: warp q owns TMEM lanes 32q .. 32q + 31
        bool ok = true;
        int it = 0, nbuf = 0;
        unsigned char *my = stg + warp * 2 * kLnStg;
        for (int u = blockIdx.x; u < sh.n_units; u += gridDim.x, ++it) {
            int mb, ks, nb;
            unit_coords(u, mb, ks, nb);
            const int a = it & 1;
            ok = mbar_wait_bounded(&accfull[a], (it >> 1) & 1, kLnSpin);
            if (!ok) break;
            tc::fence_after_sync();
            const int m0 = mb * kLnMT * kLnBM;
            const int n0 = nb * kLnBN;
            const int zi = n0 / sh.ysplit, x0 = n0 - zi * sh.ysplit;  // output matrix and column
            for (int mt = 0; mt < kLnMT; ++mt) {
                const int rbase = m0 + mt * kLnBM + 32 * warp;  // this warp's first row
                if (rbase >= sh.M) continue;                    // warp-uniform
                const int row = rbase + lane;
                const uint32_t tb = tmem + (uint32_t)(a * kLnMT * kLnBN + mt * kLnBN) + ((uint32_t)(32 * warp) << 16);
                if (sh.split == 1) {
#pragma unroll 1
                    for (int c = 0; c < kLnBN / 64; ++c) {  // 64 columns = one 128-byte store box
                        uint32_t v[64];
                        tc::tmem_ld32_nowait(tb + (uint32_t)(c * 64), v);
                        tc::tmem_ld32_nowait(tb + (uint32_t)(c * 64 + 32), v + 32);
                        tc::tmem_wait_ld();
                        float f[64];
#pragma unroll
                        for (int i = 0; i < 64; ++i) f[i] = __uint_as_float(v[i]);
                        if (res && row < sh.M) {
                            const uint4 *rp = reinterpret_cast<const uint4 *>(res + (size_t)row * sh.N + n0 + c * 64);
#pragma unroll
                            for (int q8 = 0; q8 < 8; ++q8) {
                                const uint4 rv = __ldg(rp + q8);
                                const uint32_t w4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    f[8 * q8 + 2 * e] += __uint_as_float(w4[e] << 16);
                                    f[8 * q8 + 2 * e + 1] += __uint_as_float(w4[e] & 0xFFFF0000u);
                                }
                            }
                        }
                        unsigned char *box = my + nbuf * kLnStg;
                        if (lane == 0) bulk_wait_read_all();  // this buffer's previous store has read it
                        __syncwarp();
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8)
                            *reinterpret_cast<uint4 *>(box + lane * kLnAtom + ((q8 ^ (lane & 7)) * 16)) =
                                make_uint4(ln_pack(f[8 * q8], f[8 * q8 + 1]), ln_pack(f[8 * q8 + 2], f[8 * q8 + 3]),
                                           ln_pack(f[8 * q8 + 4], f[8 * q8 + 5]), ln_pack(f[8 * q8 + 6], f[8 * q8 + 7]));
                        tc::fence_smem_to_async();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tm_y, x0 + c * 64, rbase, zi, box);
                            bulk_commit_group();
                        }
                        nbuf ^= 1;
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < kLnBN / 32; ++c) {  // 32 FP32 columns = one 128-byte store box
                        uint32_t v[32];
                        tc::tmem_ld32_nowait(tb + (uint32_t)(c * 32), v);
                        tc::tmem_wait_ld();
                        unsigned char *box = my + nbuf * kLnStg;
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
#pragma unroll
                        for (int q8 = 0; q8 < 8; ++q8)
                            *reinterpret_cast<uint4 *>(box + lane * kLnAtom + ((q8 ^ (lane & 7)) * 16)) =
                                make_uint4(v[4 * q8], v[4 * q8 + 1], v[4 * q8 + 2], v[4 * q8 + 3]);
                        tc::fence_smem_to_async();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&tm_p, n0 + c * 32, rbase, ks, box);
                            bulk_commit_group();
                        }
                        nbuf ^= 1;
                    }
                }
            }
            // every lane of this warp has read accumulator a
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty[a]);
        }
        if (lane == 0) bulk_wait_all();
        if (!ok && lane == 0) atomicExch(err, KDA_ERR_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kLnEpiWarps + 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// y = sum over the splits in split order (+ r), rounded to BF16; 8 columns per thread.
__global__ void __launch_bounds__(256)
ln_reduce_kernel(const float *__restrict__ part, const __nv_bfloat16 *__restrict__ res, __nv_bfloat16 *__restrict__ y,
                 int M, int N, int split, int ysplit)
{
    const int64_t i8 = (int64_t)blockIdx.x * 256 + threadIdx.x;  // group of 8 columns
    const int64_t total8 = (int64_t)M * N / 8;
    if (i8 >= total8) return;
    const int64_t e = i8 * 8;
    const int m = (int)(e / N), n = (int)(e - (int64_t)m * N);
    const size_t plane = (size_t)M * N;
    float acc[8];
    {
        const float4 *p = reinterpret_cast<const float4 *>(part + e);
        const float4 a = p[0], b = p[1];
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w; acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
    }
    for (int s = 1; s < split; ++s) {
        const float4 *p = reinterpret_cast<const float4 *>(part + s * plane + e);
        const float4 a = p[0], b = p[1];
        acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
        acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    if (res) {
        const uint4 rv = *reinterpret_cast<const uint4 *>(res + e);
        const uint32_t w4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc[2 * j] += __uint_as_float(w4[j] << 16);
            acc[2 * j + 1] += __uint_as_float(w4[j] & 0xFFFF0000u);
        }
    }
    const int zi = n / ysplit, xc = n - zi * ysplit;
    *reinterpret_cast<uint4 *>(y + (size_t)zi * M * ysplit + (size_t)m * ysplit + xc) =
        make_uint4(ln_pack(acc[0], acc[1]), ln_pack(acc[2], acc[3]), ln_pack(acc[4], acc[5]), ln_pack(acc[6], acc[7]));
}

// rank-3 map: dims {d0, d1, d2}, byte strides of dims 1 and 2, box {b0, b1, 1}, 128-byte swizzle
cudaError_t ln_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = encode(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// rank-2 map for the operand loads (the 2-D tensor copy): dims {d0, d1}, byte stride of dim 1,
// box {b0, b1}, 128-byte swizzle
cudaError_t ln_map2(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t s1, uint32_t b0, uint32_t b1)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {s1};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

thread_local char g_ln_msg[256];

kda_status ln_fail(kda_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_ln_msg, sizeof(g_ln_msg), fmt, ap);
    va_end(ap);
    return record_error(s, g_ln_msg);
}

// The k split for an m x n grid of tiles: the split that minimises the modelled time, the bytes
// moved (weights, plus the FP32 partials written and read back) over the fraction of the last
// wave that is busy.
int ln_choose_split(int M, int N, int K, int n_tiles, int sms)
{
    const int nk = K / kLnBK;
    int best = 1;
    double best_t = 1e300;
    for (int s = 1; s <= kLnMaxSplit && s <= nk; ++s) {
        const int per = (nk + s - 1) / s;
        const int eff_s = (nk + per - 1) / per;  // splits that get work
        if (eff_s != s) continue;
        const int64_t units = (int64_t)n_tiles * s;
        const double waves = (double)((units + sms - 1) / sms);
        const double eff = (double)units / (waves * sms);
        const double bytes = (double)N * K * 2 + (double)M * K * 2 + (s > 1 ? 2.0 * s * M * N * 4 : 0.0) +
                             (double)M * N * 2;
        const double t = bytes / eff;
        if (t < best_t * 0.999) {
            best_t = t;
            best = s;
        }
    }
    return best;
}

}  // namespace

size_t linear_workspace_bytes(int M, int N, int K, int sms)
{
    if (M < 1 || N < kLnBN || K < kLnBK) return 256;
    const int n_mblk = (M + kLnMT * kLnBM - 1) / (kLnMT * kLnBM);
    const int split = ln_choose_split(M, N, K, n_mblk * (N / kLnBN), sms);
    return 256 + (split > 1 ? (size_t)split * M * N * 4 : 0);
}

}  // namespace kda

using namespace kda;

extern "C" size_t kda_linear_workspace_bytes(int32_t M, int32_t N, int32_t K)
{
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        sms = 148;
    }
    return linear_workspace_bytes(M, N, K, sms);
}

extern "C" kda_status kda_linear(int32_t M, int32_t N, int32_t K, const void *x, const void *w, const void *r,
                                 void *y, int32_t ysplit, void *workspace, size_t workspace_bytes, void *stream)
{
    if (M < 0 || N <= 0 || K <= 0) return ln_fail(KDA_ERR_INVALID, "M must be >= 0 and N, K > 0 (got %d, %d, %d)", M, N, K);
    if (M == 0) return KDA_OK;
    if (N % kLnBN != 0) return ln_fail(KDA_ERR_INVALID, "N must be a multiple of %d (got %d)", kLnBN, N);
    if (K % kLnBK != 0) return ln_fail(KDA_ERR_INVALID, "K must be a multiple of %d (got %d)", kLnBK, K);
    if (ysplit == 0) ysplit = N;
    if (ysplit < 0 || ysplit % kLnBN != 0 || N % ysplit != 0)
        return ln_fail(KDA_ERR_INVALID, "ysplit must divide N and be a multiple of %d (got %d)", kLnBN, ysplit);
    if (r && ysplit != N) return ln_fail(KDA_ERR_INVALID, "a residual needs an unsplit output (ysplit 0 or N)");
    if (!x || !w || !y || !workspace) return ln_fail(KDA_ERR_INVALID, "x, w, y or workspace is NULL");
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
                         reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(r) |
                         reinterpret_cast<uintptr_t>(workspace);
    if (al & 15u) return ln_fail(KDA_ERR_INVALID, "x, w, r, y and workspace must be 16-byte aligned");
    if ((int64_t)M * N > INT_MAX / 2) return ln_fail(KDA_ERR_INVALID, "M * N is too large");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return ln_fail(KDA_ERR_CUDA, "%s", cudaGetErrorString(e));
    const size_t need = linear_workspace_bytes(M, N, K, sms);
    if (workspace_bytes < need)
        return ln_fail(KDA_ERR_INVALID, "workspace holds %zu bytes, %zu needed", workspace_bytes, need);

    LnShape sh;
    sh.M = M; sh.N = N; sh.K = K; sh.ysplit = ysplit;
    sh.n_mblk = (M + kLnMT * kLnBM - 1) / (kLnMT * kLnBM);
    sh.n_nblk = N / kLnBN;
    sh.split = ln_choose_split(M, N, K, sh.n_mblk * sh.n_nblk, sms);
    const int nk = K / kLnBK;
    sh.kb_per_split = (nk + sh.split - 1) / sh.split;
    sh.n_units = sh.n_mblk * sh.n_nblk * sh.split;
    const int a_rows = M < kLnBM ? M : kLnBM;  // a box is never taller than x
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *err = static_cast<int32_t *>(workspace);
    float *part = reinterpret_cast<float *>(static_cast<char *>(workspace) + 256);

    CUtensorMap tm_x, tm_w, tm_y, tm_p;
    const int st_rows = M < 32 ? M : 32;
    if ((e = ln_map2(&tm_x, x, K, M, (uint64_t)K * 2, kLnBK, a_rows)) != cudaSuccess ||
        (e = ln_map2(&tm_w, w, K, N, (uint64_t)K * 2, kLnBK, kLnBN)) != cudaSuccess ||
        (e = ln_map(&tm_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, ysplit, M, N / ysplit, (uint64_t)ysplit * 2,
                    (uint64_t)ysplit * 2 * M, 64, st_rows)) != cudaSuccess)
        return ln_fail(KDA_ERR_INVALID, "tensor map encoding failed (%s)", cudaGetErrorString(e));
    if (sh.split > 1) {
        if ((e = ln_map(&tm_p, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, part, N, M, sh.split, (uint64_t)N * 4,
                        (uint64_t)N * 4 * M, 32, st_rows)) != cudaSuccess)
            return ln_fail(KDA_ERR_INVALID, "tensor map encoding failed (%s)", cudaGetErrorString(e));
    } else {
        memcpy(&tm_p, &tm_y, sizeof(tm_p));
    }
    static bool attr_done[64];
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(ln_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLnSmem);
        if (e != cudaSuccess) return ln_fail(KDA_ERR_CUDA, "%s", cudaGetErrorString(e));
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    if ((e = cudaMemsetAsync(err, 0, sizeof(int32_t), s)) != cudaSuccess)
        return ln_fail(KDA_ERR_CUDA, "%s", cudaGetErrorString(e));
    const int grid = sh.n_units < sms ? sh.n_units : sms;
    ln_kernel<<<grid, kLnThreads, kLnSmem, s>>>(tm_x, tm_w, tm_y, tm_p,
                                                 sh.split == 1 ? static_cast<const __nv_bfloat16 *>(r) : nullptr, sh,
                                                 a_rows, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return ln_fail(KDA_ERR_CUDA, "%s", cudaGetErrorString(e));
    if (sh.split > 1) {
        const int64_t total8 = (int64_t)M * N / 8;
        ln_reduce_kernel<<<(unsigned)((total8 + 255) / 256), 256, 0, s>>>(
            part, static_cast<const __nv_bfloat16 *>(r), static_cast<__nv_bfloat16 *>(y), M, N, sh.split, ysplit);
        if ((e = cudaGetLastError()) != cudaSuccess) return ln_fail(KDA_ERR_CUDA, "%s", cudaGetErrorString(e));
    }
    return KDA_OK;
}
