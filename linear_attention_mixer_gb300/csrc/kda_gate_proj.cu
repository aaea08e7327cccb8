// kda_gate_proj.cu - the decay-gate and beta input projections of a KDA layer on
// tcgen05 tensor cores (kimi_k3.c header comment, block "KDA per-head recurrence":
// the decay gate's pre-activation is the low-rank product W_fb (W_fa x) and the
// beta logit is W_b x; struct Kda stores fa as [hd][hidden], fb as [proj][hd] and
// bp as [heads][hidden]):
//
//   f = W_fa x    d = 128 values per token
//   b = W_b x     H values per token
//   z = W_fb f    H*d values per token
//
// dt_bias and the sigmoids stay in the mixer kernels, which take z and b as inputs.
//
// Two launches on the caller's stream:
//  1. gp_in_kernel: [f | b] = x [W_fa; W_b]^T for two tiles of 128 tokens over one
//     slice of the hidden dimension (the weight boxes serve both tiles). When there
//     are too few tile pairs to fill the GPU the hidden dimension is split over up
//     to 8 CTAs (split-K), which form a thread-block cluster and add their partial
//     sums on chip, in slice order (so results do not depend on timing). The FP32
//     sums go to the caller's workspace.
//  2. gp_out_kernel: persistent, one CTA per SM, launched as a programmatic
//     dependent grid so that its prologue overlaps gp_in. Each CTA walks a
//     contiguous range of (token tile, 256-column tile of z) items. On entering a
//     token tile it reads the tile's sums, rounds f to BF16 as the A operand and,
//     if it owns the tile's first z columns, writes the tile's b. W_fb tiles stream
//     through a two-stage TMA ring into two TMEM accumulators, so one item's
//     epilogue (TMEM -> BF16 -> TMA store) runs under the next item's MMAs.
//
// Every tile in shared memory uses the 128-byte swizzled layout: a row holds 64
// BF16 (128 bytes) and its 16-byte chunk c sits at chunk c ^ (row % 8), in blocks of
// 8 rows (1024 bytes) on 1024-byte boundaries. TMA lands operand boxes of 64
// columns in that layout (few, wide requests), the MMA descriptors read it as
// K-major with 8-row groups 1024 bytes apart (a K step of 16 advances the start
// by 32 bytes), and the f tile and the z staging written by threads use it too,
// which keeps their shared-memory stores free of bank conflicts.
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

constexpr int kGpTile = 128;      // tokens per tile (MMA M)
constexpr int kGpKs = 64;         // hidden columns per pipeline stage
constexpr int kGpStages = 3;      // stages of the first product's ring
constexpr int kGpN2 = 256;        // z columns per item (MMA N of the second product)
constexpr int kGpMaxSplit = 8;    // most hidden-dimension slices per token-tile pair (one cluster)
constexpr int kGpZBox = 64;       // z columns per TMA store box (128 bytes, the swizzle span)
constexpr uint32_t kGpSpin = 1u << 26;
constexpr int kGpEpiWarps = 8;      // second product: epilogue warps (two per TMEM lane quadrant)
constexpr int kGpEpiThreads = 32 * kGpEpiWarps;
constexpr int kGpOutThreads = kGpEpiThreads + 64;  // + producer and MMA issuer warps
constexpr int kGpAlign = 1024;      // slack to align the dynamic shared memory base

__host__ __device__ constexpr int gp_n1(int H) { return kD + ((H + 15) / 16) * 16; }
__host__ __device__ constexpr int gp_in_stage_bytes(int n1) { return (2 * kGpTile + n1) * kGpKs * 2; }
constexpr int kGpAtom = 128;                        // bytes per swizzled row (64 BF16)
constexpr int kGpFBytes = kGpTile * kD * 2;         // f tile, BF16
constexpr int kGpWBytes = kGpN2 * kD * 2;           // one W_fb tile, BF16
constexpr int kGpStgWarp = 32 * 128 * 2;            // one epilogue warp's z staging (32 rows x 128 columns)
constexpr int kGpOutSmem = kGpFBytes + 2 * kGpWBytes + kGpEpiWarps * kGpStgWarp + 128 + kGpAlign;

__device__ __forceinline__ unsigned char *align_smem(unsigned char *p)
{
    const uint32_t a = smem_u32(p);
    return p + (((a + kGpAlign - 1) & ~(uint32_t)(kGpAlign - 1)) - a);
}

// AND of pred over `count` threads at named barrier `id` (also a barrier).
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred)
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

// K-major, 128-byte-swizzle shared-memory descriptor for a tile whose rows are 128
// bytes and whose 8-row groups are 1024 bytes apart (start must lie in a 1024-byte
// aligned tile; a K step moves it by 32 bytes).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;             // leading byte offset (unused by swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: 8-row groups
    d |= (uint64_t)1 << 46;             // descriptor version for this architecture
    d |= (uint64_t)2 << 61;             // layout: 128-byte swizzle
    return d;
}

// Thread-block cluster helpers: this CTA's rank, the cluster-window address of a shared
// variable in CTA `rank`, a 16-byte load through that window, and a full cluster barrier
// (release / acquire: shared-memory writes before it are visible to every CTA after it).
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// (no memory clobber: several of these may be in flight at once; the cluster barrier before
// them orders them after the peers' writes)
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// ---------------------------------------------------------------- first product
// CTA (pair, split): [f | b] partial sums of the two token tiles pair*256 .. +127 and
// pair*256+128 .. +255 over the 64-column steps split, split + splits, ... of the hidden
// dimension. Each stage brings both tiles' x boxes and one (W_fa | W_b) box, which the
// MMAs of both accumulators share. Thread 0 issues the TMA copies, thread 32 the MMAs.
// The S slices of one pair form a thread-block
// cluster: at the end each CTA puts an accumulator (TMEM lane = token) into a padded
// shared-memory tile, and after a cluster barrier CTA q adds rows q*128/S .. (q+1)*128/S - 1
// of all S slices' tiles, in slice order, through distributed shared memory, and stores the
// sums as whole rows. Only the sums leave the chip.
__global__ void __launch_bounds__(128, 1)
gp_in_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_fa,
             const __grid_constant__ CUtensorMap tm_bp, float *__restrict__ sums, int T, int ksteps, int splits,
             int n1, int x_rows, int bp_rows, int32_t *err)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem(smem_raw);
    const int sb = gp_in_stage_bytes(n1);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kGpStages * sb);
    uint64_t *empty = full + kGpStages;
    uint64_t *done = empty + kGpStages;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok0 = blockIdx.x * 2 * kGpTile, split = blockIdx.y;
    const int ntile = tok0 + kGpTile < T ? 2 : 1;  // token tiles this CTA holds
    // slice `split` takes the 64-column steps split, split + splits, ...: the CTAs of one
    // token-tile pair read neighbouring 128-byte pieces of the same rows at about the same time
    const int nk = (ksteps - split + splits - 1) / splits;
    // the second product may be scheduled now (it waits for this grid to finish before it
    // reads the sums)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGpStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tslot, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;
    bool ok = true;

    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)(ntile * x_rows + kD + bp_rows) * kGpAtom;
        int issued = 0;
        for (int i = 0; i < nk; ++i) {
            const int s = i % kGpStages;
            if (i >= kGpStages && !mbar_wait_bounded(&empty[s], ((i / kGpStages) - 1) & 1, kGpSpin)) {
                ok = false;
                break;
            }
            unsigned char *xs = smem + s * sb;                  // x of tile 0, then of tile 1
            unsigned char *ws = xs + 2 * kGpTile * kGpAtom;     // W_fa rows, then W_b rows at row 128
            mbar_arrive_expect_tx(&full[s], bytes);
            const int kx = (split + i * splits) * kGpKs;
            tma_load_2d(xs, &tm_x, kx, tok0, &full[s]);
            if (ntile == 2) tma_load_2d(xs + kGpTile * kGpAtom, &tm_x, kx, tok0 + kGpTile, &full[s]);
            tma_load_2d(ws, &tm_fa, kx, 0, &full[s]);
            tma_load_2d(ws + kD * kGpAtom, &tm_bp, kx, 0, &full[s]);
            issued = i + 1;
        }
        // the last copy into each stage has landed before the CTA can exit
        for (int i = issued > kGpStages ? issued - kGpStages : 0; i < issued; ++i)
            if (!mbar_wait_bounded(&full[i % kGpStages], (i / kGpStages) & 1, kGpSpin)) ok = false;
    } else if (threadIdx.x == 32) {
        const uint32_t idesc = tc::idesc_bf16(kGpTile, n1);
        for (int i = 0; i < nk; ++i) {
            const int s = i % kGpStages;
            if (!mbar_wait_bounded(&full[s], (i / kGpStages) & 1, kGpSpin)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const uint32_t xs = smem_u32(smem + s * sb), ws = xs + 2 * kGpTile * kGpAtom;
#pragma unroll
            for (int kk = 0; kk < kGpKs / 16; ++kk) {
                const uint64_t bd = sw128_desc(ws + kk * 32);
                tc::mma_bf16(tmem, sw128_desc(xs + kk * 32), bd, idesc, (uint32_t)(i | kk));
                if (ntile == 2)
                    tc::mma_bf16(tmem + 256, sw128_desc(xs + kGpTile * kGpAtom + kk * 32), bd, idesc,
                                 (uint32_t)(i | kk));
            }
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(done);
    }
    __syncwarp();

    if (!mbar_wait_bounded(done, 0, kGpSpin)) ok = false;
    tc::fence_after_sync();
    // the stages are free now: each accumulator goes to a [128][n1 + 4] FP32 tile (the pad
    // keeps the row-per-thread writes free of bank conflicts), then leaves as whole rows
    float *tile = reinterpret_cast<float *>(smem);
    const int pitch = n1 + 4, row = warp * 32 + lane;
    for (int a = 0; a < ntile; ++a) {
        const uint32_t ta = tmem + (uint32_t)(a * 256) + ((uint32_t)(warp * 32) << 16);
        float *dst = tile + row * pitch;
        int c = 0;
        // 64 columns per TMEM wait (its latency, not the load, is what costs)
        for (; c + 64 <= n1; c += 64) {
            uint32_t v[64];
            tc::tmem_ld32_nowait(ta + (uint32_t)c, v);
            tc::tmem_ld32_nowait(ta + (uint32_t)c + 32, v + 32);
            tc::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q)
                *reinterpret_cast<float4 *>(dst + c + 4 * q) =
                    make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
        for (; c < n1; c += 16) {
            float v[16];
            tc::tmem_ld16(ta + (uint32_t)c, v);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<float4 *>(dst + c + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        cluster_sync_all();  // every slice's tile is in place
        const int q = (int)cluster_rank(), r0 = q * kGpTile / splits, r1 = (q + 1) * kGpTile / splits;
        for (int r = r0 + warp; r < r1; r += 4) {
            const int t = tok0 + a * kGpTile + r;
            if (t >= T) break;
            float4 *dst = reinterpret_cast<float4 *>(sums + (size_t)t * n1);
            const uint32_t src = smem_u32(tile + r * pitch);
            // this lane's chunks lane and lane + 32 of the row (n1 / 4 <= 64): all slices' values
            // are requested before any is added (remote loads are slow; issued one after another
            // each would wait for the previous one), then added in slice order
            const int c4a = lane, c4b = lane + 32;
            const bool hb = c4b < n1 / 4;
            float4 ua[kGpMaxSplit], ub[kGpMaxSplit];
#pragma unroll
            for (int sp = 0; sp < kGpMaxSplit; ++sp) {
                if (sp < splits) {
                    ua[sp] = ld_cluster_f4(cluster_map(src + 16u * c4a, (uint32_t)sp));
                    if (hb) ub[sp] = ld_cluster_f4(cluster_map(src + 16u * c4b, (uint32_t)sp));
                }
            }
            float4 acc = ua[0], accb = hb ? ub[0] : acc;
#pragma unroll
            for (int sp = 1; sp < kGpMaxSplit; ++sp) {
                if (sp < splits) {
                    acc.x += ua[sp].x; acc.y += ua[sp].y; acc.z += ua[sp].z; acc.w += ua[sp].w;
                    if (hb) { accb.x += ub[sp].x; accb.y += ub[sp].y; accb.z += ub[sp].z; accb.w += ub[sp].w; }
                }
            }
            dst[c4a] = acc;
            if (hb) dst[c4b] = accb;
        }
        cluster_sync_all();  // every CTA is done reading the tiles
    }
    if (!ok) atomicExch(err, KDA_ERR_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- second product
// Warps 0-7 form the f tile (and write b) and run the epilogue: warp w reads TMEM
// lanes 32*(w%4) .. +31 (tokens) and z columns 128*(w/4) .. +127 of each item.
// Warp 8 lane 0 streams W_fb tiles, warp 9 lane 0 issues the MMAs.
__global__ void __launch_bounds__(kGpOutThreads, 1)
gp_out_kernel(const __grid_constant__ CUtensorMap tm_fb, const __grid_constant__ CUtensorMap tm_z,
              const float *__restrict__ sums, __nv_bfloat16 *__restrict__ bout, int T, int H, int HD, int n1,
              int ntiles, int items, int fb_rows, int32_t *err)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align_smem(smem_raw);
    unsigned char *f_t = smem;                       // [2 k halves][128 rows][64 BF16]
    unsigned char *wbuf = f_t + kGpFBytes;           // 2 x [2 k halves][256 rows][64 BF16]
    unsigned char *stg = wbuf + 2 * kGpWBytes;       // 8 warps x 2 boxes x [32 rows][64 BF16]
    uint64_t *bars = reinterpret_cast<uint64_t *>(stg + kGpEpiWarps * kGpStgWarp);
    uint64_t *wfull = bars, *wempty = bars + 2, *accfull = bars + 4, *ready = bars + 6, *fin = bars + 8;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 9);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = (int)((int64_t)blockIdx.x * items / gridDim.x);
    const int i1 = (int)((int64_t)(blockIdx.x + 1) * items / gridDim.x);
    const int n = i1 - i0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 9; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    if (warp == kGpEpiWarps) tc::tmem_alloc(tslot, 2 * kGpN2);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    if (warp == kGpEpiWarps) {
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            const uint32_t bytes = (uint32_t)fb_rows * kGpAtom * 2;
            for (int j = 0; j < n; ++j) {
                const int s = j & 1;
                if (j >= 2 && !mbar_wait_bounded(&wempty[s], ((j >> 1) - 1) & 1, kGpSpin)) {
                    ok = false;
                    break;
                }
                const int nt = (i0 + j) % ntiles;
                unsigned char *w = wbuf + s * kGpWBytes;
                mbar_arrive_expect_tx(&wfull[s], bytes);
                tma_load_2d(w, &tm_fb, 0, nt * kGpN2, &wfull[s]);
                tma_load_2d(w + kGpN2 * kGpAtom, &tm_fb, kGpKs, nt * kGpN2, &wfull[s]);
                issued = j + 1;
            }
            for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
                if (!mbar_wait_bounded(&wfull[j & 1], (j >> 1) & 1, kGpSpin)) ok = false;
            if (!ok) atomicExch(err, KDA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kGpEpiWarps + 1) {
        if (lane == 0) {
            bool ok = true;
            const uint32_t idesc = tc::idesc_bf16(kGpTile, kGpN2);
            const uint32_t a0 = smem_u32(f_t);
            for (int j = 0; j < n; ++j) {
                const int s = j & 1;
                const uint32_t par = (j >> 1) & 1;
                if (!mbar_wait_bounded(&ready[s], par, kGpSpin) || !mbar_wait_bounded(&wfull[s], par, kGpSpin)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t b0 = smem_u32(wbuf + s * kGpWBytes);
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t koff = (uint32_t)(kk & 3) * 32;
                    tc::mma_bf16(tmem + (uint32_t)(s * kGpN2),
                                 sw128_desc(a0 + (uint32_t)(kk >> 2) * (kGpTile * kGpAtom) + koff),
                                 sw128_desc(b0 + (uint32_t)(kk >> 2) * (kGpN2 * kGpAtom) + koff), idesc, (uint32_t)kk);
                }
                tc::mma_commit(&wempty[s]);
                tc::mma_commit(&accfull[s]);
            }
            // every MMA has finished with TMEM and shared memory before the CTA exits
            tc::mma_commit(fin);
            if (!mbar_wait_bounded(fin, 0, kGpSpin)) ok = false;
            if (!ok) atomicExch(err, KDA_ERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        const int hh = warp >> 2;              // which 128 of the item's 256 z columns
        // Round token tile m's f sums to the BF16 A operand and, when with_b, write the tile's b.
        // Warp w takes rows w, w+8, ..., and lane l f columns 4l .. 4l+3 and b heads 4l .. 4l+3
        // of each, so every load instruction reads whole rows.
        auto form = [&](int m, bool with_b) {
            const float4 *base = reinterpret_cast<const float4 *>(sums) + lane;
            const size_t rstride = (size_t)n1 / 4;
            const bool bl = with_b && 4 * lane < H;  // this lane's b heads exist
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                float4 acc[8], bacc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int t = m * kGpTile + (half * 8 + i) * 8 + warp;
                    const float4 *src = base + (size_t)t * rstride;
                    acc[i] = t < T ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
                    bacc[i] = (bl && t < T) ? src[kD / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rw = (half * 8 + i) * 8 + warp, t = m * kGpTile + rw;
                    // columns 4l .. 4l+3: k half l/16, 16-byte chunk (l%16)/2, 8-byte half l%2
                    *reinterpret_cast<uint2 *>(f_t + (lane >> 4) * (kGpTile * kGpAtom) + rw * kGpAtom +
                                               ((((lane & 15) >> 1) ^ (rw & 7)) * 16) + (lane & 1) * 8) =
                        make_uint2(pack_bf16(acc[i].x, acc[i].y), pack_bf16(acc[i].z, acc[i].w));
                    if (bl && t < T) {
                        const float bv[4] = {bacc[i].x, bacc[i].y, bacc[i].z, bacc[i].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (4 * lane + j < H) bout[(size_t)t * H + 4 * lane + j] = __float2bfloat16_rn(bv[j]);
                    }
                }
            }
            tc::fence_smem_to_async();
            named_bar_sync(1, kGpEpiThreads);
        };

        bool ok = true;
        // the first product (the previous grid in the stream) has finished and its sums are visible
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (n > 0) {
            form(i0 / ntiles, i0 % ntiles == 0);
            if (threadIdx.x == 0) mbar_arrive(&ready[0]);
        }
        unsigned char *my = stg + warp * kGpStgWarp;
        for (int j = 0; j < n; ++j) {
            const int gi = i0 + j, m = gi / ntiles, nt = gi % ntiles, s = j & 1;
            const bool next_same = j + 1 < n && (gi + 1) / ntiles == m;
            // the next item reuses this f tile: let its MMAs start now (its accumulator was
            // released by the barrier at the end of the previous item)
            if (next_same && threadIdx.x == 0) mbar_arrive(&ready[(j + 1) & 1]);
            ok = named_bar_and(2, kGpEpiThreads, mbar_wait_bounded(&accfull[s], (j >> 1) & 1, kGpSpin));
            if (!ok) break;
            tc::fence_after_sync();
            // this warp's previous stores have finished reading its staging buffer
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            const uint32_t tbase = tmem + (uint32_t)(s * kGpN2 + hh * 128) + ((uint32_t)((warp & 3) * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < 128 / kGpZBox; ++c) {
                // columns hh*128 + c*64 .. +63 = the 8 16-byte chunks of box c (two TMEM loads, one wait)
                uint32_t v[64];
                tc::tmem_ld32_nowait(tbase + (uint32_t)(c * 64), v);
                tc::tmem_ld32_nowait(tbase + (uint32_t)(c * 64 + 32), v + 32);
                tc::tmem_wait_ld();
                unsigned char *box = my + c * (32 * kGpZBox * 2) + lane * (kGpZBox * 2);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int chunk = q ^ (lane & 7);
                    *reinterpret_cast<uint4 *>(box + chunk * 16) = make_uint4(
                        pack_bf16(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                        pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                        pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                        pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
                }
            }
            tc::fence_smem_to_async();
            __syncwarp();
            if (lane == 0) {
                const int y = m * kGpTile + (warp & 3) * 32;
                if (y < T) {
#pragma unroll
                    for (int bx = 0; bx < 128 / kGpZBox; ++bx) {
                        const int x = nt * kGpN2 + hh * 128 + bx * kGpZBox;
                        if (x < HD) tma_store_2d(&tm_z, x, y, my + bx * (32 * kGpZBox * 2));
                    }
                }
                bulk_commit_group();
            }
            // every warp has read its lanes of accumulator s
            tc::fence_before_sync();
            named_bar_sync(1, kGpEpiThreads);
            if (j + 1 < n && !next_same) {
                // MMAs of item j are complete (accfull waited), so the f tile is free
                form((gi + 1) / ntiles, (gi + 1) % ntiles == 0);
                if (threadIdx.x == 0) mbar_arrive(&ready[(j + 1) & 1]);
            }
        }
        if (lane == 0) bulk_wait_all();
        if (!ok && threadIdx.x == 0) atomicExch(err, KDA_ERR_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kGpEpiWarps) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * kGpN2);
    }
}

// ---------------------------------------------------------------- first product only
// f (BF16 [T][d]) and b (BF16 [T][H]) from the FP32 sums of gp_in ([T][n1]: f then b): for a
// prefill that forms z = W_fb f itself. Thread t4 of a row rounds 4 consecutive values.
__global__ void __launch_bounds__(256)
gp_f_kernel(const float *__restrict__ sums, __nv_bfloat16 *__restrict__ f, __nv_bfloat16 *__restrict__ bout,
            int64_t T, int H, int n1)
{
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;  // (row, 4 columns of f | b)
    const int per = kD / 4 + (H + 3) / 4;
    const int64_t t = i / per;
    if (t >= T) return;
    const int c4 = (int)(i - t * per);
    const float *src = sums + (size_t)t * n1;
    if (c4 < kD / 4) {
        const float4 v = reinterpret_cast<const float4 *>(src)[c4];
        *reinterpret_cast<uint2 *>(f + (size_t)t * kD + 4 * c4) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
    } else {
        const int h0 = 4 * (c4 - kD / 4);
        for (int j = 0; j < 4 && h0 + j < H; ++j) bout[(size_t)t * H + h0 + j] = __float2bfloat16_rn(src[kD + h0 + j]);
    }
}

// ---------------------------------------------------------------- FP32 I/O path
// With FP32 I/O the same products run on CUDA cores in FP32, the correctness path for FP32
// configurations (as the FP32 prefill kernels are): C[M][N] = A[M][K] B[N][K]^T in 64 x 64
// output tiles, 256 threads with 4 x 4 outputs each, K staged through shared memory 16 at a
// time. Each output is one FP32 dot product in k order, so results do not depend on timing.
__global__ void __launch_bounds__(256)
gp_f32_gemm_kernel(const float *__restrict__ A, int lda, const float *__restrict__ B, int ldb, float *__restrict__ C,
                   int ldc, int M, int N, int K)
{
    __shared__ float As[16][68], Bs[16][68];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.x * 64, n0 = blockIdx.y * 64;  // rows on x: T may exceed 65535 tiles
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int e = threadIdx.x; e < 64 * 16; e += 256) {
            const int r = e >> 4, c = e & 15;  // 16 consecutive k of one row per 16 threads
            As[c][r] = (m0 + r < M && k0 + c < K) ? A[(size_t)(m0 + r) * lda + k0 + c] : 0.f;
            Bs[c][r] = (n0 + r < N && k0 + c < K) ? B[(size_t)(n0 + r) * ldb + k0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&As[kk][4 * ty]);
            const float4 bb = *reinterpret_cast<const float4 *>(&Bs[kk][4 * tx]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = m0 + 4 * ty + i, n = n0 + 4 * tx + j;
            if (m < M && n < N) C[(size_t)m * ldc + n] = acc[i][j];
        }
}

cudaError_t gp_f32_gemm(const float *A, int lda, const float *B, int ldb, float *C, int ldc, int M, int N, int K,
                        cudaStream_t s)
{
    const dim3 grid((unsigned)((M + 63) / 64), (unsigned)((N + 63) / 64));
    gp_f32_gemm_kernel<<<grid, 256, 0, s>>>(A, lda, B, ldb, C, ldc, M, N, K);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- host side
thread_local char g_msg[256];

kda_status gp_fail(kda_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return record_error(s, g_msg);
}

cudaError_t encode_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// hidden-dimension slices per pair of token tiles: enough CTAs to cover the SMs, at most
// kGpMaxSplit and never more than the 64-column steps there are
int gp_splits(int64_t pairs, int ksteps, int sms)
{
    int64_t s = pairs >= sms ? 1 : sms / pairs;
    if (s > kGpMaxSplit) s = kGpMaxSplit;
    if (s > ksteps) s = ksteps;
    return s < 1 ? 1 : (int)s;
}

// Host-side argument checks that need no device; returns KDA_OK or the status.
kda_status gp_check(const kda_config_t *cfg, int32_t hidden, int64_t T)
{
    if (!config_ok(cfg)) return KDA_ERR_INVALID;
    if (cfg->num_heads > 128) return gp_fail(KDA_ERR_INVALID, "kda_gate_proj needs num_heads <= 128 (got %d)", cfg->num_heads);
    if (hidden < kGpKs || hidden % kGpKs != 0)
        return gp_fail(KDA_ERR_INVALID, "hidden must be a positive multiple of %d (got %d)", kGpKs, hidden);
    if (T < 0) return gp_fail(KDA_ERR_INVALID, "T must be >= 0 (got %lld)", (long long)T);
    const int64_t ntiles = ((int64_t)cfg->num_heads * kD + kGpN2 - 1) / kGpN2;
    if (T > INT_MAX || ((T + kGpTile - 1) / kGpTile) * ntiles > INT_MAX)
        return gp_fail(KDA_ERR_INVALID, "T = %lld is too large for one call", (long long)T);
    return KDA_OK;
}

kda_status gp_sms(int *sms)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return gp_fail(KDA_ERR_CUDA, "kda_gate_proj: device query failed: %s", cudaGetErrorString(e));
    }
    return KDA_OK;
}

constexpr size_t kGpErrBytes = 256;  // the error word, padded so the partial sums stay aligned

// the error word, then the sums [T][n1] FP32 of [f | b]
size_t gp_workspace(const kda_config_t &cfg, int64_t T)
{
    return kGpErrBytes + (size_t)T * (size_t)gp_n1(cfg.num_heads) * sizeof(float);
}

}  // namespace
}  // namespace kda

extern "C" size_t kda_gate_proj_workspace_bytes(const kda_config_t *cfg, int32_t hidden, int64_t T)
{
    if (kda::gp_check(cfg, hidden, T) != KDA_OK) return 0;
    return kda::gp_workspace(*cfg, T);
}

extern "C" kda_status kda_gate_proj(const kda_config_t *cfg, int32_t hidden, int64_t T, const void *x,
                                    const void *w_fa, const void *w_fb, const void *w_b, void *z, void *b,
                                    void *workspace, size_t workspace_bytes, void *stream)
{
    using namespace kda;
    kda_status st = gp_check(cfg, hidden, T);
    if (st != KDA_OK) return st;
    if (!workspace) return gp_fail(KDA_ERR_INVALID, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return gp_fail(KDA_ERR_INVALID, "workspace is not 16-byte aligned");
    if (T == 0) return KDA_OK;
    if (!x || !w_fa || !w_fb || !w_b || !z || !b) return gp_fail(KDA_ERR_INVALID, "a tensor pointer is NULL");
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_fa) |
                         reinterpret_cast<uintptr_t>(w_fb) | reinterpret_cast<uintptr_t>(w_b) |
                         reinterpret_cast<uintptr_t>(z);
    if (al & 15u) return gp_fail(KDA_ERR_INVALID, "x, w_fa, w_fb, w_b or z is not 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(b) & (cfg->io_dtype == KDA_F32 ? 3u : 1u))
        return gp_fail(KDA_ERR_INVALID, "b is not aligned to its element size");
    int sms = 0;
    if ((st = gp_sms(&sms)) != KDA_OK) return st;
    if (cfg->io_dtype == KDA_F32) {
        // f into the workspace, b and z straight to the outputs
        cudaStream_t s32 = static_cast<cudaStream_t>(stream);
        float *f = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) + kGpErrBytes);
        const int H = cfg->num_heads, HD = H * kD;
        cudaError_t e;
        if ((e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), s32)) != cudaSuccess ||
            (e = gp_f32_gemm(static_cast<const float *>(x), hidden, static_cast<const float *>(w_fa), hidden, f, kD,
                             (int)T, kD, hidden, s32)) != cudaSuccess ||
            (e = gp_f32_gemm(static_cast<const float *>(x), hidden, static_cast<const float *>(w_b), hidden,
                             static_cast<float *>(b), H, (int)T, H, hidden, s32)) != cudaSuccess ||
            (e = gp_f32_gemm(f, kD, static_cast<const float *>(w_fb), kD, static_cast<float *>(z), HD, (int)T, HD, kD,
                             s32)) != cudaSuccess)
            return gp_fail(KDA_ERR_CUDA, "kda_gate_proj (FP32): %s", cudaGetErrorString(e));
        return KDA_OK;
    }
    const size_t need = gp_workspace(*cfg, T);
    const int splits = gp_splits((T + 2 * kGpTile - 1) / (2 * kGpTile), hidden / kGpKs, sms);
    if (workspace_bytes < need)
        return gp_fail(KDA_ERR_INVALID, "workspace holds %zu bytes; this call needs %zu", workspace_bytes, need);

    const int H = cfg->num_heads, HD = H * kD, n1 = gp_n1(H);
    const int mtiles = (int)((T + kGpTile - 1) / kGpTile);
    const int ntiles = (HD + kGpN2 - 1) / kGpN2;
    const int items = mtiles * ntiles;
    // boxes never taller than their tensor
    const int x_rows = (int)(T < kGpTile ? T : kGpTile);
    const int fb_rows = HD < kGpN2 ? HD : kGpN2;
    const int z_rows = (int)(T < 32 ? T : 32);
    CUtensorMap tm_x, tm_fa, tm_bp, tm_fb, tm_z;
    cudaError_t e;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if ((e = encode_2d(&tm_x, x, hidden, T, (uint64_t)hidden * 2, kGpKs, x_rows, sw)) != cudaSuccess ||
        (e = encode_2d(&tm_fa, w_fa, hidden, kD, (uint64_t)hidden * 2, kGpKs, kD, sw)) != cudaSuccess ||
        (e = encode_2d(&tm_bp, w_b, hidden, H, (uint64_t)hidden * 2, kGpKs, H, sw)) != cudaSuccess ||
        (e = encode_2d(&tm_fb, w_fb, kD, HD, kD * 2, kGpKs, fb_rows, sw)) != cudaSuccess ||
        (e = encode_2d(&tm_z, z, HD, T, (uint64_t)HD * 2, kGpZBox, z_rows, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "kda_gate_proj: tensor map encoding failed: %s", cudaGetErrorString(e));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *err = static_cast<int32_t *>(workspace);
    float *sums = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) + kGpErrBytes);
    const int in_smem = kGpStages * gp_in_stage_bytes(n1) + 128 + kGpAlign;
    if ((e = cudaMemsetAsync(err, 0, sizeof(int32_t), s)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(gp_in_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, in_smem)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(gp_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGpOutSmem)) !=
            cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "kda_gate_proj: %s", cudaGetErrorString(e));
    // the slices of a token-tile pair form one cluster (they reduce their sums on chip)
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute at[1];
    lc.gridDim = dim3((unsigned)((mtiles + 1) / 2), (unsigned)splits, 1);
    lc.blockDim = dim3(128, 1, 1);
    lc.dynamicSmemBytes = (size_t)in_smem;
    lc.stream = s;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = (unsigned)splits;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&lc, gp_in_kernel, tm_x, tm_fa, tm_bp, sums, (int)T, hidden / kGpKs, splits, n1,
                                x_rows, H, err)) != cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "gp_in_kernel launch: %s", cudaGetErrorString(e));
    // programmatic dependent launch: gp_out's prologue and first W_fb copies overlap the end of
    // gp_in; its epilogue warps wait for gp_in before reading the sums
    const int grid = items < sms ? items : sms;
    lc.gridDim = dim3((unsigned)grid, 1, 1);
    lc.blockDim = dim3(kGpOutThreads, 1, 1);
    lc.dynamicSmemBytes = (size_t)kGpOutSmem;
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    if ((e = cudaLaunchKernelEx(&lc, gp_out_kernel, tm_fb, tm_z, (const float *)sums, static_cast<__nv_bfloat16 *>(b),
                                (int)T, H, HD, n1, ntiles, items, fb_rows, err)) != cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "gp_out_kernel launch: %s", cudaGetErrorString(e));
    return KDA_OK;
}

extern "C" kda_status kda_gate_proj_in(const kda_config_t *cfg, int32_t hidden, int64_t T, const void *x,
                                       const void *w_fa, const void *w_b, void *f, void *b, void *workspace,
                                       size_t workspace_bytes, void *stream)
{
    using namespace kda;
    kda_status st = gp_check(cfg, hidden, T);
    if (st != KDA_OK) return st;
    if (cfg->io_dtype != KDA_BF16) return gp_fail(KDA_ERR_INVALID, "kda_gate_proj_in needs BF16 I/O");
    if (!workspace) return gp_fail(KDA_ERR_INVALID, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return gp_fail(KDA_ERR_INVALID, "workspace is not 16-byte aligned");
    if (T == 0) return KDA_OK;
    if (!x || !w_fa || !w_b || !f || !b) return gp_fail(KDA_ERR_INVALID, "a tensor pointer is NULL");
    const uintptr_t al = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_fa) |
                         reinterpret_cast<uintptr_t>(w_b) | reinterpret_cast<uintptr_t>(f);
    if (al & 15u) return gp_fail(KDA_ERR_INVALID, "x, w_fa, w_b or f is not 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(b) & 1u) return gp_fail(KDA_ERR_INVALID, "b is not aligned to its element size");
    int sms = 0;
    if ((st = gp_sms(&sms)) != KDA_OK) return st;
    const size_t need = gp_workspace(*cfg, T);
    if (workspace_bytes < need)
        return gp_fail(KDA_ERR_INVALID, "workspace holds %zu bytes; this call needs %zu", workspace_bytes, need);
    const int splits = gp_splits((T + 2 * kGpTile - 1) / (2 * kGpTile), hidden / kGpKs, sms);
    const int H = cfg->num_heads, n1 = gp_n1(H);
    const int mtiles = (int)((T + kGpTile - 1) / kGpTile);
    const int x_rows = (int)(T < kGpTile ? T : kGpTile);
    CUtensorMap tm_x, tm_fa, tm_bp;
    cudaError_t e;
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if ((e = encode_2d(&tm_x, x, hidden, T, (uint64_t)hidden * 2, kGpKs, x_rows, sw)) != cudaSuccess ||
        (e = encode_2d(&tm_fa, w_fa, hidden, kD, (uint64_t)hidden * 2, kGpKs, kD, sw)) != cudaSuccess ||
        (e = encode_2d(&tm_bp, w_b, hidden, H, (uint64_t)hidden * 2, kGpKs, H, sw)) != cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "kda_gate_proj_in: tensor map encoding failed: %s", cudaGetErrorString(e));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *err = static_cast<int32_t *>(workspace);
    float *sums = reinterpret_cast<float *>(static_cast<unsigned char *>(workspace) + kGpErrBytes);
    const int in_smem = kGpStages * gp_in_stage_bytes(n1) + 128 + kGpAlign;
    if ((e = cudaMemsetAsync(err, 0, sizeof(int32_t), s)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(gp_in_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, in_smem)) != cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "kda_gate_proj_in: %s", cudaGetErrorString(e));
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute at[1];
    lc.gridDim = dim3((unsigned)((mtiles + 1) / 2), (unsigned)splits, 1);
    lc.blockDim = dim3(128, 1, 1);
    lc.dynamicSmemBytes = (size_t)in_smem;
    lc.stream = s;
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = (unsigned)splits;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&lc, gp_in_kernel, tm_x, tm_fa, tm_bp, sums, (int)T, hidden / kGpKs, splits, n1,
                                x_rows, H, err)) != cudaSuccess)
        return gp_fail(KDA_ERR_CUDA, "gp_in_kernel launch: %s", cudaGetErrorString(e));
    const int64_t threads = T * (kD / 4 + (H + 3) / 4);
    gp_f_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(sums, static_cast<__nv_bfloat16 *>(f),
                                                                 static_cast<__nv_bfloat16 *>(b), T, H, n1);
    if ((e = cudaGetLastError()) != cudaSuccess) return gp_fail(KDA_ERR_CUDA, "gp_f_kernel launch: %s", cudaGetErrorString(e));
    return KDA_OK;
}
