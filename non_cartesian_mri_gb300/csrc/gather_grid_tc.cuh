// gather_grid_tc.cuh -- separable-grid F^H D / Q on the tensor cores.
//
// On a grid the gather of Fig. 17.11 factors (gather_grid.cuh) into
//   FhD[row][ix] = sum_m Mz[row][m] * Ex[m][ix],
//   Mz = Mu * e^{i2pi(ky y + kz z)},  Ex = e^{i2pi kx x},
// a complex matrix product over the samples: a dense contraction.  Here a CTA
// owns 128 grid rows (the MMA M) of a grid with nx = 128 columns (the MMA N).
// For each tile of 16 samples (two K = 8 steps) the warps evaluate Mz
// (128 rows x 16 samples) and Ex (16 samples x 128 columns) into shared
// memory, each value split into a tf32 high part and the float remainder;
// one thread then issues, per K step, two N = 256 products into [D_r | D_i]:
//   [D_r | D_i] += A_r [B_r | B_i]  +  A_i [-B_i | B_r],
// reading the B operands as two 256-row windows of one 384-row block
// S = [-B_i; B_r; B_i], with each real product done as hi*hi + hi*lo + lo*hi
// (12 tcgen05.mma of 128 x 256 x 8 per tile), which keeps about 21 bits of
// every product.  Shared-memory bandwidth (operand reads by the tensor core
// plus operand writes by the warps) is what binds this kernel, and the N = 256
// form reads each A operand once per pass instead of twice.  The
// accumulators live in tensor memory: D_r, D_i (columns 0-255) collect one
// block of tiles and are then added into the running sums R_r, R_i (columns
// 256-511), the blocked summation that keeps accumulation error below the
// trig error over a million samples.
//
// Operand tiles are K-major without swizzle: core matrices of 8 rows x 4
// tf32 (128 B), LBO = 128 B along K, SBO = 512 B between 8-row groups.  The
// operand stages rotate; stage s is rewritten only after the MMAs that read
// it have signalled their mbarrier, so operand generation runs ahead of the
// tensor core by up to kTcStages - 1 tiles.  Every wait is bounded; a CTA that gives
// up sets the device error word, waits (bounded) for its MMAs and copies, and
// still frees its tensor memory.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid.cuh"

namespace mri {

constexpr int kTcTile = 16;                          // samples per tile (two K = 8 steps)
constexpr int kTcRows = 128;                         // grid rows per CTA = MMA M
constexpr int kTcCols = 128;                         // grid columns = MMA N (nx = 128)
#ifndef MRI_TC_THREADS
#define MRI_TC_THREADS 256
#endif
#ifndef MRI_TC_STAGES
#define MRI_TC_STAGES 2
#endif
constexpr int kTcThreads = MRI_TC_THREADS;           // 256 or 512
// Tiles per summation block.  The tensor core's own fp32 accumulation loses
// a little with every add, with a consistent sign, so the error of a block
// grows with its length (measured on the 128^3 radial workload: rel-L2 1.4e-5
// for 64 tiles, 1.9e-6 for 8); the accurate path folds every 8 tiles (128
// samples), the fast paths every 64.
constexpr int kTcDrainAccurate = 8;
constexpr int kTcDrainFast = 64;
constexpr int kTcPartFloats = kTcRows * kTcTile;     // one A part: 128 x 16 tf32 (8 KB)
constexpr int kTcSFloats = 3 * kTcPartFloats;        // S = [-B_i; B_r; B_i]: 384 x 16 (24 KB)
constexpr int kTcStageFloats = 4 * kTcPartFloats + 2 * kTcSFloats;   // A r/i hi/lo, S hi/lo (80 KB)
constexpr int kTcStages = MRI_TC_STAGES;             // operand stages in the ring
constexpr int kTcSpt = kTcTile * kTcRows / kTcThreads;   // samples per thread per table (8 or 4)
constexpr int kTcColsPerWarp = 256 * 4 / (kTcThreads / 32);  // D columns one warp folds
constexpr uint32_t kTcTmemCols = 512;

// A parts at part * kTcPartFloats; S hi / lo after them
enum TcPart { A_RH = 0, A_RL, A_IH, A_IL };
constexpr int kTcSHi = 4 * kTcPartFloats;
constexpr int kTcSLo = kTcSHi + kTcSFloats;

inline bool grid_tc_fits(int nx) { return nx == kTcCols; }

inline size_t grid_tc_smem_bytes(bool realw)
{
    const int F = realw ? 4 : 5;
    size_t b = size_t(kTcStages) * kTcStageFloats * 4;    // operand stages
    b += size_t(kStages) * F * kTcTile * 4;               // record ring
    b += size_t(kTcRows) * 8 + size_t(kTcCols) * 4;        // (y, z) of the rows, x of the columns
    return b;
}

// float offset of element (row, k) in a [128][16] K-major no-swizzle tile
__device__ __forceinline__ int tc_kmaj(int row, int k)
{
    return (row >> 3) * 128 + (k >> 2) * 32 + (row & 7) * 4 + (k & 3);
}

// v = hi + lo with hi = v rounded to the nearest tf32 and lo the exact float
// remainder (|lo| <= 2^-11 |v|, either sign, so the dropped lo*lo term has no
// preferred sign)
__device__ __forceinline__ void tc_split(float v, float& hi, float& lo)
{
    uint32_t h;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(v));
    hi = __uint_as_float(h);
    lo = v - hi;
}

// store kTcSpt consecutive samples (k = kTcSpt*q ..) of row i into a part as hi and lo
__device__ __forceinline__ void tc_store(float* part_hi, float* part_lo, int i, int q,
                                         const float (&v)[kTcSpt])
{
#pragma unroll
    for (int c = 0; c < kTcSpt / 4; ++c) {
        float hi[4], lo[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) tc_split(v[4 * c + s], hi[s], lo[s]);
        const int o = tc_kmaj(i, kTcSpt * q + 4 * c);
        *reinterpret_cast<float4*>(part_hi + o) = make_float4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<float4*>(part_lo + o) = make_float4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// The D columns warp w folds and writes: lanes 32 (w % 4) .., columns
// kTcColsPerWarp * (w / 4) .. (D_r is columns 0-127, D_i 128-255).
__device__ __forceinline__ uint32_t tc_warp_cols(int warp)
{
    return uint32_t(kTcColsPerWarp) * uint32_t(warp >> 2);
}

// Fold D (columns 0-255) into R (256-511).
__device__ __forceinline__ void tc_drain(uint32_t tmem, int warp, bool have_r)
{
    const uint32_t lanes = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t dcol = tc_warp_cols(warp);
    const uint32_t rcol = dcol + 256u;
#pragma unroll 1
    for (uint32_t c0 = 0; c0 < uint32_t(kTcColsPerWarp); c0 += 32) {
        float d[32];
        tmem_ld32(tmem + lanes + dcol + c0, d);
        if (have_r) {
            float r[32];
            tmem_ld32(tmem + lanes + rcol + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) d[j] += r[j];
        } else {
            tmem_wait_ld();
        }
        tmem_st32(tmem + lanes + rcol + c0, d);
    }
    tmem_wait_st();
}

template <bool REALW, int TRIG>
__global__ void __launch_bounds__(kTcThreads, 1) gather_grid_tc_kernel(GridParams p)
{
    constexpr int T = kTcTile;
    constexpr int F = REALW ? 4 : 5;
    constexpr uint32_t TILE_BYTES = uint32_t(F) * T * 4;
    constexpr uint32_t ID = umma_idesc_tf32(kTcRows, 2 * kTcCols, false);   // N = 256
    constexpr int drain_tiles = (TRIG == TRIG_ACCURATE) ? kTcDrainAccurate : kTcDrainFast;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    float* const ops = reinterpret_cast<float*>(smem_raw);
    float* const ring = ops + kTcStages * kTcStageFloats;
    float2* const yz_sh = reinterpret_cast<float2*>(ring + kStages * F * T);
    float* const xs_sh = reinterpret_cast<float*>(yz_sh + kTcRows);
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t mma_bar[kTcStages];
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t total_rows = int64_t(p.ny) * p.nz;
    const int64_t row0 = int64_t(blockIdx.x) * kTcRows;

    for (int r = tid; r < kTcRows; r += kTcThreads) {
        const int64_t row = row0 + r;
        float2 yz = make_float2(0.f, 0.f);
        if (row < total_rows) {
            const int64_t iz = row / p.ny;
            const int64_t iy = row - iz * p.ny;
            yz = make_float2(p.ys[iy], p.zs[iz]);
        }
        yz_sh[r] = yz;
    }
    for (int c = tid; c < kTcCols; c += kTcThreads) xs_sh[c] = p.xs[c];
    if (warp == 0) tmem_alloc(&tmem_base_sh, kTcTmemCols);
    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&full_bar[st], 1);
#pragma unroll
        for (int st = 0; st < kTcStages; ++st) mbar_init(&mma_bar[st], 1);
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    if (tid == 0) {
        for (int st = 0; st < kStages && st < nt; ++st) {
            mbar_arrive_expect_tx(&full_bar[st], TILE_BYTES);
            tma_bulk_g2s(ring + st * F * T, p.rec + (t_begin + st) * F * T, TILE_BYTES,
                         &full_bar[st]);
        }
    }

    // generation: row / column gi, samples kTcSpt*gq .. of the tile
    const int gi = tid / (kTcTile / kTcSpt);
    const int gq = tid % (kTcTile / kTcSpt);
    const float2 yz = yz_sh[gi];
    const float xc = xs_sh[gi];

    bool have_r = false;
    int failed_at = -1;
    int issued = 0;   // tiles whose MMAs were issued
    for (int t = 0; t < nt; ++t) {
        const int st = t % kTcStages;
        const bool new_block = (t % drain_tiles) == 0;
        bool ok = true;
        // the MMAs of tile t - 3 read stage st
        if (t >= kTcStages)
            ok = mbar_wait_bounded(&mma_bar[st], uint32_t((t - kTcStages) / kTcStages) & 1u);
        // a new summation block: fold D into R once tile t - 1 is done (the
        // decision is the same in every thread, so the barrier is uniform)
        if (new_block && t > 0) {
            if (ok)
                ok = mbar_wait_bounded(&mma_bar[(t - 1) % kTcStages],
                                       uint32_t((t - 1) / kTcStages) & 1u);
            if (__syncthreads_or(!ok)) {
                failed_at = t;
                break;
            }
            tc_fence_after_sync();
            tc_drain(tmem, warp, have_r);
            have_r = true;
        }
        if (ok) ok = mbar_wait_bounded(&full_bar[t % kStages], uint32_t(t / kStages) & 1u);
        if (ok) {
            const float* rec = ring + (t % kStages) * F * T;
            float ar[kTcSpt], ai[kTcSpt], br[kTcSpt], bi[kTcSpt], nbi[kTcSpt];
            // this thread's samples are contiguous in every field of the record tile
            float kx[kTcSpt], ky[kTcSpt], kz[kTcSpt], wr[kTcSpt], wi[kTcSpt];
            const int s0 = kTcSpt * gq;
#pragma unroll
            for (int c = 0; c < kTcSpt / 4; ++c) {
                const float4 a = *reinterpret_cast<const float4*>(rec + s0 + 4 * c);
                const float4 b = *reinterpret_cast<const float4*>(rec + T + s0 + 4 * c);
                const float4 d = *reinterpret_cast<const float4*>(rec + 2 * T + s0 + 4 * c);
                const float4 e = *reinterpret_cast<const float4*>(rec + 3 * T + s0 + 4 * c);
                kx[4 * c] = a.x; kx[4 * c + 1] = a.y; kx[4 * c + 2] = a.z; kx[4 * c + 3] = a.w;
                ky[4 * c] = b.x; ky[4 * c + 1] = b.y; ky[4 * c + 2] = b.z; ky[4 * c + 3] = b.w;
                kz[4 * c] = d.x; kz[4 * c + 1] = d.y; kz[4 * c + 2] = d.z; kz[4 * c + 3] = d.w;
                wr[4 * c] = e.x; wr[4 * c + 1] = e.y; wr[4 * c + 2] = e.z; wr[4 * c + 3] = e.w;
                if (!REALW) {
                    const float4 g = *reinterpret_cast<const float4*>(rec + 4 * T + s0 + 4 * c);
                    wi[4 * c] = g.x; wi[4 * c + 1] = g.y; wi[4 * c + 2] = g.z; wi[4 * c + 3] = g.w;
                } else {
                    wi[4 * c] = wi[4 * c + 1] = wi[4 * c + 2] = wi[4 * c + 3] = 0.0f;
                }
            }
#pragma unroll
            for (int s8 = 0; s8 < kTcSpt; ++s8) {
                float sn, cs;
                table_sincos<TRIG>(fmaf(kz[s8], yz.y, ky[s8] * yz.x), sn, cs);
                if (REALW) {
                    ar[s8] = wr[s8] * cs;
                    ai[s8] = wr[s8] * sn;
                } else {
                    ar[s8] = fmaf(wr[s8], cs, -wi[s8] * sn);
                    ai[s8] = fmaf(wi[s8], cs, wr[s8] * sn);
                }
                table_sincos<TRIG>(kx[s8] * xc, bi[s8], br[s8]);
                nbi[s8] = -bi[s8];
            }
            float* const stage = ops + st * kTcStageFloats;
            tc_store(stage + A_RH * kTcPartFloats, stage + A_RL * kTcPartFloats, gi, gq, ar);
            tc_store(stage + A_IH * kTcPartFloats, stage + A_IL * kTcPartFloats, gi, gq, ai);
            // S rows: gi = -B_i, 128 + gi = B_r, 256 + gi = B_i (column gi)
            tc_store(stage + kTcSHi, stage + kTcSLo, gi, gq, nbi);
            tc_store(stage + kTcSHi + kTcPartFloats, stage + kTcSLo + kTcPartFloats, gi, gq, br);
            tc_store(stage + kTcSHi + 2 * kTcPartFloats, stage + kTcSLo + 2 * kTcPartFloats, gi, gq,
                     bi);
        }
        // generic-proxy writes of the operands -> visible to the tensor core
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(!ok)) {
            failed_at = t;
            break;
        }
        tc_fence_after_sync();
        if (tid == 0) {
            if (t + kStages < nt) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&full_bar[t % kStages], TILE_BYTES);
                tma_bulk_g2s(ring + (t % kStages) * F * T, p.rec + (t_begin + t + kStages) * F * T,
                             TILE_BYTES, &full_bar[t % kStages]);
            }
            const float* stage = ops + st * kTcStageFloats;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                // K block kb: 2 core matrices = 64 floats into every K-major tile
                auto adesc = [&](int part) {
                    return umma_desc_kmajor(stage + part * kTcPartFloats + kb * 64, 128, 512);
                };
                // window of 256 S rows starting at row r0 (16 row groups per 128 rows)
                auto sdesc = [&](int base, int r0) {
                    return umma_desc_kmajor(stage + base + (r0 / 128) * kTcPartFloats + kb * 64, 128,
                                            512);
                };
                const uint32_t acc0 = (new_block && kb == 0) ? 0u : 1u;
                // [D_r | D_i] += A_r [B_r | B_i]
                umma_tf32(tmem, adesc(A_RH), sdesc(kTcSHi, 128), ID, acc0);
                umma_tf32(tmem, adesc(A_RH), sdesc(kTcSLo, 128), ID, 1u);
                umma_tf32(tmem, adesc(A_RL), sdesc(kTcSHi, 128), ID, 1u);
                // [D_r | D_i] += A_i [-B_i | B_r]
                umma_tf32(tmem, adesc(A_IH), sdesc(kTcSHi, 0), ID, 1u);
                umma_tf32(tmem, adesc(A_IH), sdesc(kTcSLo, 0), ID, 1u);
                umma_tf32(tmem, adesc(A_IL), sdesc(kTcSHi, 0), ID, 1u);
            }
            umma_commit(&mma_bar[st]);
        }
        issued = t + 1;
    }

    bool ok = failed_at < 0;
    if (ok && nt > 0) {
        ok = mbar_wait_bounded(&mma_bar[(nt - 1) % kTcStages],
                               uint32_t((nt - 1) / kTcStages) & 1u);
        if (__syncthreads_or(!ok)) {
            ok = false;
            failed_at = nt;
        } else {
            tc_fence_after_sync();
            tc_drain(tmem, warp, have_r);
            have_r = true;
        }
    }

    if (ok) {
        // R -> outputs: warp w holds rows 32 (w % 4) + lane and its D columns
        const int row_local = 32 * (warp & 3) + lane;
        const int64_t row = row0 + row_local;
        const uint32_t wcols = tc_warp_cols(warp);
        float* const out = (wcols >= 128u ? p.out_i : p.out_r) + split * p.split_stride;
        const uint32_t taddr = tmem + (uint32_t(32 * (warp & 3)) << 16) + 256u + wcols;
        const int col0 = int(wcols & 127u);
#pragma unroll 1
        for (int c0 = 0; c0 < kTcColsPerWarp; c0 += 32) {
            float v[32];
            tmem_ld32(taddr + c0, v);
            tmem_wait_ld();
            if (row < total_rows && nt > 0) {
                float* o = out + row * kTcCols + col0 + c0;
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = p.accumulate ? o[j] + v[j] : v[j];
            }
        }
    } else {
        // Report, then let the MMAs and copies in flight finish before the
        // CTA's shared and tensor memory are released.
        if (tid == 0) {
            unsigned int bits = DEVERR_TILE_WAIT_TIMEOUT;
            if (issued > 0 && !mbar_wait_bounded(&mma_bar[(issued - 1) % kTcStages],
                                                 uint32_t((issued - 1) / kTcStages) & 1u))
                bits |= DEVERR_DRAIN_TIMEOUT;
            const int first = failed_at < nt ? failed_at : nt;
            const int last = (first + kStages < nt) ? first + kStages : nt;
            for (int u = first; u < last; ++u)
                if (!mbar_wait_bounded(&full_bar[u % kStages], uint32_t(u / kStages) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            atomicOr(p.err, bits);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace mri
