// gather_grid.cuh -- F^H D and Q for voxels on a separable grid.
//
// When the voxels form a grid xs[nx] x ys[ny] x zs[nz] (voxel n = (iz*ny + iy)*nx + ix,
// x fastest; every workload of the chapter is such a grid), the kernel of
// the register-promoted gather (Fig. 17.11) factors:
//
//   e^{i 2 pi k.x_n} = Ex[m][ix] * Eyz[m][iy, iz]
//   Ex  = e^{i 2 pi kx xs[ix]},   Eyz = e^{i 2 pi (ky ys[iy] + kz zs[iz])}.
//
// A CTA owns R = 4096 / nx whole grid rows (fixed iy, iz; all ix).  For each
// tile of kGridTile samples it builds, in shared memory,
//   Ex[s][ix]   for the tile's samples and all nx columns, and
//   Mz[r][s]    = Mu[s] * Eyz[s][row r]   for its R rows
// (Mu = conj(Phi) D for F^H D, |Phi|^2 for Q), after which every voxel-sample
// pair is one complex multiply-accumulate, acc += Mz[r][s] * Ex[s][ix]: four
// FFMA.  Each thread holds a 4 x 4 block of voxels (4 columns, 4 rows) in
// registers, so per two samples it loads four Ex and four Mz vectors
// (16-byte loads, two samples each) for 32 pairs: a quarter of a shared-memory
// load per pair.  The sin/cos work drops from two per pair to (nx + R) per
// (tile sample, CTA), i.e. 1/R + 1/nx per pair, so the accurate polynomial
// trig costs little more than the SFU one.
//
// Tables are double-buffered: the tables of tile t+1 are written while no
// thread can still read that buffer (it was last read for tile t-1, before
// the barrier that ends tile t's build), so one CTA barrier per tile
// suffices.  The records feeding the tables stream through the same
// TMA/mbarrier ring as the general kernel.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather.cuh"

namespace mri {

constexpr int kGridTile = 32;      // samples per table tile
constexpr int kGridThreads = 256;
constexpr int kGridVX = 4;         // columns per thread
constexpr int kGridVY = 4;         // rows per thread
constexpr int kGridV = kGridVX * kGridVY;                  // voxels per thread
constexpr int kGridVoxelsPerCta = kGridThreads * kGridV;   // 4096: R = 4096 / nx rows

struct GridParams {
    const float* rec;       // tile-major records, kGridTile samples per tile
    int64_t ntiles;
    int splits;
    const float *xs, *ys, *zs;
    int nx, ny, nz;
    int rows_per_cta;       // 4096 / nx
    float* out_r;           // as GatherParams, one coil
    float* out_i;
    int64_t split_stride;
    int accumulate;
    unsigned int* err;
    // tensor-core kernel: float bits of max |w_r| + |w_i| over the samples,
    // and the B operand tiles (kTcStageBytes per record tile)
    const unsigned int* wbound;
    const unsigned char* s_tab;
    // tensor-core coil groups: coils present, and the output offset of coil b
    // (out_r + b * coil_stride ..)
    int coils;
    int64_t coil_stride;
    // tensor-core kernel with the Ey table: per record tile and block of 128
    // y values, e^{i phase(ky y)} as [sample][128] float2; ny / 128 blocks
    const float2* ey_tab;
    int ey_blocks;
    // tensor-core kernel: column blocks of 128 (the last may be partly padding)
    int ncb;
};

// Forward model on a grid (tensor-core kernel, gather_grid_tc_fwd.cuh).
struct FwdParams {
    const float *kx, *ky, *kz;       // M samples
    int64_t M;
    float kscale;                    // phase units of the trig path
    const float* xs;                 // nx columns (64 or a multiple of 128)
    int nx;
    int ncb;                         // column blocks of 128
    const float2* yz_rows;           // (y, z) of every row, padded to whole blocks
    int64_t row_blocks;
    int splits;                      // CTAs along the row blocks
    const unsigned char* rho_tab;    // chunks [row block][column block][K step], 24 KB each
    const unsigned int* bound;       // float bits of max |rho_r| + |rho_i|
    float* out_r;                    // [split][M] or the caller's arrays
    float* out_i;
    int64_t split_stride;
    int accumulate;
    unsigned int* err;
};

// The table kernel takes nx in {32, 64, 128, 256}: nx / 4 column blocks
// divide the 256 threads, and the tables fit shared memory (nx = 32 gives
// R = 128 rows).  nx is a template parameter so that every table address is a
// base register plus an immediate offset.
inline bool grid_kernel_fits(int nx)
{
    return nx == 32 || nx == 64 || nx == 128 || nx == 256;
}

// Row stride of the Mz table in float2: T + 2 keeps 16-byte alignment for
// two-sample loads and puts consecutive rows in different banks.
constexpr int kMzStride = kGridTile + 2;

// Dynamic shared memory of the grid kernel for a given nx.
inline size_t grid_smem_bytes(int nx, bool realw)
{
    const int F = realw ? 4 : 5;
    const int R = kGridVoxelsPerCta / nx;
    size_t b = size_t(kStages) * F * kGridTile * 4;          // record ring
    b += 2 * size_t(kGridTile) * nx * 8;                      // Ex [T/2][nx][2], double-buffered
    b += 2 * size_t(R) * kMzStride * 8;                       // Mz [R][T+2], double-buffered
    b += size_t(R) * 8;                                       // (y, z) of the rows
    return b;
}

template <int TRIG>
__device__ __forceinline__ void table_sincos(float ph, float& s, float& c)
{
    if (TRIG == TRIG_ACCURATE) {
        sincos_quarter_turns(ph, s, c);          // records hold 4k: quarter turns
    } else if (TRIG == TRIG_FAST) {
        __sincosf(ph, &s, &c);                   // records hold 2 pi k: radians
    } else {
        const float rn = (ph + 12582912.0f) - 12582912.0f;   // records hold k: turns
        __sincosf((ph - rn) * 6.28318530717958647692f, &s, &c);
    }
}

template <bool REALW, int TRIG, int NX>
__global__ void __launch_bounds__(kGridThreads, 2) gather_grid_kernel(GridParams p)
{
    constexpr int T = kGridTile;
    constexpr int F = REALW ? 4 : 5;
    constexpr uint32_t TILE_BYTES = uint32_t(F) * T * 4;
    constexpr int VX = kGridVX, VY = kGridVY;
    constexpr int R = kGridVoxelsPerCta / NX;     // rows per CTA
    constexpr int NXB = NX / VX;                  // column blocks: column cb + NXB * i
    constexpr int SB = kGridThreads / NX;         // sample pairs per Ex-build pass
    static_assert(kGridThreads % NXB == 0 && kGridThreads % NX == 0 && T == 32 &&
                      (T / 2) % SB == 0, "grid shape");

    const int64_t total_rows = int64_t(p.ny) * p.nz;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* const ring = reinterpret_cast<float*>(smem_raw);
    float4* const ex_tab = reinterpret_cast<float4*>(ring + kStages * F * T);   // [2][T/2][NX]
    float2* const mz_tab = reinterpret_cast<float2*>(ex_tab + 2 * (T / 2) * NX); // [2][R][T+2]
    float2* const yz_sh = mz_tab + 2 * R * kMzStride;                           // [R]
    __shared__ __align__(8) uint64_t full_bar[kStages];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t row0 = int64_t(blockIdx.x) * R;

    // this thread's voxels: columns cb + NXB*i (i < 4), rows 4*rb + j (j < 4)
    const int cb = tid % NXB;
    const int rb = tid / NXB;
    // its share of the Ex build: column ix_b, sample pairs sb0 + SB*it
    const int ix_b = tid % NX;
    const int sb0 = tid / NX;
    const float x_b = p.xs[ix_b];

    for (int r = tid; r < R; r += kGridThreads) {
        const int64_t row = row0 + r;
        float2 yz = make_float2(0.f, 0.f);
        if (row < total_rows) {
            const int64_t iz = row / p.ny;
            const int64_t iy = row - iz * p.ny;
            yz = make_float2(p.ys[iy], p.zs[iz]);
        }
        yz_sh[r] = yz;
    }
    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&full_bar[st], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int st = 0; st < kStages && st < nt; ++st) {
            mbar_arrive_expect_tx(&full_bar[st], TILE_BYTES);
            tma_bulk_g2s(ring + st * F * T, p.rec + (t_begin + st) * F * T, TILE_BYTES,
                         &full_bar[st]);
        }
    }

    float run_r[VY][VX], run_i[VY][VX];
#pragma unroll
    for (int j = 0; j < VY; ++j)
#pragma unroll
        for (int i = 0; i < VX; ++i) run_r[j][i] = run_i[j][i] = 0.0f;

    int failed_at = -1;
    for (int t = 0; t < nt; ++t) {
        const int st = t % kStages;
        const bool ok = mbar_wait_bounded(&full_bar[st], uint32_t(t / kStages) & 1u);
        const float* rec = ring + st * F * T;
        float4* const ex = ex_tab + (t & 1) * (T / 2) * NX;
        float2* const mz = mz_tab + (t & 1) * R * kMzStride;
        if (ok) {
            // Ex[s][ix] = e^{i phase(kx[s] xs[ix])}, stored as (sample pair, column):
            // each thread fills whole 16-byte slots, consecutive lanes consecutive
            // columns
#pragma unroll
            for (int it = 0; it < T / (2 * SB); ++it) {
                const int q = sb0 + SB * it;          // sample pair
                float s0, c0, s1, c1;
                table_sincos<TRIG>(rec[2 * q] * x_b, s0, c0);
                table_sincos<TRIG>(rec[2 * q + 1] * x_b, s1, c1);
                ex[q * NX + ix_b] = make_float4(c0, s0, c1, s1);
            }
            // Mz[r][s] = Mu[s] * e^{i phase(ky[s] y_r + kz[s] z_r)}: lane = sample
            const float ky = rec[T + lane], kz = rec[2 * T + lane];
            const float wr = rec[3 * T + lane];
            const float wi = REALW ? 0.0f : rec[4 * T + lane];
#pragma unroll
            for (int it = 0; it < R / 8; ++it) {
                const int r = warp + 8 * it;
                const float2 yz = yz_sh[r];
                float sn, cs;
                table_sincos<TRIG>(fmaf(kz, yz.y, ky * yz.x), sn, cs);
                mz[r * kMzStride + lane] =
                    REALW ? make_float2(wr * cs, wr * sn)
                          : make_float2(fmaf(wr, cs, -wi * sn), fmaf(wi, cs, wr * sn));
            }
        }
        // tables of tile t complete; record stage st no longer read
        if (__syncthreads_or(!ok)) {
            failed_at = t;
            break;
        }
        if (tid == 0 && t + kStages < nt) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&full_bar[st], TILE_BYTES);
            tma_bulk_g2s(ring + st * F * T, p.rec + (t_begin + t + kStages) * F * T, TILE_BYTES,
                         &full_bar[st]);
        }

        float pr[VY][VX], pi[VY][VX];
#pragma unroll
        for (int j = 0; j < VY; ++j)
#pragma unroll
            for (int i = 0; i < VX; ++i) pr[j][i] = pi[j][i] = 0.0f;
        const float4* const ex_cols = ex + cb;
        const float4* const mz_rows = reinterpret_cast<const float4*>(mz + 4 * rb * kMzStride);
#pragma unroll 2
        for (int s = 0; s < T; s += 2) {
            float4 e[VX], m[VY];
#pragma unroll
            for (int i = 0; i < VX; ++i) e[i] = ex_cols[(s >> 1) * NX + NXB * i];
#pragma unroll
            for (int j = 0; j < VY; ++j) m[j] = mz_rows[(j * kMzStride + s) >> 1];
#pragma unroll
            for (int j = 0; j < VY; ++j)
#pragma unroll
                for (int i = 0; i < VX; ++i) {
                    // samples s (x, y) and s+1 (z, w): acc += Mz * Ex
                    pr[j][i] = fmaf(m[j].x, e[i].x, pr[j][i]);
                    pr[j][i] = fmaf(-m[j].y, e[i].y, pr[j][i]);
                    pi[j][i] = fmaf(m[j].x, e[i].y, pi[j][i]);
                    pi[j][i] = fmaf(m[j].y, e[i].x, pi[j][i]);
                    pr[j][i] = fmaf(m[j].z, e[i].z, pr[j][i]);
                    pr[j][i] = fmaf(-m[j].w, e[i].w, pr[j][i]);
                    pi[j][i] = fmaf(m[j].z, e[i].w, pi[j][i]);
                    pi[j][i] = fmaf(m[j].w, e[i].z, pi[j][i]);
                }
        }
#pragma unroll
        for (int j = 0; j < VY; ++j)
#pragma unroll
            for (int i = 0; i < VX; ++i) {
                run_r[j][i] += pr[j][i];
                run_i[j][i] += pi[j][i];
            }
    }

    if (failed_at >= 0) {
        if (tid == 0) {
            unsigned int bits = DEVERR_TILE_WAIT_TIMEOUT;
            const int last = (failed_at + kStages < nt) ? failed_at + kStages : nt;
            for (int u = failed_at; u < last; ++u)
                if (!mbar_wait_bounded(&full_bar[u % kStages], uint32_t(u / kStages) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            atomicOr(p.err, bits);
        }
        __syncthreads();
        return;
    }

    float* const out_r = p.out_r + split * p.split_stride;
    float* const out_i = p.out_i + split * p.split_stride;
#pragma unroll
    for (int j = 0; j < VY; ++j) {
        const int64_t row = row0 + 4 * rb + j;
        if (row < total_rows) {
#pragma unroll
            for (int i = 0; i < VX; ++i) {
                const int64_t n = row * NX + cb + NXB * i;
                float r = run_r[j][i], im = run_i[j][i];
                if (p.accumulate) {
                    r = out_r[n] + r;
                    im = out_i[n] + im;
                }
                out_r[n] = r;
                out_i[n] = im;
            }
        }
    }
}

}  // namespace mri
