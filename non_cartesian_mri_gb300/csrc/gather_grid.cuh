// gather_grid.cuh -- F^H D and Q for voxels on a separable grid.
//
// When the voxels form a grid xs[nx] x ys[ny] x zs[nz] (voxel n = (iz*ny + iy)*nx + ix,
// x fastest; every workload of the chapter is such a grid), the kernel of
// the register-promoted gather (Fig. 17.11) factors:
//
//   e^{i 2 pi k.x_n} = Ex[m][ix] * Eyz[m][iy, iz]
//   Ex  = e^{i 2 pi kx xs[ix]},   Eyz = e^{i 2 pi (ky ys[iy] + kz zs[iz])}.
//
// A CTA owns R = 2048 / nx whole grid rows (fixed iy, iz; all ix).  For each
// tile of kGridTile samples it builds, in shared memory,
//   Ex[s][ix]   for the tile's samples and all nx columns, and
//   Mz[s][r]    = Mu[s] * Eyz[s][row r]   for its R rows
// (Mu = conj(Phi) D for F^H D, |Phi|^2 for Q), after which every voxel-sample
// pair is one complex multiply-accumulate, acc += Mz[s][r] * Ex[s][ix]: four
// FFMA and one broadcast shared-memory load.  The sin/cos work drops from two
// per pair to (nx + R) per (tile sample, CTA), i.e. 1/R + 1/nx per pair, so
// the accurate polynomial trig costs little more than the SFU one.
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
constexpr int kGridV = 8;          // voxels per thread
constexpr int kGridVoxelsPerCta = kGridThreads * kGridV;   // 2048: R = 2048 / nx rows

struct GridParams {
    const float* rec;       // tile-major records, kGridTile samples per tile
    int64_t ntiles;
    int splits;
    const float *xs, *ys, *zs;
    int nx, ny, nz;
    int rows_per_cta;       // 2048 / nx
    float* out_r;           // as GatherParams, one coil
    float* out_i;
    int64_t split_stride;
    int accumulate;
    unsigned int* err;
};

// The table kernel takes nx in {16, 32, ..., 256}: nx divides 256, so each
// thread keeps one column ix for all its voxels, and the tables fit shared
// memory (nx = 16 gives R = 128 rows).
inline bool grid_kernel_fits(int nx)
{
    return nx >= 16 && nx <= 256 && (256 % nx) == 0;
}

// Dynamic shared memory of the grid kernel for a given nx.
inline size_t grid_smem_bytes(int nx, bool realw)
{
    const int F = realw ? 4 : 5;
    const int R = kGridVoxelsPerCta / nx;
    size_t b = size_t(kStages) * F * kGridTile * 4;          // record ring
    b += 2 * size_t(kGridTile) * (size_t(nx) + R) * 8;        // Ex and Mz, double-buffered
    b += size_t(nx) * 4 + size_t(R) * 8;                      // xs, (y, z) of the rows
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

template <bool REALW, int TRIG, bool FIXED_IX>
__global__ void __launch_bounds__(kGridThreads, 2) gather_grid_kernel(GridParams p)
{
    constexpr int T = kGridTile;
    constexpr int F = REALW ? 4 : 5;
    constexpr uint32_t TILE_BYTES = uint32_t(F) * T * 4;
    constexpr int V = kGridV;

    const int nx = p.nx;
    const int R = p.rows_per_cta;
    const int64_t total_rows = int64_t(p.ny) * p.nz;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* const ring = reinterpret_cast<float*>(smem_raw);
    float2* const ex_tab = reinterpret_cast<float2*>(ring + kStages * F * T);   // [2][T][nx]
    float2* const mz_tab = ex_tab + 2 * T * nx;                                 // [2][T][R]
    float2* const yz_sh = mz_tab + 2 * T * R;                                   // [R] (y, z)
    float* const xs_sh = reinterpret_cast<float*>(yz_sh + R);                   // [nx]
    __shared__ __align__(8) uint64_t full_bar[kStages];

    const int tid = threadIdx.x;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t row0 = int64_t(blockIdx.x) * R;

    // the thread's voxels: local slot j*256 + tid -> (row, ix)
    int ix_of[V], row_of[V];
#pragma unroll
    for (int j = 0; j < V; ++j) {
        const int local = j * kGridThreads + tid;
        ix_of[j] = local % nx;
        row_of[j] = local / nx;
    }

    for (int i = tid; i < nx; i += kGridThreads) xs_sh[i] = p.xs[i];
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

    float run_r[V], run_i[V];
#pragma unroll
    for (int j = 0; j < V; ++j) run_r[j] = run_i[j] = 0.0f;

    int failed_at = -1;
    for (int t = 0; t < nt; ++t) {
        const int st = t % kStages;
        const bool ok = mbar_wait_bounded(&full_bar[st], uint32_t(t / kStages) & 1u);
        const float* rec = ring + st * F * T;
        float2* const ex = ex_tab + (t & 1) * T * nx;
        float2* const mz = mz_tab + (t & 1) * T * R;
        if (ok) {
            // Ex[s][ix] = e^{i phase(kx[s] xs[ix])}
            for (int e = tid; e < T * nx; e += kGridThreads) {
                const int s = e / nx;
                const int i = e - s * nx;
                float sn, cs;
                table_sincos<TRIG>(rec[s] * xs_sh[i], sn, cs);
                ex[e] = make_float2(cs, sn);
            }
            // Mz[s][r] = Mu[s] * e^{i phase(ky[s] y_r + kz[s] z_r)}
            for (int e = tid; e < T * R; e += kGridThreads) {
                const int s = e / R;
                const int r = e - s * R;
                const float2 yz = yz_sh[r];
                float sn, cs;
                table_sincos<TRIG>(fmaf(rec[2 * T + s], yz.y, rec[T + s] * yz.x), sn, cs);
                const float wr = rec[3 * T + s];
                if (REALW) {
                    mz[e] = make_float2(wr * cs, wr * sn);
                } else {
                    const float wi = rec[4 * T + s];
                    mz[e] = make_float2(fmaf(wr, cs, -wi * sn), fmaf(wi, cs, wr * sn));
                }
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

        float pr[V], pi[V];
#pragma unroll
        for (int j = 0; j < V; ++j) pr[j] = pi[j] = 0.0f;
#pragma unroll 4
        for (int s = 0; s < T; ++s) {
            float2 e0 = make_float2(0.f, 0.f);
            if (FIXED_IX) e0 = ex[s * nx + ix_of[0]];
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const float2 e = FIXED_IX ? e0 : ex[s * nx + ix_of[j]];
                const float2 m = mz[s * R + row_of[j]];
                // (m.x + i m.y)(e.x + i e.y)
                pr[j] = fmaf(m.x, e.x, pr[j]);
                pr[j] = fmaf(-m.y, e.y, pr[j]);
                pi[j] = fmaf(m.x, e.y, pi[j]);
                pi[j] = fmaf(m.y, e.x, pi[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            run_r[j] += pr[j];
            run_i[j] += pi[j];
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
    for (int j = 0; j < V; ++j) {
        const int64_t row = row0 + row_of[j];
        if (row < total_rows) {
            const int64_t n = row * nx + ix_of[j];
            float r = run_r[j], i = run_i[j];
            if (p.accumulate) {
                r = out_r[n] + r;
                i = out_i[n] + i;
            }
            out_r[n] = r;
            out_i[n] = i;
        }
    }
}

}  // namespace mri
