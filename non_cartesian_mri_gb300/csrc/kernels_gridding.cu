// kernels_gridding.cu -- the gridding reconstruction the chapter compares the
// iterative one with (section 17.1, Fig. 17.1B; Fig. 17.19): the samples'
// Mu = conj(Phi) D interpolated onto the Cartesian k-space grid of the voxel
// grid (trilinear: the 2 x 2 x 2 grid points around a sample), then the
// inverse DFT of that grid onto the voxels x = i - n/2.
//
// The k-grid point g of an axis of n voxels sits at k_g = (g - n/2) / n;
// k is periodic with period 1 on the integer voxel grid, so grid indices wrap
// modulo n.  The centring of both grids is folded into signs:
// e^{i 2 pi k_g x} = e^{i 2 pi g i / n} (-1)^g (-1)^i (-1)^{n/2}, so the
// scatter adds Mu w (-1)^g, the library's inverse FFT (fft.cuh, unscaled)
// does the sum, and its last axis multiplies by (-1)^i (-1)^{n/2} as it
// writes the output.
#include <algorithm>
#include <cstdint>

#include "launch.h"

namespace mri {

namespace {

// The central block of the k-grid a CTA accumulates in shared memory:
// kHot^3 grid points around k = 0 (indices n/2 - kHot/2 .. n/2 + kHot/2 - 1
// of each axis of at least kHot points; a shorter axis is all central).
// Trajectories that pass through the centre (radial lines, spiral
// interleaves) put a large share of their samples' contributions on these
// few points, and atomic adds to one address are serialised in L2: summed
// per CTA first, each central point then takes one global add per CTA.
#ifndef MRI_GRID_HOT
#define MRI_GRID_HOT 8
#endif
#ifndef MRI_GRID_CTAS_PER_SM
#define MRI_GRID_CTAS_PER_SM 4
#endif
constexpr int kHot = MRI_GRID_HOT;

// Grid-point index a of an axis of n points (power of two) -> its index in
// the central block, or -1 when outside it.
__device__ __forceinline__ int hot_index(int a, int n)
{
    const int h = n < kHot ? n : kHot;
    const int r = a - (n >> 1) + (h >> 1);   // the block starts at n/2 - h/2
    return (r >= 0 && r < h) ? r : -1;
}

// Each CTA takes a contiguous run of samples (one thread per sample per
// pass): their eight corner contributions go by atomic adds of (re, im)
// pairs to the grid, those on the central block to the CTA's shared copy,
// which is added to the grid at the end.  g0 = floor(k n) + n/2 and
// f = k n - floor(k n) are exact in float (k n is k scaled by a power of
// two).
__global__ void __launch_bounds__(256) grid_scatter_kernel(
    const float* __restrict__ kx, const float* __restrict__ ky, const float* __restrict__ kz,
    const float* __restrict__ rPhi, const float* __restrict__ iPhi, const float* __restrict__ rD,
    const float* __restrict__ iD, int64_t M, int nx, int ny, int nz, float2* G)
{
    __shared__ float hot_r[kHot * kHot * kHot], hot_i[kHot * kHot * kHot];
    for (int i = threadIdx.x; i < kHot * kHot * kHot; i += blockDim.x) hot_r[i] = hot_i[i] = 0.f;
    __syncthreads();
    const int n[3] = {nx, ny, nz};
    const int64_t per = (M + gridDim.x - 1) / gridDim.x;
    const int64_t m0 = blockIdx.x * per;
    const int64_t m1 = m0 + per < M ? m0 + per : M;
    for (int64_t m = m0 + threadIdx.x; m < m1; m += blockDim.x) {
        // Mu = conj(Phi) D
        const float pr = rPhi[m], pi = iPhi[m], dr = rD[m], di = iD[m];
        const float mr = pr * dr + pi * di;
        const float mi = pr * di - pi * dr;
        int g[3];
        float f[3];
        const float k[3] = {kx[m], ky[m], kz[m]};
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            const float u = k[a] * float(n[a]);
            const float fl = floorf(u);
            f[a] = u - fl;
            // modulo n, n a power of two; the sum may be negative
            g[a] = (int(fl) + (n[a] >> 1)) & (n[a] - 1);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int cx = c & 1, cy = (c >> 1) & 1, cz = c >> 2;
            const int gx = (g[0] + cx) & (nx - 1);
            const int gy = (g[1] + cy) & (ny - 1);
            const int gz = (g[2] + cz) & (nz - 1);
            float w = (cx ? f[0] : 1.f - f[0]) * (cy ? f[1] : 1.f - f[1]) *
                      (cz ? f[2] : 1.f - f[2]);
            if ((gx + gy + gz) & 1) w = -w;   // (-1)^g of the centring
            const int hx = hot_index(gx, nx), hy = hot_index(gy, ny), hz = hot_index(gz, nz);
            if ((hx | hy | hz) >= 0) {
                const int h = (hz * kHot + hy) * kHot + hx;
                atomicAdd(&hot_r[h], w * mr);
                atomicAdd(&hot_i[h], w * mi);
            } else {
                atomicAdd(&G[(int64_t(gz) * ny + gy) * nx + gx], make_float2(w * mr, w * mi));
            }
        }
    }
    __syncthreads();
    // the CTA's central sums, one global add per point it touched
    const int hx0 = (nx >> 1) - ((nx < kHot ? nx : kHot) >> 1);
    const int hy0 = (ny >> 1) - ((ny < kHot ? ny : kHot) >> 1);
    const int hz0 = (nz >> 1) - ((nz < kHot ? nz : kHot) >> 1);
    for (int i = threadIdx.x; i < kHot * kHot * kHot; i += blockDim.x) {
        const float vr = hot_r[i], vi = hot_i[i];
        if (vr == 0.f && vi == 0.f) continue;
        const int gx = hx0 + i % kHot, gy = hy0 + (i / kHot) % kHot, gz = hz0 + i / (kHot * kHot);
        atomicAdd(&G[(int64_t(gz) * ny + gy) * nx + gx], make_float2(vr, vi));
    }
}

// The last non-trivial axis of the inverse FFT with the output folded in:
// each transformed value goes straight to out (SoA) times the centring sign
// c (-1)^(ix + iy + iz), c = (-1)^(nx/2 + ny/2 + nz/2), instead of a separate
// pass over the grid.  Lines as fft_axis_kernel's (element j of line (o, i)
// at (o L + j) inner + i, which is also the voxel index).
template <int LOG2L, bool CONTIG>
__global__ void __launch_bounds__(kFftThreads, fft_min_ctas(LOG2L))
    grid_last_axis_kernel(const float2* a, int log2inner, int64_t lines, const float2* tw,
                          int log2nx, int log2ny, int c, float* outr, float* outi,
                          int accumulate)
{
    extern __shared__ float2 fft_sm[];
    constexpr int log2W = fft_log2_lines(LOG2L);
    float2* const buf = fft_sm;
    float2* const tws = fft_sm + (fft_line_stride(LOG2L) << log2W);
    const int64_t group = int64_t(blockIdx.x) << log2W;
    const int64_t inner_mask = (int64_t(1) << log2inner) - 1;
    auto gidx = [&](int w, int j) -> int64_t {
        const int64_t line = group + w;
        if (CONTIG) return (line << LOG2L) + j;
        return ((((line >> log2inner) << LOG2L) + j) << log2inner) + (line & inner_mask);
    };
    pdl_launch_dependents();
    fft_stage_twiddles<LOG2L>(tws, tw);
    pdl_wait();
    constexpr int RL = fft_last_log2r<LOG2L, true>();
    constexpr int last_per = fft_last_per<LOG2L, true>();
    const int64_t xmask = (int64_t(1) << log2nx) - 1, ymask = (int64_t(1) << log2ny) - 1;
    fft_lines<true, LOG2L, true, !CONTIG, false>(
        buf, tws,
        [&](int w, int pos) { return group + w < lines ? a[gidx(w, pos)] : make_float2(0.f, 0.f); },
        [&](auto& y) {
#pragma unroll
            for (int it = 0; it < fft_items(LOG2L, RL); ++it) {
                int w, j;
                if (!fft_item<LOG2L, RL, !CONTIG>(it, w, j) || group + w >= lines) continue;
#pragma unroll
                for (int q = 0; q < (1 << RL); ++q) {
                    const int64_t n = gidx(w, j + q * last_per);
                    const int64_t par = (n & xmask) + ((n >> log2nx) & ymask) + (n >> (log2nx + log2ny));
                    float2 v = y[it][q];
                    if ((par + c) & 1) v = make_float2(-v.x, -v.y);
                    if (accumulate) {
                        v.x += outr[n];
                        v.y += outi[n];
                    }
                    outr[n] = v.x;
                    outi[n] = v.y;
                }
            }
        });
}

int log2_of(int n)
{
    int b = 0;
    while ((1 << b) < n) ++b;
    return b;
}

template <bool CONTIG>
cudaError_t launch_last_axis(const float2* G, int log2L, int log2inner, int64_t lines,
                             const float2* tw, int log2nx, int log2ny, int c, float* outr,
                             float* outi, int accumulate, cudaStream_t s)
{
    auto go = [&](auto kernel) -> cudaError_t {
        const size_t smem = fft_smem_total(log2L);
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        const int64_t W = int64_t(1) << fft_log2_lines(log2L);
        kernel<<<unsigned((lines + W - 1) / W), kFftThreads, smem, s>>>(
            G, log2inner, lines, tw, log2nx, log2ny, c, outr, outi, accumulate);
        return cudaGetLastError();
    };
    switch (log2L) {
        case 1: return go(grid_last_axis_kernel<1, CONTIG>);
        case 2: return go(grid_last_axis_kernel<2, CONTIG>);
        case 3: return go(grid_last_axis_kernel<3, CONTIG>);
        case 4: return go(grid_last_axis_kernel<4, CONTIG>);
        case 5: return go(grid_last_axis_kernel<5, CONTIG>);
        case 6: return go(grid_last_axis_kernel<6, CONTIG>);
        case 7: return go(grid_last_axis_kernel<7, CONTIG>);
        case 8: return go(grid_last_axis_kernel<8, CONTIG>);
        case 9: return go(grid_last_axis_kernel<9, CONTIG>);
        case 10: return go(grid_last_axis_kernel<10, CONTIG>);
    }
    return cudaErrorInvalidValue;
}

// out = c (-1)^(ix + iy + iz) G (+ out), c = (-1)^(nx/2 + ny/2 + nz/2): the
// signs alone, for a 1 x 1 x 1 grid (no FFT axis to fold them into)
__global__ void __launch_bounds__(256) grid_unshift_kernel(const float2* G, int nx, int ny, int nz,
                                                           float* outr, float* outi,
                                                           int accumulate)
{
    const int64_t N = int64_t(nx) * ny * nz;
    const int c = ((nx >> 1) + (ny >> 1) + (nz >> 1)) & 1;
    for (int64_t n = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; n < N;
         n += int64_t(gridDim.x) * blockDim.x) {
        const int64_t ix = n % nx;
        const int64_t iy = (n / nx) % ny;
        const int64_t iz = n / (int64_t(nx) * ny);
        float2 v = G[n];
        if ((ix + iy + iz + c) & 1) v = make_float2(-v.x, -v.y);
        if (accumulate) {
            v.x += outr[n];
            v.y += outi[n];
        }
        outr[n] = v.x;
        outi[n] = v.y;
    }
}

}  // namespace

cudaError_t launch_gridding(const float* kx, const float* ky, const float* kz, const float* rPhi,
                            const float* iPhi, const float* rD, const float* iD, int64_t M,
                            int nx, int ny, int nz, float* outr, float* outi, int accumulate,
                            float2* G, const float2* tw, int sms, cudaStream_t s)
{
    const int64_t N = int64_t(nx) * ny * nz;
    cudaError_t e = cudaMemsetAsync(G, 0, size_t(N) * sizeof(float2), s);
    if (e != cudaSuccess) return e;
    if (M > 0) {
        // a few CTAs per SM, each over a contiguous run of samples: the
        // central grid points take one global add per CTA
        const int64_t blocks =
            std::min<int64_t>((M + 255) / 256, int64_t(sms) * MRI_GRID_CTAS_PER_SM);
        grid_scatter_kernel<<<unsigned(blocks), 256, 0, s>>>(kx, ky, kz, rPhi, iPhi, rD, iD, M,
                                                              nx, ny, nz, G);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // the inverse FFT, its last non-trivial axis writing the output
    const int n[3] = {nx, ny, nz};
    int last = 2;
    while (last >= 0 && n[last] == 1) --last;
    if (last < 0) {
        grid_unshift_kernel<<<1, 256, 0, s>>>(G, nx, ny, nz, outr, outi, accumulate);
        return cudaGetLastError();
    }
    for (int ax = 0; ax < last; ++ax)
        if ((e = launch_fft_axis(G, nx, ny, nz, ax, true, tw, s)) != cudaSuccess) return e;
    const int log2nx = log2_of(nx), log2ny = log2_of(ny);
    const int log2inner = last == 0 ? 0 : (last == 1 ? log2nx : log2nx + log2ny);
    const int log2L = log2_of(n[last]);
    const int c = ((nx >> 1) + (ny >> 1) + (nz >> 1)) & 1;
    return last == 0 ? launch_last_axis<true>(G, log2L, 0, N >> log2L, tw, log2nx, log2ny, c,
                                              outr, outi, accumulate, s)
                     : launch_last_axis<false>(G, log2L, log2inner, N >> log2L, tw, log2nx,
                                               log2ny, c, outr, outi, accumulate, s);
}

}  // namespace mri
