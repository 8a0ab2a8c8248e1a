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
// does the sum, and the last kernel multiplies by (-1)^i (-1)^{n/2}.
#include <algorithm>
#include <cstdint>

#include "launch.h"

namespace mri {

namespace {

// One thread per sample: its eight corner contributions by atomic adds of
// (re, im) pairs.  g0 = floor(k n) + n/2 and f = k n - floor(k n) are exact
// in float (k n is k scaled by a power of two).
__global__ void __launch_bounds__(256) grid_scatter_kernel(
    const float* __restrict__ kx, const float* __restrict__ ky, const float* __restrict__ kz,
    const float* __restrict__ rPhi, const float* __restrict__ iPhi, const float* __restrict__ rD,
    const float* __restrict__ iD, int64_t M, int nx, int ny, int nz, float2* G)
{
    for (int64_t m = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; m < M;
         m += int64_t(gridDim.x) * blockDim.x) {
        // Mu = conj(Phi) D
        const float pr = rPhi[m], pi = iPhi[m], dr = rD[m], di = iD[m];
        const float mr = pr * dr + pi * di;
        const float mi = pr * di - pi * dr;
        int g[3];
        float f[3];
        const float k[3] = {kx[m], ky[m], kz[m]};
        const int n[3] = {nx, ny, nz};
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
            atomicAdd(&G[(int64_t(gz) * ny + gy) * nx + gx], make_float2(w * mr, w * mi));
        }
    }
}

// out = c (-1)^(ix + iy + iz) G (+ out), c = (-1)^(nx/2 + ny/2 + nz/2)
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
        const int64_t blocks = std::min<int64_t>((M + 255) / 256, int64_t(sms) * 16);
        grid_scatter_kernel<<<unsigned(blocks), 256, 0, s>>>(kx, ky, kz, rPhi, iPhi, rD, iD, M,
                                                              nx, ny, nz, G);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = launch_fft3(G, nx, ny, nz, true, tw, s)) != cudaSuccess) return e;
    const int64_t blocks = std::min<int64_t>((N + 255) / 256, int64_t(sms) * 16);
    grid_unshift_kernel<<<unsigned(blocks), 256, 0, s>>>(G, nx, ny, nz, outr, outi, accumulate);
    return cudaGetLastError();
}

}  // namespace mri
