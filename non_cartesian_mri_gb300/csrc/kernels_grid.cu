// kernels_grid.cu -- separable-grid F^H D / Q instantiations (gather_grid.cuh).
#include "gather_grid.cuh"
#include "launch.h"

namespace mri {

// Voxel coordinates of a separable grid, for grids the table kernel does not
// take (nx not a divisor of 256): x[n], y[n], z[n] for n = (iz*ny + iy)*nx + ix.
__global__ void __launch_bounds__(256) expand_grid_kernel(const float* xs, const float* ys,
                                                          const float* zs, int nx, int ny,
                                                          int64_t N, float* x, float* y,
                                                          float* z)
{
    for (int64_t n = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; n < N;
         n += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = n / nx;
        const int64_t ix = n - row * nx;
        const int64_t iz = row / ny;
        const int64_t iy = row - iz * ny;
        x[n] = xs[ix];
        y[n] = ys[iy];
        z[n] = zs[iz];
    }
}


cudaError_t launch_grid(bool realw, int trig, const GridParams& p, dim3 grid, cudaStream_t s)
{
    switch (p.nx) {
        case 32: return launch_grid_32(realw, trig, p, grid, s);
        case 64: return launch_grid_64(realw, trig, p, grid, s);
        case 128: return launch_grid_128(realw, trig, p, grid, s);
        case 256: return launch_grid_256(realw, trig, p, grid, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_prep_grid(bool realw, const PrepParams& p, int grid, cudaStream_t s)
{
    if (realw)
        prep_records_kernel<1, true, kGridTile><<<grid, 256, 0, s>>>(p);
    else
        prep_records_kernel<1, false, kGridTile><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_expand_grid(const float* xs, const float* ys, const float* zs, int nx, int ny,
                               int64_t N, float* x, float* y, float* z, int grid, cudaStream_t s)
{
    expand_grid_kernel<<<grid, 256, 0, s>>>(xs, ys, zs, nx, ny, N, x, y, z);
    return cudaGetLastError();
}

}  // namespace mri
