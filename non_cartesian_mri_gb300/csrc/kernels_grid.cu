// kernels_grid.cu -- voxel coordinates of a separable grid, for the grids
// the tensor-core kernels do not take (gather_grid_tc.cuh: nx < 8).
#include "gather_grid.cuh"
#include "launch.h"

namespace mri {

// x[n], y[n], z[n] for n = (iz*ny + iy)*nx + ix.
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


cudaError_t launch_expand_grid(const float* xs, const float* ys, const float* zs, int nx, int ny,
                               int64_t N, float* x, float* y, float* z, int grid, cudaStream_t s)
{
    expand_grid_kernel<<<grid, 256, 0, s>>>(xs, ys, zs, nx, ny, N, x, y, z);
    return cudaGetLastError();
}

}  // namespace mri
