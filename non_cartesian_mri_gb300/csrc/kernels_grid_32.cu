// kernels_grid_32.cu -- separable-grid kernels for nx = 32 (gather_grid.cuh).
#include "gather_grid.cuh"
#include "launch.h"

namespace mri {

namespace {
template <bool REALW, int TRIG>
cudaError_t run(const GridParams& p, dim3 grid, cudaStream_t s)
{
    const size_t smem = grid_smem_bytes(32, REALW);
    const cudaError_t attr = cudaFuncSetAttribute(
        gather_grid_kernel<REALW, TRIG, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        int(smem));
    if (attr != cudaSuccess) return attr;
    gather_grid_kernel<REALW, TRIG, 32><<<grid, kGridThreads, smem, s>>>(p);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_grid_32(bool realw, int trig, const GridParams& p, dim3 grid, cudaStream_t s)
{
    if (realw) {
        switch (trig) {
            case TRIG_ACCURATE: return run<true, TRIG_ACCURATE>(p, grid, s);
            case TRIG_FAST: return run<true, TRIG_FAST>(p, grid, s);
            case TRIG_FAST_RR: return run<true, TRIG_FAST_RR>(p, grid, s);
        }
    } else {
        switch (trig) {
            case TRIG_ACCURATE: return run<false, TRIG_ACCURATE>(p, grid, s);
            case TRIG_FAST: return run<false, TRIG_FAST>(p, grid, s);
            case TRIG_FAST_RR: return run<false, TRIG_FAST_RR>(p, grid, s);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace mri
