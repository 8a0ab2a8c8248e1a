// kernels_grid_tc.cu -- tensor-core separable-grid kernels (gather_grid_tc.cuh).
#include "gather_grid_tc.cuh"
#include "launch.h"

namespace mri {

namespace {
template <bool REALW, int TRIG>
cudaError_t run(const GridParams& p, dim3 grid, cudaStream_t s)
{
    const size_t smem = grid_tc_smem_bytes(REALW);
    const cudaError_t attr = cudaFuncSetAttribute(
        gather_grid_tc_kernel<REALW, TRIG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        int(smem));
    if (attr != cudaSuccess) return attr;
    gather_grid_tc_kernel<REALW, TRIG><<<grid, kTcThreads, smem, s>>>(p);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_grid_tc(bool realw, int trig, const GridParams& p, dim3 grid, cudaStream_t s)
{
    if (!grid_tc_fits(p.nx)) return cudaErrorInvalidValue;
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

cudaError_t launch_build_ex_tiles(int trig, const float* rec, bool realw, int64_t ntiles,
                                  const float* xs, unsigned char* s_tab, int grid, cudaStream_t s)
{
    const int fields = realw ? 4 : 5;
    switch (trig) {
        case TRIG_ACCURATE:
            build_ex_tiles_kernel<TRIG_ACCURATE><<<grid, 256, 0, s>>>(rec, fields, ntiles, xs, s_tab);
            break;
        case TRIG_FAST:
            build_ex_tiles_kernel<TRIG_FAST><<<grid, 256, 0, s>>>(rec, fields, ntiles, xs, s_tab);
            break;
        case TRIG_FAST_RR:
            build_ex_tiles_kernel<TRIG_FAST_RR><<<grid, 256, 0, s>>>(rec, fields, ntiles, xs, s_tab);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_prep_grid_tc(bool realw, const PrepParams& p, int grid, cudaStream_t s)
{
    if (realw)
        prep_records_kernel<1, true, kTcTile><<<grid, 256, 0, s>>>(p);
    else
        prep_records_kernel<1, false, kTcTile><<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mri
