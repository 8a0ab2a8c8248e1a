// kernels_grid_tc.cu -- tensor-core separable-grid kernels (gather_grid_tc.cuh).
#include "gather_grid_tc.cuh"
#include "launch.h"

namespace mri {

namespace {
template <int BC, bool REALW, int TRIG>
cudaError_t run(const GridParams& p, dim3 grid, cudaStream_t s)
{
    const size_t smem = grid_tc_smem_bytes(REALW, BC);
    const cudaError_t attr = cudaFuncSetAttribute(
        gather_grid_tc_kernel<BC, REALW, TRIG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        int(smem));
    if (attr != cudaSuccess) return attr;
    gather_grid_tc_kernel<BC, REALW, TRIG><<<grid, kTcThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int BC, bool REALW>
cudaError_t run_trig(int trig, const GridParams& p, dim3 grid, cudaStream_t s)
{
    switch (trig) {
        case TRIG_ACCURATE: return run<BC, REALW, TRIG_ACCURATE>(p, grid, s);
        case TRIG_FAST: return run<BC, REALW, TRIG_FAST>(p, grid, s);
        case TRIG_FAST_RR: return run<BC, REALW, TRIG_FAST_RR>(p, grid, s);
    }
    return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_grid_tc(bool realw, int trig, int bc, const GridParams& p, dim3 grid,
                           cudaStream_t s)
{
    if (!grid_tc_fits(p.nx)) return cudaErrorInvalidValue;
    if (realw) return bc == 1 ? run_trig<1, true>(trig, p, grid, s) : cudaErrorInvalidValue;
    switch (bc) {
        case 1: return run_trig<1, false>(trig, p, grid, s);
        case 4: return run_trig<4, false>(trig, p, grid, s);
        case 8: return run_trig<8, false>(trig, p, grid, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_build_ex_tiles(int trig, const float* rec, int fields, int64_t ntiles,
                                  const float* xs, unsigned char* s_tab, int grid, cudaStream_t s)
{
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

cudaError_t launch_prep_grid_tc(bool realw, int bc, const PrepParams& p, int grid, cudaStream_t s)
{
    if (realw) {
        if (bc != 1) return cudaErrorInvalidValue;
        prep_records_kernel<1, true, kTcTile, true><<<grid, 256, 0, s>>>(p);
    } else {
        switch (bc) {
            case 1: prep_records_kernel<1, false, kTcTile, true><<<grid, 256, 0, s>>>(p); break;
            case 4: prep_records_kernel<4, false, kTcTile, true><<<grid, 256, 0, s>>>(p); break;
            case 8: prep_records_kernel<8, false, kTcTile, true><<<grid, 256, 0, s>>>(p); break;
            default: return cudaErrorInvalidValue;
        }
    }
    return cudaGetLastError();
}

}  // namespace mri
