// kernels_coils.cu -- batched F^H D instantiations for coil groups of 2, 4, 8.
#include "launch.h"

namespace mri {

namespace {
template <int BC, int TRIG>
cudaError_t run_gather(const GatherParams& p, dim3 grid, cudaStream_t s)
{
    using Sh = PairCoilShape<BC>;
    const cudaError_t attr = cudaFuncSetAttribute(
        gather_pair_coils_kernel<BC, TRIG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        int(Sh::SMEM));
    if (attr != cudaSuccess) return attr;
    gather_pair_coils_kernel<BC, TRIG><<<grid, Sh::THREADS, Sh::SMEM, s>>>(p);
    return cudaGetLastError();
}

template <int BC>
cudaError_t by_trig(int trig, const GatherParams& p, dim3 grid, cudaStream_t s)
{
    switch (trig) {
        case TRIG_ACCURATE: return run_gather<BC, TRIG_ACCURATE>(p, grid, s);
        case TRIG_FAST: return run_gather<BC, TRIG_FAST>(p, grid, s);
        case TRIG_FAST_RR: return run_gather<BC, TRIG_FAST_RR>(p, grid, s);
    }
    return cudaErrorInvalidValue;
}
}  // namespace

cudaError_t launch_gather_coils(int bc, int trig, const GatherParams& p, dim3 grid,
                                cudaStream_t s)
{
    switch (bc) {
        case 2: return by_trig<2>(trig, p, grid, s);
        case 4: return by_trig<4>(trig, p, grid, s);
        case 8: return by_trig<8>(trig, p, grid, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_prep_coils(int bc, const PrepParams& p, int grid, cudaStream_t s)
{
    switch (bc) {
        case 2: prep_pair_coil_records_kernel<2><<<grid, 256, 0, s>>>(p); break;
        case 4: prep_pair_coil_records_kernel<4><<<grid, 256, 0, s>>>(p); break;
        case 8: prep_pair_coil_records_kernel<8><<<grid, 256, 0, s>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mri
