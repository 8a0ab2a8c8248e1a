// kernels_coils_tc.cu -- batched F^H D at arbitrary voxel coordinates on the
// tensor cores (gather_coils_tc.cuh): the weight tiles and the kernel.
#include "gather_coils_tc.cuh"
#include "launch.h"

namespace mri {

// The B tiles: for record tile t, S (24 rows: -Mu_i, Mu_r, Mu_i of coils 0-7)
// x 32 samples, f16 hi then lo, K-major core matrices (8 rows x 8 samples).
// Coil c's weights are multiplied by its power of two 2^e_c (from its bound
// word, so that every scaled weight is below 2^15 and its f16 parts keep
// their precision whatever the other coils' magnitudes).  One thread per
// (tile, row, 8-sample chunk).
__global__ void __launch_bounds__(256) build_mu_tiles_kernel(const float* rec, int64_t ntiles,
                                                             const unsigned int* bounds,
                                                             unsigned char* s_tab)
{
    constexpr int ITEMS = kCtSRows * (kTcTile / 8);   // 96 per tile
    const int64_t total = ntiles * ITEMS;
    for (int64_t item = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; item < total;
         item += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = item / ITEMS;
        const int r = int(item - t * ITEMS);
        const int row = r >> 2, kc = r & 3;           // S row, samples 8 kc ..
        const int coil = row & 7, grp = row >> 3;     // 0: -Mu_i, 1: Mu_r, 2: Mu_i
        const float* w = rec + t * kCtFields * kTcTile +
                         (3 + (grp == 1 ? 0 : kCtCoils) + coil) * kTcTile + 8 * kc;
        const float scale = exp2_int(tc_scale_exp(bounds[coil]));
        float v[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) v[s] = (grp == 0 ? -w[s] : w[s]) * scale;
        uint4 h, l;
        tc_split8(v, h, l);
        unsigned char* const tile = s_tab + t * kCtBBytes;
        const int off = (row >> 3) * 512 + kc * 128 + (row & 7) * 16;
        *reinterpret_cast<uint4*>(tile + off) = h;
        *reinterpret_cast<uint4*>(tile + kCtPartBytes + off) = l;
    }
}

namespace {
template <int TRIG>
cudaError_t run_coils_tc(const CoilTcParams& p, dim3 grid, cudaStream_t s)
{
    auto kernel = coils_tc_kernel<TRIG>;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kCtSmem));
    if (e != cudaSuccess) return e;
    kernel<<<grid, kCtThreads, kCtSmem, s>>>(p);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_build_mu_tiles(const float* rec, int64_t ntiles, const unsigned int* bounds,
                                  unsigned char* s_tab, int grid, cudaStream_t s)
{
    build_mu_tiles_kernel<<<grid, 256, 0, s>>>(rec, ntiles, bounds, s_tab);
    return cudaGetLastError();
}

cudaError_t launch_gather_coils_tc(int trig, const CoilTcParams& p, dim3 grid, cudaStream_t s)
{
    if (p.coils < 1 || p.coils > kCtCoils) return cudaErrorInvalidValue;
    switch (trig) {
        case TRIG_ACCURATE: return run_coils_tc<TRIG_ACCURATE>(p, grid, s);
        case TRIG_FAST: return run_coils_tc<TRIG_FAST>(p, grid, s);
        case TRIG_FAST_RR: return run_coils_tc<TRIG_FAST_RR>(p, grid, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mri
