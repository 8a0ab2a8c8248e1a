// kernels_coils_tc.cu -- batched F^H D at arbitrary voxel coordinates on the
// tensor cores (gather_coils_tc.cuh): the weight tiles and the kernel.
#include "gather_coils_tc.cuh"
#include "launch.h"

namespace mri {

// The weight tiles: for record tile t, eight 8-row groups (row = coil) x 32
// samples of f16 in K-major core matrices (8 rows x 8 samples, 128 B; 512 B
// per group), [-Mu_i^hi, Mu_r^hi, Mu_r^hi, Mu_i^hi, -Mu_i^lo, Mu_r^lo, Mu_r^lo,
// Mu_i^lo]: the even groups are the window the MMAs of A_i read, the odd ones
// that of A_r.  Coil c's weights are multiplied by its power of two 2^e_c
// (from its bound word, so that every scaled weight is below 2^15 and its f16
// parts keep their precision whatever the other coils' magnitudes).  One
// thread per (tile, coil, 8-sample chunk).
__global__ void __launch_bounds__(256) build_mu_tiles_kernel(const float* rec, int64_t ntiles,
                                                             const unsigned int* bounds,
                                                             unsigned char* s_tab)
{
    constexpr int ITEMS = kCtCoils * (kTcTile / 8);   // 32 per tile
    const int64_t total = ntiles * ITEMS;
    for (int64_t item = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; item < total;
         item += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = item / ITEMS;
        const int r = int(item - t * ITEMS);
        const int coil = r >> 2, kc = r & 3;          // samples 8 kc ..
        const float* wr = rec + t * kCtFields * kTcTile + (3 + coil) * kTcTile + 8 * kc;
        const float* wi = wr + kCtCoils * kTcTile;
        const float scale = exp2_int(tc_scale_exp(bounds[coil]));
        float vr[8], vi[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            vr[s] = wr[s] * scale;
            vi[s] = wi[s] * scale;
        }
        uint4 rh, rl, ih, il;
        tc_split8(vr, rh, rl);
        tc_split8(vi, ih, il);
        unsigned char* const row = s_tab + t * kCtBBytes + kc * 128 + coil * 16;
        const uint4 g[kCtGroups] = {neg_f16x8(ih), rh, rh, ih, neg_f16x8(il), rl, rl, il};
#pragma unroll
        for (int j = 0; j < kCtGroups; ++j) *reinterpret_cast<uint4*>(row + j * 512) = g[j];
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
