// gather_grid.cuh -- shared pieces of F^H D, Q and the forward model for
// voxels on a separable grid.
//
// When the voxels form a grid xs[nx] x ys[ny] x zs[nz] (voxel n = (iz*ny + iy)*nx + ix,
// x fastest; every workload of the chapter is such a grid), the kernel of
// the register-promoted gather (Fig. 17.11) factors:
//
//   e^{i 2 pi k.x_n} = Ex[m][ix] * Eyz[m][iy, iz]
//   Ex  = e^{i 2 pi kx xs[ix]},   Eyz = e^{i 2 pi (ky ys[iy] + kz zs[iz])},
//
// so F^H D over a grid is the complex matrix product
//   FhD[row][ix] = sum_m (Mu[m] Eyz[m][row]) Ex[m][ix]
// (row = (iz, iy)), which the tensor-core kernels compute
// (gather_grid_tc.cuh, gather_grid_tc_fwd.cuh for the forward model).  The
// sin/cos work drops from two per voxel-sample pair to one pair per
// (sample, column) and per (sample, row).  This header holds their launch
// parameters and the per-factor sin/cos of each trig path.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather.cuh"

namespace mri {

// F^H D / Q on a grid (tensor-core kernel, gather_grid_tc.cuh).
struct GridParams {
    const float* rec;       // tile-major records, 32 samples per tile
    int64_t ntiles;
    int splits;
    const float *xs, *ys, *zs;
    int nx, ny, nz;
    int rows_per_cta;       // 128 / coils per CTA
    float* out_r;           // as GatherParams; coil b at out_r + b * coil_stride
    float* out_i;
    int64_t split_stride;
    int accumulate;
    unsigned int* err;
    // per coil of the group: float bits of max |w_r| + |w_i| over the
    // samples (the coil's weights are scaled by their own power of two); and
    // the B operand tiles (kTcStageBytes per record tile and column block)
    const unsigned int* wbound;
    const unsigned char* s_tab;
    // coil groups: coils present, and the output offset of one coil
    int coils;
    int64_t coil_stride;
    // column blocks of 128 (the last may be partly padding)
    int ncb;
    // Row folding (nx <= 64): with fold > 1 and the check word `fold_ok`
    // set, a block's 128 columns are `fold` consecutive grid rows of
    // 2^log2_fw columns each (column c: row offset c >> log2_fw, x index
    // c & (2^log2_fw - 1)), and an MMA row is a group of `fold` grid rows;
    // with the word clear the unfolded layout runs (a CTA whose rows lie past
    // the folded row count exits at once).
    int fold;
    int log2_fw;
    const unsigned int* fold_ok;
};

// Forward model on a grid (tensor-core kernel, gather_grid_tc_fwd.cuh).
struct FwdParams {
    const float *kx, *ky, *kz;       // M samples
    int64_t M;
    float kscale;                    // phase units of the trig path
    const float* xs;                 // nx columns
    int nx;
    int ncb;                         // column blocks of 128
    const float2* yz_rows;           // (y, z) of every row, padded to whole blocks
    const float* row_step;           // per group of 8 rows: the y step when the group's
                                     // rows share z and are evenly spaced in y, else NaN
    int64_t row_blocks;
    int splits;                      // CTAs along the row blocks
    const unsigned char* rho_tab;    // chunks [row block][column block][chunk], kFwChunkBytes each
    const unsigned int* bound;       // float bits of max |rho_r| + |rho_i|
    float* out_r;                    // [split][M] or the caller's arrays
    float* out_i;
    int64_t split_stride;
    int accumulate;
    unsigned int* err;
};

template <int TRIG>
__device__ __forceinline__ void table_sincos(float ph, float& s, float& c)
{
    if (TRIG == TRIG_ACCURATE) {
        sincos_half_turns(ph, s, c);             // records hold 2k: half turns
    } else if (TRIG == TRIG_FAST) {
        __sincosf(ph, &s, &c);                   // records hold 2 pi k: radians
    } else {
        const float rn = (ph + 12582912.0f) - 12582912.0f;   // records hold k: turns
        __sincosf((ph - rn) * 6.28318530717958647692f, &s, &c);
    }
}

}  // namespace mri
