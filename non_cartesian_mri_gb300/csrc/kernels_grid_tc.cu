// kernels_grid_tc.cu -- tensor-core separable-grid kernels (gather_grid_tc_ws.cuh,
// gather_grid_tc_fwd.cuh) and their per-call operand tables (gather_grid_tc.cuh).
#include "gather_grid_tc.cuh"
#include "gather_grid_tc_fwd.cuh"
#include "gather_grid_tc_ws.cuh"
#include "launch.h"

namespace mri {

namespace {
template <int BC, bool REALW, int TRIG>
cudaError_t run_ws(const GridParams& p, dim3 grid, cudaStream_t s)
{
    auto kernel = gather_grid_tc_ws_kernel<BC, REALW, TRIG>;
    // the warpgroup register budgets must fit the registers the CTA is
    // launched with, or a budget increase would wait forever
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kWsThreads < 32 * kWsGenWarps * kWsGenRegs + 128 * kWsAuxRegs)
        return cudaErrorInvalidConfiguration;
    const size_t smem = grid_tc_ws_smem_bytes(REALW, BC);
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    kernel<<<grid, kWsThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int BC, bool REALW>
cudaError_t run_trig(int trig, const GridParams& p, dim3 grid, cudaStream_t s)
{
    switch (trig) {
        case TRIG_ACCURATE: return run_ws<BC, REALW, TRIG_ACCURATE>(p, grid, s);
        case TRIG_FAST: return run_ws<BC, REALW, TRIG_FAST>(p, grid, s);
        case TRIG_FAST_RR: return run_ws<BC, REALW, TRIG_FAST_RR>(p, grid, s);
    }
    return cudaErrorInvalidValue;
}
}  // namespace

int grid_tc_threads()
{
    return kWsThreads;
}


// One CTA: *ok = 1 when the offsets of every group of G rows from its first
// row equal those of the first group exactly and are floats themselves;
// dy[j] = those offsets.  Otherwise *ok = 0 and the unfolded layout runs.
// The differences are taken in double, where the difference of two floats is
// exact unless their exponents are far apart; a - d == b confirms it.
__global__ void __launch_bounds__(256) grid_fold_check_kernel(const float* ys, int ny, int G,
                                                              unsigned int* ok, float* dy)
{
    bool good = true;
    for (int i = threadIdx.x; i < ny; i += blockDim.x) {
        const int j = i % G;
        const double a = ys[i], b = ys[i - j], a0 = ys[j], b0 = ys[0];
        const double d = a - b, d0 = a0 - b0;
        good = good && a - d == b && a0 - d0 == b0 && d == d0 && double(float(d0)) == d0;
    }
    good = __syncthreads_and(good) != 0;
    if (int(threadIdx.x) < G) dy[threadIdx.x] = float(double(ys[threadIdx.x]) - double(ys[0]));
    if (threadIdx.x == 0) *ok = good ? 1u : 0u;
}

cudaError_t launch_grid_fold_check(const float* ys, int ny, int G, unsigned int* ok, float* dy,
                                   cudaStream_t s)
{
    if (G < 2 || G > kTcCols / kTcMinCols || ny % G != 0) return cudaErrorInvalidValue;
    grid_fold_check_kernel<<<1, 256, 0, s>>>(ys, ny, G, ok, dy);
    return cudaGetLastError();
}

cudaError_t launch_grid_tc(bool realw, int trig, int bc, const GridParams& p, dim3 grid,
                           cudaStream_t s)
{
    if (!grid_tc_fits(p.nx)) return cudaErrorInvalidValue;
    if (p.fold > 1 && (p.fold != grid_tc_fold(p.nx, p.ny) || p.fold_ok == nullptr ||
                       p.log2_fw != grid_tc_fold_log2_width(p.fold)))
        return cudaErrorInvalidValue;
    if (realw) {
        if (bc != 1) return cudaErrorInvalidValue;
        return run_trig<1, true>(trig, p, grid, s);
    }
    switch (bc) {
        case 1: return run_trig<1, false>(trig, p, grid, s);
        case 4: return run_trig<4, false>(trig, p, grid, s);
        case 8: return run_trig<8, false>(trig, p, grid, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_build_ex_tiles(int trig, bool mub, const float* rec, int fields,
                                  int64_t ntiles, const float* xs, int nx, unsigned char* s_tab,
                                  int grid, cudaStream_t s, int fold,
                                  const unsigned int* fold_ok, const float* fold_dy)
{
    const int ncb = grid_tc_col_blocks(nx);
    if (fold > 1 && (ncb != 1 || fold_ok == nullptr || fold_dy == nullptr))
        return cudaErrorInvalidValue;
    const int log2_fw = grid_tc_fold_log2_width(fold);
    auto go = [&](auto kernel) {
        kernel<<<grid, 256, 0, s>>>(rec, fields, ntiles, xs, nx, ncb, s_tab, fold, log2_fw,
                                    fold_ok, fold_dy);
        return cudaGetLastError();
    };
    switch (trig) {
        case TRIG_ACCURATE:
            return mub ? go(build_ex_tiles_kernel<TRIG_ACCURATE, true>)
                       : go(build_ex_tiles_kernel<TRIG_ACCURATE, false>);
        case TRIG_FAST:
            return mub ? go(build_ex_tiles_kernel<TRIG_FAST, true>)
                       : go(build_ex_tiles_kernel<TRIG_FAST, false>);
        case TRIG_FAST_RR:
            return mub ? go(build_ex_tiles_kernel<TRIG_FAST_RR, true>)
                       : go(build_ex_tiles_kernel<TRIG_FAST_RR, false>);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_forward_grid_tc(int trig, const FwdParams& p, dim3 grid, cudaStream_t s)
{
    const size_t smem = grid_tc_fwd_smem_bytes();
    auto go = [&](auto kernel) -> cudaError_t {
        const cudaError_t attr =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (attr != cudaSuccess) return attr;
        kernel<<<grid, kFwThreads, smem, s>>>(p);
        return cudaGetLastError();
    };
    switch (trig) {
        case TRIG_ACCURATE: return go(forward_grid_tc_kernel<TRIG_ACCURATE>);
        case TRIG_FAST: return go(forward_grid_tc_kernel<TRIG_FAST>);
        case TRIG_FAST_RR: return go(forward_grid_tc_kernel<TRIG_FAST_RR>);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_forward_grid_prep(const float* rr, const float* ri, int64_t rows, int nx,
                                     int64_t row_blocks, const float* ys, int ny, const float* zs,
                                     unsigned int* bound, unsigned char* tab, float2* yz_rows,
                                     float* row_step, int grid, cudaStream_t s)
{
    if (cudaMemsetAsync(bound, 0, sizeof(unsigned int), s) != cudaSuccess)
        return cudaErrorUnknown;
    rho_bound_kernel<<<grid, 256, 0, s>>>(rr, ri, rows * nx, bound);
    build_rho_tiles_kernel<<<grid, 256, 0, s>>>(rr, ri, rows, nx, grid_tc_col_blocks(nx),
                                                row_blocks, bound, tab);
    build_row_coords_kernel<<<grid, 256, 0, s>>>(ys, ny, zs, rows, row_blocks * kFwRows, yz_rows,
                                                 row_step);
    return cudaGetLastError();
}

// Multiply the weights of the records (fields 3 .. fields - 1 of every
// tile) by the power of two 2^e taken from the bound word, so that every A
// value the kernel makes from them is below 2^kTcAExp (see tc_scale_exp); the
// kernel multiplies its results by 2^-e.
__global__ void __launch_bounds__(256) scale_records_kernel(float* rec, int fields,
                                                            int64_t ntiles,
                                                            const unsigned int* bound, int bc)
{
    const int per_tile = (fields - 3) * kTcTile;
    const int64_t total = ntiles * per_tile;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = i / per_tile;
        const int j = int(i - t * per_tile);
        // weight field (j / kTcTile) belongs to coil (j / kTcTile) % bc
        rec[t * fields * kTcTile + 3 * kTcTile + j] *=
            exp2_int(tc_scale_exp(bound[(j / kTcTile) % bc]));
    }
}

cudaError_t launch_scale_records(float* rec, int fields, int64_t ntiles,
                                 const unsigned int* bound, int bc, int grid, cudaStream_t s)
{
    if (bc < 1 || (fields - 3) % bc != 0) return cudaErrorInvalidValue;
    scale_records_kernel<<<grid, 256, 0, s>>>(rec, fields, ntiles, bound, bc);
    return cudaGetLastError();
}

cudaError_t launch_prep_grid_tc(bool realw, int bc, const PrepParams& p, int grid, cudaStream_t s)
{
    if (realw) {
        if (bc != 1) return cudaErrorInvalidValue;
        prep_records_kernel<1, true, kTcTile><<<grid, 256, 0, s>>>(p);
    } else {
        switch (bc) {
            case 1: prep_records_kernel<1, false, kTcTile><<<grid, 256, 0, s>>>(p); break;
            case 4: prep_records_kernel<4, false, kTcTile><<<grid, 256, 0, s>>>(p); break;
            case 8: prep_records_kernel<8, false, kTcTile><<<grid, 256, 0, s>>>(p); break;
            default: return cudaErrorInvalidValue;
        }
    }
    return cudaGetLastError();
}

}  // namespace mri
