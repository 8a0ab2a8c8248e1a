// launch.h -- internal host-side interface between the C ABI and the kernel
// translation units.  Not part of the public API.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gather.cuh"
#include "gather_pair.cuh"
#include "gather_grid.cuh"
#include "gather_grid_tc.cuh"
#include "fft.cuh"

namespace mri {

struct CoilTcParams;

struct KernelShape {
    int threads;
    int v;                  // voxels per thread
    int voxels_per_cta;
    int min_blocks;         // CTAs per SM the kernel is built for
    size_t smem;            // dynamic shared memory per CTA
    int tile_floats;        // floats per record tile
    int fast_fp32_voxels;   // of the v voxels of a thread, those whose fast-path trig is
                            // the polynomial on the FMA pipe (the rest use the SFU)
};

// bc: coils in one group (1, 2, 4, 8); realw: Q's real weight (bc == 1).
KernelShape gather_shape(int bc, bool realw);

cudaError_t launch_prep(int bc, bool realw, const PrepParams& p, int grid, cudaStream_t s);
// phase units the records of a general gather launch hold (k is multiplied by it)
float gather_kscale(int bc, int trig);
cudaError_t launch_gather(int bc, bool realw, int trig, const GatherParams& p, dim3 grid,
                          cudaStream_t s);
cudaError_t launch_reduce(const float* part, int splits, int bc, int64_t N, float* out_r,
                          float* out_i, int64_t out_coil_stride, int accumulate, int grid,
                          cudaStream_t s);
cudaError_t launch_mu(const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                      float* rMu, float* iMu, int64_t M, int grid, cudaStream_t s);

cudaError_t launch_zero(float* a, int64_t n, int grid, cudaStream_t s);

// tensor-core grid path (kernels_grid_tc.cu), nx >= 8 in column blocks of 128
// tensor-core grid kernel over a group of bc coils (1, or 4 / 8 for F^H D)
cudaError_t launch_grid_tc(bool realw, int trig, int bc, const GridParams& p, dim3 grid,
                           cudaStream_t s);
cudaError_t launch_prep_grid_tc(bool realw, int bc, const PrepParams& p, int grid, cudaStream_t s);
// forward model on a grid (nx >= 8) on the tensor cores:
// the rho table, row coordinates and scale word, then the kernel
cudaError_t launch_forward_grid_prep(const float* rr, const float* ri, int64_t rows, int nx,
                                     int64_t row_blocks, const float* ys, int ny, const float* zs,
                                     unsigned int* bound, unsigned char* tab, float2* yz_rows,
                                     float* row_step, int grid, cudaStream_t s);
cudaError_t launch_forward_grid_tc(int trig, const FwdParams& p, dim3 grid, cudaStream_t s);
// weights of tensor-core grid records (bc coils) times each coil's power of
// two, from its bound word bound[coil]
cudaError_t launch_scale_records(float* rec, int fields, int64_t ntiles,
                                 const unsigned int* bound, int bc, int grid, cudaStream_t s);
// threads per CTA of the tensor-core grid kernel
int grid_tc_threads();
// the row-folding check of a narrow grid (grid_tc_fold(nx, ny) = G > 1): *ok
// and the G row offsets dy, read by the B-tile build and the kernel
cudaError_t launch_grid_fold_check(const float* ys, int ny, int G, unsigned int* ok, float* dy,
                                   cudaStream_t s);
// B operand tiles of the tensor-core grid kernel from its records (kx) and
// xs; mub: times the records' (scaled) weight, for single-coil launches
cudaError_t launch_build_ex_tiles(int trig, bool mub, const float* rec, int fields,
                                  int64_t ntiles, const float* xs, int nx, unsigned char* s_tab,
                                  int grid, cudaStream_t s, int fold = 1,
                                  const unsigned int* fold_ok = nullptr,
                                  const float* fold_dy = nullptr);
// voxel coordinates of a grid the tensor-core kernels do not take (kernels_grid.cu)
cudaError_t launch_expand_grid(const float* xs, const float* ys, const float* zs, int nx, int ny,
                               int64_t N, float* x, float* y, float* z, int grid, cudaStream_t s);

// the find-rho step on a grid (kernels_toeplitz.cu): FFT twiddle table,
// 3-D FFTs of the doubled grid, difference axes, Toeplitz product, CG
cudaError_t launch_fft_twiddles(float2* tw, cudaStream_t s);
cudaError_t launch_fft3(float2* a, int Lx, int Ly, int Lz, bool inverse, const float2* tw,
                        cudaStream_t s);
// one axis (0 = x, 1 = y, 2 = z) of that 3-D FFT; nothing for a length of 1
cudaError_t launch_fft_axis(float2* a, int Lx, int Ly, int Lz, int axis, bool inverse,
                            const float2* tw, cudaStream_t s);
cudaError_t launch_diff_axes(int nx, int ny, int nz, float hx, float hy, float hz, float* axes,
                             cudaStream_t s);
// Q (SoA, doubled grid) into the complex array whose spectrum is K, the
// planes at index n of every axis zeroed; K = the real part of a spectrum
cudaError_t launch_spectrum_input(const float* r, const float* i, int nx, int ny, int nz,
                                  float2* out, int grid, cudaStream_t s);
cudaError_t launch_real_part(const float2* spec, int64_t n, float* K, int grid, cudaStream_t s);
// CTAs of the last Toeplitz stage: the p.Ap partial sums launch_cg keeps
int64_t toeplitz_dot_blocks(int nx, int ny, int nz);
cudaError_t launch_toeplitz_apply(const float* K, int nx, int ny, int nz, float lambda,
                                  const float* ir, const float* ii, float* outr, float* outi,
                                  int accumulate, float2* work, const float2* tw,
                                  cudaStream_t s);
// the gridding reconstruction (kernels_gridding.cu): G (nx*ny*nz complex
// scratch) zeroed, the samples' trilinear scatter, the inverse FFT, the
// centring signs into out
cudaError_t launch_gridding(const float* kx, const float* ky, const float* kz, const float* rPhi,
                            const float* iPhi, const float* rD, const float* iD, int64_t M,
                            int nx, int ny, int nz, float* outr, float* outi, int accumulate,
                            float2* G, const float2* tw, int sms, cudaStream_t s);
cudaError_t launch_cg(const float* K, int nx, int ny, int nz, float lambda, const float* br,
                      const float* bi, float* xr, float* xi, int iters, double* rr,
                      float* vec, float2* work, double* scal, const float2* tw, int grid,
                      int dot_blocks, cudaStream_t s);

// per-TU dispatchers
cudaError_t launch_gather_single(bool realw, int trig, const GatherParams& p, dim3 grid,
                                 cudaStream_t s);
cudaError_t launch_gather_coils(int bc, int trig, const GatherParams& p, dim3 grid,
                                cudaStream_t s);
cudaError_t launch_prep_coils(int bc, const PrepParams& p, int grid, cudaStream_t s);
// batched F^H D of up to 8 coils on the tensor cores (kernels_coils_tc.cu;
// CoilTcParams in gather_coils_tc.cuh, which only the TUs that launch or fill
// it include: its kernel's shared-memory alignment stays out of the others):
// the weight tiles from the grid-path records of 8 coils and their 8 bound
// words (each coil scaled by its own power of two), the kernel
cudaError_t launch_build_mu_tiles(const float* rec, int64_t ntiles, const unsigned int* bounds,
                                  unsigned char* s_tab, int grid, cudaStream_t s);
cudaError_t launch_gather_coils_tc(int trig, const CoilTcParams& p, dim3 grid, cudaStream_t s);

}  // namespace mri
