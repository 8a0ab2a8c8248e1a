/*
 * mri.h -- C ABI of the GB300 F^H D / Q gather library (libmri.so).
 *
 * The operations are the data-parallel core of iterative non-Cartesian MRI
 * reconstruction as the chapter "Iterative MRI reconstruction" (PMPP ch. 17)
 * describes it:
 *
 *   cmpMu  (section 17.3, Figs. 17.6-17.7):  Mu[m] = conj(Phi[m]) * D[m]
 *   cmpFhD (section 17.3, Figs. 17.9-17.11): FhD[n] = sum_m Mu[m] * e^{+i 2 pi k_m . x_n}
 *   Q      (section 17.2):                   Q[n]   = sum_m |Phi[m]|^2 * e^{+i 2 pi k_m . x_n}
 *
 * The sign +i and k in cycles per unit of x follow Eq. 17.1 and the phase
 * 2*PI*(kx*x + ky*y + kz*z) of the register-promoted kernel (Fig. 17.11).
 * The pages print no formula for Mu or Q; the readings above are the ones
 * this library implements.
 *
 * Conventions for every entry point
 *   - Arrays are float32, structure of arrays, caller-owned DEVICE memory on
 *     the current CUDA device, each at least 4-byte aligned.  Nothing is kept
 *     after a call returns.
 *   - Sample arrays have M elements, voxel arrays N elements; batched data and
 *     outputs are coil-major [B][M] and [B][N].
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  The return value covers argument checks and launch
 *     errors; errors during execution surface at the caller's next
 *     synchronisation or through mri_device_errors().
 *   - Scratch memory (tile records, per-split partial sums) is taken from a
 *     library-owned stream-ordered memory pool on `stream` and returned to it
 *     before the call returns; the pool keeps freed memory for reuse.
 *   - No C++ exception crosses this interface; no call traps or aborts.
 *   - The kernels are built for sm_103a only; any other device gives
 *     MRI_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef MRI_H
#define MRI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mri_status {
    MRI_OK = 0,
    MRI_ERR_NULL = 1,               /* a required pointer is NULL */
    MRI_ERR_SIZE = 2,               /* M, N or B negative or too large */
    MRI_ERR_ALIGN = 3,              /* a pointer is not 4-byte aligned */
    MRI_ERR_NOT_DEVICE = 4,         /* a pointer is not device memory of the current device */
    MRI_ERR_MODE = 5,               /* unknown trig mode or accumulate flag not 0/1 */
    MRI_ERR_CUDA = 6,               /* a CUDA runtime call failed (launch, pool, query) */
    MRI_ERR_UNSUPPORTED_DEVICE = 7  /* the current device is not compute capability 10.3 */
} mri_status;

typedef enum mri_trig {
    /* sin/cos in software on the FP32 pipe, the role of the software trig
     * of the chapter's sequential and early kernels: the phase in half
     * turns, reduced exactly to [-1/2, 1/2], then the library's own minimax
     * polynomials (sin degree 9, cos degree 8, within 2.6e-7). */
    MRI_TRIG_ACCURATE = 0,
    /* hardware sin/cos on the SFU (MUFU), the chapter's step 3 (Fig. 17.17);
     * the phase is formed in radians directly. */
    MRI_TRIG_FAST = 1,
    /* MUFU sin/cos after exact reduction of the phase to [-1/2, 1/2] turn;
     * slower than MRI_TRIG_FAST, for phases far beyond 100*pi. */
    MRI_TRIG_FAST_RR = 2
} mri_trig;

/* Kinds understood by mri_plan_gather. */
typedef enum mri_kind {
    MRI_KIND_FHD = 0,
    MRI_KIND_Q = 1,
    MRI_KIND_FHD_BATCHED = 2
} mri_kind;

/*
 * cmpMu (section 17.3, Fig. 17.7; loop fission of Fig. 17.6):
 *   rMu[m] = rPhi[m]*rD[m] + iPhi[m]*iD[m]
 *   iMu[m] = rPhi[m]*iD[m] - iPhi[m]*rD[m]        for 0 <= m < M.
 * Inputs rPhi, iPhi, rD, iD [M]; outputs rMu, iMu [M] (may not alias the
 * inputs).  M == 0 is a no-op.  mri_fhd does this internally; this entry
 * point exposes it on its own.
 */
mri_status mri_mu(const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                  float* rMu, float* iMu, int64_t M, void* stream);

/*
 * F^H D (section 17.3: cmpMu, then the voxel gather of Figs. 17.10-17.11):
 *   rFhD[n] + i*iFhD[n] = sum_{m<M} conj(Phi[m]) D[m] e^{+i 2 pi (kx[m] x[n] + ky[m] y[n] + kz[m] z[n])}
 * Inputs kx, ky, kz, rPhi, iPhi, rD, iD [M]; x, y, z [N].  Outputs rFhD,
 * iFhD [N] are overwritten, or added to when accumulate == 1 (the kernel of
 * Fig. 17.11 reads rFhD[n] first and adds to it, so chunks of k-space can be
 * processed by successive calls).  M == 0 writes zeros (accumulate == 0) or
 * leaves the outputs unchanged; N == 0 is a no-op.  Outputs may not alias
 * inputs.
 */
mri_status mri_fhd(const float* kx, const float* ky, const float* kz,
                   const float* x, const float* y, const float* z,
                   const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                   int64_t M, int64_t N, float* rFhD, float* iFhD,
                   mri_trig trig, int accumulate, void* stream);

/*
 * Q (section 17.2; "the same core structure as F^H D", once per trajectory):
 *   rQ[n] + i*iQ[n] = sum_{m<M} (rPhi[m]^2 + iPhi[m]^2) e^{+i 2 pi k_m . x_n}
 * Arguments and edge cases as mri_fhd, without D.
 */
mri_status mri_q(const float* kx, const float* ky, const float* kz,
                 const float* x, const float* y, const float* z,
                 const float* rPhi, const float* iPhi,
                 int64_t M, int64_t N, float* rQ, float* iQ,
                 mri_trig trig, int accumulate, void* stream);

/*
 * Batched F^H D: B data vectors (e.g. coils) acquired on one trajectory,
 *   FhD_b[n] = sum_m conj(Phi[m]) D_b[m] e^{+i 2 pi k_m . x_n},   0 <= b < B.
 * rD, iD are coil-major [B][M]; rFhD, iFhD are coil-major [B][N].  Each
 * sin/cos pair is computed once and used for up to 8 coils: groups of 3 to
 * 8 coils run the multiply-accumulate over the coils on the tensor cores
 * (each coil's weights scaled by its own power of two, undone exactly), a
 * remainder of 1 or 2 coils the per-pair kernels.  The pages do not
 * describe this variant; it is F^H D applied to several D.
 * B >= 1.  Other arguments and edge cases as mri_fhd.
 */
mri_status mri_fhd_batched(const float* kx, const float* ky, const float* kz,
                           const float* x, const float* y, const float* z,
                           const float* rPhi, const float* iPhi,
                           const float* rD, const float* iD,
                           int64_t B, int64_t M, int64_t N,
                           float* rFhD, float* iFhD,
                           mri_trig trig, int accumulate, void* stream);

/*
 * Forward model: D[m] = sum_n rho[n] e^{-i 2 pi k_m . x_n}, the F of Fig. 17.3
 * (section 17.1: F models the physics of the imaging process; F^H D above is
 * its conjugate transpose applied to the data), e.g. to synthesise k-space
 * from a phantom or for the F rho products of an iterative solver.  rho
 * (rRho, iRho) has N elements at voxels (x, y, z); D (rD, iD) has M, one per
 * k-space sample.  It is the same gather as mri_fhd with the roles of samples
 * and voxels exchanged and the exponent's sign reversed; launch shape as
 * mri_plan_gather(MRI_KIND_FHD, 1, N, M).  Edge cases as mri_fhd with M and N
 * exchanged: M == 0 is a no-op, N == 0 zeroes D (or leaves it when
 * accumulating).
 */
mri_status mri_forward(const float* kx, const float* ky, const float* kz,
                       const float* x, const float* y, const float* z,
                       const float* rRho, const float* iRho,
                       int64_t M, int64_t N, float* rD, float* iD,
                       mri_trig trig, int accumulate, void* stream);

/*
 * F^H D without any memory allocation.  The pages have no counterpart: this
 * is an interface for callers that may not allocate GPU memory while they
 * run -- a process whose device memory is reserved up front, a real-time
 * reconstruction loop that must not stall in an allocator, or a framework
 * that owns every allocation.  Arguments, results and edge cases are those
 * of mri_fhd; the scratch it needs (the tile records and, when it splits the
 * samples, the partial sums) lives in one fixed array of
 * MRI_FHD_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU
 * that loads the library holds until the process exits.
 *   - The call makes no cudaMalloc, cudaFree, pool or other allocating call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array: calls that may overlap on
 *     the GPU (different streams, or different host threads) race and must be
 *     serialised by the caller.  Each call rewrites every byte of the array it
 *     reads, so nothing in it needs to start at zero.
 *   - M is limited by the records: ceil(M/256) * 12288 bytes must fit in the
 *     array (M <= 698,880 for 32 MiB), else MRI_ERR_SIZE.  The sample
 *     splits are capped to the partial sums that fit after the records (for
 *     a 128^3 grid none do, and the call runs unsplit).
 */
#define MRI_FHD_NOALLOC_SCRATCH_BYTES (32ll * 1024 * 1024)
mri_status mri_fhd_noalloc(const float* kx, const float* ky, const float* kz,
                           const float* x, const float* y, const float* z,
                           const float* rPhi, const float* iPhi,
                           const float* rD, const float* iD,
                           int64_t M, int64_t N, float* rFhD, float* iFhD,
                           mri_trig trig, int accumulate, void* stream);

/*
 * F^H D and Q on a separable voxel grid: voxel n = (iz*ny + iy)*nx + ix sits
 * at (xs[ix], ys[iy], zs[iz]) (x fastest), the layout of every image the
 * chapter reconstructs.  Same sums as mri_fhd / mri_q over those N = nx*ny*nz
 * voxels; xs, ys, zs are device arrays of nx, ny, nz floats, outputs [N].
 * The exponential factors, e^{i2pi k.x} = e^{i2pi kx x} e^{i2pi (ky y + kz z)}
 * (the grid form of the gather's phase, Fig. 17.11), so per tile of samples
 * the kernel tabulates the x factor per column and Mu times the (y, z)
 * factor per row and spends one complex multiply-accumulate per
 * voxel-sample pair; sin/cos are evaluated per (sample, column) and
 * (sample, row) only.  For nx >= 8 the sum over samples is done as a
 * complex matrix product on the tensor cores (tcgen05, f16 operands split
 * into high and low parts so that each product keeps ~22 bits, fp32
 * accumulation, blocked summation): columns in blocks of 128, the last one
 * padded; a grid 8 to 64 wide folds G = 128 / (nx rounded up to a power of
 * two) rows into one block when every group of G rows has the same y
 * offsets from its first row (checked on the device; otherwise the padded
 * layout runs).  The results meet the same tolerances as the other paths.
 * Grids with nx < 8 are expanded to coordinates and take the general
 * kernel.  nx up to 8,388,480 (65,535 blocks of columns; a wider grid's
 * launch is refused: MRI_ERR_CUDA).  Edge cases as mri_fhd.
 */
mri_status mri_fhd_grid(const float* kx, const float* ky, const float* kz,
                        const float* xs, int nx, const float* ys, int ny,
                        const float* zs, int nz,
                        const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                        int64_t M, float* rFhD, float* iFhD,
                        mri_trig trig, int accumulate, void* stream);
mri_status mri_q_grid(const float* kx, const float* ky, const float* kz,
                      const float* xs, int nx, const float* ys, int ny,
                      const float* zs, int nz,
                      const float* rPhi, const float* iPhi,
                      int64_t M, float* rQ, float* iQ,
                      mri_trig trig, int accumulate, void* stream);

/*
 * Batched F^H D on a separable grid: mri_fhd_batched's B coils (rD, iD
 * coil-major [B][M]; outputs rFhD, iFhD coil-major [B][N], N = nx*ny*nz,
 * voxel order as mri_fhd_grid).  One trajectory, so the x factor of the
 * phase is tabulated once per call and the (y, z) factor once per (row,
 * sample) for up to 8 coils at a time, each sin/cos pair serving every coil
 * of the group.  As for mri_fhd_batched, the pages do not describe this
 * variant; it is F^H D applied to several D.  nx >= 8 runs on the tensor
 * cores as mri_fhd_grid does, with the coils of a group sharing each MMA's
 * rows (groups of 8, and the remainder as a group padded to 4 or 8 coils;
 * a remainder of one coil takes the single-coil kernel); grids with nx < 8 are expanded to coordinates and
 * take mri_fhd_batched.  Edge cases as mri_fhd_batched.
 */
mri_status mri_fhd_batched_grid(const float* kx, const float* ky, const float* kz,
                                const float* xs, int nx, const float* ys, int ny,
                                const float* zs, int nz,
                                const float* rPhi, const float* iPhi,
                                const float* rD, const float* iD, int64_t B, int64_t M,
                                float* rFhD, float* iFhD,
                                mri_trig trig, int accumulate, void* stream);

/*
 * The forward model of mri_forward on a separable grid: rho (rRho, iRho) on
 * the grid xs x ys x zs (voxel order as mri_fhd_grid, N = nx*ny*nz), D (rD,
 * iD) at the M samples.  For nx >= 8 (columns in blocks of 128, the last
 * one padded) the sum over the columns is a complex matrix product on the
 * tensor cores (the samples are the MMA rows; f16 operands split into high
 * and low parts, fp32 accumulation) and the sum over rows follows in the
 * epilogue with blocked summation; grids with nx < 8 are expanded to
 * coordinates and take mri_forward.  Edge cases as mri_forward.
 */
mri_status mri_forward_grid(const float* kx, const float* ky, const float* kz,
                            const float* xs, int nx, const float* ys, int ny,
                            const float* zs, int nz,
                            const float* rRho, const float* iRho, int64_t M,
                            float* rD, float* iD,
                            mri_trig trig, int accumulate, void* stream);

/*
 * The "find rho" step (chapter "Iterative MRI reconstruction", background
 * section, Fig. 17.3): rho = (F^H F + lambda W^H W)^{-1} F^H D solved by
 * conjugate gradients, whose cost per iteration is the product of
 * F^H F + lambda W^H W with the current rho.  F^H F is Toeplitz, so that
 * product goes through FFTs, built from Q (the chapter's Q).  Readings: F
 * carries the sensitivity, F[m][n] = Phi_m e^{-i2pi k_m . x_n}, so F^H D is
 * mri_fhd's and (F^H F)[n][n'] = Q(x_n - x_n') with Q of mri_q; W (from
 * patient scans, not given) is the identity, lambda >= 0 from the caller.
 * The voxels form a regular grid x = (ix hx, iy hy, iz hz), ix < nx etc.,
 * with nx, ny, nz powers of two up to 512 (voxel order as mri_fhd_grid;
 * any offset of the grid cancels in the differences).
 *
 * mri_toeplitz_kernel: Q on the circular grid of voxel differences of the
 * doubled grid (2nx x 2ny x 2nz: difference i h for i < n, (i - 2n) h for
 * i >= n per axis), computed by the grid Q path with trig mode `trig` on
 * the z planes below nz and taken as Q(-d) = conj Q(d) of the mirrored
 * point on the others, with the planes at index n of every axis set to zero
 * (the difference -n h occurs between no two voxels of the grid, so the
 * product does not use them; without them the grid is Hermitian-symmetric),
 * then the real part of its 3-D FFT (the imaginary part is rounding),
 * written to K: a device array of 8 * nx*ny*nz floats, 8-byte aligned, x
 * fastest.  Samples as mri_q (kx, ky, kz, rPhi, iPhi: M floats each; M = 0
 * gives K = 0).  Scratch from the stream-ordered pool: 12 bytes per point of
 * the doubled grid.
 *
 * mri_toeplitz_apply: out = (F^H F + lambda I) in, from K, for SoA complex
 * vectors of nx*ny*nz floats (rIn, iIn; rOut, iOut, which may be the same
 * arrays as the inputs); accumulate = 1 adds into out.  Zero-padding to the
 * doubled grid, forward FFT, product with K, inverse FFT, crop -- in five
 * kernels that never form the padding's zeros nor the part of the result
 * the crop drops.  Scratch: 4 nx*ny*nz complex values.
 *
 * mri_cg_solve: `iters` conjugate-gradient iterations on
 * (F^H F + lambda I) x = b from K: rB, iB the right-hand side (typically
 * F^H D from mri_fhd_grid), rX, iX the starting point on entry and the
 * iterate on return; rnorms (device, iters + 1 doubles, 8-byte aligned)
 * receives ||r_0|| .. ||r_iters||, r = b - (F^H F + lambda I) x.  The
 * iteration's scalars stay on the device (no host synchronisation); once
 * r = 0 the iterate stops changing.  Scratch from the stream-ordered pool:
 * 4 nx*ny*nz complex values plus 6 nx*ny*nz floats.
 *
 * These calls are asynchronous on `stream`.  MRI_ERR_SIZE for a grid edge that
 * is not a power of two in 1 .. 512, a non-finite spacing or lambda, iters
 * outside 0 .. 2^20; MRI_ERR_ALIGN for K or rnorms not 8-byte aligned; the
 * other pointer checks as mri_fhd.
 */
/*
 * The 3-D FFT under mri_toeplitz_*: in place on `data`, Lz x Ly x Lx complex
 * values interleaved (re, im), x fastest, each length a power of two in
 * 1 .. 1024; forward X[k] = sum_j x[j] e^{-2 pi i j.k / L}, inverse with
 * e^{+...} and no scaling.  Asynchronous on `stream`.
 */
mri_status mri_fft3(float* data, int Lx, int Ly, int Lz, int inverse, void* stream);
mri_status mri_toeplitz_kernel(const float* kx, const float* ky, const float* kz,
                               const float* rPhi, const float* iPhi, int64_t M,
                               int nx, int ny, int nz, float hx, float hy, float hz,
                               float* K, mri_trig trig, void* stream);
mri_status mri_toeplitz_apply(const float* K, int nx, int ny, int nz, float lambda,
                              const float* rIn, const float* iIn, float* rOut, float* iOut,
                              int accumulate, void* stream);
mri_status mri_cg_solve(const float* K, int nx, int ny, int nz, float lambda,
                        const float* rB, const float* iB, float* rX, float* iX,
                        int iters, double* rnorms, void* stream);

/*
 * The gridding reconstruction (the chapter's comparison method: section
 * 17.1, Fig. 17.1B; its accuracy in Fig. 17.19).  Each sample's
 * Mu = conj(Phi) D is interpolated trilinearly onto the 2 x 2 x 2 nearest
 * points of the Cartesian k-space grid k_g = (g - n/2) / n, g < n, of the
 * voxel grid (indices modulo n: k is periodic with period 1 on that grid),
 * then out[iz][iy][ix] = sum_g G[g] e^{+i 2 pi k_g . x} at the voxels
 * x = (ix - nx/2, iy - ny/2, iz - nz/2) (the integer coordinates of a grid
 * centred on 0, x fastest).  No density or deapodisation correction beyond
 * what Phi carries.  Samples as mri_fhd (M floats each, device); rOut, iOut:
 * nx*ny*nz floats (device); accumulate = 1 adds into them.  nx, ny, nz powers
 * of two in 1 .. 1024 (MRI_ERR_SIZE otherwise).  Scratch: nx*ny*nz complex
 * values from the stream-ordered pool.  The grid is summed with atomic adds,
 * so the summation order (and the last bits of the result) is not fixed.
 * Asynchronous on `stream`.
 */
mri_status mri_gridding(const float* kx, const float* ky, const float* kz,
                        const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                        int64_t M, int nx, int ny, int nz, float* rOut, float* iOut,
                        int accumulate, void* stream);

/* A static, NUL-terminated description of a status code. */
const char* mri_status_string(mri_status status);

/*
 * How a gather call will be launched (host-only; no CUDA call is made when
 * num_sms > 0).  The chapter tunes threads per block and unrolling jointly
 * (section 17.3 step 4); this reports the shape the library picks.
 *   kind: MRI_KIND_*; B: coils (1 unless batched); num_sms: SM count of the
 *   target device, or 0 for the current device.
 */
typedef struct mri_plan {
    int threads_per_cta;      /* threads per CTA */
    int voxels_per_thread;    /* V: voxels held in registers by each thread */
    int samples_per_tile;     /* samples per shared-memory k-tile */
    int splits;               /* CTAs along the sample axis (1: no split) */
    int64_t voxel_ctas;       /* CTAs along the voxel axis */
    int64_t tiles;            /* k-tiles covering M */
    int coil_groups;          /* gather launches over coil groups (batched) */
    int launches;             /* kernel launches one call makes */
    int64_t scratch_bytes;    /* pool memory one call takes */
    int tensor_cores;         /* 1: the gather runs on the tcgen05 tensor cores */
    int grid_fold;            /* grid calls with 8 <= nx <= 64: grid rows whose columns share
                                 one block of 128 when the y axis is evenly spaced within
                                 groups of that many rows (checked on the device; voxel_ctas
                                 counts the folded blocks), else 1 */
    int fast_fp32_voxels;     /* general gather, fast trig: of voxels_per_thread, how many
                                 take sin/cos from the polynomial on the FMA pipe instead of
                                 the SFU (both units then share the trig work) */
    int voxels_per_cta;       /* output voxels of one coil that one CTA covers, padding
                                 included: threads_per_cta * voxels_per_thread on the per-pair
                                 kernels, 128 on the tensor-core coil kernel (one voxel per
                                 tensor-memory lane), grid rows per CTA * 128 columns on the
                                 tensor-core grid kernels */
} mri_plan;

mri_status mri_plan_gather(int kind, int64_t B, int64_t M, int64_t N, int num_sms,
                           mri_plan* plan);

/* The same for mri_fhd_grid (kind MRI_KIND_FHD) and mri_q_grid (MRI_KIND_Q),
 * for any trig mode. */
mri_status mri_plan_grid(int kind, int64_t M, int nx, int ny, int nz, int num_sms,
                         mri_plan* plan);

/* The same for mri_fhd_batched_grid with B coils (first coil group's shape). */
mri_status mri_plan_grid_batched(int64_t B, int64_t M, int nx, int ny, int nz, int num_sms,
                                 mri_plan* plan);

/*
 * Device-side error bits of the current device (bit 0: a k-tile wait timed
 * out; bit 1: in-flight copies did not drain; bit 2, MRI_DEBUG builds only: a
 * copy's tile index was outside its table and the copy was skipped).
 * Synchronises the device.
 * clear != 0 resets the bits.  Kernels never trap; a non-zero word means the
 * outputs of some earlier call are not valid.
 */
mri_status mri_device_errors(unsigned int* bits, int clear);

/*
 * Gather-kernel timing, for benchmarks and profiling.  Between
 * mri_timing_begin() and mri_timing_end(), every gather-kernel launch made on
 * the current device is bracketed by two CUDA events recorded on the
 * launch's own stream (the events are the library's; at most 4096 launches
 * per window are timed).  mri_timing_end() waits for those events and
 * returns the summed gather-kernel time in milliseconds and the number of
 * launches timed.  The prep and split-reduction kernels are not included.
 * Timing adds two event records per launch and changes nothing else.
 */
mri_status mri_timing_begin(void);
mri_status mri_timing_end(double* gather_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* MRI_H */
