/*
 * oracle.c -- plain fp64 CPU oracle for the F^H D / Q gather.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no source, header, table or helper with the CUDA
 * library.
 *
 * What it computes (sources are the pages on iterative non-Cartesian MRI
 * reconstruction):
 *
 *   Eq. 17.1 (section 17.1) sums k-space samples into an image with the
 *   kernel e^{+i 2 pi k_j . r}.
 *
 *   Section 17.3 splits F^H D by loop fission into a per-sample stage that
 *   forms (rMu, iMu) (cmpMu, Fig. 17.7) and a gather stage in which each voxel
 *   n sums, over all samples m, Mu[m] times cos/sin of 2*PI*(kx*x + ky*y +
 *   kz*z) (Figs. 17.9-17.11; the register-promoted kernel printed in the
 *   study notes on step 2 accumulates rMu*c - iMu*s into the real part and
 *   iMu*c + rMu*s into the imaginary part).
 *
 *   The pages leave cmpMu's formula and Q's definition out; the readings used
 *   here are Mu = conj(Phi) * D and Q[n] = sum_m |Phi[m]|^2 e^{+i 2 pi k_m.x_n}
 *   (section 17.2 says Q has "the same core structure" as F^H D).
 *
 * Every input element is a float promoted exactly to double; all arithmetic
 * is double; sin and cos are the C library's double functions; sums run in
 * sample order m = 0 .. M-1.  Voxels are independent (section 17.3), so the
 * voxel loop is shared among OpenMP threads; this does not change any
 * voxel's arithmetic.
 *
 * Parity status: every function here is pinned by CPU tests against closed
 * forms (see the test suite's oracle pins); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static const double TWO_PI = 6.283185307179586476925286766559;

static void set_threads(int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

/* Number of threads an OpenMP parallel region will use (1 without OpenMP). */
int oracle_threads(int threads)
{
    set_threads(threads);
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * cmpMu (Fig. 17.7, first loop after fission, Fig. 17.6):
 *   Mu[m] = conj(Phi[m]) * D[m]
 *   rMu = rPhi*rD + iPhi*iD,  iMu = rPhi*iD - iPhi*rD.
 */
void oracle_mu(int64_t M, const float *rPhi, const float *iPhi,
               const float *rD, const float *iD, double *rMu, double *iMu)
{
    for (int64_t m = 0; m < M; ++m) {
        double rp = rPhi[m], ip = iPhi[m], rd = rD[m], id = iD[m];
        rMu[m] = rp * rd + ip * id;
        iMu[m] = rp * id - ip * rd;
    }
}

/*
 * One voxel of the gather (Fig. 17.10 / 17.11 loop body):
 *   phase = 2*pi*(kx[m]*x + ky[m]*y + kz[m]*z)
 *   re += wr[m]*cos(phase) - wi[m]*sin(phase)
 *   im += wi[m]*cos(phase) + wr[m]*sin(phase)
 * with (wr, wi) = (rMu, iMu) for F^H D, (|Phi|^2, 0) for Q.
 */
static void gather_one(int64_t M, const float *kx, const float *ky,
                       const float *kz, const double *wr, const double *wi,
                       double x, double y, double z, double *re, double *im)
{
    double sr = 0.0, si = 0.0;
    for (int64_t m = 0; m < M; ++m) {
        double phase = TWO_PI * ((double)kx[m] * x + (double)ky[m] * y
                                 + (double)kz[m] * z);
        double c = cos(phase), s = sin(phase);
        sr += wr[m] * c - wi[m] * s;
        si += wi[m] * c + wr[m] * s;
    }
    *re = sr;
    *im = si;
}

/*
 * Gather over a list of voxels.  idx == NULL means voxels 0 .. nout-1;
 * otherwise output j is voxel idx[j].  wi == NULL means a real weight.
 */
static void gather(int64_t M, const float *kx, const float *ky, const float *kz,
                   const double *wr, const double *wi,
                   const float *x, const float *y, const float *z,
                   int64_t nout, const int64_t *idx, double *re, double *im)
{
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t j = 0; j < nout; ++j) {
        int64_t n = idx ? idx[j] : j;
        double r, i;
        if (wi) {
            gather_one(M, kx, ky, kz, wr, wi, x[n], y[n], z[n], &r, &i);
        } else {
            /* real weight: the imaginary weight is identically zero */
            double sr = 0.0, si = 0.0;
            for (int64_t m = 0; m < M; ++m) {
                double phase = TWO_PI * ((double)kx[m] * x[n]
                                         + (double)ky[m] * y[n]
                                         + (double)kz[m] * z[n]);
                sr += wr[m] * cos(phase);
                si += wr[m] * sin(phase);
            }
            r = sr;
            i = si;
        }
        re[j] = r;
        im[j] = i;
    }
}

/*
 * F^H D (section 17.3): cmpMu, then the voxel gather.
 * mu_r, mu_i: caller-provided double scratch of length M.
 */
void oracle_fhd(int64_t M, const float *kx, const float *ky, const float *kz,
                const float *rPhi, const float *iPhi,
                const float *rD, const float *iD,
                const float *x, const float *y, const float *z,
                int64_t nout, const int64_t *idx,
                double *rFhD, double *iFhD, double *mu_r, double *mu_i,
                int threads)
{
    set_threads(threads);
    oracle_mu(M, rPhi, iPhi, rD, iD, mu_r, mu_i);
    gather(M, kx, ky, kz, mu_r, mu_i, x, y, z, nout, idx, rFhD, iFhD);
}

/*
 * Q (section 17.2): Q[n] = sum_m |Phi[m]|^2 e^{+i 2 pi k_m . x_n}.
 * w: caller-provided double scratch of length M.
 */
void oracle_q(int64_t M, const float *kx, const float *ky, const float *kz,
              const float *rPhi, const float *iPhi,
              const float *x, const float *y, const float *z,
              int64_t nout, const int64_t *idx,
              double *rQ, double *iQ, double *w, int threads)
{
    set_threads(threads);
    for (int64_t m = 0; m < M; ++m) {
        double rp = rPhi[m], ip = iPhi[m];
        w[m] = rp * rp + ip * ip;
    }
    gather(M, kx, ky, kz, w, NULL, x, y, z, nout, idx, rQ, iQ);
}

/*
 * Several data vectors on one trajectory: D is coil-major [B][M], the
 * outputs are [B][nout].  Each coil is an independent F^H D.
 */
void oracle_fhd_batched(int64_t B, int64_t M,
                        const float *kx, const float *ky, const float *kz,
                        const float *rPhi, const float *iPhi,
                        const float *rD, const float *iD,
                        const float *x, const float *y, const float *z,
                        int64_t nout, const int64_t *idx,
                        double *rFhD, double *iFhD, double *mu_r, double *mu_i,
                        int threads)
{
    for (int64_t b = 0; b < B; ++b)
        oracle_fhd(M, kx, ky, kz, rPhi, iPhi, rD + b * M, iD + b * M,
                   x, y, z, nout, idx, rFhD + b * nout, iFhD + b * nout,
                   mu_r, mu_i, threads);
}

/*
 * Forward model D = F rho (the "inverse process" that turns a phantom into
 * synthetic k-space data for the PSNR check of section 17.3 step 3):
 *   D[m] = sum_n rho[n] e^{-i 2 pi k_m . x_n}.
 * F^H is the conjugate transpose of this F, which is where the +i of Eq. 17.1
 * comes from.  Voxels with rho == 0 contribute nothing and are skipped.
 */
void oracle_forward(int64_t M, const float *kx, const float *ky, const float *kz,
                    int64_t N, const float *x, const float *y, const float *z,
                    const double *rRho, const double *iRho,
                    double *rD, double *iD, int threads)
{
    set_threads(threads);
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double sr = 0.0, si = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            if (rRho[n] == 0.0 && iRho[n] == 0.0) continue;
            double phase = -TWO_PI * ((double)kx[m] * x[n] + (double)ky[m] * y[n]
                                      + (double)kz[m] * z[n]);
            double c = cos(phase), s = sin(phase);
            sr += rRho[n] * c - iRho[n] * s;
            si += iRho[n] * c + rRho[n] * s;
        }
        rD[m] = sr;
        iD[m] = si;
    }
}
