// kernels_toeplitz.cu -- the "find rho" step on a regular grid: F^H F as a
// Toeplitz product through FFTs (fft.cuh), and the conjugate-gradient
// iteration around it (the chapter's background section, Fig. 17.3:
// rho = (F^H F + lambda W^H W)^{-1} F^H D, W = I here).
//
// The grid has n = (nx, ny, nz) voxels; the doubled grid 2n holds Q on the
// circular grid of voxel differences and, zero-padded, the vector being
// multiplied; (F^H F v)[x] = sum_x' Q(x - x') v[x'] is then the corner of
// IFFT(FFT(Q) * FFT(pad v)) / |2n|.  All buffers are device memory; the
// CG scalars stay on the device (no host round trip per iteration).
#include <cstdint>
#include <type_traits>

#include "fft.cuh"
#include "launch.h"

namespace mri {

namespace {

// tw[k] = e^{-2 pi i k / kFftMaxLen}, k < kFftMaxLen / 2, from double precision
__global__ void __launch_bounds__(256) fft_twiddle_kernel(float2* tw)
{
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < kFftMaxLen / 2) {
        double s, c;
        sincospi(-2.0 * double(k) / double(kFftMaxLen), &s, &c);
        tw[k] = make_float2(float(c), float(s));
    }
}

// circular difference axes of the doubled grid: i h for i < n, (i - 2n) h
// for i >= n; x at axes[0 .. 2nx), y after it, z after that
__global__ void __launch_bounds__(256) diff_axes_kernel(int nx, int ny, int nz, float hx,
                                                        float hy, float hz, float* axes)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int total = 2 * (nx + ny + nz);
    if (t >= total) return;
    int n, i;
    float h;
    if (t < 2 * nx) { n = nx; i = t; h = hx; }
    else if (t < 2 * (nx + ny)) { n = ny; i = t - 2 * nx; h = hy; }
    else { n = nz; i = t - 2 * (nx + ny); h = hz; }
    axes[t] = float(i < n ? i : i - 2 * n) * h;
}

__global__ void __launch_bounds__(256) interleave_kernel(const float* r, const float* i,
                                                         int64_t n, float2* out)
{
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x)
        out[k] = make_float2(r[k], i[k]);
}

// v (n grid, SoA) into the corner of the doubled grid, zeros elsewhere
__global__ void __launch_bounds__(256) pad_kernel(const float* vr, const float* vi, int nx,
                                                  int ny, int nz, float2* out)
{
    const int64_t Lx = 2 * nx, Ly = 2 * ny;
    const int64_t total = Lx * Ly * 2 * nz;
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < total;
         k += int64_t(gridDim.x) * blockDim.x) {
        const int64_t ix = k % Lx;
        const int64_t rest = k / Lx;
        const int64_t iy = rest % Ly;
        const int64_t iz = rest / Ly;
        float2 v = make_float2(0.0f, 0.0f);
        if (ix < nx && iy < ny && iz < nz) {
            const int64_t n = (iz * ny + iy) * nx + ix;
            v = make_float2(vr[n], vi[n]);
        }
        out[k] = v;
    }
}

// a *= K (complex), the spectrum of Q times the spectrum of the padded vector
__global__ void __launch_bounds__(256) spectrum_mul_kernel(float2* a, const float2* K, int64_t n)
{
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x) {
        const float2 x = a[k];
        const float2 y = K[k];
        a[k] = make_float2(x.x * y.x - x.y * y.y, x.x * y.y + x.y * y.x);
    }
}

// out = scale * corner(a) + lambda * in (+ out when accumulating)
__global__ void __launch_bounds__(256) crop_kernel(const float2* a, int nx, int ny, int nz,
                                                   float scale, float lambda, const float* ir,
                                                   const float* ii, float* outr, float* outi,
                                                   int accumulate)
{
    const int64_t N = int64_t(nx) * ny * nz;
    for (int64_t n = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; n < N;
         n += int64_t(gridDim.x) * blockDim.x) {
        const int64_t ix = n % nx;
        const int64_t rest = n / nx;
        const int64_t iy = rest % ny;
        const int64_t iz = rest / ny;
        const float2 v = a[(iz * 2 * ny + iy) * 2 * nx + ix];
        float r = fmaf(lambda, ir[n], v.x * scale);
        float i = fmaf(lambda, ii[n], v.y * scale);
        if (accumulate) {
            r += outr[n];
            i += outi[n];
        }
        outr[n] = r;
        outi[n] = i;
    }
}

// ---- conjugate gradients: Re <a, b> in double, per block, then one block sums
constexpr int kDotThreads = 256;

__device__ __forceinline__ double block_sum(double v, double* sm)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sm[warp] = v;
    __syncthreads();
    double s = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kDotThreads / 32; ++w) s += sm[w];
    return s;   // thread 0
}

__global__ void __launch_bounds__(kDotThreads) dot_partial_kernel(const float* ar, const float* ai,
                                                                  const float* br, const float* bi,
                                                                  int64_t n, double* partial)
{
    __shared__ double sm[kDotThreads / 32];
    double v = 0.0;
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x)
        v += double(ar[k]) * br[k] + double(ai[k]) * bi[k];
    const double s = block_sum(v, sm);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kDotThreads) sum_partials_kernel(const double* partial, int n,
                                                                   double* out)
{
    __shared__ double sm[kDotThreads / 32];
    double v = 0.0;
    for (int k = threadIdx.x; k < n; k += kDotThreads) v += partial[k];   // fixed order
    const double s = block_sum(v, sm);
    if (threadIdx.x == 0) *out = s;
}

// step alpha = r.r / p.Ap (0 once r = 0 or p.Ap = 0)
__device__ __forceinline__ float cg_ratio(const double* num, const double* den)
{
    const double a = *num, b = *den;
    return (a > 0.0 && b != 0.0) ? float(a / b) : 0.0f;
}

// x += alpha p, r -= alpha Ap, partial sums of |r|^2
__global__ void __launch_bounds__(kDotThreads) cg_xr_kernel(float* xr, float* xi, float* rr_,
                                                            float* ri, const float* pr,
                                                            const float* pi, const float* apr,
                                                            const float* api, int64_t n,
                                                            const double* rr, const double* pap,
                                                            double* partial)
{
    __shared__ double sm[kDotThreads / 32];
    const float alpha = cg_ratio(rr, pap);
    double v = 0.0;
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x) {
        xr[k] = fmaf(alpha, pr[k], xr[k]);
        xi[k] = fmaf(alpha, pi[k], xi[k]);
        const float a = fmaf(-alpha, apr[k], rr_[k]);
        const float b = fmaf(-alpha, api[k], ri[k]);
        rr_[k] = a;
        ri[k] = b;
        v += double(a) * a + double(b) * b;
    }
    const double s = block_sum(v, sm);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

// p = r + beta p, beta = new r.r / old r.r
__global__ void __launch_bounds__(256) cg_p_kernel(float* pr, float* pi, const float* rr_,
                                                   const float* ri, int64_t n,
                                                   const double* rr_new, const double* rr_old)
{
    const float beta = cg_ratio(rr_new, rr_old);
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x) {
        pr[k] = fmaf(beta, pr[k], rr_[k]);
        pi[k] = fmaf(beta, pi[k], ri[k]);
    }
}

// r = b - r (r holds A x), p = r
__global__ void __launch_bounds__(256) cg_start_kernel(const float* br, const float* bi,
                                                       float* rr_, float* ri, float* pr,
                                                       float* pi, int64_t n)
{
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x) {
        const float a = br[k] - rr_[k];
        const float b = bi[k] - ri[k];
        rr_[k] = a;
        ri[k] = b;
        pr[k] = a;
        pi[k] = b;
    }
}

__global__ void __launch_bounds__(256) sqrt_kernel(double* v, int n)
{
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < n) v[k] = sqrt(v[k]);
}

int log2i(int L)
{
    int b = 0;
    while ((1 << b) < L) ++b;
    return b;
}

}  // namespace

cudaError_t launch_fft_twiddles(float2* tw, cudaStream_t s)
{
    fft_twiddle_kernel<<<(kFftMaxLen / 2 + 255) / 256, 256, 0, s>>>(tw);
    return cudaGetLastError();
}

cudaError_t launch_fft3(float2* a, int Lx, int Ly, int Lz, bool inverse, const float2* tw,
                        cudaStream_t s)
{
    if (!fft_len_ok(Lx) || !fft_len_ok(Ly) || !fft_len_ok(Lz)) return cudaErrorInvalidValue;
    const int64_t L[3] = {Lx, Ly, Lz};
    const int64_t inner[3] = {1, Lx, int64_t(Lx) * Ly};
    const int64_t outer[3] = {int64_t(Ly) * Lz, Lz, 1};
    for (int ax = 0; ax < 3; ++ax) {
        if (L[ax] == 1) continue;
        const int len = int(L[ax]);
        const int log2L = log2i(len);
        const size_t smem = fft_smem_total(log2L);
        const int64_t lines = outer[ax] * inner[ax];
        const int64_t W = int64_t(1) << fft_log2_lines(log2L);
        const int64_t groups = (lines + W - 1) / W;
        auto go = [&](auto kernel) -> cudaError_t {
            const cudaError_t e = cudaFuncSetAttribute(
                kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
            if (e != cudaSuccess) return e;
            kernel<<<unsigned(groups), kFftThreads, smem, s>>>(a, log2i(int(inner[ax])), lines,
                                                               tw);
            return cudaGetLastError();
        };
        auto by_length = [&](auto inv) -> cudaError_t {
            constexpr bool I = decltype(inv)::value;
            switch (log2L) {
                case 1: return go(fft_axis_kernel<I, 1>);
                case 2: return go(fft_axis_kernel<I, 2>);
                case 3: return go(fft_axis_kernel<I, 3>);
                case 4: return go(fft_axis_kernel<I, 4>);
                case 5: return go(fft_axis_kernel<I, 5>);
                case 6: return go(fft_axis_kernel<I, 6>);
                case 7: return go(fft_axis_kernel<I, 7>);
                case 8: return go(fft_axis_kernel<I, 8>);
                case 9: return go(fft_axis_kernel<I, 9>);
                case 10: return go(fft_axis_kernel<I, 10>);
            }
            return cudaErrorInvalidValue;
        };
        const cudaError_t e = inverse ? by_length(std::true_type{}) : by_length(std::false_type{});
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_diff_axes(int nx, int ny, int nz, float hx, float hy, float hz, float* axes,
                             cudaStream_t s)
{
    const int total = 2 * (nx + ny + nz);
    diff_axes_kernel<<<(total + 255) / 256, 256, 0, s>>>(nx, ny, nz, hx, hy, hz, axes);
    return cudaGetLastError();
}

cudaError_t launch_interleave(const float* r, const float* i, int64_t n, float2* out, int grid,
                              cudaStream_t s)
{
    interleave_kernel<<<grid, 256, 0, s>>>(r, i, n, out);
    return cudaGetLastError();
}

cudaError_t launch_toeplitz_apply(const float2* K, int nx, int ny, int nz, float lambda,
                                  const float* ir, const float* ii, float* outr, float* outi,
                                  int accumulate, float2* work, const float2* tw, int grid,
                                  cudaStream_t s)
{
    const int64_t n8 = int64_t(8) * nx * ny * nz;
    pad_kernel<<<grid, 256, 0, s>>>(ir, ii, nx, ny, nz, work);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_fft3(work, 2 * nx, 2 * ny, 2 * nz, false, tw, s);
    if (e == cudaSuccess) {
        spectrum_mul_kernel<<<grid, 256, 0, s>>>(work, K, n8);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = launch_fft3(work, 2 * nx, 2 * ny, 2 * nz, true, tw, s);
    if (e == cudaSuccess) {
        crop_kernel<<<grid, 256, 0, s>>>(work, nx, ny, nz, float(1.0 / double(n8)), lambda, ir,
                                         ii, outr, outi, accumulate);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_cg(const float2* K, int nx, int ny, int nz, float lambda, const float* br,
                      const float* bi, float* xr, float* xi, int iters, double* rr,
                      float* vec, float2* work, double* scal, const float2* tw, int grid,
                      int dot_blocks, cudaStream_t s)
{
    // vec: r (2 N), p (2 N), Ap (2 N); scal: dot partials (dot_blocks), p.Ap
    const int64_t N = int64_t(nx) * ny * nz;
    float *r_r = vec, *r_i = vec + N, *p_r = vec + 2 * N, *p_i = vec + 3 * N;
    float *a_r = vec + 4 * N, *a_i = vec + 5 * N;
    double* partial = scal;
    double* pap = scal + dot_blocks;
    // r = b - A x, p = r, rr[0] = r.r
    cudaError_t e = launch_toeplitz_apply(K, nx, ny, nz, lambda, xr, xi, r_r, r_i, 0, work, tw,
                                          grid, s);
    if (e != cudaSuccess) return e;
    cg_start_kernel<<<grid, 256, 0, s>>>(br, bi, r_r, r_i, p_r, p_i, N);
    dot_partial_kernel<<<dot_blocks, kDotThreads, 0, s>>>(r_r, r_i, r_r, r_i, N, partial);
    sum_partials_kernel<<<1, kDotThreads, 0, s>>>(partial, dot_blocks, rr);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int it = 0; it < iters; ++it) {
        e = launch_toeplitz_apply(K, nx, ny, nz, lambda, p_r, p_i, a_r, a_i, 0, work, tw, grid,
                                  s);
        if (e != cudaSuccess) return e;
        dot_partial_kernel<<<dot_blocks, kDotThreads, 0, s>>>(p_r, p_i, a_r, a_i, N, partial);
        sum_partials_kernel<<<1, kDotThreads, 0, s>>>(partial, dot_blocks, pap);
        cg_xr_kernel<<<dot_blocks, kDotThreads, 0, s>>>(xr, xi, r_r, r_i, p_r, p_i, a_r, a_i,
                                                        N, rr + it, pap, partial);
        sum_partials_kernel<<<1, kDotThreads, 0, s>>>(partial, dot_blocks, rr + it + 1);
        cg_p_kernel<<<grid, 256, 0, s>>>(p_r, p_i, r_r, r_i, N, rr + it + 1, rr + it);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    sqrt_kernel<<<(iters + 1 + 255) / 256, 256, 0, s>>>(rr, iters + 1);
    return cudaGetLastError();
}

}  // namespace mri
