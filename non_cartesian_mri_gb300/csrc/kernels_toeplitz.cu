// kernels_toeplitz.cu -- the "find rho" step on a regular grid: F^H F as a
// Toeplitz product through FFTs (fft.cuh), and the conjugate-gradient
// iteration around it (the chapter's background section, Fig. 17.3:
// rho = (F^H F + lambda W^H W)^{-1} F^H D, W = I here).
//
// The grid has n = (nx, ny, nz) voxels; the doubled grid 2n holds Q on the
// circular grid of voxel differences and, zero-padded, the vector being
// multiplied; (F^H F v)[x] = sum_x' Q(x - x') v[x'] is then the corner of
// IFFT(FFT(Q) * FFT(pad v)) / |2n|, computed in five fused FFT stages that
// skip the padding's zeros and the part of the result that is cut away.
// All buffers are device memory; the CG scalars stay on the device (no host
// round trip per iteration).
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <set>
#include <type_traits>
#include <utility>

#include "fft.cuh"
#include "launch.h"

namespace mri {

namespace {

// Every kernel of a product and of a CG iteration is launched with
// programmatic dependent launch (see pdl_wait in fft.cuh): each lets the next
// one launch once its CTAs have started, and waits for the previous one
// before it touches any buffer.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

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

// The complex array the spectrum is taken of, on the doubled grid, from Q
// (SoA) on its z planes iz < nz: the planes at index n of every axis are
// zero (they hold Q at the difference -n h, which no voxel pair of the n
// grid has, and without them the grid is Hermitian-symmetric, so its
// spectrum is real), and a point with iz > nz is the conjugate of its mirror
// image (2nz - iz, -iy, -ix) mod 2n, because Q(-d) = conj Q(d).
__global__ void __launch_bounds__(256) spectrum_input_kernel(const float* r, const float* i,
                                                             int nx, int ny, int nz,
                                                             float2* out)
{
    const int64_t Lx = 2 * nx, Ly = 2 * ny;
    const int64_t n = Lx * Ly * 2 * nz;
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x) {
        const int64_t ix = k % Lx;
        const int64_t iy = (k / Lx) % Ly;
        const int64_t iz = k / (Lx * Ly);
        float2 v = make_float2(0.f, 0.f);
        if (ix != nx && iy != ny && iz != nz) {
            if (iz < nz) {
                v = make_float2(r[k], i[k]);
            } else {
                const int64_t src = ((2 * nz - iz) * Ly + ((Ly - iy) & (Ly - 1))) * Lx +
                                    ((Lx - ix) & (Lx - 1));
                v = make_float2(r[src], -i[src]);
            }
        }
        out[k] = v;
    }
}

// K = Re(spectrum); the imaginary part is rounding (Hermitian input)
__global__ void __launch_bounds__(256) real_part_kernel(const float2* spec, int64_t n, float* K)
{
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x)
        K[k] = spec[k].x;
}

// ---- sums for the conjugate-gradient scalars: per thread in float with
// compensated addition (the FP64 units are few: a conversion and a double
// FMA per element would bound these kernels), per block and across blocks in
// double
constexpr int kDotThreads = 256;
static_assert(kDotThreads == kFftThreads, "the stage kernels reduce with block_sum");

// s + c += x exactly up to the final rounding (TwoSum, Knuth): c collects
// the rounding error of every addition
struct FloatSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x)
    {
        const float t = s + x;
        const float z = t - s;
        c += (s - (t - z)) + (x - z);
        s = t;
    }
    __device__ __forceinline__ double value() const { return double(s) + double(c); }
};

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

// Once every CTA of the grid has written partial[blockIdx.x] (thread 0),
// the last CTA to arrive adds them up in index order (a fixed order, so the
// result does not depend on which CTA is last) into *out and resets *count
// for the next use: the total without a separate launch.  Every thread of
// the CTA calls it.
__device__ __forceinline__ void finish_sum(const double* partial, double* out,
                                           unsigned int* count, double* sm)
{
    __shared__ unsigned int ticket;
    if (threadIdx.x == 0) {
        __threadfence();   // this CTA's partial is visible before its ticket
        ticket = atomicAdd(count, 1u);
    }
    __syncthreads();
    if (ticket != gridDim.x - 1) return;
    __threadfence();
    double v = 0.0;
    for (int k = threadIdx.x; k < int(gridDim.x); k += kDotThreads) v += __ldcg(partial + k);
    const double total = block_sum(v, sm);
    if (threadIdx.x == 0) {
        *out = total;
        *count = 0u;
    }
}

// a CG step ratio, alpha = r.r / p.Ap or beta = new r.r / old r.r (0 once
// r = 0 or p.Ap = 0)
__device__ __forceinline__ float cg_ratio(const double* num, const double* den)
{
    const double a = *num, b = *den;
    return (a > 0.0 && b != 0.0) ? float(a / b) : 0.0f;
}

// ---- the Toeplitz product in five FFT stages over the doubled grid L = 2n.
// The padded vector is zero outside the corner n and only the corner of the
// result is kept, so no stage touches more than it must:
//   x forward   lines (iy < ny, iz < nz): read v (SoA, zero for ix >= nx),
//               write work[iz][iy][0 .. Lx)
//   y forward   lines (ix, iz < nz): read iy < ny (zero above), write all Ly
//   z           lines (ix, iy): read iz < nz (zero above), forward FFT, times
//               K (the spectrum of Q), inverse FFT, write iz < nz
//   y inverse   lines (ix, iz < nz): read all Ly, write iy < ny
//   x inverse   lines (iy < ny, iz < nz): read all Lx, write
//               out = scale * value + lambda * v (+ out) for ix < nx
// work is [nz][Ly][Lx] complex (half the doubled grid); K is [Lz][Ly][Lx]
// real.  The x inverse stage can also sum Re <v, result> per CTA (the p.Ap
// of conjugate gradients).
enum ToeplitzStage : int { kXFwd = 0, kYFwd = 1, kZConv = 2, kYInv = 3, kXInv = 4 };

struct ToeplitzArgs {
    const float* ir;        // v, real and imaginary, [nz][ny][nx]
    const float* ii;
    float* outr;            // result, [nz][ny][nx] (may alias ir / ii)
    float* outi;
    float2* work;           // [nz][2 ny][2 nx]
    const float* K;         // [2 nz][2 ny][2 nx], real
    double* dot;            // x inverse: per CTA Re <v, result> (nullptr: none)
    double* dot_total;      // and their sum, by the last CTA (nullptr: not formed)
    unsigned int* dot_count;   // its arrival counter (zero between uses)
    // x forward, conjugate gradients: v = r + beta v, beta = *rr_new /
    // *rr_old, is formed, written back to (vw_r, vw_i) = (ir, ii) and
    // transformed (upd_r == nullptr: v as it is)
    const float* upd_r;
    const float* upd_i;
    const double* rr_new;
    const double* rr_old;
    float* vw_r;
    float* vw_i;
    int log2nx, log2ny, log2nz;
    float scale;            // 1 / |2n|, the inverse transform's normalisation
    float lambda;
    int accumulate;
};

// Every index below fits in 32 bits: the grid is at most 512 per axis, so
// K has at most 2^30 values.  Transforms use the plan with the odd radix
// first; the inverse transform of the z stage, which starts from the forward
// transform's registers, uses the plan with the odd radix last, so that its
// first pass has the forward transform's last radix and butterflies.
template <int STAGE, int LOG2L>
__global__ void __launch_bounds__(kFftThreads, fft_min_ctas(LOG2L))
    toeplitz_stage_kernel(ToeplitzArgs p, int64_t lines64, const float2* tw)
{
    extern __shared__ float2 fft_sm[];
    constexpr int log2W = fft_log2_lines(LOG2L);
    float2* const buf = fft_sm;
    float2* const tws = fft_sm + (fft_line_stride(LOG2L) << log2W);
    const uint32_t lines = uint32_t(lines64);
    const uint32_t group = blockIdx.x << log2W;
    const int log2Lx = p.log2nx + 1, log2Ly = p.log2ny + 1;
    const float2 zero = make_float2(0.f, 0.f);
    // the last pass of a transform: radix, butterflies a thread holds, and
    // the stride of its outputs
    constexpr int RL = fft_last_log2r<LOG2L, true>();
    constexpr int IL = fft_items(LOG2L, RL);
    constexpr int per = fft_last_per<LOG2L, true>();
    pdl_launch_dependents();
    fft_stage_twiddles<LOG2L>(tws, tw);
    pdl_wait();
    if constexpr (STAGE == kXFwd || STAGE == kXInv) {
        const uint32_t ymask = (1u << p.log2ny) - 1;
        // line l = iz ny + iy: its row of work, and its row of v
        auto widx = [&](int w, int j) -> uint32_t {
            const uint32_t l = group + w;
            return ((((l >> p.log2ny) << log2Ly) | (l & ymask)) << log2Lx) + j;
        };
        auto vidx = [&](int w, int j) -> uint32_t { return ((group + w) << p.log2nx) + j; };
        if constexpr (STAGE == kXFwd) {
            const bool upd = p.upd_r != nullptr;
            const float beta = upd ? cg_ratio(p.rr_new, p.rr_old) : 0.f;
            // the positions ix >= nx of the padded line are zero: not loaded
            fft_lines<false, LOG2L, true, false, true>(
                buf, tws,
                [&](int w, int pos) {
                    if (group + w >= lines) return zero;
                    const uint32_t n = vidx(w, pos);
                    float vr = p.ir[n], vi = p.ii[n];
                    if (upd) {
                        vr = fmaf(beta, vr, p.upd_r[n]);
                        vi = fmaf(beta, vi, p.upd_i[n]);
                    }
                    return make_float2(vr, vi);
                },
                [&](auto& y) {
#pragma unroll
                    for (int it = 0; it < IL; ++it) {
                        int w, j;
                        if (fft_item<LOG2L, RL, false>(it, w, j) && group + w < lines) {
#pragma unroll
                            for (int q = 0; q < (1 << RL); ++q) p.work[widx(w, j + q * per)] = y[it][q];
                        }
                    }
                },
                [&](int w, int pos, float2 v) {
                    // the new direction, written back once every load is
                    // issued (each v[n] is read and written by this thread only)
                    if (!upd || group + w >= lines) return;
                    const uint32_t n = vidx(w, pos);
                    p.vw_r[n] = v.x;
                    p.vw_i[n] = v.y;
                });
        } else {
            FloatSum dot;
            fft_lines<true, LOG2L, true, false, false>(
                buf, tws,
                [&](int w, int pos) { return group + w < lines ? p.work[widx(w, pos)] : zero; },
                [&](auto& y) {
#pragma unroll
                    for (int it = 0; it < IL; ++it) {
                        int w, j;
                        if (!fft_item<LOG2L, RL, false>(it, w, j) || group + w >= lines) continue;
                        // the corner ix < nx: outputs q < R / 2.  Every v[n] of
                        // the item is loaded before the first out[n] is stored
                        // (v and out may be one array, each n this thread's
                        // only; a load after a store would wait for it)
                        constexpr int H = (1 << RL) / 2;
                        float vr_[H], vi_[H];
#pragma unroll
                        for (int q = 0; q < H; ++q) {
                            const uint32_t n = vidx(w, j + q * per);
                            vr_[q] = p.ir[n];
                            vi_[q] = p.ii[n];
                        }
#pragma unroll
                        for (int q = 0; q < H; ++q) {
                            const uint32_t n = vidx(w, j + q * per);
                            const float vr = vr_[q], vi = vi_[q];
                            float r = fmaf(p.lambda, vr, y[it][q].x * p.scale);
                            float i = fmaf(p.lambda, vi, y[it][q].y * p.scale);
                            if (p.accumulate) {
                                r += p.outr[n];
                                i += p.outi[n];
                            }
                            p.outr[n] = r;
                            p.outi[n] = i;
                            dot.add(vr * r);
                            dot.add(vi * i);
                        }
                    }
                });
            if (p.dot != nullptr) {
                __shared__ double sm[kDotThreads / 32];
                const double total = block_sum(dot.value(), sm);
                if (threadIdx.x == 0) p.dot[blockIdx.x] = total;
                if (p.dot_total != nullptr) finish_sum(p.dot, p.dot_total, p.dot_count, sm);
            }
        }
    } else {
        // y: line l = iz Lx + ix at stride Lx; z: line l = iy Lx + ix at
        // stride Lx Ly.  work holds the positions < L / 2 of a z line (and of
        // a y line before the y forward stage).
        const int log2inner = STAGE == kZConv ? log2Lx + log2Ly : log2Lx;
        const uint32_t imask = (1u << log2inner) - 1;
        auto gidx = [&](int w, int j) -> uint32_t {
            const uint32_t l = group + w;
            return ((((l >> log2inner) << LOG2L) + j) << log2inner) + (l & imask);
        };
        // cache hints, measured: the strided stages' work loads in L2 only
        // (__ldcg) and the once-read spectrum as streaming (__ldcs, evict
        // first), CG iteration 0.168 -> 0.160 ms at 128^3
        auto load = [&](int w, int pos) {
            return group + w < lines ? __ldcg(p.work + gidx(w, pos)) : zero;
        };
        // the lower half of every line to work
        auto store_half = [&](auto& y, auto rl, auto per_c) {
            constexpr int R_ = decltype(rl)::value, PER = decltype(per_c)::value;
#pragma unroll
            for (int it = 0; it < fft_items(LOG2L, R_); ++it) {
                int w, j;
                if (fft_item<LOG2L, R_, true>(it, w, j) && group + w < lines) {
#pragma unroll
                    for (int q = 0; q < (1 << R_) / 2; ++q) p.work[gidx(w, j + q * PER)] = y[it][q];
                }
            }
        };
        if constexpr (STAGE == kZConv) {
            // the (real) spectrum at the positions of the forward transform's
            // last pass, loaded first so that it arrives during the transform
            // (streaming: each value is read once per product)
            float kreg[IL][1 << RL];
#pragma unroll
            for (int it = 0; it < IL; ++it) {
                int w, j;
                const bool on = fft_item<LOG2L, RL, true>(it, w, j) && group + w < lines;
#pragma unroll
                for (int q = 0; q < (1 << RL); ++q)
                    kreg[it][q] = on ? __ldcs(p.K + gidx(w, j + q * per)) : 0.f;
            }
            fft_lines<false, LOG2L, true, true, true>(buf, tws, load, [&](auto& y) {
#pragma unroll
                for (int it = 0; it < IL; ++it) {
#pragma unroll
                    for (int q = 0; q < (1 << RL); ++q)
                        y[it][q] = make_float2(y[it][q].x * kreg[it][q], y[it][q].y * kreg[it][q]);
                    // the inverse transform's first pass (Ns = 1, no twiddles)
                    fft_dft_regs<true, RL, false>(y[it]);
                }
                constexpr int RI = fft_last_log2r<LOG2L, false>();
                fft_run_from<true, LOG2L, false, true, 0>(buf, tws, y, [&](auto& yo) {
                    store_half(yo, std::integral_constant<int, RI>{},
                               std::integral_constant<int, fft_last_per<LOG2L, false>()>{});
                });
            });
        } else if constexpr (STAGE == kYFwd) {
            fft_lines<false, LOG2L, true, true, true>(buf, tws, load, [&](auto& y) {
#pragma unroll
                for (int it = 0; it < IL; ++it) {
                    int w, j;
                    if (fft_item<LOG2L, RL, true>(it, w, j) && group + w < lines) {
#pragma unroll
                        for (int q = 0; q < (1 << RL); ++q) p.work[gidx(w, j + q * per)] = y[it][q];
                    }
                }
            });
        } else {
            fft_lines<true, LOG2L, true, true, false>(buf, tws, load, [&](auto& y) {
                store_half(y, std::integral_constant<int, RL>{}, std::integral_constant<int, per>{});
            });
        }
    }
}

// ---- the strided stages (y forward, z, y inverse) as persistent CTAs.
// Loaded one tile at a time, these stages leave DRAM mostly idle (ncu at
// 128^3: 31-36 % of its cycles active, the warps waiting on their loads):
// each CTA loads, transforms, then stores.  Here each CTA walks over the
// tiles g = blockIdx.x, + gridDim.x, ... and copies the inputs of its next
// tile (the work lines' loaded positions, and in the z stage the spectrum)
// into a second shared-memory buffer with cp.async while it transforms the
// current one, so the copies are in flight during the passes.  The staged
// values sit at [position][line] (the W lines of a tile are adjacent in
// memory at every position), read back by the first pass as the loads of
// toeplitz_stage_kernel read global memory.
__device__ __forceinline__ void cp_async8(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// positions of a line the stage loads (complex; the spectrum: all L, z only)
template <int STAGE, int LOG2L>
__host__ __device__ constexpr int strided_cpos() { return STAGE == kYInv ? 1 << LOG2L : 1 << (LOG2L - 1); }
template <int STAGE, int LOG2L>
__host__ __device__ constexpr int strided_kpos() { return STAGE == kZConv ? 1 << LOG2L : 0; }
// bytes of one staging buffer
template <int STAGE, int LOG2L>
__host__ __device__ constexpr size_t strided_stage_bytes()
{
    return (size_t(strided_cpos<STAGE, LOG2L>()) * 8 + size_t(strided_kpos<STAGE, LOG2L>()) * 4)
           << fft_log2_lines(LOG2L);
}
template <int STAGE, int LOG2L>
size_t strided_smem_total()
{
    return fft_smem_total(LOG2L) + 2 * strided_stage_bytes<STAGE, LOG2L>();
}

// CTAs per SM the persistent kernels are compiled for: two up to L = 256
// (about 100 KB of shared memory each), then one
__host__ __device__ constexpr int strided_min_ctas(int log2L) { return log2L <= 8 ? 2 : 1; }

template <int STAGE, int LOG2L>
__global__ void __launch_bounds__(kFftThreads, strided_min_ctas(LOG2L))
    toeplitz_strided_kernel(ToeplitzArgs p, int64_t lines64, const float2* tw)
{
    static_assert(STAGE == kYFwd || STAGE == kZConv || STAGE == kYInv, "strided stages");
    extern __shared__ float2 fft_sm[];
    constexpr int log2W = fft_log2_lines(LOG2L);
    constexpr int W = 1 << log2W;
    constexpr int CPOS = strided_cpos<STAGE, LOG2L>();
    constexpr int KPOS = strided_kpos<STAGE, LOG2L>();
    constexpr size_t SB = strided_stage_bytes<STAGE, LOG2L>();
    float2* const buf = fft_sm;
    float2* const tws = fft_sm + (fft_line_stride(LOG2L) << log2W);
    unsigned char* const stage0 =
        reinterpret_cast<unsigned char*>(tws + (1 << LOG2L));   // 8-byte aligned
    const uint32_t lines = uint32_t(lines64);
    const uint32_t ngroups = (lines + W - 1) >> log2W;
    const int log2Lx = p.log2nx + 1, log2Ly = p.log2ny + 1;
    const float2 zero = make_float2(0.f, 0.f);
    constexpr int RL = fft_last_log2r<LOG2L, true>();
    constexpr int IL = fft_items(LOG2L, RL);
    constexpr int per = fft_last_per<LOG2L, true>();
    const int log2inner = STAGE == kZConv ? log2Lx + log2Ly : log2Lx;
    const uint32_t imask = (1u << log2inner) - 1;
    auto gidx = [&](uint32_t l, int j) -> uint32_t {
        return ((((l >> log2inner) << LOG2L) + j) << log2inner) + (l & imask);
    };
    // the staged complex values and spectrum of a buffer
    auto cst = [&](int b) { return reinterpret_cast<float2*>(stage0 + b * SB); };
    auto kst = [&](int b) { return reinterpret_cast<float*>(stage0 + b * SB + size_t(CPOS) * 8 * W); };
    // 16-byte copies when a tile's W lines are adjacent at every position
    // (inner >= W and the tile whole), else one element per copy
    const bool wide = (1u << log2inner) >= uint32_t(W);
    auto prefetch = [&](uint32_t g, int b) {
        const uint32_t l0 = g << log2W;
        float2* const c = cst(b);
        if (wide && l0 + W <= lines) {
            for (int e = threadIdx.x; e < CPOS * W / 2; e += kFftThreads) {
                const int w = (2 * e) & (W - 1), pos = (2 * e) >> log2W;
                cp_async16(c + 2 * e, p.work + gidx(l0 + w, pos));
            }
        } else {
            for (int e = threadIdx.x; e < CPOS * W; e += kFftThreads) {
                const int w = e & (W - 1), pos = e >> log2W;
                if (l0 + w < lines) cp_async8(c + e, p.work + gidx(l0 + w, pos));
                else c[e] = zero;
            }
        }
        if constexpr (KPOS > 0) {
            float* const k = kst(b);
            if (wide && l0 + W <= lines) {
                for (int e = threadIdx.x; e < KPOS * W / 4; e += kFftThreads) {
                    const int w = (4 * e) & (W - 1), pos = (4 * e) >> log2W;
                    cp_async16(k + 4 * e, p.K + gidx(l0 + w, pos));
                }
            } else {
                for (int e = threadIdx.x; e < KPOS * W; e += kFftThreads) {
                    const int w = e & (W - 1), pos = e >> log2W;
                    if (l0 + w < lines) cp_async4(k + e, p.K + gidx(l0 + w, pos));
                    else k[e] = 0.f;
                }
            }
        }
    };
    pdl_launch_dependents();
    fft_stage_twiddles<LOG2L>(tws, tw);
    pdl_wait();

    int it = 0;
    if (blockIdx.x < ngroups) prefetch(blockIdx.x, 0);
    cp_async_commit();
    for (uint32_t g = blockIdx.x; g < ngroups; g += gridDim.x, ++it) {
        const int b = it & 1;
        if (g + gridDim.x < ngroups) prefetch(g + gridDim.x, b ^ 1);
        cp_async_commit();
        cp_async_wait<1>();           // this tile's copies have landed
        __syncthreads();              // everyone's, and the zeros written beside them
        const uint32_t group = g << log2W;
        const float2* const c = cst(b);
        auto load = [&](int w, int pos) { return c[(pos << log2W) + w]; };
        // the lower half of every line to work
        auto store_half = [&](auto& y, auto rl, auto per_c) {
            constexpr int R_ = decltype(rl)::value, PER = decltype(per_c)::value;
#pragma unroll
            for (int i2 = 0; i2 < fft_items(LOG2L, R_); ++i2) {
                int w, j;
                if (fft_item<LOG2L, R_, true>(i2, w, j) && group + w < lines) {
#pragma unroll
                    for (int q = 0; q < (1 << R_) / 2; ++q)
                        p.work[gidx(group + w, j + q * PER)] = y[i2][q];
                }
            }
        };
        if constexpr (STAGE == kZConv) {
            const float* const k = kst(b);
            float kreg[IL][1 << RL];
#pragma unroll
            for (int i2 = 0; i2 < IL; ++i2) {
                int w, j;
                const bool on = fft_item<LOG2L, RL, true>(i2, w, j);
#pragma unroll
                for (int q = 0; q < (1 << RL); ++q)
                    kreg[i2][q] = on ? k[((j + q * per) << log2W) + w] : 0.f;
            }
            fft_lines<false, LOG2L, true, true, true>(buf, tws, load, [&](auto& y) {
#pragma unroll
                for (int i2 = 0; i2 < IL; ++i2) {
#pragma unroll
                    for (int q = 0; q < (1 << RL); ++q)
                        y[i2][q] = make_float2(y[i2][q].x * kreg[i2][q], y[i2][q].y * kreg[i2][q]);
                    // the inverse transform's first pass (Ns = 1, no twiddles)
                    fft_dft_regs<true, RL, false>(y[i2]);
                }
                constexpr int RI = fft_last_log2r<LOG2L, false>();
                fft_run_from<true, LOG2L, false, true, 0>(buf, tws, y, [&](auto& yo) {
                    store_half(yo, std::integral_constant<int, RI>{},
                               std::integral_constant<int, fft_last_per<LOG2L, false>()>{});
                });
            });
        } else if constexpr (STAGE == kYFwd) {
            fft_lines<false, LOG2L, true, true, true>(buf, tws, load, [&](auto& y) {
#pragma unroll
                for (int i2 = 0; i2 < IL; ++i2) {
                    int w, j;
                    if (fft_item<LOG2L, RL, true>(i2, w, j) && group + w < lines) {
#pragma unroll
                        for (int q = 0; q < (1 << RL); ++q)
                            p.work[gidx(group + w, j + q * per)] = y[i2][q];
                    }
                }
            });
        } else {
            fft_lines<true, LOG2L, true, true, false>(buf, tws, load, [&](auto& y) {
                store_half(y, std::integral_constant<int, RL>{}, std::integral_constant<int, per>{});
            });
        }
        __syncthreads();              // this buffer is read; the next prefetch may refill it
    }
    cp_async_wait<0>();
}

// ---- conjugate gradients
__global__ void __launch_bounds__(kDotThreads) dot_partial_kernel(const float* ar, const float* ai,
                                                                  const float* br, const float* bi,
                                                                  int64_t n, double* partial)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ double sm[kDotThreads / 32];
    FloatSum v;
    for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n;
         k += int64_t(gridDim.x) * blockDim.x) {
        v.add(ar[k] * br[k]);
        v.add(ai[k] * bi[k]);
    }
    const double s = block_sum(v.value(), sm);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kDotThreads) sum_partials_kernel(const double* partial, int n,
                                                                   double* out)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ double sm[kDotThreads / 32];
    double v = 0.0;
    for (int k = threadIdx.x; k < n; k += kDotThreads) v += partial[k];   // fixed order
    const double s = block_sum(v, sm);
    if (threadIdx.x == 0) *out = s;
}


__device__ __forceinline__ float4 fma4(float a, float4 x, float4 y)
{
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

// x += alpha p, r -= alpha Ap, partial sums of |r|^2 and (the last CTA)
// their total into *rr_next; VEC: four values per
// access (n a multiple of 4, every array 16-byte aligned).  Every load of an
// element comes before its stores: the arrays may alias as far as the
// compiler knows, so a load after a store would wait for it, one access in
// flight at a time.
template <bool VEC>
__global__ void __launch_bounds__(kDotThreads) cg_xr_kernel(float* xr, float* xi, float* rr_,
                                                            float* ri, const float* pr,
                                                            const float* pi, const float* apr,
                                                            const float* api, int64_t n,
                                                            const double* rr, const double* pap,
                                                            double* partial, double* rr_next,
                                                            unsigned int* count)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ double sm[kDotThreads / 32];
    const float alpha = cg_ratio(rr, pap);
    FloatSum v;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    if constexpr (VEC) {
        float4* const x4r = reinterpret_cast<float4*>(xr);
        float4* const x4i = reinterpret_cast<float4*>(xi);
        float4* const r4r = reinterpret_cast<float4*>(rr_);
        float4* const r4i = reinterpret_cast<float4*>(ri);
        for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < (n >> 2);
             k += stride) {
            const float4 p_r = reinterpret_cast<const float4*>(pr)[k];
            const float4 p_i = reinterpret_cast<const float4*>(pi)[k];
            const float4 a_r = reinterpret_cast<const float4*>(apr)[k];
            const float4 a_i = reinterpret_cast<const float4*>(api)[k];
            const float4 x_r = x4r[k], x_i = x4i[k], r_r = r4r[k], r_i = r4i[k];
            x4r[k] = fma4(alpha, p_r, x_r);
            x4i[k] = fma4(alpha, p_i, x_i);
            const float4 a = fma4(-alpha, a_r, r_r);
            const float4 b = fma4(-alpha, a_i, r_i);
            r4r[k] = a;
            r4i[k] = b;
            v.add(a.x * a.x);
            v.add(a.y * a.y);
            v.add(a.z * a.z);
            v.add(a.w * a.w);
            v.add(b.x * b.x);
            v.add(b.y * b.y);
            v.add(b.z * b.z);
            v.add(b.w * b.w);
        }
    } else {
        for (int64_t k = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; k < n; k += stride) {
            const float p_r = pr[k], p_i = pi[k], a_r = apr[k], a_i = api[k];
            const float x_r = xr[k], x_i = xi[k], r_r = rr_[k], r_i = ri[k];
            xr[k] = fmaf(alpha, p_r, x_r);
            xi[k] = fmaf(alpha, p_i, x_i);
            const float a = fmaf(-alpha, a_r, r_r);
            const float b = fmaf(-alpha, a_i, r_i);
            rr_[k] = a;
            ri[k] = b;
            v.add(a * a);
            v.add(b * b);
        }
    }
    const double s = block_sum(v.value(), sm);
    if (threadIdx.x == 0) partial[blockIdx.x] = s;
    finish_sum(partial, rr_next, count, sm);   // the new r.r
}

// r = b - r (r holds A x), p = r
__global__ void __launch_bounds__(256) cg_start_kernel(const float* br, const float* bi,
                                                       float* rr_, float* ri, float* pr,
                                                       float* pi, int64_t n)
{
    pdl_launch_dependents();
    pdl_wait();
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
    pdl_launch_dependents();
    pdl_wait();
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

namespace {

// Kernels whose launch attributes have been set, per device (the attributes
// are per device; a process may use several).
std::mutex g_attr_mutex;
std::set<std::pair<int, const void*>> g_attr_done;

bool attributes_set(const void* kernel)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    return g_attr_done.count({dev, kernel}) != 0;
}

void mark_attributes_set(const void* kernel)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    g_attr_done.insert({dev, kernel});
}

// dynamic shared memory, then the launch, of one FFT kernel over `lines`
// lines of length 2^log2L (the per-length kernels are picked by `pick`)
template <class Pick>
cudaError_t launch_by_length(int log2L, int64_t lines, cudaStream_t s, Pick pick)
{
    auto go = [&](auto kernel, auto... args) -> cudaError_t {
        const size_t smem = fft_smem_total(log2L);
        // once per kernel and device: the dynamic shared memory, and all of
        // the unified L1 / shared memory as shared memory, so that
        // fft_min_ctas tiles fit on an SM
        if (!attributes_set(reinterpret_cast<const void*>(kernel))) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 int(smem));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         int(cudaSharedmemCarveoutMaxShared));
            if (e != cudaSuccess) return e;
            mark_attributes_set(reinterpret_cast<const void*>(kernel));
        }
        const int64_t W = int64_t(1) << fft_log2_lines(log2L);
        return launch_pdl(kernel, unsigned((lines + W - 1) / W), kFftThreads, smem, s, args...);
    };
    switch (log2L) {
        case 1: return pick(std::integral_constant<int, 1>{}, go);
        case 2: return pick(std::integral_constant<int, 2>{}, go);
        case 3: return pick(std::integral_constant<int, 3>{}, go);
        case 4: return pick(std::integral_constant<int, 4>{}, go);
        case 5: return pick(std::integral_constant<int, 5>{}, go);
        case 6: return pick(std::integral_constant<int, 6>{}, go);
        case 7: return pick(std::integral_constant<int, 7>{}, go);
        case 8: return pick(std::integral_constant<int, 8>{}, go);
        case 9: return pick(std::integral_constant<int, 9>{}, go);
        case 10: return pick(std::integral_constant<int, 10>{}, go);
    }
    return cudaErrorInvalidValue;
}

template <bool INVERSE>
cudaError_t fft_axis(float2* a, int log2L, int log2inner, int64_t lines, const float2* tw,
                     cudaStream_t s)
{
    return launch_by_length(log2L, lines, s, [&](auto len, auto go) {
        constexpr int L2 = decltype(len)::value;
        return log2inner == 0 ? go(fft_axis_kernel<INVERSE, L2, true>, a, log2inner, lines, tw)
                              : go(fft_axis_kernel<INVERSE, L2, false>, a, log2inner, lines, tw);
    });
}

// Lines of at least 2^MRI_TOEPLITZ_PERSISTENT_LOG2L take the persistent
// strided stages (measured: 256^3 grid, doubled grid 512^3, product 1.65 ->
// 1.49 ms; 128^3 0.128 -> 0.129 ms, 64^3 0.042 -> 0.046: shorter lines
// keep one tile per CTA, four CTAs per SM).
#ifndef MRI_TOEPLITZ_PERSISTENT_LOG2L
#define MRI_TOEPLITZ_PERSISTENT_LOG2L 9
#endif

// A strided stage as persistent CTAs (toeplitz_strided_kernel): as many as
// fit on the SMs at once, at most one per tile.
template <int STAGE, int LOG2L>
cudaError_t launch_strided(const ToeplitzArgs& p, int64_t lines, const float2* tw, cudaStream_t s)
{
    auto kernel = toeplitz_strided_kernel<STAGE, LOG2L>;
    const size_t smem = strided_smem_total<STAGE, LOG2L>();
    if (!attributes_set(reinterpret_cast<const void*>(kernel))) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     int(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return e;
        mark_attributes_set(reinterpret_cast<const void*>(kernel));
    }
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFftThreads, smem);
    if (e != cudaSuccess) return e;
    const int64_t W = int64_t(1) << fft_log2_lines(LOG2L);
    const int64_t groups = (lines + W - 1) / W;
    const int64_t grid = std::min<int64_t>(groups, int64_t(sms) * std::max(per_sm, 1));
    return launch_pdl(kernel, unsigned(grid), kFftThreads, smem, s, p, lines, tw);
}

template <int STAGE>
cudaError_t toeplitz_stage(const ToeplitzArgs& p, int log2L, int64_t lines, const float2* tw,
                           cudaStream_t s)
{
    return launch_by_length(log2L, lines, s, [&](auto len, auto go) {
        constexpr int L2 = decltype(len)::value;
        if constexpr (STAGE != kXFwd && STAGE != kXInv && L2 >= MRI_TOEPLITZ_PERSISTENT_LOG2L)
            return launch_strided<STAGE, L2>(p, lines, tw, s);
        else
            return go(toeplitz_stage_kernel<STAGE, L2>, p, lines, tw);
    });
}

}  // namespace

cudaError_t launch_fft_axis(float2* a, int Lx, int Ly, int Lz, int axis, bool inverse,
                            const float2* tw, cudaStream_t s)
{
    if (!fft_len_ok(Lx) || !fft_len_ok(Ly) || !fft_len_ok(Lz) || axis < 0 || axis > 2)
        return cudaErrorInvalidValue;
    const int len[3] = {Lx, Ly, Lz};
    const int log2L = log2i(len[axis]);
    if (log2L == 0) return cudaSuccess;
    int log2inner = 0;
    for (int ax = 0; ax < axis; ++ax) log2inner += log2i(len[ax]);
    const int64_t lines = (int64_t(Lx) * Ly * Lz) >> log2L;
    return inverse ? fft_axis<true>(a, log2L, log2inner, lines, tw, s)
                   : fft_axis<false>(a, log2L, log2inner, lines, tw, s);
}

cudaError_t launch_fft3(float2* a, int Lx, int Ly, int Lz, bool inverse, const float2* tw,
                        cudaStream_t s)
{
    for (int ax = 0; ax < 3; ++ax) {
        const cudaError_t e = launch_fft_axis(a, Lx, Ly, Lz, ax, inverse, tw, s);
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

cudaError_t launch_spectrum_input(const float* r, const float* i, int nx, int ny, int nz,
                                  float2* out, int grid, cudaStream_t s)
{
    spectrum_input_kernel<<<grid, 256, 0, s>>>(r, i, nx, ny, nz, out);
    return cudaGetLastError();
}

cudaError_t launch_real_part(const float2* spec, int64_t n, float* K, int grid, cudaStream_t s)
{
    real_part_kernel<<<grid, 256, 0, s>>>(spec, n, K);
    return cudaGetLastError();
}

int64_t toeplitz_dot_blocks(int nx, int ny, int nz)
{
    const int64_t W = int64_t(1) << fft_log2_lines(log2i(2 * nx));
    return (int64_t(ny) * nz + W - 1) / W;
}

namespace {

// upd_r != nullptr: v = (vw_r, vw_i) is first replaced by upd + beta v (the
// CG direction update, see ToeplitzArgs)
cudaError_t toeplitz_apply(const float* K, int nx, int ny, int nz, float lambda, const float* ir,
                           const float* ii, float* outr, float* outi, int accumulate,
                           float2* work, double* dot, const float2* tw, cudaStream_t s,
                           double* dot_total = nullptr, unsigned int* dot_count = nullptr,
                           const float* upd_r = nullptr, const float* upd_i = nullptr,
                           const double* rr_new = nullptr, const double* rr_old = nullptr,
                           float* vw_r = nullptr, float* vw_i = nullptr)
{
    ToeplitzArgs p;
    p.upd_r = upd_r;
    p.upd_i = upd_i;
    p.rr_new = rr_new;
    p.rr_old = rr_old;
    p.vw_r = vw_r;
    p.vw_i = vw_i;
    p.ir = ir;
    p.ii = ii;
    p.outr = outr;
    p.outi = outi;
    p.work = work;
    p.K = K;
    p.dot = dot;
    p.dot_total = dot_total;
    p.dot_count = dot_count;
    p.log2nx = log2i(nx);
    p.log2ny = log2i(ny);
    p.log2nz = log2i(nz);
    p.scale = float(1.0 / (8.0 * double(nx) * ny * nz));
    p.lambda = lambda;
    p.accumulate = accumulate;
    const int64_t Lx = 2 * nx, Ly = 2 * ny;
    cudaError_t e = toeplitz_stage<kXFwd>(p, p.log2nx + 1, int64_t(ny) * nz, tw, s);
    if (e == cudaSuccess) e = toeplitz_stage<kYFwd>(p, p.log2ny + 1, Lx * nz, tw, s);
    if (e == cudaSuccess) e = toeplitz_stage<kZConv>(p, p.log2nz + 1, Lx * Ly, tw, s);
    if (e == cudaSuccess) e = toeplitz_stage<kYInv>(p, p.log2ny + 1, Lx * nz, tw, s);
    if (e == cudaSuccess) e = toeplitz_stage<kXInv>(p, p.log2nx + 1, int64_t(ny) * nz, tw, s);
    return e;
}

}  // namespace

cudaError_t launch_toeplitz_apply(const float* K, int nx, int ny, int nz, float lambda,
                                  const float* ir, const float* ii, float* outr, float* outi,
                                  int accumulate, float2* work, const float2* tw, cudaStream_t s)
{
    return toeplitz_apply(K, nx, ny, nz, lambda, ir, ii, outr, outi, accumulate, work, nullptr,
                          tw, s);
}

cudaError_t launch_cg(const float* K, int nx, int ny, int nz, float lambda, const float* br,
                      const float* bi, float* xr, float* xi, int iters, double* rr,
                      float* vec, float2* work, double* scal, const float2* tw, int grid,
                      int dot_blocks, cudaStream_t s)
{
    // vec: r (2 N), p (2 N), Ap (2 N); scal: dot partials (max(dot_blocks,
    // toeplitz_dot_blocks)), p.Ap, then two arrival counters (one double's room)
    const int64_t N = int64_t(nx) * ny * nz;
    float *r_r = vec, *r_i = vec + N, *p_r = vec + 2 * N, *p_i = vec + 3 * N;
    float *a_r = vec + 4 * N, *a_i = vec + 5 * N;
    const int64_t apply_blocks = toeplitz_dot_blocks(nx, ny, nz);
    double* partial = scal;
    double* pap = scal + std::max<int64_t>(dot_blocks, apply_blocks);
    unsigned int* count = reinterpret_cast<unsigned int*>(pap + 1);   // [0]: p.Ap, [1]: r.r
    const bool vec4 = N % 4 == 0 && (reinterpret_cast<uintptr_t>(xr) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(xi) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(vec) & 15u) == 0;
    cudaError_t e = cudaMemsetAsync(count, 0, 2 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    // r = b - A x, p = r, rr[0] = r.r
    e = toeplitz_apply(K, nx, ny, nz, lambda, xr, xi, r_r, r_i, 0, work, nullptr, tw, s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(cg_start_kernel, grid, 256, 0, s, br, bi, r_r, r_i, p_r, p_i, N);
    if (e == cudaSuccess)
        e = launch_pdl(dot_partial_kernel, dot_blocks, kDotThreads, 0, s, r_r, r_i, r_r, r_i, N,
                       partial);
    if (e == cudaSuccess)
        e = launch_pdl(sum_partials_kernel, 1, kDotThreads, 0, s, partial, dot_blocks, rr);
    if (e != cudaSuccess) return e;
    for (int it = 0; it < iters; ++it) {
        // Ap, with p.Ap summed by the last CTA of its last stage; from the
        // second iteration on, its first stage also forms the new direction
        // p = r + beta p, beta = rr[it] / rr[it - 1]
        if (it == 0)
            e = toeplitz_apply(K, nx, ny, nz, lambda, p_r, p_i, a_r, a_i, 0, work, partial, tw, s,
                               pap, count);
        else
            e = toeplitz_apply(K, nx, ny, nz, lambda, p_r, p_i, a_r, a_i, 0, work, partial, tw, s,
                               pap, count, r_r, r_i, rr + it, rr + it - 1, p_r, p_i);
        // x += alpha p, r -= alpha Ap, rr[it + 1] = r.r (by its last CTA)
        if (e == cudaSuccess)
            e = launch_pdl(vec4 ? cg_xr_kernel<true> : cg_xr_kernel<false>, dot_blocks,
                           kDotThreads, 0, s, xr, xi, r_r, r_i, p_r, p_i, a_r, a_i, N, rr + it,
                           pap, partial, rr + it + 1, count + 1);
        if (e != cudaSuccess) return e;
    }
    e = launch_pdl(sqrt_kernel, (iters + 1 + 255) / 256, 256, 0, s, rr, iters + 1);
    return e;
}

}  // namespace mri
