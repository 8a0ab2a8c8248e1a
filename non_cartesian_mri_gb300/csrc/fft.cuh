// fft.cuh -- complex FFTs along one axis of a 3-D array, for the Toeplitz
// product F^H F of the "find rho" step (the chapter's background section:
// F^H F is Toeplitz, so its product with rho goes through FFTs).
//
// Layout: float2 (re, im) interleaved, x fastest; an axis of length L (a
// power of two, 2 .. kFftMaxLen) sits between `outer` slabs and `inner`
// consecutive elements: element j of line (o, i) is a[(o L + j) inner + i].
// A CTA transforms W lines (16, or 8 for L = 1024): W consecutive i when
// inner > 1 (so that a warp's loads cover consecutive addresses), W
// consecutive o when inner == 1 (each line contiguous).  The lines go to
// shared memory in natural order and the transform is a Stockham
// auto-sorting FFT: radix-4 passes (one radix-2 pass when log2 L is odd),
// each thread reading 4 values of a line at stride L / 4, multiplying by
// the twiddles of the pass and doing the 4-point DFT in registers, then,
// after a barrier, writing them back in place where the final output ends
// up in natural order -- no bit reversal, one buffer (six CTAs per SM at
// L = 256).  Twiddles e^{-2 pi i k / kFftMaxLen} come from a per-device table
// evaluated in double precision (the twiddle kernel of kernels_toeplitz.cu)
// and are staged for the line length in shared memory; the inverse
// transform conjugates them where it uses them and does not scale (the
// caller divides by the size).  The pieces (stage the twiddles, load a tile,
// run the passes, store a tile) are separate so that a kernel can do more
// than one transform on a tile, or fuse the work on either side of one.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mri {

constexpr int kFftMaxLen = 1024;              // 2^10
constexpr int kFftThreads = 256;

inline bool fft_len_ok(int64_t L) { return L >= 1 && L <= kFftMaxLen && (L & (L - 1)) == 0; }

// lines per CTA: 16 (2^4), 8 at the largest length (shared memory)
__host__ __device__ constexpr int fft_log2_lines(int log2L) { return log2L >= 10 ? 3 : 4; }

// Shared memory: W lines of L + 1 values (the pad keeps the W lines of a
// strided axis, stored column by column, in different banks), then L
// twiddles.
inline size_t fft_smem_total(int log2L)
{
    const size_t L = size_t(1) << log2L;
    return (size_t(1) << fft_log2_lines(log2L)) * (L + 1) * sizeof(float2) + L * sizeof(float2);
}

// One Stockham pass of radix R = 2^LOG2R over the W lines in `buf`, in
// place: every thread first reads its butterflies' R inputs (times the
// pass's twiddles) and does the R-point DFTs in registers, then, after a
// barrier, writes the outputs.  Ns = 2^log2Ns is the length of the
// sub-transforms already done.
template <bool INVERSE, int LOG2R, int LOG2L>
__device__ __forceinline__ void fft_pass(float2* buf, const float2* tws, int log2Ns)
{
    constexpr int R = 1 << LOG2R;
    constexpr int log2L = LOG2L;
    constexpr int log2W = fft_log2_lines(LOG2L);
    constexpr int log2per = LOG2L - LOG2R;          // butterflies per line
    constexpr int per = 1 << log2per;
    constexpr int work = 1 << (log2W + log2per);
    // butterflies one thread holds between the read and the write half
    constexpr int ITEMS = work >= kFftThreads ? work / kFftThreads : 1;
    const int sh = log2L - log2Ns - LOG2R;          // twiddle index unit
    const int ns_mask = (1 << log2Ns) - 1;
    float2 y[ITEMS][R];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int b = threadIdx.x + it * kFftThreads;
        if (b < work) {
            const int w = b >> log2per;
            const int j = b & (per - 1);
            const int jm = j & ns_mask;
            const float2* in = buf + w * (per << LOG2R | 1);
            float2 v[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float2 x = in[j + r * per];
                if (r > 0) {
                    const float2 t = tws[(jm * r) << sh];
                    if (INVERSE)   // x * conj(t)
                        x = make_float2(x.x * t.x + x.y * t.y, x.y * t.x - x.x * t.y);
                    else
                        x = make_float2(x.x * t.x - x.y * t.y, x.x * t.y + x.y * t.x);
                }
                v[r] = x;
            }
            if (R == 4) {
                const float2 a0 = make_float2(v[0].x + v[2].x, v[0].y + v[2].y);
                const float2 a1 = make_float2(v[0].x - v[2].x, v[0].y - v[2].y);
                const float2 a2 = make_float2(v[1].x + v[3 % R].x, v[1].y + v[3 % R].y);
                const float2 a3 = make_float2(v[1].x - v[3 % R].x, v[1].y - v[3 % R].y);
                // a3 times -i (forward) or +i (inverse)
                const float2 b3 = INVERSE ? make_float2(-a3.y, a3.x) : make_float2(a3.y, -a3.x);
                y[it][0] = make_float2(a0.x + a2.x, a0.y + a2.y);
                y[it][1 % R] = make_float2(a1.x + b3.x, a1.y + b3.y);
                y[it][2 % R] = make_float2(a0.x - a2.x, a0.y - a2.y);
                y[it][3 % R] = make_float2(a1.x - b3.x, a1.y - b3.y);
            } else {
                y[it][0] = make_float2(v[0].x + v[1 % R].x, v[0].y + v[1 % R].y);
                y[it][1 % R] = make_float2(v[0].x - v[1 % R].x, v[0].y - v[1 % R].y);
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int b = threadIdx.x + it * kFftThreads;
        if (b < work) {
            const int w = b >> log2per;
            const int j = b & (per - 1);
            float2* out = buf + w * (per << LOG2R | 1);
            const int base = ((j >> log2Ns) << (log2Ns + LOG2R)) + (j & ns_mask);
#pragma unroll
            for (int r = 0; r < R; ++r) out[base + (r << log2Ns)] = y[it][r];
        }
    }
    __syncthreads();
}

// The tile of a CTA: W lines of L values.  Element e of the tile is line
// w, position j: on a contiguous axis w = e / L, j = e % L (a warp reads 32
// consecutive values of one line); on a strided axis j = e / W, w = e % W (a
// warp reads the same position of W consecutive lines, which are adjacent
// in memory).
template <int LOG2L>
__device__ __forceinline__ void fft_tile_elem(bool contiguous, int e, int& w, int& j)
{
    constexpr int log2W = fft_log2_lines(LOG2L);
    if (contiguous) { w = e >> LOG2L; j = e & ((1 << LOG2L) - 1); }
    else { j = e >> log2W; w = e & ((1 << log2W) - 1); }
}

// Twiddles of length L in shared memory: tws[m] = e^{-2 pi i m / L}, m < L,
// from the per-device table of e^{-2 pi i k / 2^10}, k < 2^9 (the upper half
// of the circle is its negation).
template <int LOG2L>
__device__ __forceinline__ void fft_stage_twiddles(float2* tws, const float2* tw)
{
    constexpr int L = 1 << LOG2L;
    for (int m = threadIdx.x; m < L; m += kFftThreads) {
        const int h = m < (L >> 1) ? m : m - (L >> 1);
        float2 t = tw[h << (10 - LOG2L)];
        if (m >= (L >> 1)) t = make_float2(-t.x, -t.y);
        tws[m] = t;
    }
}

// Fill the tile: buf[w][j] = get(w, j) for every element, eight loads in
// flight per thread before their shared-memory stores.  get returns zero
// for lines past the end and for positions known to be zero.
template <int LOG2L, class Get>
__device__ __forceinline__ void fft_load_tile(float2* buf, bool contiguous, Get get)
{
    constexpr int total = (1 << fft_log2_lines(LOG2L)) << LOG2L;
    constexpr int stride = (1 << LOG2L) + 1;
    constexpr int U = 8;
    for (int e0 = threadIdx.x; e0 < total; e0 += U * kFftThreads) {
        float2 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * kFftThreads;
            int w, j;
            fft_tile_elem<LOG2L>(contiguous, e, w, j);
            v[u] = e < total ? get(w, j) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * kFftThreads;
            int w, j;
            fft_tile_elem<LOG2L>(contiguous, e, w, j);
            if (e < total) buf[w * stride + j] = v[u];
        }
    }
}

// Hand every element of the tile to put(w, j, value).
template <int LOG2L, class Put>
__device__ __forceinline__ void fft_store_tile(const float2* buf, bool contiguous, Put put)
{
    constexpr int total = (1 << fft_log2_lines(LOG2L)) << LOG2L;
    constexpr int stride = (1 << LOG2L) + 1;
    for (int e = threadIdx.x; e < total; e += kFftThreads) {
        int w, j;
        fft_tile_elem<LOG2L>(contiguous, e, w, j);
        put(w, j, buf[w * stride + j]);
    }
}

// The whole transform of the W lines in buf (natural order in and out).
template <bool INVERSE, int LOG2L>
__device__ __forceinline__ void fft_tile_passes(float2* buf, const float2* tws)
{
    int log2Ns = 0;
    if constexpr (LOG2L >= 2) {
#pragma unroll
        for (; LOG2L - log2Ns >= 2; log2Ns += 2) fft_pass<INVERSE, 2, LOG2L>(buf, tws, log2Ns);
    }
    if constexpr (LOG2L % 2 == 1) fft_pass<INVERSE, 1, LOG2L>(buf, tws, log2Ns);
}

// One axis of a 3-D FFT in place, `lines` lines of length L = 2^LOG2L at
// element stride inner = 2^log2inner: element j of line (o, i) is
// a[(o L + j) inner + i].
template <bool INVERSE, int LOG2L>
__global__ void __launch_bounds__(kFftThreads) fft_axis_kernel(float2* a, int log2inner,
                                                               int64_t lines, const float2* tw)
{
    extern __shared__ float2 fft_sm[];
    constexpr int log2W = fft_log2_lines(LOG2L);
    constexpr int stride = (1 << LOG2L) + 1;
    float2* const buf = fft_sm;
    float2* const tws = fft_sm + (stride << log2W);
    const int64_t group = int64_t(blockIdx.x) << log2W;
    const bool contiguous = log2inner == 0;
    const int64_t inner_mask = (int64_t(1) << log2inner) - 1;
    auto gidx = [&](int w, int j) -> int64_t {
        const int64_t line = group + w;
        const int64_t o = line >> log2inner;
        return (((o << LOG2L) + j) << log2inner) + (line & inner_mask);
    };
    fft_stage_twiddles<LOG2L>(tws, tw);
    fft_load_tile<LOG2L>(buf, contiguous, [&](int w, int j) {
        return group + w < lines ? a[gidx(w, j)] : make_float2(0.f, 0.f);
    });
    __syncthreads();
    fft_tile_passes<INVERSE, LOG2L>(buf, tws);
    fft_store_tile<LOG2L>(buf, contiguous, [&](int w, int j, float2 v) {
        if (group + w < lines) a[gidx(w, j)] = v;
    });
}

}  // namespace mri
