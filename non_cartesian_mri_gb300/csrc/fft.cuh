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
// auto-sorting FFT: one pass of radix 2^(log2 L mod 4) when that is not 0,
// then radix-16 passes, each thread reading R values of a line at stride
// L / R, multiplying by the twiddles of the pass and doing the R-point DFT
// in registers, then, after a barrier, writing them back in place where the
// final output ends up in natural order -- no bit reversal, one buffer, two
// passes at L = 256 (four CTAs per SM at that length).
// Twiddles e^{-2 pi i k / kFftMaxLen} come from a per-device table
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

// CTAs per SM the kernels are compiled for: five up to L = 256 (at most 51
// registers a thread; 5 x 37 KB of shared memory), else as registers allow.
__host__ __device__ constexpr int fft_min_ctas(int log2L) { return log2L <= 8 ? 5 : 1; }

// Shared-memory layout of a tile: value i of line w at fft_at(w, i) =
// w S + i + i / 16, S = L + L / 16 + 1.  The slot after every 16 values
// spreads a radix-16 pass's stores (16 consecutive values per thread) over
// the banks, and the extra slot per line does the same for the column
// accesses of a strided axis.  Then the L twiddles.
__host__ __device__ constexpr int fft_line_stride(int log2L)
{
    return (1 << log2L) + ((1 << log2L) >> 4) + 1;
}

__device__ __forceinline__ int fft_at(int S, int w, int i) { return w * S + i + (i >> 4); }

inline size_t fft_smem_total(int log2L)
{
    return (size_t(1) << fft_log2_lines(log2L)) * size_t(fft_line_stride(log2L)) * sizeof(float2) +
           (size_t(1) << log2L) * sizeof(float2);
}

// cos(2 pi m / 16), a chain of selects that folds to a constant for a
// constant m
__device__ __forceinline__ float fft_cos16(int m)
{
    constexpr float c1 = 0.923879532511286756f;   // cos(pi / 8)
    constexpr float s1 = 0.382683432365089772f;   // sin(pi / 8)
    constexpr float h = 0.707106781186547524f;    // cos(pi / 4)
    m &= 15;
    const int q = m > 8 ? 16 - m : m;             // cos is even
    return q == 0 ? 1.f : q == 1 ? c1 : q == 2 ? h : q == 3 ? s1 : q == 4 ? 0.f
         : q == 5 ? -s1 : q == 6 ? -h : q == 7 ? -c1 : -1.f;
}

// e^{-2 pi i m / 16} (conjugated for the inverse): the roots inside one
// radix-16 butterfly.  m is a constant once the caller's loops are unrolled.
template <bool INVERSE>
__device__ __forceinline__ float2 fft_mul_root16(float2 x, int m)
{
    if (m == 0) return x;
    if (m == 8) return make_float2(-x.x, -x.y);
    const bool fwd = !INVERSE;
    if (m == 4) return fwd ? make_float2(x.y, -x.x) : make_float2(-x.y, x.x);     // -+i
    if (m == 12) return fwd ? make_float2(-x.y, x.x) : make_float2(x.y, -x.x);    // +-i
    const float c = fft_cos16(m), sn = fft_cos16(m + 12);   // sin = cos(. - pi / 2)
    const float si = fwd ? -sn : sn;
    return make_float2(x.x * c - x.y * si, x.x * si + x.y * c);
}

__host__ __device__ constexpr int fft_bitrev(int i, int bits)
{
    int r = 0;
    for (int b = 0; b < bits; ++b) r |= ((i >> b) & 1) << (bits - 1 - b);
    return r;
}

// Stage LS of a radix-2 decimation-in-frequency DFT of 2^LOG2R values in
// registers (butterflies at span 2^LS), then the stages below it.
// ZERO_UPPER: the upper half of v is zero on entry (only the first stage,
// whose butterflies pair v[k] with v[k + R / 2], sees that).
template <bool INVERSE, int LOG2R, int LS, bool ZERO_UPPER>
__device__ __forceinline__ void fft_dif_stage(float2 (&v)[1 << LOG2R])
{
    constexpr int span = 1 << LS;
#pragma unroll
    for (int q = 0; q < (1 << LOG2R) / 2; ++q) {
        const int lo = ((q >> LS) << (LS + 1)) + (q & (span - 1));
        const int m = ((q & (span - 1)) * 8) >> LS;
        const float2 a = v[lo], b = v[lo + span];
        // times e^{-+2 pi i k / (2 span)}, k = q mod span: root16^(8 k / span)
        if (ZERO_UPPER) {
            v[lo + span] = fft_mul_root16<INVERSE>(a, m);
        } else {
            v[lo] = make_float2(a.x + b.x, a.y + b.y);
            v[lo + span] = fft_mul_root16<INVERSE>(make_float2(a.x - b.x, a.y - b.y), m);
        }
    }
    if constexpr (LS > 0) fft_dif_stage<INVERSE, LOG2R, LS - 1, false>(v);
}

// In-register DFT of R = 2^LOG2R values (R <= 16), natural order in and
// out: radix-2 decimation in frequency, whose bit-reversed output order is
// undone by renaming registers.
template <bool INVERSE, int LOG2R, bool ZERO_UPPER>
__device__ __forceinline__ void fft_dft_regs(float2 (&v)[1 << LOG2R])
{
    constexpr int R = 1 << LOG2R;
    if constexpr (LOG2R > 0) fft_dif_stage<INVERSE, LOG2R, LOG2R - 1, ZERO_UPPER>(v);
    float2 t[R];
#pragma unroll
    for (int i = 0; i < R; ++i) t[fft_bitrev(i, LOG2R)] = v[i];
#pragma unroll
    for (int i = 0; i < R; ++i) v[i] = t[i];
}

// One Stockham pass of radix R = 2^LOG2R over the W lines in `buf`, in
// place, Ns = 2^LOG2NS the length of the sub-transforms already done:
// butterfly j (< L / R) of a line takes the R values j + r L / R, times
// e^{-+2 pi i (j mod Ns) r / (Ns R)}, does their R-point DFT and stores
// output r at (j / Ns) Ns R + (j mod Ns) + r Ns.  Every thread first reads
// its butterflies into registers and transforms them, then, after a
// barrier, writes them back.  HALF_IN (first pass only): the values at
// positions >= L / 2 are zero and are not read.  HALF_OUT (last pass only):
// only the outputs at positions < L / 2 are written.
template <bool INVERSE, int LOG2R, int LOG2L, int LOG2NS, bool HALF_IN, bool HALF_OUT>
__device__ __forceinline__ void fft_pass(float2* buf, const float2* tws)
{
    static_assert(!HALF_IN || LOG2NS == 0, "zero inputs are known in the first pass only");
    static_assert(!HALF_OUT || LOG2NS + LOG2R == LOG2L, "a half is dropped in the last pass only");
    constexpr int R = 1 << LOG2R;
    constexpr int log2W = fft_log2_lines(LOG2L);
    constexpr int S = fft_line_stride(LOG2L);
    constexpr int log2per = LOG2L - LOG2R;          // butterflies per line
    constexpr int per = 1 << log2per;
    constexpr int work = 1 << (log2W + log2per);
    // butterflies one thread holds between the read and the write half
    constexpr int ITEMS = work >= kFftThreads ? work / kFftThreads : 1;
    constexpr int sh = LOG2L - LOG2NS - LOG2R;      // twiddle index unit
    constexpr int ns_mask = (1 << LOG2NS) - 1;
    float2 y[ITEMS][R];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int b = threadIdx.x + it * kFftThreads;
        if (b < work) {
            const int w = b >> log2per;
            const int j = b & (per - 1);
            const int jm = j & ns_mask;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (HALF_IN && r >= R / 2) {   // position j + r L / R >= L / 2
                    y[it][r] = make_float2(0.f, 0.f);
                    continue;
                }
                float2 x = buf[fft_at(S, w, j + r * per)];
                if (LOG2NS > 0 && r > 0) {
                    const float2 t = tws[(jm * r) << sh];
                    if (INVERSE)   // x * conj(t)
                        x = make_float2(x.x * t.x + x.y * t.y, x.y * t.x - x.x * t.y);
                    else
                        x = make_float2(x.x * t.x - x.y * t.y, x.x * t.y + x.y * t.x);
                }
                y[it][r] = x;
            }
            fft_dft_regs<INVERSE, LOG2R, HALF_IN>(y[it]);
        }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
        const int b = threadIdx.x + it * kFftThreads;
        if (b < work) {
            const int w = b >> log2per;
            const int j = b & (per - 1);
            const int base = ((j >> LOG2NS) << (LOG2NS + LOG2R)) + (j & ns_mask);
#pragma unroll
            for (int r = 0; r < (HALF_OUT ? R / 2 : R); ++r)
                buf[fft_at(S, w, base + (r << LOG2NS))] = y[it][r];
        }
    }
    __syncthreads();
}

// The passes from sub-transform length 2^LOG2NS up: first the odd part
// (radix 2^(log2 L mod 4)), then radix-16 passes.
template <bool INVERSE, int LOG2L, int LOG2NS, bool HALF_IN, bool HALF_OUT>
__device__ __forceinline__ void fft_passes_from(float2* buf, const float2* tws)
{
    if constexpr (LOG2NS < LOG2L) {
        constexpr int LOG2R = (LOG2NS == 0 && LOG2L % 4 != 0) ? LOG2L % 4 : 4;
        constexpr bool last = LOG2NS + LOG2R == LOG2L;
        fft_pass<INVERSE, LOG2R, LOG2L, LOG2NS, HALF_IN && LOG2NS == 0, HALF_OUT && last>(buf,
                                                                                           tws);
        fft_passes_from<INVERSE, LOG2L, LOG2NS + LOG2R, HALF_IN, HALF_OUT>(buf, tws);
    }
}

// The tile of a CTA: W lines of L values.  Element e of the tile is line
// w, position j: on a contiguous axis w = e / L, j = e % L (a warp reads 32
// consecutive values of one line); on a strided axis j = e / W, w = e % W (a
// warp reads the same position of W consecutive lines, which are adjacent
// in memory).
template <int LOG2L, bool HALF = false>
__device__ __forceinline__ void fft_tile_elem(bool contiguous, int e, int& w, int& j)
{
    constexpr int log2W = fft_log2_lines(LOG2L);
    constexpr int log2row = HALF ? LOG2L - 1 : LOG2L;   // values per line visited
    if (contiguous) { w = e >> log2row; j = e & ((1 << log2row) - 1); }
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

// Fill the tile: buf[w][j] = get(w, j) for every element (HALF: for the
// lower half of every line only), eight loads in flight per thread before
// their shared-memory stores.  get returns zero for lines past the end and
// for positions known to be zero.
template <int LOG2L, bool HALF = false, class Get>
__device__ __forceinline__ void fft_load_tile(float2* buf, bool contiguous, Get get)
{
    constexpr int total = (1 << fft_log2_lines(LOG2L)) << (HALF ? LOG2L - 1 : LOG2L);
    constexpr int S = fft_line_stride(LOG2L);
    constexpr int U = 8;
    for (int e0 = threadIdx.x; e0 < total; e0 += U * kFftThreads) {
        float2 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * kFftThreads;
            int w, j;
            fft_tile_elem<LOG2L, HALF>(contiguous, e, w, j);
            v[u] = e < total ? get(w, j) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * kFftThreads;
            int w, j;
            fft_tile_elem<LOG2L, HALF>(contiguous, e, w, j);
            if (e < total) buf[fft_at(S, w, j)] = v[u];
        }
    }
}

// Hand every element of the tile (HALF: of the lower half of every line)
// to put(w, j, value).
template <int LOG2L, bool HALF = false, class Put>
__device__ __forceinline__ void fft_store_tile(const float2* buf, bool contiguous, Put put)
{
    constexpr int total = (1 << fft_log2_lines(LOG2L)) << (HALF ? LOG2L - 1 : LOG2L);
    constexpr int S = fft_line_stride(LOG2L);
    for (int e = threadIdx.x; e < total; e += kFftThreads) {
        int w, j;
        fft_tile_elem<LOG2L, HALF>(contiguous, e, w, j);
        put(w, j, buf[fft_at(S, w, j)]);
    }
}

// The whole transform of the W lines in buf (natural order in and out).
// HALF_IN: the upper half of every line is zero (and need not be in buf);
// HALF_OUT: only the lower half of the result is wanted.
template <bool INVERSE, int LOG2L, bool HALF_IN = false, bool HALF_OUT = false>
__device__ __forceinline__ void fft_tile_passes(float2* buf, const float2* tws)
{
    fft_passes_from<INVERSE, LOG2L, 0, HALF_IN, HALF_OUT>(buf, tws);
}

// One axis of a 3-D FFT in place, `lines` lines of length L = 2^LOG2L at
// element stride inner = 2^log2inner: element j of line (o, i) is
// a[(o L + j) inner + i].
template <bool INVERSE, int LOG2L>
__global__ void __launch_bounds__(kFftThreads, fft_min_ctas(LOG2L)) fft_axis_kernel(float2* a, int log2inner,
                                                               int64_t lines, const float2* tw)
{
    extern __shared__ float2 fft_sm[];
    constexpr int log2W = fft_log2_lines(LOG2L);
    float2* const buf = fft_sm;
    float2* const tws = fft_sm + (fft_line_stride(LOG2L) << log2W);
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
