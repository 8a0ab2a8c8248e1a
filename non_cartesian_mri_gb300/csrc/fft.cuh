// fft.cuh -- complex FFTs along one axis of a 3-D array, for the Toeplitz
// product F^H F of the "find rho" step (the chapter's background section:
// F^H F is Toeplitz, so its product with rho goes through FFTs).
//
// Layout: float2 (re, im) interleaved, x fastest; an axis of length L (a
// power of two, 2 .. kFftMaxLen) sits between `outer` slabs and `inner`
// consecutive elements: element j of line (o, i) is a[(o L + j) inner + i].
// A CTA transforms W lines (16, or 8 for L = 1024): W consecutive i when
// inner > 1 (so that a warp's accesses at one position of its lines are
// contiguous), W consecutive o when inner == 1 (each line contiguous).  The
// transform is a Stockham auto-sorting FFT (natural order in and out, no bit
// reversal): one pass of radix 2^(log2 L mod 4) when that is not 0 and
// radix-16 passes, each thread doing the R-point DFTs of its butterflies in
// registers.  The first pass reads its inputs straight from global memory
// into registers and the last pass hands its outputs over in registers;
// shared memory only carries the values from one pass to the next (one
// exchange at L = 256), so a kernel can fuse the work on either side of a
// transform, or keep the result of one transform in registers as the input
// of the next (the z stage of the Toeplitz product: forward transform,
// product with the spectrum, inverse transform).  Twiddles
// e^{-2 pi i k / kFftMaxLen} come from a per-device table evaluated in double
// precision (the twiddle kernel of kernels_toeplitz.cu) and are staged for
// the line length in shared memory; the inverse transform conjugates them
// where it uses them and does not scale (the caller divides by the size).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mri {

constexpr int kFftMaxLen = 1024;              // 2^10
constexpr int kFftThreads = 256;

inline bool fft_len_ok(int64_t L) { return L >= 1 && L <= kFftMaxLen && (L & (L - 1)) == 0; }

// Programmatic dependent launch: kernels that run back to back on one
// stream, each short (the FFT passes, the Toeplitz stages, the CG kernels),
// are launched with the programmatic-serialisation attribute.  Each one lets
// the next one launch as soon as all of its CTAs have started
// (pdl_launch_dependents), and each one waits for the previous one to
// finish, with its writes visible (pdl_wait), before it touches any buffer;
// what comes before the wait (twiddle staging, index set-up) reads nothing
// the previous kernel writes.  Launched without the attribute, both are
// no-ops.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// lines per CTA: 16 (2^4), 8 at the largest length (shared memory)
__host__ __device__ constexpr int fft_log2_lines(int log2L) { return log2L >= 10 ? 3 : 4; }

// CTAs per SM the kernels are compiled for: four up to L = 256 (at most 64
// registers a thread: a radix-16 butterfly and, in the z stage of the
// Toeplitz product, the 16 spectrum values loaded ahead), else as registers
// allow.
__host__ __device__ constexpr int fft_min_ctas(int log2L) { return log2L <= 8 ? 4 : 1; }

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

// ---- passes
//
// A plan is the sequence of radices of the passes: the odd part
// 2^(log2 L mod 4) first (ODD_FIRST) or last, radix 16 otherwise.  Pass k
// with radix R = 2^r and Ns = the product of the radices before it (the
// length of the sub-transforms done) has L / R butterflies per line;
// butterfly j takes the values at positions j + q L / R, q < R, times
// e^{-+2 pi i (j mod Ns) q / (Ns R)}, does their R-point DFT and puts output
// q at (j / Ns) Ns R + (j mod Ns) + q Ns (Stockham: the result of the last
// pass is in natural order, at j + q L / R).
template <int LOG2L, bool ODD_FIRST>
struct FftPlan {
    static constexpr int odd = LOG2L % 4;
    static constexpr int passes = LOG2L / 4 + (odd != 0 ? 1 : 0);
    __host__ __device__ static constexpr int log2r(int k)
    {
        if (odd == 0) return 4;
        return ODD_FIRST ? (k == 0 ? odd : 4) : (k == passes - 1 ? odd : 4);
    }
    __host__ __device__ static constexpr int log2ns(int k)
    {
        int s = 0;
        for (int i = 0; i < k; ++i) s += log2r(i);
        return s;
    }
};

// butterflies of a pass of radix 2^LOG2R one thread holds
__host__ __device__ constexpr int fft_items(int log2L, int log2r)
{
    return (1 << (fft_log2_lines(log2L) + log2L - log2r)) >= kFftThreads
               ? (1 << (fft_log2_lines(log2L) + log2L - log2r)) / kFftThreads
               : 1;
}

// Butterfly `it` of this thread in a pass of radix 2^LOG2R: line w, index j
// (< L / R).  WFAST: consecutive lanes take consecutive lines (a strided
// axis, whose W lines of a CTA are adjacent in memory: a warp's global
// accesses at one position are contiguous); otherwise consecutive lanes take
// consecutive j of one line (a contiguous axis).  Returns false for a
// thread without that butterfly.
template <int LOG2L, int LOG2R, bool WFAST>
__device__ __forceinline__ bool fft_item(int it, int& w, int& j)
{
    constexpr int log2W = fft_log2_lines(LOG2L);
    constexpr int log2per = LOG2L - LOG2R;
    const int b = threadIdx.x + it * kFftThreads;
    if (WFAST) { w = b & ((1 << log2W) - 1); j = b >> log2W; }
    else { w = b >> log2per; j = b & ((1 << log2per) - 1); }
    return b < (1 << (log2W + log2per));
}

// the pass twiddles of butterfly j, times its inputs 1 .. R - 1
template <bool INVERSE, int LOG2L, int LOG2R, int LOG2NS>
__device__ __forceinline__ void fft_twiddle(float2 (&v)[1 << LOG2R], int j, const float2* tws)
{
    if constexpr (LOG2NS > 0) {
        constexpr int sh = LOG2L - LOG2NS - LOG2R;     // twiddle index unit
        const int jm = j & ((1 << LOG2NS) - 1);
#pragma unroll
        for (int q = 1; q < (1 << LOG2R); ++q) {
            const float2 t = tws[(jm * q) << sh];
            const float2 x = v[q];
            v[q] = INVERSE ? make_float2(x.x * t.x + x.y * t.y, x.y * t.x - x.x * t.y)   // x conj(t)
                           : make_float2(x.x * t.x - x.y * t.y, x.x * t.y + x.y * t.x);
        }
    }
}

// Between pass A and pass B: A's outputs (ya) to shared memory, then B's
// inputs (yb) from it, times B's twiddles, and B's DFTs.  The barrier in
// front keeps the writes behind every read of the previous exchange.
template <bool INVERSE, int LOG2L, int LOG2RA, int LOG2NSA, int LOG2RB, bool WFAST, int IA, int IB>
__device__ __forceinline__ void fft_exchange(float2* buf, const float2* tws,
                                             const float2 (&ya)[IA][1 << LOG2RA],
                                             float2 (&yb)[IB][1 << LOG2RB])
{
    constexpr int S = fft_line_stride(LOG2L);
    constexpr int nsa_mask = (1 << LOG2NSA) - 1;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < IA; ++it) {
        int w, j;
        if (fft_item<LOG2L, LOG2RA, WFAST>(it, w, j)) {
            const int base = ((j >> LOG2NSA) << (LOG2NSA + LOG2RA)) + (j & nsa_mask);
#pragma unroll
            for (int q = 0; q < (1 << LOG2RA); ++q)
                buf[fft_at(S, w, base + (q << LOG2NSA))] = ya[it][q];
        }
    }
    __syncthreads();
    constexpr int perb = 1 << (LOG2L - LOG2RB);
#pragma unroll
    for (int it = 0; it < IB; ++it) {
        int w, j;
        if (fft_item<LOG2L, LOG2RB, WFAST>(it, w, j)) {
#pragma unroll
            for (int q = 0; q < (1 << LOG2RB); ++q) yb[it][q] = buf[fft_at(S, w, j + q * perb)];
            fft_twiddle<INVERSE, LOG2L, LOG2RB, LOG2NSA + LOG2RA>(yb[it], j, tws);
            fft_dft_regs<INVERSE, LOG2RB, false>(yb[it]);
        }
    }
}

// The passes after pass K, whose outputs are in y; then fin(y) with the last
// pass's outputs: butterfly (w, j) of fft_item, output q at position
// j + q L / R_last.
template <bool INVERSE, int LOG2L, bool ODD_FIRST, bool WFAST, int K, int I, int R, class Fin>
__device__ __forceinline__ void fft_run_from(float2* buf, const float2* tws, float2 (&y)[I][R],
                                             Fin&& fin)
{
    using P = FftPlan<LOG2L, ODD_FIRST>;
    if constexpr (K + 1 == P::passes) {
        fin(y);
    } else {
        constexpr int RB = P::log2r(K + 1);
        constexpr int IB = fft_items(LOG2L, RB);
        float2 z[IB][1 << RB];
        fft_exchange<INVERSE, LOG2L, P::log2r(K), P::log2ns(K), RB, WFAST>(buf, tws, y, z);
        fft_run_from<INVERSE, LOG2L, ODD_FIRST, WFAST, K + 1>(buf, tws, z, fin);
    }
}

struct FftNoKeep {
    __device__ __forceinline__ void operator()(int, int, float2) const {}
};

// The transform of the CTA's W lines: the first pass takes its inputs from
// load(w, position) straight into registers (HALF_IN: the positions >= L / 2
// are zero and not loaded, and the first DFT stage skips them), shared
// memory carries the values between passes only, and fin gets the last
// pass's outputs in registers (see fft_run_from).  Lines past the end are
// the loader's, keep's and fin's to skip.  The first pass has Ns = 1: no
// twiddles.  keep(w, position, value) sees every loaded value once all the
// loads are issued: a store it makes (the CG direction written back) holds
// back no load, which a store inside load would (the compiler cannot tell
// the arrays apart).
template <bool INVERSE, int LOG2L, bool ODD_FIRST, bool WFAST, bool HALF_IN, class Load, class Fin,
          class Keep>
__device__ __forceinline__ void fft_lines(float2* buf, const float2* tws, Load&& load, Fin&& fin,
                                          Keep&& keep)
{
    using P = FftPlan<LOG2L, ODD_FIRST>;
    constexpr int R0 = P::log2r(0);
    constexpr int I0 = fft_items(LOG2L, R0);
    constexpr int per0 = 1 << (LOG2L - R0);
    float2 y[I0][1 << R0];
    // every load of the thread in flight before the first use
#pragma unroll
    for (int it = 0; it < I0; ++it) {
        int w, j;
        const bool on = fft_item<LOG2L, R0, WFAST>(it, w, j);
#pragma unroll
        for (int q = 0; q < (1 << R0); ++q)
            y[it][q] = (on && !(HALF_IN && q >= (1 << R0) / 2)) ? load(w, j + q * per0)
                                                                 : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int it = 0; it < I0; ++it) {
        int w, j;
        if (!fft_item<LOG2L, R0, WFAST>(it, w, j)) continue;
#pragma unroll
        for (int q = 0; q < (HALF_IN ? (1 << R0) / 2 : (1 << R0)); ++q)
            keep(w, j + q * per0, y[it][q]);
    }
#pragma unroll
    for (int it = 0; it < I0; ++it) fft_dft_regs<INVERSE, R0, HALF_IN>(y[it]);
    fft_run_from<INVERSE, LOG2L, ODD_FIRST, WFAST, 0>(buf, tws, y, fin);
}

template <bool INVERSE, int LOG2L, bool ODD_FIRST, bool WFAST, bool HALF_IN, class Load, class Fin>
__device__ __forceinline__ void fft_lines(float2* buf, const float2* tws, Load&& load, Fin&& fin)
{
    fft_lines<INVERSE, LOG2L, ODD_FIRST, WFAST, HALF_IN>(buf, tws, load, fin, FftNoKeep{});
}

// The last pass of a plan: its log2 radix, and the stride of its outputs
// (output q of butterfly j sits at position j + q * fft_last_per).
template <int LOG2L, bool ODD_FIRST>
__host__ __device__ constexpr int fft_last_log2r()
{
    return FftPlan<LOG2L, ODD_FIRST>::log2r(FftPlan<LOG2L, ODD_FIRST>::passes - 1);
}

template <int LOG2L, bool ODD_FIRST>
__host__ __device__ constexpr int fft_last_per()
{
    return 1 << (LOG2L - fft_last_log2r<LOG2L, ODD_FIRST>());
}

// Twiddles of length L in shared memory: tws[m] = e^{-2 pi i m / L}, m < L,
// from the per-device table of e^{-2 pi i k / 2^10}, k < 2^9 (the upper half
// of the circle is its negation).  The first exchange's barrier makes them
// visible before any pass uses them.
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

// One axis of a 3-D FFT in place, `lines` lines of length L = 2^LOG2L at
// element stride inner = 2^log2inner (CONTIG: inner = 1): element j of line
// (o, i) is a[(o L + j) inner + i].
template <bool INVERSE, int LOG2L, bool CONTIG>
__global__ void __launch_bounds__(kFftThreads, fft_min_ctas(LOG2L))
    fft_axis_kernel(float2* a, int log2inner, int64_t lines, const float2* tw)
{
    extern __shared__ float2 fft_sm[];
    constexpr int log2W = fft_log2_lines(LOG2L);
    float2* const buf = fft_sm;
    float2* const tws = fft_sm + (fft_line_stride(LOG2L) << log2W);
    const int64_t group = int64_t(blockIdx.x) << log2W;
    const int64_t inner_mask = (int64_t(1) << log2inner) - 1;
    auto gidx = [&](int w, int j) -> int64_t {
        const int64_t line = group + w;
        if (CONTIG) return (line << LOG2L) + j;
        return ((((line >> log2inner) << LOG2L) + j) << log2inner) + (line & inner_mask);
    };
    pdl_launch_dependents();
    fft_stage_twiddles<LOG2L>(tws, tw);
    pdl_wait();
    constexpr int RL = fft_last_log2r<LOG2L, true>();
    constexpr int last_per = fft_last_per<LOG2L, true>();
    fft_lines<INVERSE, LOG2L, true, !CONTIG, false>(
        buf, tws,
        [&](int w, int pos) { return group + w < lines ? a[gidx(w, pos)] : make_float2(0.f, 0.f); },
        [&](auto& y) {
#pragma unroll
            for (int it = 0; it < fft_items(LOG2L, RL); ++it) {
                int w, j;
                if (fft_item<LOG2L, RL, !CONTIG>(it, w, j) && group + w < lines) {
#pragma unroll
                    for (int q = 0; q < (1 << RL); ++q) a[gidx(w, j + q * last_per)] = y[it][q];
                }
            }
        });
}

}  // namespace mri
