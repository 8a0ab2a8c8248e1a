// fft.cuh -- complex FFTs along one axis of a 3-D array, for the Toeplitz
// product F^H F of the "find rho" step (the chapter's background section:
// F^H F is Toeplitz, so its product with rho goes through FFTs).
//
// Layout: float2 (re, im) interleaved, x fastest; an axis of length L (a
// power of two, 2 .. kFftMaxLen) sits between `outer` slabs and `inner`
// consecutive elements: element j of line (o, i) is a[(o L + j) inner + i].
// A CTA transforms kFftLines lines: kFftLines consecutive i (inner > 1, so
// that a warp's loads cover consecutive addresses) or kFftLines consecutive
// o (inner == 1, each line contiguous).  The lines go to shared memory in
// bit-reversed order; log2 L radix-2 butterfly stages run in place, one CTA
// barrier per stage; the result is stored back in natural order.  Twiddles
// e^{-2 pi i k / kFftMaxLen} come from a per-device table evaluated in double
// precision (the twiddle kernel of kernels_toeplitz.cu); the inverse
// transform conjugates them and does not scale (the caller divides by the
// size).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace mri {

constexpr int kFftMaxLen = 1024;
constexpr int kFftLines = 16;                   // lines per CTA
constexpr int kFftThreads = 256;

inline bool fft_len_ok(int64_t L) { return L >= 1 && L <= kFftMaxLen && (L & (L - 1)) == 0; }

inline size_t fft_smem_bytes(int L) { return size_t(kFftLines) * (L + 1) * sizeof(float2); }

__device__ __forceinline__ unsigned int bit_reverse(unsigned int j, int bits)
{
    return __brev(j) >> (32 - bits);
}

template <bool INVERSE>
__global__ void __launch_bounds__(kFftThreads) fft_axis_kernel(float2* a, int L, int log2L,
                                                               int64_t outer, int64_t inner,
                                                               const float2* tw)
{
    extern __shared__ float2 fft_sm[];
    const int stride = L + 1;                         // one pad element per line
    const int64_t lines = outer * inner;
    const int64_t group = int64_t(blockIdx.x) * kFftLines;
    const bool contiguous = inner == 1;
    // global index of element j of this CTA's line w
    auto gidx = [&](int w, int j) -> int64_t {
        if (contiguous) return (group + w) * L + j;
        const int64_t line = group + w;               // line = o * inner + i
        const int64_t o = line / inner;
        const int64_t i = line - o * inner;
        return (o * L + j) * inner + i;
    };
    const int total = kFftLines * L;
    for (int e = threadIdx.x; e < total; e += kFftThreads) {
        int w, j;
        if (contiguous) { w = e / L; j = e - w * L; }
        else { j = e / kFftLines; w = e - j * kFftLines; }
        if (group + w < lines)
            fft_sm[w * stride + bit_reverse(unsigned(j), log2L)] = a[gidx(w, j)];
    }
    __syncthreads();
    const int half_total = kFftLines * (L >> 1);
    for (int s = 1; s <= log2L; ++s) {
        const int half = 1 << (s - 1);
        const int tw_step = kFftMaxLen >> s;          // e^{-2 pi i pos / 2 half}
        for (int b = threadIdx.x; b < half_total; b += kFftThreads) {
            const int w = b / (L >> 1);
            const int bb = b - w * (L >> 1);
            const int pos = bb & (half - 1);
            const int i0 = ((bb >> (s - 1)) << s) + pos;
            float2* line = fft_sm + w * stride;
            float2 t = tw[pos * tw_step];
            if (INVERSE) t.y = -t.y;
            const float2 u = line[i0];
            const float2 v0 = line[i0 + half];
            const float2 v = make_float2(v0.x * t.x - v0.y * t.y, v0.x * t.y + v0.y * t.x);
            line[i0] = make_float2(u.x + v.x, u.y + v.y);
            line[i0 + half] = make_float2(u.x - v.x, u.y - v.y);
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < total; e += kFftThreads) {
        int w, j;
        if (contiguous) { w = e / L; j = e - w * L; }
        else { j = e / kFftLines; w = e - j * kFftLines; }
        if (group + w < lines) a[gidx(w, j)] = fft_sm[w * stride + j];
    }
}

}  // namespace mri
