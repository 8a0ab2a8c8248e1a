// gather_grid_tc.cuh -- shared pieces of separable-grid F^H D / Q on the
// tensor cores: shapes, operand layouts, the per-call operand tables and the
// per-element helpers.  The kernel is gather_grid_tc_ws_kernel
// (gather_grid_tc_ws.cuh).
//
// On a grid the gather of Fig. 17.11 factors (gather_grid.cuh) into
//   FhD[row][ix] = sum_m Mz[row][m] * Ex[m][ix],
//   Mz = Mu * e^{i2pi(ky y + kz z)},  Ex = e^{i2pi kx x},
// a complex matrix product over the samples: a dense contraction.  A CTA
// owns 128 MMA rows (grid rows, or coils x grid rows) and one block of 128
// columns (the last block of an nx that is not a multiple of 128 is padded
// with zero columns, which are computed and not stored).  Per tile of 32
// samples the B operand (32 samples x 128 columns) is the same for every CTA
// of a column block: build_ex_tiles_kernel evaluates it once per call into a
// table of operand tiles in the tensor core's shared-memory layout, fetched
// with one TMA bulk copy per tile.  The A operand (128 rows x 32 samples) is
// evaluated by the CTA into tensor memory.  Every value is split into an f16
// high part and the f16-rounded remainder, and per K step (two per tile) two
// N = 256 products go into [D_r | D_i]:
//   [D_r | D_i] += A_r [B_r | B_i]  +  A_i [-B_i | B_r],
// reading B as two 256-row windows of one 384-row block S = [-B_i; B_r; B_i],
// with each real product done as hi*hi + hi*lo + lo*hi (12 tcgen05.mma of
// 128 x 256 x 16 per tile).  The two f16 parts carry about 22 significant
// bits, and the dropped lo*lo term is below 2^-22 of a product, so every
// product keeps close to fp32 accuracy.  f16 has a narrow exponent range: the
// weights are multiplied (once per call, in the records) by a power of two
// chosen from the largest |w_r| + |w_i| of the call so that every weighted
// operand is below 2^15, and the results are multiplied back exactly; the
// phase factors (|e^{i phi}| = 1) need no scale.  In a coil group every coil
// has its own bound and power of two, so a coil far smaller than the others
// keeps the full precision of its f16 parts.
//
// Where the weight goes.  With one coil per CTA (F^H D, Q) the weight Mu is
// folded into the B table (B = Mu e^{i2pi kx x}, once per call), and A is the
// bare row factor e^{i2pi(ky y + kz z)}: per (row, sample) element the CTA
// evaluates one sin/cos pair and splits it, with no weight loads and no
// complex multiply.  With a coil group (batched F^H D) B is shared by the
// group's coils, so A = Mu_coil e^{i2pi(ky y + kz z)}.
//
// Tensor memory: D (columns 0-255) collects one block of tiles and is then
// added into running sums held in registers (each generating thread owns 128
// of the 128 x 256 sums: its warp's lane quarter and half of the columns),
// the blocked summation that keeps accumulation error below the trig error
// over a million samples; columns 256.. hold the A stages (64 columns each).
// B tiles are K-major without swizzle: core matrices of 8 rows x 8 f16
// (128 B), LBO = 128 B along K, SBO = 512 B between 8-row groups.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid.cuh"

namespace mri {

constexpr int kTcTile = 32;                          // samples per tile (two K = 16 steps)
constexpr int kTcRows = 128;                         // grid rows per CTA = MMA M
constexpr int kTcCols = 128;                         // grid columns per CTA = MMA N / 2
constexpr int kTcThreads = 256;                      // threads generating A
constexpr int kTcWarps = kTcThreads / 32;
#ifndef MRI_TC_STAGES
#define MRI_TC_STAGES 4
#endif
// Tiles per summation block.  The tensor core's own fp32 accumulation loses
// a little with every add, with a consistent sign, so the error of a block
// grows with its length (accurate F^H D on the 128^3 radial workload, rel-L2
// against the oracle: 1.0e-6 for blocks of 128 samples, 1.9e-6 for 256,
// 4.0e-6 for 512; 1.4e-5 for 1024), while every fold stalls the tensor core
// (accurate F^H D: 65.5, 74.6, 77.9 Tpairs/s for 128, 256, 512).  The
// accurate path folds every 256 samples, the fast paths (trig error ~1e-5)
// every 1024.
#ifndef MRI_TC_DRAIN_ACCURATE
#define MRI_TC_DRAIN_ACCURATE 8
#endif
#ifndef MRI_TC_DRAIN_FAST
#define MRI_TC_DRAIN_FAST 32
#endif
constexpr int kTcDrainAccurate = MRI_TC_DRAIN_ACCURATE;
constexpr int kTcDrainFast = MRI_TC_DRAIN_FAST;
constexpr int kTcPartBytes = kTcRows * kTcTile * 2;  // 128 S rows x 32 f16 (8 KB)
constexpr int kTcSBytes = 3 * kTcPartBytes;          // S = [-B_i; B_r; B_i]: 384 x 32 (24 KB)
constexpr int kTcStageBytes = 2 * kTcSBytes;         // S hi, S lo (48 KB)
constexpr int kTcStages = MRI_TC_STAGES;             // operand stages in the ring
constexpr int kTcColsPerWarp = 256 * 4 / kTcWarps;  // D columns one warp folds (128)
constexpr uint32_t kTcDCols = 256;                   // D_r | D_i
constexpr uint32_t kTcAPartCols = kTcTile / 2;       // one A part: 32 f16 per lane (16 columns)
constexpr uint32_t kTcAStageCols = 4 * kTcAPartCols; // A r/i hi/lo (64 columns)
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcAExp = 15;                          // |A| * scale < 2^kTcAExp
constexpr int kTcAChunks = kTcTile / 8 / (kTcWarps / 4);   // 8-sample A chunks per thread
static_assert(kTcStages >= 1 && kTcDCols + kTcStages * kTcAStageCols <= kTcTmemCols,
              "A stages fit tensor memory");

// A parts (tensor-memory column offset / kTcAPartCols within a stage)
enum TcPart { A_RH = 0, A_RL, A_IH, A_IL };
constexpr int kTcSHi = 0;
constexpr int kTcSLo = kTcSBytes;

// Any nx >= 8 runs in column blocks of 128, the last one padded with zero
// columns.  The MMA work is that of the padded width, so the rate in
// voxel-sample pairs is nx / (128 ceil(nx / 128)) of the full one: at nx = 8
// still about twice the general kernel's; narrower grids take the general
// kernel on expanded coordinates.
constexpr int kTcMinCols = 8;
inline bool grid_tc_fits(int nx) { return nx >= kTcMinCols; }
inline int grid_tc_col_blocks(int nx) { return (nx + kTcCols - 1) / kTcCols; }

// Shape of the forward-model kernel (gather_grid_tc_fwd.cuh), which takes the
// same nx.
constexpr int kFwSamples = 128;                 // samples per CTA = MMA M
constexpr int kFwRows = 64;                     // grid rows per block = MMA N / 2
constexpr int kFwCols = 128;                    // grid columns per block = K
constexpr int kFwKSteps = kFwCols / 16;         // 8 K steps of 16 per column block
constexpr int kFwKPerChunk = 4;                 // K steps per rho chunk
constexpr int kFwChunks = kFwKSteps / kFwKPerChunk;           // 2 chunks per block
constexpr int kFwChunkHalf = 3 * kFwRows * 32 * kFwKPerChunk; // 192 rows x 64 f16 = 24 KB
constexpr int kFwChunkBytes = 2 * kFwChunkHalf;               // hi, lo: 48 KB
inline bool grid_tc_fwd_fits(int nx) { return grid_tc_fits(nx); }

// Coils per CTA (a coil group): the MMA's 128 rows are bc coils x 128 / bc
// grid rows, m = b * (128 / bc) + r.
inline bool grid_tc_coils_ok(int bc) { return bc == 1 || bc == 4 || bc == 8; }

// e[s * RC + r] = e^{i phase(ky[s] y_r + kz[s] z_r)} for the RC grid
// rows of a CTA and the samples of one record tile: with several coils per
// CTA the (y, z) factor of a row is shared by its coils, so it is evaluated
// once per (row, sample) and read back by each coil's thread.
template <int TRIG, int RC>
__device__ __forceinline__ void tc_row_factors(const float* rec, const float2* yz_sh, float2* e,
                                               int tid)
{
    constexpr int ITEMS = kTcTile * RC;
    static_assert(ITEMS % kTcThreads == 0, "row-factor items");
#pragma unroll
    for (int k = 0; k < ITEMS / kTcThreads; ++k) {
        const int i = tid + k * kTcThreads;
        const int s = i / RC;
        const int r = i % RC;
        const float2 yz = yz_sh[r];
        float sn, cs;
        table_sincos<TRIG>(fmaf(rec[2 * kTcTile + s], yz.y, rec[kTcTile + s] * yz.x), sn, cs);
        e[i] = make_float2(cs, sn);
    }
}

// byte offset of samples 8 kc .. 8 kc + 7 of row `row` in a [128][32] K-major
// no-swizzle f16 tile (one 16-byte core-matrix row)
__device__ __forceinline__ int tc_kmaj_bytes(int row, int kc)
{
    return (row >> 3) * 512 + kc * 128 + (row & 7) * 16;
}

// Exponent e of the power-of-two scale 2^e applied to the A operand, from the
// float bits of the bound b = max |w_r| + |w_i|: b < 2^(E - 126) for the
// biased exponent E, so |A| <= b 2^e < 2^kTcAExp.  Clamped so that 2^e and
// 2^-e are normal floats (b = 0 or subnormal, or b = inf / NaN, whose results
// are then inf / NaN anyway).
__device__ __forceinline__ int tc_scale_exp(unsigned int bound_bits)
{
    const int E = int((bound_bits >> 23) & 0xFFu);
    int e = kTcAExp - (E - 126);
    e = e < -120 ? -120 : (e > 120 ? 120 : e);
    return e;
}

__device__ __forceinline__ float exp2_int(int e)   // 2^e, |e| <= 126
{
    return __uint_as_float(uint32_t(e + 127) << 23);
}

// two floats -> packed f16x2 (round to nearest even), `lo_elem` in bits 0-15
__device__ __forceinline__ uint32_t pack_f16x2(float lo_elem, float hi_elem)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi_elem), "f"(lo_elem));
    return d;
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t d)
{
    float a, b;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(a), "=f"(b)
        : "r"(d));
    return make_float2(a, b);
}

// The low f16 parts of a and b given their high parts h (pack_f16x2(a, b)):
// the remainders a - hi and b - hi, each formed in fp32 by one
// mixed-precision FMA (the f16 hi times -1 plus the fp32 value: exact, since
// hi is the value rounded), rounded to f16 and packed.
__device__ __forceinline__ uint32_t split_lo_f16x2(float a, float b, uint32_t h)
{
    uint32_t l;
    asm("{\n\t.reg .b16 h0, h1, m;\n\t.reg .f32 l0, l1;\n\t"
        "mov.b32 {h0, h1}, %3;\n\t"
        "mov.b16 m, 0xBC00;\n\t"            // f16 -1
        "fma.rn.f32.f16 l0, h0, m, %1;\n\t"
        "fma.rn.f32.f16 l1, h1, m, %2;\n\t"
        "cvt.rn.f16x2.f32 %0, l1, l0;\n\t}"
        : "=r"(l)
        : "f"(a), "f"(b), "r"(h));
    return l;
}

// v = hi + lo for 8 values, two per word: hi = v rounded to f16, lo = the
// exact float remainder v - hi rounded to f16 (|lo| <= 2^-11 |v|, either
// sign, so the dropped lo*lo term has no preferred sign).  The remainder by
// the mixed-precision FMA (split_lo_f16x2).
__device__ __forceinline__ void tc_split8(const float (&v)[8], uint4& hi, uint4& lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        h[j] = pack_f16x2(v[2 * j], v[2 * j + 1]);
        l[j] = split_lo_f16x2(v[2 * j], v[2 * j + 1], h[j]);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// The same parts, bit for bit, with the remainder taken after converting hi
// back to fp32 (two conversions and two subtractions per word instead of two
// FMAs).  The coil-group generators of the grid kernel run 1-2 % faster with
// it; everywhere else the FMA form is as fast or faster (single-coil grid
// paths 1-2 %, the coil kernel at arbitrary coordinates 3 %).
__device__ __forceinline__ void tc_split8_rt(const float (&v)[8], uint4& hi, uint4& lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        h[j] = pack_f16x2(v[2 * j], v[2 * j + 1]);
        const float2 hf = unpack_f16x2(h[j]);
        l[j] = pack_f16x2(v[2 * j] - hf.x, v[2 * j + 1] - hf.y);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ uint4 neg_f16x8(uint4 v)
{
    constexpr uint32_t S = 0x80008000u;
    return make_uint4(v.x ^ S, v.y ^ S, v.z ^ S, v.w ^ S);
}

__device__ __forceinline__ void st_shared16(unsigned char* p, uint4 v)
{
    *reinterpret_cast<uint4*>(p) = v;
}

// The D columns warp w folds and writes: lanes 32 (w % 4) .., columns
// kTcColsPerWarp * (w / 4) .. (D_r is columns 0-127, D_i 128-255).
__device__ __forceinline__ uint32_t tc_warp_cols(int warp)
{
    return uint32_t(kTcColsPerWarp) * uint32_t(warp >> 2);
}

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity)
{
    return mbar_wait_bounded(bar, parity);
}

// The B operand tiles: tile t holds, for every grid column c and sample s of
// record tile t, the f16 hi / lo parts of B = e^{i phase(kx[s] x[c])} (MUB:
// B = w[s] e^{i phase(kx[s] x[c])}, the sample's scaled weight folded in) as
// -B_i, B_r and B_i in S = [-B_i; B_r; B_i] row order (hi block, then lo
// block), each block K-major as the MMA reads it.  One thread per (tile,
// 8-row group, 8-sample chunk, row): consecutive threads write consecutive
// 16-byte core-matrix rows, so a warp's stores are contiguous.
//
// Folded rows (fold > 1 and *fold_ok set, one column block): column gi is x
// index gi & (2^log2_fw - 1) of grid row offset j = gi >> log2_fw within a row
// group, and B = e^{i phase(kx[s] x + ky[s] dy[j])} with dy[j] the exact y
// offset of the group's row j from its first row (fold_dy, from the check).
template <int TRIG, bool MUB>
__global__ void __launch_bounds__(256) build_ex_tiles_kernel(const float* rec, int fields,
                                                             int64_t ntiles, const float* xs,
                                                             int nx, int ncb,
                                                             unsigned char* s_tab, int fold,
                                                             int log2_fw,
                                                             const unsigned int* fold_ok,
                                                             const float* fold_dy)
{
    // MUB: one weight per sample (fields 3, and 4 unless the weight is real)
    const bool complex_w = fields > 4;
    const bool folded = fold > 1 && *fold_ok != 0u;
    const int fmask = (1 << log2_fw) - 1;
    constexpr int ITEMS = kTcCols * kTcTile / 8;       // 512 (column, chunk) items per tile
    const int64_t total = ntiles * ncb * ITEMS;
    for (int64_t item = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; item < total;
         item += int64_t(gridDim.x) * blockDim.x) {
        const int64_t tc = item / ITEMS;              // (tile, column block)
        const int64_t t = tc / ncb;
        const int cb = int(tc - t * ncb);
        const int r = int(item - tc * ITEMS);
        const int gi = ((r >> 5) << 3) | (r & 7);     // column within the block
        const int kc = (r >> 3) & 3;                  // samples 8 kc ..
        const float* kx = rec + t * fields * kTcTile + 8 * kc;
        float br[8], bi[8];
        if (folded) {
            const int ix = gi & fmask;
            const float xc = ix < nx ? xs[ix] : 0.0f;  // padding columns are never written
            const float dy = fold_dy[gi >> log2_fw];
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8)
                table_sincos<TRIG>(fmaf(kx[kTcTile + s8], dy, kx[s8] * xc), bi[s8], br[s8]);
        } else {
            const int col = cb * kTcCols + gi;
            const float xc = col < nx ? xs[col] : 0.0f;   // padding columns are never written
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8) table_sincos<TRIG>(kx[s8] * xc, bi[s8], br[s8]);
        }
        if constexpr (MUB) {
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8) {
                const float wr = kx[3 * kTcTile + s8];
                const float wi = complex_w ? kx[4 * kTcTile + s8] : 0.0f;
                const float c = br[s8], sn = bi[s8];
                br[s8] = fmaf(wr, c, -wi * sn);
                bi[s8] = fmaf(wr, sn, wi * c);
            }
        }
        unsigned char* const tile = s_tab + tc * kTcStageBytes;
        const int off = tc_kmaj_bytes(gi, kc);        // == 16 r
        uint4 h, l;
        tc_split8(bi, h, l);
        *reinterpret_cast<uint4*>(tile + kTcSHi + 2 * kTcPartBytes + off) = h;
        *reinterpret_cast<uint4*>(tile + kTcSLo + 2 * kTcPartBytes + off) = l;
        *reinterpret_cast<uint4*>(tile + kTcSHi + off) = neg_f16x8(h);
        *reinterpret_cast<uint4*>(tile + kTcSLo + off) = neg_f16x8(l);
        tc_split8(br, h, l);
        *reinterpret_cast<uint4*>(tile + kTcSHi + kTcPartBytes + off) = h;
        *reinterpret_cast<uint4*>(tile + kTcSLo + kTcPartBytes + off) = l;
    }
}

// Row folding for narrow grids.  A block holds 128 columns; for nx <= 64
// the columns of G = 128 / fw consecutive grid rows (fw = nx rounded up to a
// power of two) share one block, so the MMA work is that of the real width
// instead of 128 padded columns.  It is exact when every group of G rows has
// the same y offsets from its first row: ys[G g + j] - ys[G g] = dy[j] for
// every g, as real numbers (then ky ys[G g + j] = ky ys[G g] + ky dy[j]).
inline int grid_tc_fold(int nx, int ny)
{
    if (nx < kTcMinCols || nx > kTcCols / 2) return 1;
    int fw = kTcMinCols;
    while (fw < nx) fw *= 2;
    const int G = kTcCols / fw;
    return ny % G == 0 ? G : 1;
}

inline int grid_tc_fold_log2_width(int G)
{
    int l = 7;
    while ((1 << (7 - l)) < G) --l;
    return l;   // fw = 128 / G = 2^l
}

// Bounded wait that also gives up once any role of the CTA has given up (the
// kernels with warp roles share an abort flag in shared memory).
__device__ __forceinline__ bool ws_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            return false;
        }
    }
}

// this thread's 8 samples s0 .. s0 + 7 of record field f (contiguous in the tile)
__device__ __forceinline__ void tc_load8(const float* rec, int f, int s0, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(rec + f * kTcTile + s0);
    const float4 b = *reinterpret_cast<const float4*>(rec + f * kTcTile + s0 + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

}  // namespace mri
