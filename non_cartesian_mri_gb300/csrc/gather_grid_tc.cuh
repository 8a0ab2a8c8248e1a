// gather_grid_tc.cuh -- separable-grid F^H D / Q on the tensor cores.
//
// On a grid the gather of Fig. 17.11 factors (gather_grid.cuh) into
//   FhD[row][ix] = sum_m Mz[row][m] * Ex[m][ix],
//   Mz = Mu * e^{i2pi(ky y + kz z)},  Ex = e^{i2pi kx x},
// a complex matrix product over the samples: a dense contraction.  Here a CTA
// owns 128 grid rows (the MMA M) and one block of 128 columns (the MMA N;
// blockIdx.z picks the block; the last block of an nx that is not a multiple
// of 128 is padded with zero columns, which are computed and not stored).  Ex (32 samples x 128 columns per tile of 32 samples and column
// block, the B operand) is the same for every CTA of a column block:
// build_ex_tiles_kernel evaluates it once per call into
// a table of operand tiles in the tensor core's shared-memory layout, and a
// CTA fetches each tile with one TMA bulk copy.  The warps evaluate Mz (128
// rows x 32 samples, the A operand) into tensor memory.  Every value is split
// into an f16 high part and the f16-rounded remainder; one thread then
// issues, per K step (two per tile), two N = 256 products into [D_r | D_i]:
//   [D_r | D_i] += A_r [B_r | B_i]  +  A_i [-B_i | B_r],
// reading the B operands as two 256-row windows of one 384-row block
// S = [-B_i; B_r; B_i], with each real product done as hi*hi + hi*lo + lo*hi
// (12 tcgen05.mma of 128 x 256 x 16 per tile).  The two f16 parts carry about
// 22 significant bits, and the dropped lo*lo term is below 2^-22 of a
// product, so every product keeps close to fp32 accuracy.  f16 has a narrow
// exponent range: the weights are multiplied (once per call, in the records)
// by a power of two chosen from the largest |w_r| + |w_i| of the call so that
// every weighted operand is below 2^15, and the results are multiplied back
// exactly; the phase factors (|e^{i phi}| = 1) need no scale.
//
// Where the weight goes.  With one coil per CTA (F^H D, Q) the weight Mu is
// folded into the B table (B = Mu e^{i2pi kx x}, once per call), and A is the
// bare row factor e^{i2pi(ky y + kz z)}: per (row, sample) element the CTA
// evaluates one sin/cos pair and splits it, with no weight loads and no
// complex multiply -- operand generation, not the tensor core, is what a
// tile waits for.  With a coil group (batched F^H D) B is shared by the
// group's coils, so A = Mu_coil e^{i2pi(ky y + kz z)} as written above.
//
// Shared-memory bandwidth binds a kernel whose operands all pass through
// shared memory (operand writes plus operand reads by the tensor core); with
// A in tensor memory only B takes that path, written by the TMA.  D (tensor
// memory columns 0-255) collects one block of tiles and is then added into
// running sums R held in registers (each thread owns 128 of the 128 x 256
// sums: its warp's lane quarter and half of the columns), the blocked
// summation that keeps accumulation error below the trig error over a
// million samples.  Columns 256.. hold the A stages (64 columns each).
//
// B tiles are K-major without swizzle: core matrices of 8 rows x 8 f16
// (128 B), LBO = 128 B along K, SBO = 512 B between 8-row groups.  The
// operand stages rotate; stage s is rewritten only after the MMAs that read
// it have signalled their mbarrier, so operand generation runs ahead of the
// tensor core by up to kTcStages - 1 tiles.  Every wait is bounded; a CTA
// that gives up sets the device error word, waits (bounded) for its MMAs and
// copies, and still frees its tensor memory.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid.cuh"

namespace mri {

constexpr int kTcTile = 32;                          // samples per tile (two K = 16 steps)
constexpr int kTcRows = 128;                         // grid rows per CTA = MMA M
constexpr int kTcCols = 128;                         // grid columns per CTA = MMA N / 2
#ifndef MRI_TC_THREADS
#define MRI_TC_THREADS 256
#endif
constexpr int kTcThreads = MRI_TC_THREADS;           // 256 or 512
constexpr int kTcWarps = kTcThreads / 32;
#ifndef MRI_TC_STAGES
#define MRI_TC_STAGES 4
#endif
// How many tiles ahead of the MMAs the B tile copies run (1 or 2); the stage
// a copy fills must have been released by the MMAs of tile u - kTcStages.
#ifndef MRI_TC_S_LEAD
#define MRI_TC_S_LEAD 2
#endif
// Tiles per summation block.  The tensor core's own fp32 accumulation loses
// a little with every add, with a consistent sign, so the error of a block
// grows with its length (measured on the 128^3 radial workload: rel-L2 1.4e-5
// for blocks of 1024 samples, 1.9e-6 for 128); the accurate path folds every
// 128 samples, the fast paths every 1024.
#ifndef MRI_TC_DRAIN_ACCURATE
#define MRI_TC_DRAIN_ACCURATE 4
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
constexpr int kTcSLead = MRI_TC_S_LEAD;
// The Ey table replaces the per-(row, sample) sin/cos of the accurate path
// (and of the fast paths when MRI_TC_EY_FAST is 1).
#ifndef MRI_TC_EY_FAST
#define MRI_TC_EY_FAST 0
#endif
// With the Ey table two 32 KB Ey stages take shared memory from the B ring.
constexpr int kTcStagesEy = 3;
constexpr int kTcEyBytes = kTcTile * kTcRows * 8;   // 32 samples x 128 rows of float2
constexpr int kTcColsPerWarp = 256 * 4 / kTcWarps;  // D columns one warp folds (128 or 64)
constexpr uint32_t kTcDCols = 256;                   // D_r | D_i
constexpr uint32_t kTcAPartCols = kTcTile / 2;       // one A part: 32 f16 per lane (16 columns)
constexpr uint32_t kTcAStageCols = 4 * kTcAPartCols; // A r/i hi/lo (64 columns)
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcAExp = 15;                          // |A| * scale < 2^kTcAExp
static_assert(kTcThreads == 256 || kTcThreads == 512, "generation mapping");
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
constexpr int kFwRows = 128;                    // grid rows per block = MMA N / 2
constexpr int kFwCols = 128;                    // grid columns per block = K
constexpr int kFwKSteps = kFwCols / 16;         // 8
constexpr int kFwChunkHalf = 3 * kFwRows * 32;  // 384 rows x 16 f16 = 12 KB (hi or lo)
constexpr int kFwChunkBytes = 2 * kFwChunkHalf; // 24 KB
inline bool grid_tc_fwd_fits(int nx) { return grid_tc_fits(nx); }

// Coils per CTA (a coil group): the MMA's 128 rows are bc coils x 128 / bc
// grid rows, m = b * (128 / bc) + r.
inline bool grid_tc_coils_ok(int bc) { return bc == 1 || bc == 4 || bc == 8; }

inline size_t grid_tc_smem_bytes(bool realw, int bc = 1, bool eyt = false)
{
    const int F = realw ? 4 : 3 + 2 * bc;
    const int rc = kTcRows / bc;
    size_t b = size_t(eyt ? kTcStagesEy : kTcStages) * kTcStageBytes;   // B operand stages
    if (eyt) b += size_t(2) * kTcEyBytes + size_t(2) * kTcTile * 8;   // Ey tiles, z factors
    b += size_t(kStages) * F * kTcTile * 4;                // record ring
    b += size_t(rc) * 8;                                   // (y, z) of the rows
    if (bc > 1) b += size_t(2) * kTcTile * rc * 8;         // row factors, two tiles
    return b;
}

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

// v = hi + lo for 8 values, two per word: hi = v rounded to f16, lo = the
// exact float remainder v - hi rounded to f16 (|lo| <= 2^-11 |v|, either
// sign, so the dropped lo*lo term has no preferred sign)
__device__ __forceinline__ void tc_split8(const float (&v)[8], uint4& hi, uint4& lo)
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
template <int TRIG, bool MUB>
__global__ void __launch_bounds__(256) build_ex_tiles_kernel(const float* rec, int fields,
                                                             int64_t ntiles, const float* xs,
                                                             int nx, int ncb,
                                                             unsigned char* s_tab)
{
    // MUB: one weight per sample (fields 3, and 4 unless the weight is real)
    const bool complex_w = fields > 4;
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
        const int col = cb * kTcCols + gi;
        const float xc = col < nx ? xs[col] : 0.0f;   // padding columns are never written
        float br[8], bi[8];
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) table_sincos<TRIG>(kx[s8] * xc, bi[s8], br[s8]);
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

// The Ey table: for record tile t and block yb of 128 y values,
// e^{i phase(ky[s] ys[128 yb + r])} at [(t * nyb + yb) * 32 + s] * 128 + r
// (float2: cos, sin).  Consecutive threads take consecutive r.
template <int TRIG>
__global__ void __launch_bounds__(256) build_ey_tiles_kernel(const float* rec, int fields,
                                                             int64_t ntiles, const float* ys,
                                                             int nyb, float2* ey_tab)
{
    const int64_t per_tile = int64_t(nyb) * kTcTile * kTcRows;
    const int64_t total = ntiles * per_tile;
    for (int64_t item = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; item < total;
         item += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = item / per_tile;
        const int rem = int(item - t * per_tile);
        const int yb = rem / (kTcTile * kTcRows);
        const int s = (rem / kTcRows) % kTcTile;
        const int r = rem % kTcRows;
        float sn, cs;
        table_sincos<TRIG>(rec[t * fields * kTcTile + kTcTile + s] * ys[yb * kTcRows + r], sn, cs);
        ey_tab[item] = make_float2(cs, sn);
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

template <int BC, bool REALW, int TRIG, bool EYT>
__global__ void __launch_bounds__(kTcThreads, 1) gather_grid_tc_kernel(GridParams p)
{
    // EYT: the y factor of Mz comes from the Ey table (one z-plane per CTA)
    static_assert(!EYT || BC == 1, "Ey table for single-weight calls");
    constexpr int kS = EYT ? kTcStagesEy : kTcStages;   // B / A stages
    constexpr int kLead = EYT ? 1 : kTcSLead;
    static_assert(BC == 1 || (!REALW && (BC == 4 || BC == 8)), "coil group");
    constexpr int T = kTcTile;
    constexpr int F = REALW ? 4 : 3 + 2 * BC;
    constexpr int RC = kTcRows / BC;                  // grid rows per CTA
    constexpr uint32_t TILE_BYTES = uint32_t(F) * T * 4;
    constexpr uint32_t ID = umma_idesc_f16(kTcRows, 2 * kTcCols);   // N = 256
    constexpr int drain_tiles = (TRIG == TRIG_ACCURATE) ? kTcDrainAccurate : kTcDrainFast;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const ops = smem_raw;
    float2* const ey_sh = reinterpret_cast<float2*>(ops + kS * kTcStageBytes);   // EYT: 2 Ey tiles
    float* const ring = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(ey_sh) +
                                                 (EYT ? 2 * kTcEyBytes : 0));
    float2* const yz_sh = reinterpret_cast<float2*>(ring + kStages * F * T);
    // BC > 1: row factors of two tiles; EYT: Mu e^{i phase(kz z)} of two tiles
    float2* const e_sh = yz_sh + RC;
    __shared__ __align__(8) uint64_t full_bar[kStages];     // record tile landed
    __shared__ __align__(8) uint64_t ey_bar[2];             // EYT: Ey tile landed
    __shared__ __align__(8) uint64_t s_bar[kS];      // B operand tile landed
    __shared__ __align__(8) uint64_t mma_bar[kS];    // MMAs of the stage done
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t total_rows = int64_t(p.ny) * p.nz;
    const int64_t row0 = int64_t(blockIdx.x) * RC;
    const int scale_e = tc_scale_exp(*p.wbound);

    for (int r = tid; r < RC; r += kTcThreads) {
        const int64_t row = row0 + r;
        float2 yz = make_float2(0.f, 0.f);
        if (row < total_rows) {
            const int64_t iz = row / p.ny;
            const int64_t iy = row - iz * p.ny;
            yz = make_float2(p.ys[iy], p.zs[iz]);
        }
        yz_sh[r] = yz;
    }
    if (warp == 0) tmem_alloc(&tmem_base_sh, kTcTmemCols);
    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&full_bar[st], 1);
        mbar_init(&ey_bar[0], 1);
        mbar_init(&ey_bar[1], 1);
#pragma unroll
        for (int st = 0; st < kS; ++st) {
            mbar_init(&s_bar[st], 1);
            mbar_init(&mma_bar[st], 1);
        }
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    // B tile u into stage u % kS (thread 0 only)
    auto load_s = [&](int u) {
        uint64_t* bar = &s_bar[u % kS];
        mbar_arrive_expect_tx(bar, uint32_t(kTcStageBytes));
        tma_bulk_g2s(ops + (u % kS) * kTcStageBytes,
                     p.s_tab + ((t_begin + u) * p.ncb + blockIdx.z) * kTcStageBytes,
                     uint32_t(kTcStageBytes), bar);
    };
    // EYT: this CTA's 128 rows are grid rows iy0 .. iy0 + 127 of plane iz
    const int ey_block = EYT ? int((row0 % p.ny) / kTcRows) : 0;
    const float z_plane = EYT ? p.zs[row0 / p.ny] : 0.0f;
    auto load_ey = [&](int u) {
        uint64_t* bar = &ey_bar[u & 1];
        mbar_arrive_expect_tx(bar, uint32_t(kTcEyBytes));
        tma_bulk_g2s(ey_sh + (u & 1) * (T * kTcRows),
                     p.ey_tab + ((t_begin + u) * p.ey_blocks + ey_block) * (T * kTcRows),
                     uint32_t(kTcEyBytes), bar);
    };
    int ey_loaded = 0;    // Ey tiles whose copy thread 0 has issued
    int s_loaded = 0;     // B tiles whose copy thread 0 has issued
    int s_consumed = 0;   // B tiles thread 0 has seen land
    if (tid == 0) {
        for (int st = 0; st < kStages && st < nt; ++st) {
            mbar_arrive_expect_tx(&full_bar[st], TILE_BYTES);
            tma_bulk_g2s(ring + st * F * T, p.rec + (t_begin + st) * F * T, TILE_BYTES,
                         &full_bar[st]);
        }
        for (; s_loaded < kS && s_loaded < nt; ++s_loaded) load_s(s_loaded);
        if constexpr (EYT)
            for (; ey_loaded < 2 && ey_loaded < nt; ++ey_loaded) load_ey(ey_loaded);
    }
    // EYT: e[s] = e^{i phase(kz[s] z)} of this CTA's plane (the weight is in
    // the B table), by warp 0
    auto z_factors = [&](const float* rec, float2* e) {
        if (warp == 0) {
            const int s = lane;
            float sn, cs;
            table_sincos<TRIG>(rec[2 * T + s] * z_plane, sn, cs);
            e[s] = make_float2(cs, sn);
        }
    };

    // A (Mz) generation: row ra = this thread's tensor-memory lane (a warp
    // reaches only its own lane quarter), samples 8 kTcAChunks ah .., which
    // are columns 4 kTcAChunks ah .. of every A part (two f16 per column).
    // With BC coils, lane ra is coil ra / RC of grid row ra % RC.
    const int ra = 32 * (warp & 3) + lane;
    const int ah = warp >> 2;
    const int coil = ra / RC;
    const int rr = ra % RC;
    const uint32_t lanes = uint32_t(32 * (warp & 3)) << 16;
    const float2 yz = yz_sh[rr];

    // running sums: lanes of this warp's quarter, D columns tc_warp_cols(warp) ..
    float R[kTcColsPerWarp];
#pragma unroll
    for (int j = 0; j < kTcColsPerWarp; ++j) R[j] = 0.0f;
    const uint32_t dcols = tmem + lanes + tc_warp_cols(warp);
    auto drain = [&]() {
#pragma unroll
        for (int c = 0; c < kTcColsPerWarp / 32; ++c) {
            float d[32];
            tmem_ld32(dcols + uint32_t(32 * c), d);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) R[32 * c + j] += d[j];
        }
    };

    int failed_at = -1;
    bool s_fail = false;   // thread 0: a B tile or stage wait timed out
    if constexpr (BC > 1 || EYT) {
        // row (or plane) factors of tile 0; later tiles' are made one tile ahead
        bool ok0 = true;
        if (nt > 0) {
            ok0 = mbar_wait_bounded(&full_bar[0], 0u);
            if (ok0) {
                if constexpr (EYT)
                    z_factors(ring, e_sh);
                else
                    tc_row_factors<TRIG, RC>(ring, yz_sh, e_sh, tid);
            }
        }
        if (__syncthreads_or(!ok0)) failed_at = 0;
    }
    for (int t = 0; t < nt && failed_at < 0; ++t) {
        const int st = t % kS;
        const bool new_block = (t % drain_tiles) == 0;
        const uint32_t acol = tmem + kTcDCols + uint32_t(st) * kTcAStageCols;
        bool ok = true;
        // the MMAs of tile t - kS read stage st
        if (t >= kS)
            ok = tc_wait(&mma_bar[st], uint32_t((t - kS) / kS) & 1u);
        if (ok) ok = tc_wait(&full_bar[t % kStages], uint32_t(t / kStages) & 1u);
        if (EYT && ok) ok = tc_wait(&ey_bar[t & 1], uint32_t(t >> 1) & 1u);
        // warp-uniform: the tensor-memory store below is .sync.aligned
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            const float* rec = ring + (t % kStages) * F * T;
#pragma unroll
            for (int c = 0; c < kTcAChunks; ++c) {
                const int s0 = 8 * (kTcAChunks * ah + c);
                float ar[8], ai[8];
                if constexpr (EYT) {
                    // A = e^{i phase(kz z)} e^{i phase(ky y)}
                    const float2* ez = e_sh + (t & 1) * T;
                    const float2* ey = ey_sh + (t & 1) * (T * kTcRows);
#pragma unroll
                    for (int s8 = 0; s8 < 8; ++s8) {
                        const float2 f = ez[s0 + s8];
                        const float2 e = ey[(s0 + s8) * kTcRows + ra];
                        ar[s8] = fmaf(f.x, e.x, -f.y * e.y);
                        ai[s8] = fmaf(f.x, e.y, f.y * e.x);
                    }
                } else if constexpr (BC == 1) {
                    // A = e^{i phase(ky y + kz z)} (the weight is in the B table)
                    float ky[8], kz[8];
                    tc_load8(rec, 1, s0, ky);
                    tc_load8(rec, 2, s0, kz);
#pragma unroll
                    for (int s8 = 0; s8 < 8; ++s8)
                        table_sincos<TRIG>(fmaf(kz[s8], yz.y, ky[s8] * yz.x), ai[s8], ar[s8]);
                } else {
                    // Mu of this thread's coil times the row's shared factor
                    const float2* e = e_sh + (t & 1) * T * RC;
                    float wr[8], wi[8];
                    tc_load8(rec, 3 + coil, s0, wr);
                    tc_load8(rec, 3 + BC + coil, s0, wi);
#pragma unroll
                    for (int s8 = 0; s8 < 8; ++s8) {
                        const float2 f = e[(s0 + s8) * RC + rr];
                        ar[s8] = fmaf(wr[s8], f.x, -wi[s8] * f.y);
                        ai[s8] = fmaf(wi[s8], f.x, wr[s8] * f.y);
                    }
                }
                // samples s0 .. s0 + 7 = columns s0 / 2 .. of each part
                const uint32_t col = acol + uint32_t(s0 / 2);
                uint4 h, l;
                tc_split8(ar, h, l);
                tmem_st4(col + A_RH * kTcAPartCols, h);
                tmem_st4(col + A_RL * kTcAPartCols, l);
                tc_split8(ai, h, l);
                tmem_st4(col + A_IH * kTcAPartCols, h);
                tmem_st4(col + A_IL * kTcAPartCols, l);
            }
            tmem_wait_st();
            if constexpr (BC > 1 || EYT) {
                // row (or plane) factors of the next tile (its buffer was last
                // read by tile t - 1, before the previous barrier)
                if (t + 1 < nt) {
                    ok = mbar_wait_bounded(&full_bar[(t + 1) % kStages],
                                           uint32_t((t + 1) / kStages) & 1u);
                    if (ok) {
                        const float* rec1 = ring + ((t + 1) % kStages) * F * T;
                        if constexpr (EYT)
                            z_factors(rec1, e_sh + ((t + 1) & 1) * T);
                        else
                            tc_row_factors<TRIG, RC>(rec1, yz_sh, e_sh + ((t + 1) & 1) * T * RC,
                                                     tid);
                    }
                }
            }
        }
        // a new summation block: fold D into R once tile t - 1 is done, before
        // the first MMA of tile t overwrites D (the decision is the same in
        // every thread, so the barrier is uniform)
        if (new_block && t > 0) {
            if (ok)
                ok = tc_wait(&mma_bar[(t - 1) % kS], uint32_t((t - 1) / kS) & 1u);
            if (__syncthreads_or(!ok || s_fail)) {
                failed_at = t;
                break;
            }
            tc_fence_after_sync();
            drain();
        }
        // A written to tensor memory -> visible to the MMAs
        tc_fence_before_sync();
        if (__syncthreads_or(!ok || s_fail)) {
            failed_at = t;
            break;
        }
        tc_fence_after_sync();
        if (tid == 0) {
            // Ey tile t + 2 into the buffer tile t has just finished with
            if constexpr (EYT) {
                if (t + 2 < nt && ey_loaded == t + 2) {
                    load_ey(t + 2);
                    ++ey_loaded;
                }
            }
            if (t + kStages < nt) {
                mbar_arrive_expect_tx(&full_bar[t % kStages], TILE_BYTES);
                tma_bulk_g2s(ring + (t % kStages) * F * T, p.rec + (t_begin + t + kStages) * F * T,
                             TILE_BYTES, &full_bar[t % kStages]);
            }
            bool s_ok = mbar_wait_bounded(&s_bar[st], uint32_t(t / kS) & 1u);
            if (s_ok) {
                s_consumed = t + 1;
                const unsigned char* stage = ops + st * kTcStageBytes;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    // K step kb: 8 columns of every A part, 2 core matrices = 256 B of S
                    auto a = [&](int part) {
                        return acol + uint32_t(part) * kTcAPartCols + uint32_t(8 * kb);
                    };
                    // window of 256 S rows starting at row r0 (16 row groups per 128 rows)
                    auto sdesc = [&](int base, int r0) {
                        return umma_desc_kmajor(stage + base + (r0 / 128) * kTcPartBytes + kb * 256,
                                                128, 512);
                    };
                    const uint32_t acc0 = (new_block && kb == 0) ? 0u : 1u;
                    // [D_r | D_i] += A_r [B_r | B_i]
                    umma_f16_ta(tmem, a(A_RH), sdesc(kTcSHi, 128), ID, acc0);
                    umma_f16_ta(tmem, a(A_RH), sdesc(kTcSLo, 128), ID, 1u);
                    umma_f16_ta(tmem, a(A_RL), sdesc(kTcSHi, 128), ID, 1u);
                    // [D_r | D_i] += A_i [-B_i | B_r]
                    umma_f16_ta(tmem, a(A_IH), sdesc(kTcSHi, 0), ID, 1u);
                    umma_f16_ta(tmem, a(A_IH), sdesc(kTcSLo, 0), ID, 1u);
                    umma_f16_ta(tmem, a(A_IL), sdesc(kTcSHi, 0), ID, 1u);
                }
                umma_commit(&mma_bar[st]);
                // refill a stage for tile t + lead as soon as the MMAs that
                // read it (tile t + lead - kS) are done
                const int u = t + kLead;
                if (u >= kS && u < nt && s_loaded == u) {
                    s_ok = mbar_wait_bounded(&mma_bar[u % kS],
                                             uint32_t((u - kS) / kS) & 1u);
                    if (s_ok) {
                        load_s(u);
                        ++s_loaded;
                    }
                }
            }
            // a timeout here stops every thread at the next barrier
            if (!s_ok) s_fail = true;
        }
    }

    bool ok = failed_at < 0;
    if (ok && nt > 0) {
        if (!s_fail)
            ok = tc_wait(&mma_bar[(nt - 1) % kS], uint32_t((nt - 1) / kS) & 1u);
        if (__syncthreads_or(!ok || s_fail)) {
            ok = false;
            failed_at = nt;
        } else {
            tc_fence_after_sync();
            drain();
        }
    }

    if (ok) {
        // R -> outputs: this thread holds grid row rr of coil `coil` and its
        // warp's D columns
        const float inv_scale = exp2_int(-scale_e);
        const int64_t row = row0 + rr;
        const uint32_t wcols = tc_warp_cols(warp);
        float* const out = (wcols >= 128u ? p.out_i : p.out_r) + split * p.split_stride +
                           coil * p.coil_stride;
        if (row < total_rows && coil < p.coils && nt > 0) {
            const int col0 = int(blockIdx.z) * kTcCols;
            const int ncols = p.nx - col0 < kTcCols ? p.nx - col0 : kTcCols;
            float* o = out + row * p.nx + col0 + (wcols & 127u);
            // a thread's outputs are contiguous: 16-byte accesses when the
            // block is whole and every row starts on a 16-byte boundary
            const float keep = p.accumulate ? 1.0f : 0.0f;
            if (ncols == kTcCols && (p.nx & 3) == 0 &&
                (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
                float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
                for (int j = 0; j < kTcColsPerWarp / 4; ++j) {
                    const float4 a = p.accumulate ? o4[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                    o4[j] = make_float4(fmaf(R[4 * j], inv_scale, keep * a.x),
                                        fmaf(R[4 * j + 1], inv_scale, keep * a.y),
                                        fmaf(R[4 * j + 2], inv_scale, keep * a.z),
                                        fmaf(R[4 * j + 3], inv_scale, keep * a.w));
                }
            } else {
#pragma unroll
                for (int j = 0; j < kTcColsPerWarp; ++j)
                    if (int(wcols & 127u) + j < ncols)
                        o[j] = fmaf(R[j], inv_scale, p.accumulate ? o[j] : 0.0f);
            }
        }
    } else {
        // Report, then let the MMAs and copies in flight finish before the
        // CTA's shared and tensor memory are released.
        if (tid == 0) {
            // thread 0 issued the MMAs of exactly the first s_consumed tiles
            unsigned int bits = DEVERR_TILE_WAIT_TIMEOUT;
            const int issued = s_consumed;
            if (issued > 0 && !mbar_wait_bounded(&mma_bar[(issued - 1) % kS],
                                                 uint32_t((issued - 1) / kS) & 1u))
                bits |= DEVERR_DRAIN_TIMEOUT;
            const int first = failed_at < nt ? failed_at : nt;
            const int last = (first + kStages < nt) ? first + kStages : nt;
            for (int u = first; u < last; ++u)
                if (!mbar_wait_bounded(&full_bar[u % kStages], uint32_t(u / kStages) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            for (int u = s_consumed; u < s_loaded; ++u)
                if (!mbar_wait_bounded(&s_bar[u % kS], uint32_t(u / kS) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            // the last Ey copy into each buffer
            for (int u = ey_loaded > 2 ? ey_loaded - 2 : 0; u < ey_loaded; ++u)
                if (!mbar_wait_bounded(&ey_bar[u & 1], uint32_t(u >> 1) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            atomicOr(p.err, bits);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace mri
