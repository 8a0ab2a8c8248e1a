// gather_grid_tc_fwd.cuh -- the forward model D = F rho on a separable grid,
// on the tensor cores (nx >= 8).
//
// D[m] = sum_n rho[n] e^{-i2pi k_m . x_n} (F of Fig. 17.3) over the voxels of
// a grid factors like F^H D does (gather_grid_tc.cuh), with the roles of the
// two sums exchanged:
//   T[m][row] = sum_ix Ex*[m][ix] rho[row][ix],   Ex* = e^{-i2pi kx x},
//   D[m]      = sum_row T[m][row] e^{-i2pi (ky y + kz z)}_row.
// The first is a complex matrix product (samples x nx columns) by (nx
// columns x rows): a CTA owns 128 samples (the MMA M) and walks the columns
// in blocks of 128 (K, 8 steps of 16; the last block padded with zero
// columns) and, inside each, the grid rows in blocks of 64 (the MMA N,
// [T_r | T_i] = 128 columns).  A = Ex* of the CTA's samples for one column
// block is evaluated into tensor memory (columns 0-255, f16 hi / lo parts)
// and serves every row block; B = rho arrives per (row block, column block,
// group of K steps) as a chunk of the per-call table built by
// build_rho_tiles_kernel (rows [-rho_i; rho_r; rho_i], f16 hi / lo,
// K-major), by TMA into a ring of shared-memory stages.  Per K step 6
// tcgen05.mma of 128 x 128 x 16 do
//   [T_r | T_i] += A_r [B_r | B_i] + A_i [-B_i | B_r]
// with each real product as hi*hi + hi*lo + lo*hi (about 22 bits).  rho is
// scaled by one power of two so that every |rho| < 2^15 (f16 range) and the
// result is scaled back exactly.
// The second sum is the epilogue of each (column block, row block): a thread
// reads T of its sample for 32 of the block's rows from tensor memory,
// multiplies by e^{-i2pi(ky y + kz z)} of each row and adds the block's
// total to its running sums (blocked summation; the row factor distributes
// over the column blocks); the two threads of a sample combine at the end.
// The row factors go by groups of 8 rows: a group whose rows share z and are
// evenly spaced in y (marked in the row table) takes one sin/cos and seven
// rotations by e^{-i2pi ky d}, any other group a sin/cos per row.
//
// Warp roles, as in the F^H D kernel (gather_grid_tc_ws.cuh): D is double
// buffered (tensor-memory columns 256-383 and 384-511), so the MMAs of row
// block b + 1 run while the epilogue of block b reads its buffer.
//   warps 0-7  build A (once per column block, after the last MMA of the
//              previous one), then per row block: wait d_full, copy their
//              part of D to registers, signal d_free, fold into the sums;
//   warp 8     lane 0: issues the MMAs (waiting a_full, the chunk, d_free),
//              commits to the chunk's c_bar and to the buffer's d_full;
//   warp 9     lane 0: TMA copies of the rho chunks, a stage reused once its
//              MMAs are done;
//   warps 10-11 idle.
// Every wait is bounded and gives up when another role has given up; the
// issuing and copying threads wait (bounded) for their MMAs and copies in
// flight before tensor and shared memory are released.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid_tc.cuh"

namespace mri {

constexpr int kFwThreads = 384;                 // 8 epilogue warps + a warpgroup of helpers
constexpr int kFwGenWarps = 8;
constexpr int kFwStages = 4;                    // rho chunks resident (48 KB each)
constexpr uint32_t kFwDCol = 256;               // D buffers at columns 256-383, 384-511
constexpr uint32_t kFwDBufCols = 2 * kFwRows;   // [T_r | T_i] of one row block
static_assert(kFwDCol + 2 * kFwDBufCols <= kTcTmemCols, "two D buffers fit tensor memory");

inline size_t grid_tc_fwd_smem_bytes()
{
    return size_t(kFwStages) * kFwChunkBytes + size_t(kFwSamples) * 8;
}

// float bits of max |rho_r| + |rho_i| into *bound (zeroed by the caller)
__global__ void __launch_bounds__(256) rho_bound_kernel(const float* rr, const float* ri,
                                                        int64_t n, unsigned int* bound)
{
    float w = 0.0f;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        w = fmaxf(w, fabsf(rr[i]) + fabsf(ri[i]));
    const unsigned int b = __reduce_max_sync(0xffffffffu, __float_as_uint(w));
    if ((threadIdx.x & 31) == 0 && b != 0u) atomicMax(bound, b);
}

// (y, z) of grid row r = iz * ny + iy, zero past the last row; and per group
// of 8 rows the y step d when the group's rows share z and y_i = y_0 + i d
// exactly (checked in double; d exact in float), else NaN
__global__ void __launch_bounds__(256) build_row_coords_kernel(const float* ys, int ny,
                                                               const float* zs, int64_t rows,
                                                               int64_t padded, float2* yz,
                                                               float* step)
{
    for (int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; r < padded;
         r += int64_t(gridDim.x) * blockDim.x) {
        float2 v = make_float2(0.0f, 0.0f);
        if (r < rows) v = make_float2(ys[r % ny], zs[r / ny]);
        yz[r] = v;
    }
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < padded / 8;
         g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r0 = 8 * g;
        float st = __int_as_float(0x7fc00000);   // NaN: rows one by one
        if (r0 + 7 < rows && r0 / ny == (r0 + 7) / ny) {
            const int64_t i0 = r0 % ny;
            const double y0 = ys[i0];
            const double d = double(ys[i0 + 1]) - y0;
            bool even = double(float(d)) == d;
            for (int i = 2; i < 8; ++i) even = even && double(ys[i0 + i]) == y0 + i * d;
            if (even) st = float(d);
        }
        step[g] = st;
    }
}

// The rho table: chunk (block b, column block cb, chunk kp) holds rows
// [-rho_i; rho_r; rho_i] of grid rows 64 b .. 64 b + 63 and columns
// 128 cb + 16 kFwKPerChunk kp .. (kFwKPerChunk K steps; zero past nx or the
// last row), scaled by 2^e, split into f16 hi (first half) and lo.  K-major
// without swizzle: core matrices of 8 rows x 8 f16, LBO = 128 B (along K),
// SBO = 256 kFwKPerChunk B (8-row groups).  One thread per (block, column block, chunk, row,
// 8-column quarter).
__global__ void __launch_bounds__(256) build_rho_tiles_kernel(const float* rr, const float* ri,
                                                              int64_t rows, int nx, int ncb,
                                                              int64_t row_blocks,
                                                              const unsigned int* bound,
                                                              unsigned char* tab)
{
    const float scale = exp2_int(tc_scale_exp(*bound));
    constexpr int Q = 2 * kFwKPerChunk;                       // 8-column groups per chunk
    constexpr int ITEMS = kFwChunks * kFwRows * Q;            // per (row block, column block)
    const int64_t total = row_blocks * ncb * ITEMS;
    for (int64_t item = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; item < total;
         item += int64_t(gridDim.x) * blockDim.x) {
        const int64_t bc = item / ITEMS;                      // b * ncb + cb
        const int cb = int(bc % ncb);
        int rem = int(item - bc * ITEMS);
        const int kp = rem / (kFwRows * Q);
        rem -= kp * kFwRows * Q;
        const int r = rem / Q;
        const int kc = rem - r * Q;
        const int64_t row = (bc / ncb) * kFwRows + r;
        float vr[8], vi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = cb * kFwCols + 16 * kFwKPerChunk * kp + 8 * kc + j;
            const bool in = row < rows && col < nx;
            const int64_t n = row * nx + col;
            vr[j] = in ? rr[n] * scale : 0.0f;
            vi[j] = in ? ri[n] * scale : 0.0f;
        }
        unsigned char* chunk = tab + (bc * kFwChunks + kp) * int64_t(kFwChunkBytes);
        auto off = [&](int srow) { return (srow >> 3) * (128 * Q) + kc * 128 + (srow & 7) * 16; };
        uint4 h, l;
        tc_split8(vi, h, l);
        *reinterpret_cast<uint4*>(chunk + off(2 * kFwRows + r)) = h;
        *reinterpret_cast<uint4*>(chunk + kFwChunkHalf + off(2 * kFwRows + r)) = l;
        *reinterpret_cast<uint4*>(chunk + off(r)) = neg_f16x8(h);
        *reinterpret_cast<uint4*>(chunk + kFwChunkHalf + off(r)) = neg_f16x8(l);
        tc_split8(vr, h, l);
        *reinterpret_cast<uint4*>(chunk + off(kFwRows + r)) = h;
        *reinterpret_cast<uint4*>(chunk + kFwChunkHalf + off(kFwRows + r)) = l;
    }
}

template <int TRIG>
__global__ void __launch_bounds__(kFwThreads, 1) forward_grid_tc_kernel(FwdParams p)
{
    constexpr uint32_t ID = umma_idesc_f16(kFwSamples, 2 * kFwRows);   // N = 128
    constexpr int NS = kFwStages;
    constexpr uint32_t kSbo = 256 * kFwKPerChunk;    // bytes per 8-row group of a chunk

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const ring = smem_raw;
    float2* const half_sh = reinterpret_cast<float2*>(ring + NS * kFwChunkBytes);
    __shared__ __align__(8) uint64_t s_bar[NS];     // chunk landed
    __shared__ __align__(8) uint64_t c_bar[NS];     // MMAs of the chunk done
    __shared__ __align__(8) uint64_t d_full[2];     // MMAs of the buffer's row block done
    __shared__ __align__(8) uint64_t d_free[2];     // buffer read by every epilogue warp
    __shared__ __align__(8) uint64_t a_full;        // A of the column block written
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    volatile int* const abort_flag = &abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.y;
    const int64_t b_begin = (p.row_blocks * split) / p.splits;
    const int64_t b_end = (p.row_blocks * (split + 1)) / p.splits;
    const int nb = int(b_end - b_begin);
    const int nblk = nb * p.ncb;                      // (column block, row block) pairs
    const int nc = nblk * kFwChunks;                  // chunks of this CTA, column block outer

    if (warp == 0) tmem_alloc(&tmem_base_sh, kTcTmemCols);
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            mbar_init(&s_bar[i], 1);
            mbar_init(&c_bar[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_free[i], kFwGenWarps);
        }
        mbar_init(&a_full, kFwGenWarps);
        abort_sh = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    bool failed = false;
    float run_r = 0.0f, run_i = 0.0f;   // epilogue warps: running sums over blocks
    if (warp >= kFwGenWarps) {
        if (warp == kFwGenWarps && lane == 0 && nc > 0) {
            // ---- MMA issue: column block outer, row block, K step ----
            int c = 0;          // chunks whose MMAs are issued
            bool ok = true;
            for (int blk = 0; blk < nblk && ok; ++blk) {
                const int cb = blk / nb;
                const int buf = blk & 1;
                if (blk - cb * nb == 0)   // a new column block: its A is written
                    ok = ws_wait(&a_full, uint32_t(cb) & 1u, abort_flag);
                // the buffer's previous row block has been read by the epilogue
                if (ok && blk >= 2)
                    ok = ws_wait(&d_free[buf], uint32_t((blk - 2) >> 1) & 1u, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t d = tmem + kFwDCol + uint32_t(buf) * kFwDBufCols;
                for (int kp = 0; kp < kFwChunks; ++kp, ++c) {
                    if (!ws_wait(&s_bar[c % NS], uint32_t(c / NS) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    // one descriptor per chunk; the windows are constant offsets
                    const uint64_t d0 =
                        umma_desc_kmajor(ring + (c % NS) * kFwChunkBytes, 128, kSbo);
                    const uint32_t a0 = tmem + uint32_t(kFwKPerChunk * kp * 8);
#pragma unroll
                    for (int j = 0; j < kFwKPerChunk; ++j) {
                        const int kb = kFwKPerChunk * kp + j;
                        auto a = [&](int part) { return a0 + uint32_t(part * 64 + j * 8); };
                        // window of 128 S rows from row r0 (8-row groups of kSbo
                        // bytes), K step j of the chunk (two core matrices of 128 B)
                        auto sdesc = [&](int half, int r0) {
                            return umma_desc_add(
                                d0, uint32_t(half * kFwChunkHalf + (r0 / 8) * kSbo + j * 256));
                        };
                        const uint32_t acc0 = kb > 0 ? 1u : 0u;
                        // [T_r | T_i] += A_r [B_r | B_i]   (S rows 64 .. 191)
                        umma_f16_ta(d, a(0), sdesc(0, kFwRows), ID, acc0);
                        umma_f16_ta(d, a(0), sdesc(1, kFwRows), ID, 1u);
                        umma_f16_ta(d, a(1), sdesc(0, kFwRows), ID, 1u);
                        // [T_r | T_i] += A_i [-B_i | B_r]  (S rows 0 .. 127)
                        umma_f16_ta(d, a(2), sdesc(0, 0), ID, 1u);
                        umma_f16_ta(d, a(2), sdesc(1, 0), ID, 1u);
                        umma_f16_ta(d, a(3), sdesc(0, 0), ID, 1u);
                    }
                    umma_commit(&c_bar[c % NS]);
                }
                if (ok) umma_commit(&d_full[buf]);
            }
            // the MMAs issued finish before tensor memory is released (the
            // last commit covers all of them; the phase before it on the same
            // barrier completed before that chunk's stage was refilled)
            if (c > 0 && !mbar_wait_bounded(&c_bar[(c - 1) % NS], uint32_t((c - 1) / NS) & 1u))
                atomicOr(p.err, DEVERR_DRAIN_TIMEOUT);
            if (!ok) atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
        } else if (warp == kFwGenWarps + 1 && lane == 0 && nc > 0) {
            // ---- copies: chunk u into stage u % NS once its MMAs are done ----
            int loaded = 0;
            for (int u = 0; u < nc; ++u) {
                if (u >= NS &&
                    !ws_wait(&c_bar[u % NS], uint32_t((u - NS) / NS) & 1u, abort_flag))
                    break;
                const int blk = u / kFwChunks;
                const int cb = blk / nb;
                const int64_t b = b_begin + (blk - cb * nb);
                const int64_t chunk = (b * p.ncb + cb) * kFwChunks + (u - blk * kFwChunks);
                tma_load_checked(ring + (u % NS) * kFwChunkBytes, p.rho_tab, chunk,
                                 p.row_blocks * p.ncb * kFwChunks, uint32_t(kFwChunkBytes),
                                 &s_bar[u % NS], p.err);
                loaded = u + 1;
            }
            // the latest copy into each stage lands before shared memory is
            // released (the copy before it in the stage was consumed)
            unsigned int bits = loaded < nc ? DEVERR_TILE_WAIT_TIMEOUT : 0u;
            for (int u = loaded > NS ? loaded - NS : 0; u < loaded; ++u)
                if (!mbar_wait_bounded(&s_bar[u % NS], uint32_t(u / NS) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            if (bits) atomicOr(p.err, bits);
        }
        __syncwarp();
    }
    else if (nc > 0) {
        // ---- epilogue warps: thread = tensor-memory lane = sample ms; the
        // warps w and w + 4 share the lanes and take rows 32 h .. of a block ----
        const int h = warp >> 2;
        const int ms = 32 * (warp & 3) + lane;
        const int64_t m = int64_t(blockIdx.x) * kFwSamples + ms;
        const uint32_t lanes = uint32_t(32 * (warp & 3)) << 16;
        // this thread's sample, phases pre-negated for e^{-i ...}
        float nkx = 0.0f, nky = 0.0f, nkz = 0.0f;
        if (m < p.M) {
            nkx = -p.kx[m] * p.kscale;
            nky = -p.ky[m] * p.kscale;
            nkz = -p.kz[m] * p.kscale;
        }
        bool ok = true;
        // the rotation of the last evenly spaced row group (NaN: none yet)
        float rot_step = __int_as_float(0x7fc00000), rot_s = 0.0f, rot_c = 1.0f;
        for (int blk = 0; blk < nblk && ok; ++blk) {
            const int cb = blk / nb;
            const int b = blk - cb * nb;
            const int buf = blk & 1;
            if (b == 0) {
                // A = Ex*[m][ix] for ix = 128 cb + 64 h .. + 63 (zero past nx,
                // where rho is zero too): columns 32 h .. of every part.  The
                // previous column block's MMAs are all done: its last row
                // block was waited for below.
                const int col0 = cb * kFwCols + 64 * h;
                const uint32_t a0 = tmem + lanes + uint32_t(32 * h);
#pragma unroll 2
                for (int c8 = 0; c8 < 8; ++c8) {
                    float ar[8], ai[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int col = col0 + 8 * c8 + j;
                        table_sincos<TRIG>(nkx * (col < p.nx ? p.xs[col] : 0.0f), ai[j], ar[j]);
                    }
                    // columns 8 c8 .. = 32-bit columns 4 c8 .. of each part
                    const uint32_t col = a0 + uint32_t(4 * c8);
                    uint4 hh, ll;
                    tc_split8(ar, hh, ll);
                    tmem_st4(col + 0 * 64, hh);   // A_RH
                    tmem_st4(col + 1 * 64, ll);   // A_RL
                    tc_split8(ai, hh, ll);
                    tmem_st4(col + 2 * 64, hh);   // A_IH
                    tmem_st4(col + 3 * 64, ll);   // A_IL
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full);
            }
            // the block's MMAs are done: copy this thread's part of T, free the buffer
            ok = __all_sync(0xffffffffu,
                            ws_wait(&d_full[buf], uint32_t(blk >> 1) & 1u, abort_flag));
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t dcol = tmem + lanes + kFwDCol + uint32_t(buf) * kFwDBufCols +
                                  uint32_t(32 * h);
            float tr[32], ti[32];
            tmem_ld32(dcol, tr);
            tmem_ld32(dcol + uint32_t(kFwRows), ti);
            tmem_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_free[buf]);
            // rows 32 h .. 32 h + 31 of block b_begin + b, in groups of 8: a
            // group of evenly spaced rows sharing z takes one sin/cos and
            // seven rotations by e^{i 2 pi ky d} (rounding drift of at most
            // seven complex products), any other group a sin/cos per row
            const int64_t row0 = (b_begin + b) * kFwRows + 32 * h;
            const float2* yz = p.yz_rows + row0;
            const float* gst = p.row_step + row0 / 8;
            float bs_r = 0.0f, bs_i = 0.0f;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float st = gst[g];
                if (st == st) {
                    if (st != rot_step) {
                        table_sincos<TRIG>(nky * st, rot_s, rot_c);
                        rot_step = st;
                    }
                    const float2 c = yz[8 * g];
                    float sn, cs;
                    table_sincos<TRIG>(fmaf(nkz, c.y, nky * c.x), sn, cs);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 8 * g + i;
                        bs_r = fmaf(tr[r], cs, fmaf(-ti[r], sn, bs_r));
                        bs_i = fmaf(tr[r], sn, fmaf(ti[r], cs, bs_i));
                        const float nc = fmaf(cs, rot_c, -sn * rot_s);
                        sn = fmaf(cs, rot_s, sn * rot_c);
                        cs = nc;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 8 * g + i;
                        const float2 c = yz[r];
                        float sn, cs;
                        table_sincos<TRIG>(fmaf(nkz, c.y, nky * c.x), sn, cs);
                        bs_r = fmaf(tr[r], cs, fmaf(-ti[r], sn, bs_r));
                        bs_i = fmaf(tr[r], sn, fmaf(ti[r], cs, bs_i));
                    }
                }
            }
            run_r += bs_r;
            run_i += bs_i;
        }
        if (!ok) {
            failed = true;
            if (lane == 0) atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
        }
        // the two threads of a sample (h = 0, 1) combine after the barrier below
        if (h == 1) half_sh[ms] = make_float2(run_r, run_i);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp < 4 && nc > 0 && !failed && !*abort_flag) {
        const int ms = 32 * warp + lane;
        const int64_t m = int64_t(blockIdx.x) * kFwSamples + ms;
        if (m < p.M) {
            const float2 o = half_sh[ms];
            const float inv = exp2_int(-tc_scale_exp(*p.bound));
            const float vr = (run_r + o.x) * inv;
            const float vi = (run_i + o.y) * inv;
            float* orr = p.out_r + split * p.split_stride + m;
            float* oi = p.out_i + split * p.split_stride + m;
            *orr = p.accumulate ? *orr + vr : vr;
            *oi = p.accumulate ? *oi + vi : vi;
        }
    }
    if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace mri
