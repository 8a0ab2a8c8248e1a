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
// columns) and, inside each, the grid rows in blocks of 128 (the MMA N,
// [T_r | T_i] = 256 columns).  A = Ex* of the CTA's samples for one column
// block is evaluated into tensor memory (columns 0-255, f16 hi / lo parts)
// and serves every row block; B = rho arrives per (row block, column block,
// K step) as a 24 KB chunk of the per-call table built by
// build_rho_tiles_kernel (rows [-rho_i; rho_r; rho_i], f16 hi / lo,
// K-major), by TMA into a ring of shared-memory stages.
// Per K step 6 tcgen05.mma of 128 x 256 x 16 do
//   [T_r | T_i] += A_r [B_r | B_i] + A_i [-B_i | B_r]
// with each real product as hi*hi + hi*lo + lo*hi (about 22 bits).  rho is
// scaled by one power of two so that every |rho| < 2^15 (f16 range) and the
// result is scaled back exactly.
// The second sum is the epilogue of each (column block, row block): every
// thread reads the T of its sample for 64 of the block's rows from tensor
// memory (columns 256-511), multiplies by e^{-i2pi(ky y + kz z)} of each row
// and adds the block's total to its running sums (blocked summation; the
// row factor distributes over the column blocks); the two threads of a
// sample (two halves of the rows) combine at the end.
// Every wait is bounded; a CTA that gives up sets the device error word,
// waits (bounded) for its MMAs and copies, and frees its tensor memory.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid_tc.cuh"

namespace mri {

constexpr int kFwThreads = 256;
#ifndef MRI_FW_STAGES
#define MRI_FW_STAGES 6
#endif
#ifndef MRI_FW_LEAD
#define MRI_FW_LEAD 4
#endif
constexpr int kFwStages = MRI_FW_STAGES;        // B chunks resident
constexpr int kFwLead = MRI_FW_LEAD;            // chunk copies issued ahead of the MMAs
static_assert(kFwLead >= 1 && kFwLead < kFwStages, "chunk lead");
constexpr uint32_t kFwACols = 256;              // A: 4 parts x 64 columns
constexpr uint32_t kFwDCol = 256;               // D = [T_r | T_i] at columns 256-511

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

// (y, z) of grid row r = iz * ny + iy, zero past the last row
__global__ void __launch_bounds__(256) build_row_coords_kernel(const float* ys, int ny,
                                                               const float* zs, int64_t rows,
                                                               int64_t padded, float2* yz)
{
    for (int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; r < padded;
         r += int64_t(gridDim.x) * blockDim.x) {
        float2 v = make_float2(0.0f, 0.0f);
        if (r < rows) v = make_float2(ys[r % ny], zs[r / ny]);
        yz[r] = v;
    }
}

// The rho table: chunk (block b, column block cb, K step kb) holds rows
// [-rho_i; rho_r; rho_i] of grid rows 128 b .. 128 b + 127 and columns
// 128 cb + 16 kb .. + 15 (zero past nx or the last row), scaled by 2^e,
// split into f16 hi (first 12 KB) and lo.  K-major without swizzle: core
// matrices of 8 rows x 8 f16, LBO = 128 B (along K), SBO = 256 B.  One
// thread per (block, column block, K step, row, 8-column half).
__global__ void __launch_bounds__(256) build_rho_tiles_kernel(const float* rr, const float* ri,
                                                              int64_t rows, int nx, int ncb,
                                                              int64_t row_blocks,
                                                              const unsigned int* bound,
                                                              unsigned char* tab)
{
    const float scale = exp2_int(tc_scale_exp(*bound));
    constexpr int ITEMS = kFwKSteps * kFwRows * 2;            // per (row block, column block)
    const int64_t total = row_blocks * ncb * ITEMS;
    for (int64_t item = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; item < total;
         item += int64_t(gridDim.x) * blockDim.x) {
        const int64_t bc = item / ITEMS;                      // b * ncb + cb
        const int cb = int(bc % ncb);
        int rem = int(item - bc * ITEMS);
        const int kb = rem / (kFwRows * 2);
        rem -= kb * kFwRows * 2;
        const int r = rem >> 1;
        const int kc = rem & 1;
        const int64_t row = (bc / ncb) * kFwRows + r;
        float vr[8], vi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = cb * kFwCols + 16 * kb + 8 * kc + j;
            const bool in = row < rows && col < nx;
            const int64_t n = row * nx + col;
            vr[j] = in ? rr[n] * scale : 0.0f;
            vi[j] = in ? ri[n] * scale : 0.0f;
        }
        unsigned char* chunk = tab + (bc * kFwKSteps + kb) * int64_t(kFwChunkBytes);
        auto off = [&](int srow) { return (srow >> 3) * 256 + kc * 128 + (srow & 7) * 16; };
        uint4 h, l;
        tc_split8(vi, h, l);
        *reinterpret_cast<uint4*>(chunk + off(256 + r)) = h;
        *reinterpret_cast<uint4*>(chunk + kFwChunkHalf + off(256 + r)) = l;
        constexpr uint32_t S = 0x80008000u;
        *reinterpret_cast<uint4*>(chunk + off(r)) = make_uint4(h.x ^ S, h.y ^ S, h.z ^ S, h.w ^ S);
        *reinterpret_cast<uint4*>(chunk + kFwChunkHalf + off(r)) =
            make_uint4(l.x ^ S, l.y ^ S, l.z ^ S, l.w ^ S);
        tc_split8(vr, h, l);
        *reinterpret_cast<uint4*>(chunk + off(128 + r)) = h;
        *reinterpret_cast<uint4*>(chunk + kFwChunkHalf + off(128 + r)) = l;
    }
}

template <int TRIG>
__global__ void __launch_bounds__(kFwThreads, 1) forward_grid_tc_kernel(FwdParams p)
{
    constexpr uint32_t ID = umma_idesc_f16(kFwSamples, 2 * kFwRows);   // N = 256
    constexpr int NS = kFwStages;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const ring = smem_raw;
    float2* const half_sh = reinterpret_cast<float2*>(ring + NS * kFwChunkBytes);
    __shared__ __align__(8) uint64_t s_bar[NS];     // chunk landed
    __shared__ __align__(8) uint64_t c_bar[NS];     // MMAs of the chunk done
    __shared__ __align__(8) uint64_t d_bar;         // MMAs of the row block done
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int h = warp >> 2;                          // column half: rows 64 h .. of a block
    const int split = blockIdx.y;
    const int64_t b_begin = (p.row_blocks * split) / p.splits;
    const int64_t b_end = (p.row_blocks * (split + 1)) / p.splits;
    const int nb = int(b_end - b_begin);
    const int nblk = nb * p.ncb;                      // (column block, row block) pairs
    const int nc = nblk * kFwKSteps;                  // chunks of this CTA, column block outer
    const int ms = 32 * (warp & 3) + lane;            // this thread's sample = TMEM lane
    const int64_t m = int64_t(blockIdx.x) * kFwSamples + ms;
    const uint32_t lanes = uint32_t(32 * (warp & 3)) << 16;

    if (warp == 0) tmem_alloc(&tmem_base_sh, kTcTmemCols);
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            mbar_init(&s_bar[i], 1);
            mbar_init(&c_bar[i], 1);
        }
        mbar_init(&d_bar, 1);
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    auto load_chunk = [&](int c) {
        uint64_t* bar = &s_bar[c % NS];
        const int blk = c / kFwKSteps;
        const int cb = blk / nb;
        const int64_t b = b_begin + (blk - cb * nb);
        const int64_t chunk = (b * p.ncb + cb) * kFwKSteps + (c - blk * kFwKSteps);
        mbar_arrive_expect_tx(bar, uint32_t(kFwChunkBytes));
        tma_bulk_g2s(ring + (c % NS) * kFwChunkBytes, p.rho_tab + chunk * int64_t(kFwChunkBytes),
                     uint32_t(kFwChunkBytes), bar);
    };
    int loaded = 0;     // chunks whose copy thread 0 issued
    int consumed = 0;   // chunks whose MMAs thread 0 issued
    if (tid == 0)
        for (; loaded < NS && loaded < nc; ++loaded) load_chunk(loaded);

    // this thread's sample, phases pre-negated for e^{-i ...}
    float nkx = 0.0f, nky = 0.0f, nkz = 0.0f;
    if (m < p.M) {
        nkx = -p.kx[m] * p.kscale;
        nky = -p.ky[m] * p.kscale;
        nkz = -p.kz[m] * p.kscale;
    }
    // A = Ex*[m][ix] for ix = 128 cb + 64 h .. + 63 (zero past nx, where rho
    // is zero too): columns 32 h .. of every part
    auto build_a = [&](int cb) {
        uint32_t hr[32], lr[32], hi_[32], li[32];
        const int col0 = cb * kFwCols + 64 * h;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
            float ar[8], ai[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = col0 + 8 * c8 + j;
                table_sincos<TRIG>(nkx * (col < p.nx ? p.xs[col] : 0.0f), ai[j], ar[j]);
            }
            uint4 hh, ll;
            tc_split8(ar, hh, ll);
            hr[4 * c8] = hh.x; hr[4 * c8 + 1] = hh.y; hr[4 * c8 + 2] = hh.z; hr[4 * c8 + 3] = hh.w;
            lr[4 * c8] = ll.x; lr[4 * c8 + 1] = ll.y; lr[4 * c8 + 2] = ll.z; lr[4 * c8 + 3] = ll.w;
            tc_split8(ai, hh, ll);
            hi_[4 * c8] = hh.x; hi_[4 * c8 + 1] = hh.y; hi_[4 * c8 + 2] = hh.z; hi_[4 * c8 + 3] = hh.w;
            li[4 * c8] = ll.x; li[4 * c8 + 1] = ll.y; li[4 * c8 + 2] = ll.z; li[4 * c8 + 3] = ll.w;
        }
        const uint32_t a0 = tmem + lanes + uint32_t(32 * h);
        tmem_st32u(a0 + 0 * 64, hr);     // A_RH
        tmem_st32u(a0 + 1 * 64, lr);     // A_RL
        tmem_st32u(a0 + 2 * 64, hi_);    // A_IH
        tmem_st32u(a0 + 3 * 64, li);     // A_IL
        tmem_wait_st();
    };

    float run_r = 0.0f, run_i = 0.0f;   // running sums over blocks
    bool ok = true;
    bool c_fail = false;                // thread 0: a chunk wait timed out
    int failed = 0;
#pragma unroll 1
    for (int blk = 0; blk < nblk; ++blk) {
        const int cb = blk / nb;
        const int b = blk - cb * nb;
        if (b == 0) {
            // a new column block: every MMA of the previous one has completed
            // (its last block's commit was waited for), so A may be rewritten
            build_a(cb);
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
        }
        if (tid == 0) {
            for (int kb = 0; kb < kFwKSteps && !c_fail; ++kb) {
                const int c = blk * kFwKSteps + kb;
                if (!mbar_wait_bounded(&s_bar[c % NS], uint32_t(c / NS) & 1u)) {
                    c_fail = true;
                    break;
                }
                const unsigned char* ch = ring + (c % NS) * kFwChunkBytes;
                auto a = [&](int part) { return tmem + uint32_t(part * 64 + kb * 8); };
                auto sdesc = [&](int half, int r0) {
                    return umma_desc_kmajor(ch + half * kFwChunkHalf + (r0 >> 3) * 256, 128, 256);
                };
                const uint32_t d = tmem + kFwDCol;
                // [T_r | T_i] += A_r [B_r | B_i]   (S rows 128 .. 383)
                umma_f16_ta(d, a(0), sdesc(0, 128), ID, kb > 0 ? 1u : 0u);
                umma_f16_ta(d, a(0), sdesc(1, 128), ID, 1u);
                umma_f16_ta(d, a(1), sdesc(0, 128), ID, 1u);
                // [T_r | T_i] += A_i [-B_i | B_r]  (S rows 0 .. 255)
                umma_f16_ta(d, a(2), sdesc(0, 0), ID, 1u);
                umma_f16_ta(d, a(2), sdesc(1, 0), ID, 1u);
                umma_f16_ta(d, a(3), sdesc(0, 0), ID, 1u);
                umma_commit(&c_bar[c % NS]);
                consumed = c + 1;
                // chunk c + lead into the stage chunk c + lead - NS used
                const int u = c + kFwLead;
                if (u >= NS && u < nc && loaded == u) {
                    if (!mbar_wait_bounded(&c_bar[u % NS], uint32_t((u - NS) / NS) & 1u)) {
                        c_fail = true;
                        break;
                    }
                    load_chunk(u);
                    ++loaded;
                }
            }
            if (!c_fail) umma_commit(&d_bar);
        }
        // every thread: wait for the block's MMAs (thread 0's failure reaches
        // the others through the barrier; their own wait then gives up too)
        ok = c_fail ? false : mbar_wait_bounded(&d_bar, uint32_t(blk) & 1u);
        if (__syncthreads_or(!ok)) {
            failed = 1;
            break;
        }
        tc_fence_after_sync();
        // epilogue: rows 64 h .. 64 h + 63 of block b_begin + b
        const float2* yz = p.yz_rows + (b_begin + b) * kFwRows + 64 * h;
        float bs_r = 0.0f, bs_i = 0.0f;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float tr[16], ti[16];
            tmem_ld16(tmem + lanes + kFwDCol + uint32_t(64 * h + 16 * j), tr);
            tmem_ld16(tmem + lanes + kFwDCol + uint32_t(kFwRows + 64 * h + 16 * j), ti);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 c = yz[16 * j + i];
                float sn, cs;
                table_sincos<TRIG>(fmaf(nkz, c.y, nky * c.x), sn, cs);
                bs_r = fmaf(tr[i], cs, fmaf(-ti[i], sn, bs_r));
                bs_i = fmaf(tr[i], sn, fmaf(ti[i], cs, bs_i));
            }
        }
        run_r += bs_r;
        run_i += bs_i;
        // D is read: the next block's first MMA may overwrite it
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
    }

    if (!failed) {
        // the two threads of a sample (h = 0, 1) combine; h = 0 writes
        if (h == 1) half_sh[ms] = make_float2(run_r, run_i);
        __syncthreads();
        if (h == 0 && m < p.M && nb > 0) {
            const float2 o = half_sh[ms];
            const float inv = exp2_int(-tc_scale_exp(*p.bound));
            const float vr = (run_r + o.x) * inv;
            const float vi = (run_i + o.y) * inv;
            float* orr = p.out_r + split * p.split_stride + m;
            float* oi = p.out_i + split * p.split_stride + m;
            *orr = p.accumulate ? *orr + vr : vr;
            *oi = p.accumulate ? *oi + vi : vi;
        }
    } else if (tid == 0) {
        unsigned int bits = DEVERR_TILE_WAIT_TIMEOUT;
        if (consumed > 0 && !mbar_wait_bounded(&c_bar[(consumed - 1) % NS],
                                               uint32_t((consumed - 1) / NS) & 1u))
            bits |= DEVERR_DRAIN_TIMEOUT;
        for (int u = loaded > NS ? loaded - NS : 0; u < loaded; ++u)
            if (!mbar_wait_bounded(&s_bar[u % NS], uint32_t(u / NS) & 1u))
                bits |= DEVERR_DRAIN_TIMEOUT;
        atomicOr(p.err, bits);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace mri
