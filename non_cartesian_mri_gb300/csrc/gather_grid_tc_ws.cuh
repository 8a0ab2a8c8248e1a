// gather_grid_tc_ws.cuh -- the tensor-core grid F^H D / Q kernel, with warp
// roles (operand layouts, tables and helpers in gather_grid_tc.cuh).
//
// Per tile of 32 samples, A (128 MMA rows: BC coils x 128 / BC grid rows) goes to tensor
// memory as f16 hi / lo parts, B (one block of 128 columns) comes from the
// per-call table by TMA, and 12 tcgen05.mma of 128 x 256 x 16 add A B into
// D; D is folded into running sums in registers every block of tiles
// (blocked summation).  A per case:
//   BC = 1:         A = e^{i2pi(ky y + kz z)} (the weight is in the B table),
//                   one sin/cos per element (accurate: the polynomial on
//                   pairs of samples);
//   BC = 4 or 8:    A = Mu_coil e^{i2pi(ky y + kz z)}: the row factor of each
//                   (grid row, sample) evaluated once into shared memory one
//                   tile ahead, by all generator threads (a named barrier of
//                   the generator warps makes it visible), times each coil's
//                   weight.
//
// Who waits for whom.  tcgen05.mma is issued by one thread and stalls that
// thread while the tensor core's instruction queue is full -- for most of a
// tile's MMA time.  Were the issuing thread also generating operands, with
// the CTA meeting at a barrier every tile, every warp would wait for it and
// operand generation and the MMAs would run one after the other (measured:
// 963 of 2,460 cycles per tile in the issue, 67 against 89 Tpairs/s).  So
// the roles are separate and meet only at mbarriers:
//   warps 0-7   (two warpgroups, 232 registers each thread): generate A into
//               the tensor-memory stage of tile t once the MMAs of tile
//               t - kS are done, signal a_full; fold D into the running sums
//               when a block's last MMA is done, signal d_free; epilogue.
//   warp 8      lane 0: waits a_full and the B tile, issues the MMAs,
//               commits to mma_bar; waits d_free before the first MMA of a
//               block (the first MMA of a block overwrites D).
//   warp 9      lane 0: TMA copies of the record tiles (slot reused once
//               every generator warp has signalled rec_free) and of the B
//               tiles (stage reused once its MMAs are done).
//   warps 10-11 idle (they complete the third warpgroup, which gives up its
//               registers to the generators: 32 each).
// Launch: 384 threads at 168 registers (the whole register file); the host
// checks the compiled count before launching, since the warpgroup budgets
// (2 x 128 x 232 + 128 x 32 = 63,488 of 64,512) must fit what the CTA holds.
//
// Every wait is bounded and also gives up when another role has given up
// (a shared abort flag); a role that gives up reports through the device
// error word, and the issuing and copying threads wait (bounded) for their
// MMAs and copies in flight before tensor and shared memory are released.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid_tc.cuh"

// Accurate single-coil A generation on pairs of samples (.f32x2).
#ifndef MRI_TC_PACKED_A
#define MRI_TC_PACKED_A 1
#endif

namespace mri {

constexpr int kWsGenWarps = 8;                        // two warpgroups
constexpr int kWsThreads = 32 * kWsGenWarps + 128;    // + one warpgroup of helpers
constexpr int kWsLaunchRegs = 168;                    // 65,536 / 384, a multiple of 8
constexpr int kWsGenRegs = 232;
constexpr int kWsAuxRegs = 32;
static_assert(32 * kWsGenWarps * kWsGenRegs + 128 * kWsAuxRegs <= kWsThreads * kWsLaunchRegs,
              "warpgroup register budgets exceed the launch");
static_assert(kWsGenWarps == kTcWarps, "generator warps own the D columns by tc_warp_cols");

inline size_t grid_tc_ws_smem_bytes(bool realw, int bc)
{
    const int F = realw ? 4 : 3 + 2 * bc;
    const int rc = kTcRows / bc;
    size_t b = size_t(kTcStages) * kTcStageBytes;                       // B operand stages
    b += size_t(kStages) * F * kTcTile * 4;                             // record ring
    b += size_t(rc) * 8;                                                // (y, z) of the rows
    if (bc > 1) b += size_t(2) * kTcTile * rc * 8;                      // row factors, two tiles
    return b;
}

// Barrier of the generator warps alone (named barrier 1; 0 is __syncthreads)
// that also returns whether `v` holds in every generator thread.  Every
// generator warp reaches it the same number of times: a failure is carried
// to the next one as v = false, and all leave together.
__device__ __forceinline__ bool ws_gen_sync_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q, p;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v)), "n"(32 * kWsGenWarps)
        : "memory");
    return r != 0;
}

template <int BC, bool REALW, int TRIG>
__global__ void __launch_bounds__(kWsThreads, 1) gather_grid_tc_ws_kernel(GridParams p)
{
    static_assert(BC == 1 || (!REALW && (BC == 4 || BC == 8)), "coil group");
    constexpr int kS = kTcStages;                     // A / B stages
    constexpr int T = kTcTile;
    constexpr int F = REALW ? 4 : 3 + 2 * BC;
    constexpr int RC = kTcRows / BC;                  // grid rows per CTA
    constexpr uint32_t TILE_BYTES = uint32_t(F) * T * 4;
    constexpr uint32_t ID = umma_idesc_f16(kTcRows, 2 * kTcCols);   // N = 256
    constexpr int drain_tiles = (TRIG == TRIG_ACCURATE) ? kTcDrainAccurate : kTcDrainFast;
    static_assert(drain_tiles >= kS, "at most one block waits for its drain");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* const ops = smem_raw;
    float* const ring = reinterpret_cast<float*>(ops + kS * kTcStageBytes);
    float2* const yz_sh = reinterpret_cast<float2*>(ring + kStages * F * T);
    float2* const e_sh = yz_sh + RC;                  // BC > 1: row factors of two tiles
    __shared__ __align__(8) uint64_t full_bar[kStages];   // record tile landed
    __shared__ __align__(8) uint64_t rec_free[kStages];   // record tile read by every generator
    __shared__ __align__(8) uint64_t s_bar[kS];           // B tile landed
    __shared__ __align__(8) uint64_t a_full[kS];          // A tile written by every generator
    __shared__ __align__(8) uint64_t mma_bar[kS];         // MMAs of the tile done
    __shared__ __align__(8) uint64_t d_free;              // D folded by every generator
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    __shared__ int fold_sh[3];                            // G, log2 of its width, row groups
    __shared__ unsigned int bound_sh[BC];                 // each coil's weight bound word
    volatile int* const abort_flag = &abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    // row folding: an MMA row is a group of G grid rows (the check word says
    // whether the y axis allows it; the grid is sized for the unfolded rows)
    int G = 1, log2_fw = 7;
    if (p.fold > 1 && *p.fold_ok != 0u) {
        G = p.fold;
        log2_fw = p.log2_fw;
    }
    const int64_t row0 = int64_t(blockIdx.x) * RC;
    {
        const int nyg = p.ny / G;                      // row groups per z plane
        const int64_t total_rows = int64_t(nyg) * p.nz;   // MMA rows over the grid
        if (row0 >= total_rows) return;                // folded: nothing for this CTA
        for (int r = tid; r < RC; r += kWsThreads) {
            const int64_t row = row0 + r;
            float2 yz = make_float2(0.f, 0.f);
            if (row < total_rows) {
                const int64_t iz = row / nyg;
                const int64_t iy = (row - iz * nyg) * G;   // the group's first grid row
                yz = make_float2(p.ys[iy], p.zs[iz]);
            }
            yz_sh[r] = yz;
        }
        if (tid < BC) bound_sh[tid] = p.wbound[tid];
        if (tid == 0) {
            fold_sh[0] = G;
            fold_sh[1] = log2_fw;
            fold_sh[2] = nyg;
        }
    }
    if (warp == 0) tmem_alloc(&tmem_base_sh, kTcTmemCols);
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&rec_free[i], kWsGenWarps);
        }
#pragma unroll
        for (int i = 0; i < kS; ++i) {
            mbar_init(&s_bar[i], 1);
            mbar_init(&a_full[i], kWsGenWarps);
            mbar_init(&mma_bar[i], 1);
        }
        mbar_init(&d_free, kWsGenWarps);
        abort_sh = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp >= kWsGenWarps) {
        setmaxnreg_dec<kWsAuxRegs>();
        if (warp == kWsGenWarps && lane == 0) {
            // ---- MMA issue ----
            int issued = 0;
            for (int t = 0; t < nt; ++t) {
                const int st = t % kS;
                const bool first = (t % drain_tiles) == 0;
                bool ok = true;
                // the first MMA of a block overwrites D: the previous block is folded
                if (first && t > 0)
                    ok = ws_wait(&d_free, uint32_t(t / drain_tiles - 1) & 1u, abort_flag);
                if (ok) ok = ws_wait(&a_full[st], uint32_t(t / kS) & 1u, abort_flag);
                if (ok) ok = ws_wait(&s_bar[st], uint32_t(t / kS) & 1u, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                // one descriptor per stage; the windows are constant offsets
                const uint64_t d0 = umma_desc_kmajor(ops + st * kTcStageBytes, 128, 512);
                const uint32_t acol = tmem + kTcDCols + uint32_t(st) * kTcAStageCols;
#pragma unroll
                for (int kb = 0; kb < 2; ++kb) {
                    auto a = [&](int part) {
                        return acol + uint32_t(part) * kTcAPartCols + uint32_t(8 * kb);
                    };
                    auto sdesc = [&](int base, int r0) {
                        return umma_desc_add(
                            d0, uint32_t(base + (r0 / 128) * kTcPartBytes + kb * 256));
                    };
                    const uint32_t acc0 = (first && kb == 0) ? 0u : 1u;
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
                issued = t + 1;
            }
            // the MMAs issued finish before tensor memory is released (the
            // last commit covers all of them; the phase before it completed
            // before its tile's A was written)
            if (issued > 0 && !mbar_wait_bounded(&mma_bar[(issued - 1) % kS],
                                                 uint32_t((issued - 1) / kS) & 1u))
                atomicOr(p.err, DEVERR_DRAIN_TIMEOUT);
            if (issued < nt) atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
        } else if (warp == kWsGenWarps + 1 && lane == 0) {
            // ---- copies: record tile u, B tile u ----
            int r_issued = 0, b_issued = 0;
            for (int u = 0; u < nt; ++u) {
                bool ok = true;
                if (u >= kStages)
                    ok = ws_wait(&rec_free[u % kStages], uint32_t((u - kStages) / kStages) & 1u,
                                 abort_flag);
                if (!ok) break;
                tma_load_checked(ring + (u % kStages) * F * T, p.rec, t_begin + u, p.ntiles,
                                 TILE_BYTES, &full_bar[u % kStages], p.err);
                r_issued = u + 1;
                if (u >= kS)
                    ok = ws_wait(&mma_bar[u % kS], uint32_t((u - kS) / kS) & 1u, abort_flag);
                if (!ok) break;
                tma_load_checked(ops + (u % kS) * kTcStageBytes, p.s_tab,
                                 (t_begin + u) * p.ncb + blockIdx.z, p.ntiles * p.ncb,
                                 uint32_t(kTcStageBytes), &s_bar[u % kS], p.err);
                b_issued = u + 1;
            }
            // the latest copy into each slot and stage lands before shared
            // memory is released, whatever the other roles did (the copy
            // before it in the same slot was consumed, so the phase is
            // unambiguous; in a run without failure these have landed)
            unsigned int bits = 0;
            for (int u = r_issued > kStages ? r_issued - kStages : 0; u < r_issued; ++u)
                if (!mbar_wait_bounded(&full_bar[u % kStages], uint32_t(u / kStages) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            for (int u = b_issued > kS ? b_issued - kS : 0; u < b_issued; ++u)
                if (!mbar_wait_bounded(&s_bar[u % kS], uint32_t(u / kS) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            if (b_issued < nt) bits |= DEVERR_TILE_WAIT_TIMEOUT;
            if (bits) atomicOr(p.err, bits);
        }
        __syncwarp();
    } else {
        setmaxnreg_inc<kWsGenRegs>();
        // ---- generators: thread = tensor-memory lane ra = coil ra / RC of
        // grid row ra % RC ----
        const int ra = 32 * (warp & 3) + lane;
        const int ah = warp >> 2;                     // samples 16 ah .. 16 ah + 15 of a tile
        const int coil = ra / RC;
        const int rr = ra % RC;
        const uint32_t lanes = uint32_t(32 * (warp & 3)) << 16;
        const float2 yz = yz_sh[rr];
        float R[kTcColsPerWarp];
#pragma unroll
        for (int j = 0; j < kTcColsPerWarp; ++j) R[j] = 0.0f;
        const uint32_t dcols = tmem + lanes + tc_warp_cols(warp);
        // fold D into R, then tell the issuer that D may be overwritten
        auto fold = [&](bool signal) {
            tc_fence_after_sync();
#pragma unroll
            for (int c = 0; c < kTcColsPerWarp / 32; ++c) {
                float d[32];
                tmem_ld32(dcols + uint32_t(32 * c), d);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) R[32 * c + j] += d[j];
            }
            if (signal) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_free);
            }
        };

        bool ok = true;
        if constexpr (BC > 1) {
            // row factors of tile 0; later tiles' are made one tile ahead
            if (nt > 0) {
                ok = __all_sync(0xffffffffu, ws_wait(&full_bar[0], 0u, abort_flag));
                if (ok) tc_row_factors<TRIG, RC>(ring, yz_sh, e_sh, tid);
            }
            ok = ws_gen_sync_and(ok);
        }
        int pend = -1;   // last tile of a block whose D is not folded yet (another block follows)
        // no early exit inside a tile: with coil groups every generator warp
        // meets the others at the named barrier closing each tile
        for (int t = 0; t < nt && ok; ++t) {
            const int st = t % kS;
            if (pend >= 0) {
                // fold as soon as the block's last MMA is done; at the latest
                // before A of tile pend + kS (which waits for it anyway)
                const bool must = t - kS >= pend;
                bool done = must ? ws_wait(&mma_bar[pend % kS], uint32_t(pend / kS) & 1u,
                                           abort_flag)
                                 : mbar_try_wait(&mma_bar[pend % kS], uint32_t(pend / kS) & 1u);
                done = __all_sync(0xffffffffu, done);
                if (must && !done) {
                    ok = false;
                } else if (done) {
                    fold(true);
                    pend = -1;
                }
            }
            // the stage's previous A (tile t - kS) has been read; the records have landed
            if (ok && t >= kS)
                ok = ws_wait(&mma_bar[st], uint32_t((t - kS) / kS) & 1u, abort_flag);
            if (ok) ok = ws_wait(&full_bar[t % kStages], uint32_t(t / kStages) & 1u, abort_flag);
            // warp-uniform: the tensor-memory stores below are .sync.aligned
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after_sync();
                const float* rec = ring + (t % kStages) * F * T;
                const uint32_t acol = tmem + lanes + kTcDCols + uint32_t(st) * kTcAStageCols;
#pragma unroll
                for (int c = 0; c < kTcAChunks; ++c) {
                    const int s0 = 8 * (kTcAChunks * ah + c);
                    float ar[8], ai[8];
                    if constexpr (BC == 1 && TRIG == TRIG_ACCURATE && MRI_TC_PACKED_A) {
                        // the polynomial on pairs of samples (.f32x2)
                        float ky[8], kz[8];
                        tc_load8(rec, 1, s0, ky);
                        tc_load8(rec, 2, s0, kz);
                        const f2 y2 = f2_splat(yz.x), z2 = f2_splat(yz.y);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const f2 ph = f2_fma(f2_pack(kz[2 * h], kz[2 * h + 1]), z2,
                                                 f2_mul(f2_pack(ky[2 * h], ky[2 * h + 1]), y2));
                            f2 sn, cs;
                            sincos_half_turns2(ph, sn, cs);
                            f2_unpack(sn, ai[2 * h], ai[2 * h + 1]);
                            f2_unpack(cs, ar[2 * h], ar[2 * h + 1]);
                        }
                    } else if constexpr (BC == 1) {
                        float ky[8], kz[8];
                        tc_load8(rec, 1, s0, ky);
                        tc_load8(rec, 2, s0, kz);
#pragma unroll
                        for (int s8 = 0; s8 < 8; ++s8)
                            table_sincos<TRIG>(fmaf(kz[s8], yz.y, ky[s8] * yz.x), ai[s8], ar[s8]);
                    } else {
                        // this coil's weight times the row's shared factor
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
                    if constexpr (BC == 1) tc_split8(ar, h, l); else tc_split8_rt(ar, h, l);
                    tmem_st4(col + A_RH * kTcAPartCols, h);
                    tmem_st4(col + A_RL * kTcAPartCols, l);
                    if constexpr (BC == 1) tc_split8(ai, h, l); else tc_split8_rt(ai, h, l);
                    tmem_st4(col + A_IH * kTcAPartCols, h);
                    tmem_st4(col + A_IL * kTcAPartCols, l);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[st]);
                    mbar_arrive(&rec_free[t % kStages]);
                }
                if (t % drain_tiles == drain_tiles - 1 && t + 1 < nt) pend = t;
                if constexpr (BC > 1) {
                    // row factors of tile t + 1 into the buffer tile t - 1 used
                    // (every generator finished with it before the previous
                    // named barrier)
                    if (t + 1 < nt) {
                        ok = __all_sync(0xffffffffu, ws_wait(&full_bar[(t + 1) % kStages],
                                                             uint32_t((t + 1) / kStages) & 1u,
                                                             abort_flag));
                        if (ok)
                            tc_row_factors<TRIG, RC>(ring + ((t + 1) % kStages) * F * T, yz_sh,
                                                     e_sh + ((t + 1) & 1) * T * RC, tid);
                    }
                }
            }
            if constexpr (BC > 1) ok = ws_gen_sync_and(ok);
        }
        // the block still waiting for its fold, then the last block
        if (ok && pend >= 0) {
            ok = __all_sync(0xffffffffu,
                            ws_wait(&mma_bar[pend % kS], uint32_t(pend / kS) & 1u, abort_flag));
            if (ok) fold(true);
        }
        if (ok && nt > 0) {
            ok = __all_sync(0xffffffffu, ws_wait(&mma_bar[(nt - 1) % kS],
                                                 uint32_t((nt - 1) / kS) & 1u, abort_flag));
            if (ok) fold(false);
        }
        if (!ok) {
            if (lane == 0) atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
        } else if (nt > 0) {
            // R -> outputs: grid row ra, this warp's D columns (the fold
            // state is read back from shared memory, not kept in registers)
            const float inv_scale = exp2_int(-tc_scale_exp(bound_sh[coil]));   // this coil's
            const volatile int* fs = fold_sh;
            const int G = fs[0], log2_fw = fs[1], nyg = fs[2];
            const int64_t total_rows = int64_t(nyg) * p.nz;
            const int64_t row = row0 + rr;
            const uint32_t wcols = tc_warp_cols(warp);
            float* const out = (wcols >= 128u ? p.out_i : p.out_r) + split * p.split_stride +
                               coil * p.coil_stride;
            if (G > 1 && row < total_rows && coil < p.coils) {
                // column c of the block: grid row G * (row group) + (c >> log2_fw),
                // x index c & (fw - 1); padding columns (x index >= nx) are not stored
                const int64_t iz = row / nyg;
                const int64_t iy = (row - iz * nyg) * G;
                float* const o = out + (iz * p.ny + iy) * p.nx;
                const int fmask = (1 << log2_fw) - 1;
#pragma unroll
                for (int j = 0; j < kTcColsPerWarp; ++j) {
                    const int ix = j & fmask;
                    if (ix < p.nx) {
                        float* oj = o + int64_t(j >> log2_fw) * p.nx + ix;
                        *oj = fmaf(R[j], inv_scale, p.accumulate ? *oj : 0.0f);
                    }
                }
            } else if (row < total_rows && coil < p.coils) {
                const int col0 = int(blockIdx.z) * kTcCols;
                const int ncols = p.nx - col0 < kTcCols ? p.nx - col0 : kTcCols;
                float* o = out + row * p.nx + col0 + (wcols & 127u);
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
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kTcTmemCols);
}

}  // namespace mri
