// gather_coils_tc.cuh -- batched F^H D for arbitrary voxel coordinates on the
// tensor cores: a group of up to 8 coils per launch.
//
// For a coil group the gather of Fig. 17.11 is, per voxel n and coil c,
//   FhD_c[n] = sum_m E[n][m] Mu_c[m],   E[n][m] = e^{i 2 pi k_m . x_n}:
// a complex matrix product (voxels x samples) by (samples x coils).  The
// per-pair work that remains on the SM is E -- one sin/cos per voxel-sample
// pair, shared by the coils -- and the multiply-accumulate of every coil goes
// to the tensor core.  On the SIMT cores the multiply-accumulate (4 FP32
// operations per pair and coil) binds; here the SFU (fast) or the FP32
// polynomial (accurate) of E does, once per pair for all coils.
//
// A CTA owns 128 voxels (the MMA's M) and a range of the samples.  Per tile of
// 32 samples its generator warps evaluate A = E (128 voxels x 32 samples),
// split every value into f16 high and low parts, and store them to tensor
// memory (thread = MMA row = voxel); B holds the group's weights (8 coils,
// zero for absent ones), built once per call into a table of operand tiles
// fetched by TMA.  The f16 parts of the weights lie along N: one MMA of
// N = 32 multiplies one A part by the high and the low part of the weights
// at once, into D = [D_r | D_i | D_r' | D_i'] (8 coils each; the fold adds
// the primed low-part columns).  Per K step of 16 samples four products:
//   D += A_r^hi W_r + A_r^lo W_r + A_i^hi W_i + A_i^lo W_i,
//   W_r = [Mu_r^hi | Mu_i^hi | Mu_r^lo | Mu_i^lo],
//   W_i = [-Mu_i^hi | Mu_r^hi | -Mu_i^lo | Mu_r^lo],
// i.e. every product of the parts, lo*lo included (the split-f16 scheme of
// the grid kernels, gather_grid_tc.cuh; the weights of each coil are scaled
// by their own power of two, so coils of very different magnitude keep full
// precision each, and D's columns are scaled back per coil).  W_r and W_i are
// two windows of one tile of eight 8-row groups, taken with a stride of two
// groups: [-Mu_i^hi, Mu_r^hi, Mu_r^hi, Mu_i^hi, -Mu_i^lo, Mu_r^lo, Mu_r^lo,
// Mu_i^lo], W_i the even groups, W_r the odd ones.  The tensor core's time
// per MMA at these small N follows the A operand it reads (about 64 bytes of
// A per clock), so the fewer, wider products are the cheaper form: 8 MMAs
// per tile where three N = 16 passes per part pair took 12.  D is folded
// into running sums in registers every block of tiles (blocked summation).
// Roles meet at mbarriers, every wait bounded: warps 0-7 generate A (warps
// 0-3 also fold D and write the outputs), warp 8 lane 0 issues the MMAs,
// warp 9 lane 0 copies the record and B tiles.  Two CTAs per SM (256
// tensor-memory columns each).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather_grid_tc.cuh"

namespace mri {

constexpr int kCtRows = 128;                        // voxels per CTA = MMA M
constexpr int kCtCoils = 8;                         // coils per launch (padded)
constexpr int kCtN = 2 * kCtCoils;                  // D_r, D_i
constexpr int kCtMmaN = 2 * kCtN;                   // MMA N: D_r, D_i and their low parts
constexpr int kCtGroups = 8;                        // 8-row groups of a weight tile
constexpr int kCtBBytes = kCtGroups * 512;          // one weight tile: 4 KB
constexpr int kCtFields = 3 + 2 * kCtCoils;         // record fields (grid-path layout)
constexpr int kCtRecBytes = kCtFields * kTcTile * 4; // one record tile: 2,432 B
constexpr int kCtKBytes = 3 * kTcTile * 4;          // its k fields: 384 B
constexpr int kCtStages = 3;                        // A stages (tensor memory)
#ifndef MRI_CT_RING
#define MRI_CT_RING 8
#endif
// Shared-memory stages of the copied k fields and weight tiles: more than the
// A stages, so that the copies run far enough ahead to hide their latency
// (a stage is refilled once the MMAs of the tile it held are done).
constexpr int kCtRing = MRI_CT_RING;
constexpr int kCtGenWarps = 8;
constexpr int kCtThreads = 32 * kCtGenWarps + 64;   // + the MMA and copy warps
constexpr uint32_t kCtTmemCols = 256;               // two CTAs per SM
constexpr uint32_t kCtACol = 64;                    // A stages after D (columns 0-31)
// Dynamic shared memory (operand rings) padded so that at most two CTAs fit an SM,
// the number whose tensor-memory allocations fit together.
constexpr size_t kCtSmem = 96 * 1024;
static_assert(kCtACol + kCtStages * kTcAStageCols <= kCtTmemCols, "A stages fit");
static_assert(size_t(kCtRing) * (kCtKBytes + kCtBBytes) <= kCtSmem, "rings fit");
static_assert(kCtRing >= kCtStages, "the ring holds every tile with an A stage");

struct CoilTcParams {
    const float* rec;               // grid-path records [tile][19][32]; the kernel reads the
                                    // k fields (scaled to the trig unit)
    const unsigned char* s_tab;     // weight tiles (scaled per coil), kCtBBytes each
    const unsigned int* bounds;     // per coil: float bits of max |w_r| + |w_i| (its scale)
    int64_t ntiles;
    int splits;
    const float *x, *y, *z;
    int64_t N;
    float* out_r;                   // coil c of split s at out + s * split_stride + c * coil_stride
    float* out_i;
    int64_t coil_stride;
    int64_t split_stride;
    int coils;                      // coils present (the rest of the 8 have weight 0)
    int accumulate;
    unsigned int* err;
};

// A's split, accurate trig: 0 floating with the remainder after converting hi
// back (tc_split8_rt), 1 fixed point, 2 floating with the remainder by a
// mixed-precision FMA (tc_split8) (measured on 8 coils, 128^3 voxels: 2 is
// 4.6 % faster than 1, which is 3 % faster than 0)
#ifndef MRI_CT_SPLIT
#define MRI_CT_SPLIT 2
#endif
// the same for the fast trig paths (2 is 2.7 % faster than 0, which is 1 %
// faster than 1)
#ifndef MRI_CT_SPLIT_FAST
#define MRI_CT_SPLIT_FAST 2
#endif
#ifndef MRI_CT_PHASE2
#define MRI_CT_PHASE2 1   // fast trig: the phase on pairs of samples (.f32x2)
#endif

// v = hi + lo for 8 values of magnitude at most 1 (a sine or cosine), in
// fixed point: hi = v rounded to a multiple of 2^-11 (adding and removing
// 1.5 * 2^12 rounds there), which f16 holds exactly, and lo = v - hi (exact,
// |lo| <= 2^-12) rounded to f16, so that |v - hi - lo| <= 2^-24: the
// absolute error of fp32's own rounding of a unit-modulus value.  All on
// pairs of floats, no conversion back from f16.
__device__ __forceinline__ void ct_split8_unit(const float (&v)[8], uint4& hi, uint4& lo)
{
    const f2 magic = f2_splat(6144.0f);
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const f2 x = f2_pack(v[2 * j], v[2 * j + 1]);
        const f2 hv = f2_sub(f2_add(x, magic), magic);
        const f2 lv = f2_sub(x, hv);
        float a, b;
        f2_unpack(hv, a, b);
        h[j] = pack_f16x2(a, b);
        f2_unpack(lv, a, b);
        l[j] = pack_f16x2(a, b);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

template <int TRIG>
__device__ __forceinline__ void ct_split8(const float (&v)[8], uint4& hi, uint4& lo)
{
    constexpr int kind = TRIG == TRIG_ACCURATE ? MRI_CT_SPLIT : MRI_CT_SPLIT_FAST;
    if constexpr (kind == 1) {
        ct_split8_unit(v, hi, lo);
    } else if constexpr (kind == 2) {
        tc_split8(v, hi, lo);
    } else {
        tc_split8_rt(v, hi, lo);
    }
}

// sin and cos of 8 phases (the records' trig units) into ar (cos) and ai (sin)
template <int TRIG>
__device__ __forceinline__ void ct_phase_trig8(const float (&kx)[8], const float (&ky)[8],
                                               const float (&kz)[8], float x, float y, float z,
                                               float (&ar)[8], float (&ai)[8])
{
    if constexpr (TRIG == TRIG_ACCURATE) {
        // the polynomial on pairs of samples (.f32x2)
        const f2 x2 = f2_splat(x), y2 = f2_splat(y), z2 = f2_splat(z);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const f2 ph = f2_fma(f2_pack(kz[2 * h], kz[2 * h + 1]), z2,
                                 f2_fma(f2_pack(ky[2 * h], ky[2 * h + 1]), y2,
                                        f2_mul(f2_pack(kx[2 * h], kx[2 * h + 1]), x2)));
            f2 sn, cs;
            sincos_half_turns2(ph, sn, cs);
            f2_unpack(sn, ai[2 * h], ai[2 * h + 1]);
            f2_unpack(cs, ar[2 * h], ar[2 * h + 1]);
        }
    } else if constexpr (MRI_CT_PHASE2 != 0) {
        const f2 x2 = f2_splat(x), y2 = f2_splat(y), z2 = f2_splat(z);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const f2 ph = f2_fma(f2_pack(kz[2 * h], kz[2 * h + 1]), z2,
                                 f2_fma(f2_pack(ky[2 * h], ky[2 * h + 1]), y2,
                                        f2_mul(f2_pack(kx[2 * h], kx[2 * h + 1]), x2)));
            float p0, p1;
            f2_unpack(ph, p0, p1);
            table_sincos<TRIG>(p0, ai[2 * h], ar[2 * h]);
            table_sincos<TRIG>(p1, ai[2 * h + 1], ar[2 * h + 1]);
        }
    } else {
#pragma unroll
        for (int s = 0; s < 8; ++s)
            table_sincos<TRIG>(fmaf(kz[s], z, fmaf(ky[s], y, kx[s] * x)), ai[s], ar[s]);
    }
}

// The four MMAs of one K step, D += A_r^hi W_r + A_r^lo W_r + A_i^hi W_i +
// A_i^lo W_i, in one block: a = tensor-memory address of A_r^hi (the other
// parts 16, 32, 48 columns on), wr_lo / wi_lo the low words of the two
// window descriptors (dhi their common high word), acc = 0: the first
// overwrites D.  The issuing thread shares its scheduler with the
// generating warps, so its instructions per MMA are kept to a minimum.
__device__ __forceinline__ void ct_mma4(uint32_t d, uint32_t a, uint32_t wr_lo, uint32_t wi_lo,
                                        uint32_t dhi, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 wr, wi;\n\t.reg .b32 a1, a2, a3;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.eq.b32 q, %6, %6;\n\t"
        "mov.b64 wr, {%2, %4};\n\t"
        "mov.b64 wi, {%3, %4};\n\t"
        "add.u32 a1, %1, 16;\n\t"
        "add.u32 a2, %1, 32;\n\t"
        "add.u32 a3, %1, 48;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], wr, %5, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], wr, %5, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], wi, %5, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], wi, %5, q;\n\t}" ::"r"(d),
        "r"(a), "r"(wr_lo), "r"(wi_lo), "r"(dhi), "r"(idesc), "r"(acc)
        : "memory");
}

template <int TRIG>
__global__ void __launch_bounds__(kCtThreads, 2) coils_tc_kernel(CoilTcParams p)
{
    constexpr int kS = kCtStages;
    constexpr int T = kTcTile;
    constexpr uint32_t ID = umma_idesc_f16(kCtRows, kCtMmaN);   // N = 32
    constexpr int drain_tiles = (TRIG == TRIG_ACCURATE) ? kTcDrainAccurate : kTcDrainFast;
    static_assert(drain_tiles >= kS, "at most one block waits for its fold");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    constexpr int kR = kCtRing;
    unsigned char* const bring = smem_raw;                          // weight tiles
    float* const kring = reinterpret_cast<float*>(smem_raw + kR * kCtBBytes);   // k fields
    __shared__ __align__(8) uint64_t full_bar[kR];    // k fields and weight tile landed
    __shared__ __align__(8) uint64_t ring_free[kR];   // MMAs of the stage's tile done
    __shared__ __align__(8) uint64_t a_full[kS];      // A written by every generator warp
    __shared__ __align__(8) uint64_t mma_bar[kS];     // MMAs of the tile done
    __shared__ __align__(8) uint64_t d_free;          // D folded (warps 0-3)
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    volatile int* const abort_flag = &abort_sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t n0 = int64_t(blockIdx.x) * kCtRows;

    if (warp == 0) tmem_alloc(&tmem_base_sh, kCtTmemCols);
    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < kR; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&ring_free[i], 1);
        }
#pragma unroll
        for (int i = 0; i < kS; ++i) {
            mbar_init(&a_full[i], kCtGenWarps);
            mbar_init(&mma_bar[i], 1);
        }
        mbar_init(&d_free, 4);
        abort_sh = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    if (warp == kCtGenWarps) {
        if (lane == 0) {
            // ---- MMA issue ----
            static_assert(kTcAPartCols == 16 && A_RL == 1 && A_IH == 2 && A_IL == 3,
                          "ct_mma4's part offsets");
            // ring stage 0's descriptor (8-row groups 1024 B apart: every
            // other group of a tile); the other stages are 4096 B further on
            const uint64_t desc0 = umma_desc_kmajor(bring, 128, 1024);
            const uint32_t dlo0 = uint32_t(desc0), dhi = uint32_t(desc0 >> 32);
            int issued = 0;
            int st = 0, rs = 0, tb = 0;               // t % kS, t % kR, t % drain_tiles
            uint32_t ph_s = 0, ph_r = 0, ph_d = 0;    // (t / kS), (t / kR), (t / drain - 1) & 1
            for (int t = 0; t < nt; ++t) {
                bool ok = true;
                // the first MMA of a block overwrites D: the previous block is folded
                if (tb == 0 && t > 0) {
                    ok = ws_wait(&d_free, ph_d, abort_flag);
                    ph_d ^= 1u;
                }
                if (ok) ok = ws_wait(&a_full[st], ph_s, abort_flag);
                if (ok) ok = ws_wait(&full_bar[rs], ph_r, abort_flag);
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t dlo = dlo0 + uint32_t(rs) * uint32_t(kCtBBytes >> 4);
                const uint32_t acol = tmem + kCtACol + uint32_t(st) * kTcAStageCols;
                // K steps of 16 samples: 8 columns of A, 256 B of each weight group
                ct_mma4(tmem, acol, dlo + (512 >> 4), dlo, dhi, ID, tb == 0 ? 0u : 1u);
                ct_mma4(tmem, acol + 8, dlo + ((512 + 256) >> 4), dlo + (256 >> 4), dhi, ID, 1u);
                umma_commit(&mma_bar[st]);
                umma_commit(&ring_free[rs]);
                issued = t + 1;
                if (++st == kS) { st = 0; ph_s ^= 1u; }
                if (++rs == kR) { rs = 0; ph_r ^= 1u; }
                if (++tb == drain_tiles) tb = 0;
            }
            // the MMAs issued finish before tensor memory is released
            if (issued > 0 && !mbar_wait_bounded(&mma_bar[(issued - 1) % kS],
                                                 uint32_t((issued - 1) / kS) & 1u))
                atomicOr(p.err, DEVERR_DRAIN_TIMEOUT);
            if (issued < nt) atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kCtGenWarps + 1) {
        if (lane == 0) {
            // ---- copies: the k fields of record tile u and B tile u ----
            int issued = 0;
            for (int u = 0; u < nt; ++u) {
                const int rs = u % kR;
                if (u >= kR &&
                    !ws_wait(&ring_free[rs], uint32_t((u - kR) / kR) & 1u, abort_flag))
                    break;
                const int64_t tile = t_begin + u;
                if (MRI_DEBUG && (tile < 0 || tile >= p.ntiles)) {
                    // a bad index copies nothing; the consumers' waits report too
                    atomicOr(p.err, DEVERR_BOUNDS);
                    break;
                }
                mbar_arrive_expect_tx(&full_bar[rs], uint32_t(kCtKBytes + kCtBBytes));
                tma_bulk_g2s(kring + rs * 3 * T,
                             reinterpret_cast<const unsigned char*>(p.rec) + tile * kCtRecBytes,
                             uint32_t(kCtKBytes), &full_bar[rs]);
                tma_bulk_g2s(bring + rs * kCtBBytes, p.s_tab + tile * kCtBBytes,
                             uint32_t(kCtBBytes), &full_bar[rs]);
                issued = u + 1;
            }
            // copies still in flight land before shared memory is released
            unsigned int bits = 0;
            for (int u = issued > kR ? issued - kR : 0; u < issued; ++u)
                if (!mbar_wait_bounded(&full_bar[u % kR], uint32_t(u / kR) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            if (issued < nt) bits |= DEVERR_TILE_WAIT_TIMEOUT;
            if (bits) atomicOr(p.err, bits);
        }
        __syncwarp();
    } else {
        // ---- generators: thread = tensor-memory lane ra = voxel n0 + ra ----
        const int ra = 32 * (warp & 3) + lane;
        const int ah = warp >> 2;                     // samples 16 ah .. 16 ah + 15 of a tile
        const uint32_t lanes = uint32_t(32 * (warp & 3)) << 16;
        const int64_t n = n0 + ra;
        const bool in = n < p.N;
        const float vx = in ? p.x[n] : 0.0f, vy = in ? p.y[n] : 0.0f, vz = in ? p.z[n] : 0.0f;
        const bool folds = warp < 4;                  // warps 0-3 hold the running sums
        float R[kCtN];
#pragma unroll
        for (int j = 0; j < kCtN; ++j) R[j] = 0.0f;
        auto fold = [&](bool signal) {
            tc_fence_after_sync();
            float d[32];
            tmem_ld32(tmem + lanes, d);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < kCtN; ++j) R[j] += d[j] + d[kCtN + j];
            if (signal) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_free);
            }
        };

        bool ok = true;
        int pend = -1;   // last tile of a block whose D is not folded yet
        // t % kS, t % kR, t % drain_tiles and the parities (t / kS) & 1,
        // (t / kR) & 1, kept incrementally
        int st = 0, rs = 0, tb = 0;
        uint32_t ph_s = 0, ph_r = 0;
        for (int t = 0; t < nt && ok; ++t) {
            if (folds && pend >= 0) {
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
            // the stage's previous A (tile t - kS) has been read; the k fields have landed
            if (ok && t >= kS) ok = ws_wait(&mma_bar[st], ph_s ^ 1u, abort_flag);
            if (ok) ok = ws_wait(&full_bar[rs], ph_r, abort_flag);
            ok = __all_sync(0xffffffffu, ok);   // the tensor-memory stores are .sync.aligned
            if (!ok) break;
            tc_fence_after_sync();
            const float* kt = kring + rs * 3 * T;
            const uint32_t acol = tmem + lanes + kCtACol + uint32_t(st) * kTcAStageCols;
#pragma unroll
            for (int c = 0; c < kTcAChunks; ++c) {
                const int s0 = 8 * (kTcAChunks * ah + c);
                float kx[8], ky[8], kz[8], ar[8], ai[8];
                tc_load8(kt, 0, s0, kx);
                tc_load8(kt, 1, s0, ky);
                tc_load8(kt, 2, s0, kz);
                ct_phase_trig8<TRIG>(kx, ky, kz, vx, vy, vz, ar, ai);
                // samples s0 .. s0 + 7 = columns s0 / 2 .. of each part
                const uint32_t col = acol + uint32_t(s0 / 2);
                uint4 h, l;
                ct_split8<TRIG>(ar, h, l);
                tmem_st4(col + A_RH * kTcAPartCols, h);
                tmem_st4(col + A_RL * kTcAPartCols, l);
                ct_split8<TRIG>(ai, h, l);
                tmem_st4(col + A_IH * kTcAPartCols, h);
                tmem_st4(col + A_IL * kTcAPartCols, l);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[st]);
            if (tb == drain_tiles - 1 && t + 1 < nt) pend = t;
            if (++st == kS) {
                st = 0;
                ph_s ^= 1u;
            }
            if (++rs == kR) {
                rs = 0;
                ph_r ^= 1u;
            }
            if (++tb == drain_tiles) tb = 0;
        }
        if (folds) {
            // the block still waiting for its fold, then the last block
            if (ok && pend >= 0) {
                ok = __all_sync(0xffffffffu, ws_wait(&mma_bar[pend % kS],
                                                     uint32_t(pend / kS) & 1u, abort_flag));
                if (ok) fold(true);
            }
            if (ok && nt > 0) {
                ok = __all_sync(0xffffffffu, ws_wait(&mma_bar[(nt - 1) % kS],
                                                     uint32_t((nt - 1) / kS) & 1u, abort_flag));
                if (ok) fold(false);
            }
            if (!ok) {
                if (lane == 0) atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
            } else if (nt > 0 && in) {
                float* const out_r = p.out_r + split * p.split_stride;
                float* const out_i = p.out_i + split * p.split_stride;
#pragma unroll
                for (int c = 0; c < kCtCoils; ++c) {
                    if (c < p.coils) {
                        const float inv_scale = exp2_int(-tc_scale_exp(p.bounds[c]));
                        float* rp = out_r + c * p.coil_stride + n;
                        float* ip = out_i + c * p.coil_stride + n;
                        *rp = fmaf(R[c], inv_scale, p.accumulate ? *rp : 0.0f);
                        *ip = fmaf(R[kCtCoils + c], inv_scale, p.accumulate ? *ip : 0.0f);
                    }
                }
            }
        } else if (!ok && lane == 0) {
            atomicOr(p.err, DEVERR_TILE_WAIT_TIMEOUT);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, kCtTmemCols);
}

}  // namespace mri
