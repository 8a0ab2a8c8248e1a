// gather_pair.cuh -- the single-weight F^H D / Q gather on pairs of floats.
//
// Method (section 17.3, the register-promoted gather of Fig. 17.11):
//   FhD[n] = sum_m Mu[m] e^{+i 2 pi (kx[m] x[n] + ky[m] y[n] + kz[m] z[n])},
//   Q[n]   = the same with the real weight |Phi[m]|^2.
//
// The work per voxel-sample pair is a few floating-point operations and one
// sin/cos, so the kernel is bound by how many instructions the SM can issue
// (four warp instructions per clock) and by the SFU.  sm_103a executes
// add / mul / fma on PAIRS of floats (.f32x2) in one instruction, each half
// rounded exactly as the scalar instruction would be.  This kernel keeps the
// V voxels of a thread as V/2 packed pairs, so the phase, the polynomial trig
// and the complex multiply-accumulate of two voxels cost one instruction each:
//   * the phase t = kx x + ky y + kz z: 3 packed instructions per two pairs;
//   * accurate trig: reduction to half turns f = u - rint(u) in [-1/2, 1/2],
//     minimax polynomials of pi f (SinCosHalf, gen_sincospi.py), then the sign
//     (-1)^rint(u) -- all packed except the sign flip (a shift and two xors
//     per voxel on the integer pipe);
//   * fast trig: the phase in radians unpacked into the SFU's __sincosf;
//   * the multiply-accumulate: 4 packed fmas (Q: 2) per two pairs.
// To feed packed operands without moves, the tile records hold every sample
// value twice (f, f): one 16-byte shared-memory load gives two samples, each
// already a packed pair.  F^H D keeps -iMu as a field of its own so that the
// multiply-accumulate needs no negation.  The tiles stream through a
// kStages-deep ring filled by 1-D TMA bulk copies (as in gather.cuh), every
// wait is bounded, partial sums restart every tile (blocked summation).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "gather.cuh"

namespace mri {

// Records of one tile: field f of sample j at [f][2 j] and [f][2 j + 1].
//   F^H D: kx ky kz rMu iMu -iMu        Q: kx ky kz w
template <bool REALW>
struct PairRec {
    static constexpr int F = REALW ? 4 : 6;
    static constexpr int TILE_FLOATS = F * 2 * kTile;
    static constexpr uint32_t TILE_BYTES = TILE_FLOATS * 4u;
};

#ifndef MRI_PAIR_V
#define MRI_PAIR_V 8
#endif
// Accurate trig in quarter turns (fewer FMA-pipe operations, a quadrant
// rotation on the integer pipe) instead of half turns.
#ifndef MRI_PAIR_QUARTER
#define MRI_PAIR_QUARTER 0
#endif
// Fast trig: of the V / 2 voxel pairs of a thread, the last NP_FP32 take the
// polynomial on the FMA pipe instead of the SFU (F^H D and Q separately).
#ifndef MRI_PAIR_NP_FP32
#define MRI_PAIR_NP_FP32 0
#endif
#ifndef MRI_PAIR_NP_FP32_Q
#define MRI_PAIR_NP_FP32_Q 1
#endif

struct PairShape {
    static constexpr int THREADS = 256;
    static constexpr int V = MRI_PAIR_V;            // voxels per thread (V / 2 packed pairs)
    static constexpr int MIN_BLOCKS = 2;
    static constexpr int VOXELS_PER_CTA = THREADS * V;
    static_assert(V % 2 == 0, "voxels come in pairs");
    template <bool REALW>
    __host__ __device__ static constexpr size_t smem()
    {
        return size_t(kStages) * PairRec<REALW>::TILE_BYTES;
    }
    // voxel pairs whose fast-path trig runs on the FMA pipe
    template <bool REALW>
    __host__ __device__ static constexpr int np_fp32()
    {
        return REALW ? MRI_PAIR_NP_FP32_Q : MRI_PAIR_NP_FP32;
    }
    static_assert(MRI_PAIR_NP_FP32 <= V / 2 && MRI_PAIR_NP_FP32_Q <= V / 2, "pairs per thread");
};

// Units of the phase the records hold (the factor k is multiplied by): half
// turns for the polynomial, radians for the SFU, turns for the SFU after an
// explicit reduction.
__host__ __device__ constexpr float pair_kscale(int trig)
{
    return trig == TRIG_ACCURATE ? (MRI_PAIR_QUARTER ? 4.0f : 2.0f)
           : trig == TRIG_FAST   ? 6.28318530717958647692f
                                 : 1.0f;
}

// cmpMu and the duplicated record layout.  One thread per sample slot
// (zero-padded to whole tiles: a padded sample has k = 0 and weight 0).
template <bool REALW>
__global__ void __launch_bounds__(256) prep_pair_records_kernel(PrepParams p)
{
    using R = PairRec<REALW>;
    const int64_t total = p.ntiles * kTile;
    for (int64_t m = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; m < total;
         m += int64_t(gridDim.x) * blockDim.x) {
        const int64_t tile = m / kTile;
        const int j = int(m - tile * kTile);
        float f[R::F];
#pragma unroll
        for (int i = 0; i < R::F; ++i) f[i] = 0.0f;
        if (m < p.M) {
            f[0] = p.kx[m] * p.kscale;
            f[1] = p.ky[m] * p.kscale;
            f[2] = p.kz[m] * p.kscale;
            const float rp = p.unit_phi ? 1.0f : p.rPhi[m];
            const float ip = p.unit_phi ? 0.0f : p.iPhi[m];
            if constexpr (REALW) {
                f[3] = fmaf(ip, ip, rp * rp);                       // |Phi|^2
            } else {
                const float rd = p.rD[p.b0 * p.M + m];
                const float id = p.iD[p.b0 * p.M + m];
                f[3] = fmaf(ip, id, rp * rd);                       // Re conj(Phi) D
                f[4] = fmaf(-ip, rd, rp * id);                      // Im conj(Phi) D
                f[5] = -f[4];
            }
        }
        float2* base = reinterpret_cast<float2*>(p.rec + tile * R::TILE_FLOATS) + j;
#pragma unroll
        for (int i = 0; i < R::F; ++i) base[i * kTile] = make_float2(f[i], f[i]);
    }
}

// sin and cos of (pi/2) u for a pair of phases u in quarter turns: the
// reduction and polynomials packed (SinCosQuarter), then per half the
// rotation by q quarter turns (odd q swaps sin and cos; the signs follow bits
// 0 and 1 of q) on the integer pipe.
__device__ __forceinline__ void sincos_quarter_turns2(f2 u, f2& s, f2& c)
{
    using Coef = SinCosQuarter;
    const f2 magic = f2_splat(12582912.0f);
    const f2 v = f2_add(u, magic);
    const f2 f = f2_sub(u, f2_sub(v, magic));
    const f2 f2sq = f2_mul(f, f);
    f2 p = f2_splat(Coef::P(Coef::P_TERMS - 1));
#pragma unroll
    for (int i = Coef::P_TERMS - 2; i >= 0; --i) p = f2_fma(p, f2sq, f2_splat(Coef::P(i)));
    f2 q = f2_splat(Coef::Q(Coef::Q_TERMS - 1));
#pragma unroll
    for (int i = Coef::Q_TERMS - 2; i >= 0; --i) q = f2_fma(q, f2sq, f2_splat(Coef::Q(i)));
    const f2 sf = f2_mul(f, p);
    uint32_t vh[2], sh[2], ch[2], so[2], co[2];
    f2_halves(v, vh[0], vh[1]);
    f2_halves(sf, sh[0], sh[1]);
    f2_halves(q, ch[0], ch[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const bool odd = (vh[h] & 1u) != 0u;
        const uint32_t s_sel = odd ? ch[h] : sh[h];
        const uint32_t c_sel = odd ? sh[h] : ch[h];
        const uint32_t m1 = vh[h] << 30, m0 = vh[h] << 31;
        so[h] = s_sel ^ (m1 & 0x80000000u);
        co[h] = c_sel ^ ((m1 ^ m0) & 0x80000000u);
    }
    s = f2_from_halves(so[0], so[1]);
    c = f2_from_halves(co[0], co[1]);
}

// ON_FP32: a fast-path voxel pair that takes the polynomial (the records hold
// radians; 1/pi turns them into half turns).
template <int TRIG, bool ON_FP32 = false>
__device__ __forceinline__ void phase_sincos2(f2 ph, f2& s, f2& c)
{
    if (TRIG == TRIG_ACCURATE) {
        if (MRI_PAIR_QUARTER)
            sincos_quarter_turns2(ph, s, c);          // records hold 4k: quarter turns
        else
            sincos_half_turns2(ph, s, c);             // records hold 2k: half turns
    } else if (TRIG == TRIG_FAST && ON_FP32) {
        sincos_half_turns2(f2_mul(ph, f2_splat(0.318309886183790671538f)), s, c);
    } else {
        float a, b;
        f2_unpack(ph, a, b);
        if (TRIG == TRIG_FAST_RR) {
            // records hold k in turns; subtract the nearest integer exactly
            const f2 magic = f2_splat(12582912.0f);
            f2 r = f2_sub(ph, f2_sub(f2_add(ph, magic), magic));
            r = f2_mul(r, f2_splat(6.28318530717958647692f));
            f2_unpack(r, a, b);
        }
        float sa, ca, sb, cb;                         // radians on the SFU
        __sincosf(a, &sa, &ca);
        __sincosf(b, &sb, &cb);
        s = f2_pack(sa, sb);
        c = f2_pack(ca, cb);
    }
}

template <bool REALW, int TRIG>
__global__ void __launch_bounds__(PairShape::THREADS, PairShape::MIN_BLOCKS)
    gather_pair_kernel(GatherParams p)
{
    using R = PairRec<REALW>;
    constexpr int V = PairShape::V;
    constexpr int VP = V / 2;
    constexpr int T = PairShape::THREADS;
    constexpr int FS = 2 * kTile;                     // floats between fields of a tile

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* const ring = reinterpret_cast<float*>(smem_raw);
    __shared__ __align__(8) uint64_t full_bar[kStages];

    const int tid = threadIdx.x;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t n0 = int64_t(blockIdx.x) * PairShape::VOXELS_PER_CTA + tid;

    // voxels n0 + v T, v < V, as V / 2 packed pairs (v = 2 i, 2 i + 1)
    f2 x2[VP], y2[VP], z2[VP];
#pragma unroll
    for (int i = 0; i < VP; ++i) {
        float c[2][3];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + int64_t(2 * i + h) * T;
            const bool in = n < p.N;
            c[h][0] = in ? p.x[n] : 0.0f;
            c[h][1] = in ? p.y[n] : 0.0f;
            c[h][2] = in ? p.z[n] : 0.0f;
        }
        x2[i] = f2_pack(c[0][0], c[1][0]);
        y2[i] = f2_pack(c[0][1], c[1][1]);
        z2[i] = f2_pack(c[0][2], c[1][2]);
    }

    float* const out_r = p.out_r + split * p.split_stride;
    float* const out_i = p.out_i + split * p.split_stride;

    f2 run_r[VP], run_i[VP];
#pragma unroll
    for (int i = 0; i < VP; ++i) run_r[i] = run_i[i] = f2_splat(0.0f);

    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&full_bar[st], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int st = 0; st < kStages && st < nt; ++st) {
            tma_load_checked(ring + st * R::TILE_FLOATS, p.rec, t_begin + st, p.ntiles,
                             R::TILE_BYTES, &full_bar[st], p.err);
        }
    }

    int failed_at = -1;
    for (int t = 0; t < nt; ++t) {
        const int st = t % kStages;
        const uint32_t parity = uint32_t(t / kStages) & 1u;
        const bool ok = mbar_wait_bounded(&full_bar[st], parity);
        const float* tile = ring + st * R::TILE_FLOATS;

        f2 pr[VP], pi[VP];
#pragma unroll
        for (int i = 0; i < VP; ++i) pr[i] = pi[i] = f2_splat(0.0f);

        if (ok) {
            // two samples per step: one 16-byte broadcast load per field
#pragma unroll 1
            for (int j = 0; j < kTile; j += 2) {
                f2 f[R::F][2];
#pragma unroll
                for (int k = 0; k < R::F; ++k) {
                    const ulonglong2 d =
                        *reinterpret_cast<const ulonglong2*>(tile + k * FS + 2 * j);
                    f[k][0] = d.x;
                    f[k][1] = d.y;
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
#pragma unroll
                    for (int i = 0; i < VP; ++i) {
                        const f2 ph =
                            f2_fma(f[2][q], z2[i], f2_fma(f[1][q], y2[i], f2_mul(f[0][q], x2[i])));
                        f2 sn, cs;
                        if (i >= VP - PairShape::np_fp32<REALW>())
                            phase_sincos2<TRIG, true>(ph, sn, cs);
                        else
                            phase_sincos2<TRIG, false>(ph, sn, cs);
                        if constexpr (REALW) {
                            pr[i] = f2_fma(f[3][q], cs, pr[i]);
                            pi[i] = f2_fma(f[3][q], sn, pi[i]);
                        } else {
                            // (rMu + i iMu)(cos + i sin)
                            pr[i] = f2_fma(f[3][q], cs, pr[i]);
                            pr[i] = f2_fma(f[5][q], sn, pr[i]);
                            pi[i] = f2_fma(f[4][q], cs, pi[i]);
                            pi[i] = f2_fma(f[3][q], sn, pi[i]);
                        }
                    }
                }
            }
        }

        // every thread is done with this stage (and agrees on success)
        if (__syncthreads_or(!ok)) {
            failed_at = t;
            break;
        }

        // fold the tile's partial sums into the running sums
#pragma unroll
        for (int i = 0; i < VP; ++i) {
            run_r[i] = f2_add(run_r[i], pr[i]);
            run_i[i] = f2_add(run_i[i], pi[i]);
        }

        // refill the stage just released with the tile kStages ahead
        if (tid == 0 && t + kStages < nt) {
            fence_proxy_async_smem();
            tma_load_checked(ring + st * R::TILE_FLOATS, p.rec, t_begin + t + kStages, p.ntiles,
                             R::TILE_BYTES, &full_bar[st], p.err);
        }
    }

    if (failed_at >= 0) {
        // Report, then let every copy still in flight land before the CTA's
        // shared memory is released.
        if (tid == 0) {
            unsigned int bits = DEVERR_TILE_WAIT_TIMEOUT;
            const int last = (failed_at + kStages < nt) ? failed_at + kStages : nt;
            for (int u = failed_at; u < last; ++u)
                if (!mbar_wait_bounded(&full_bar[u % kStages], uint32_t(u / kStages) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            atomicOr(p.err, bits);
        }
        __syncthreads();
        return;
    }

#pragma unroll
    for (int i = 0; i < VP; ++i) {
        float r[2], im[2];
        f2_unpack(run_r[i], r[0], r[1]);
        f2_unpack(run_i[i], im[0], im[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + int64_t(2 * i + h) * T;
            if (n < p.N) {
                float a = r[h], b = im[h];
                if (p.accumulate) {
                    a = out_r[n] + a;
                    b = out_i[n] + b;
                }
                out_r[n] = a;
                out_i[n] = b;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Coil groups (batched F^H D): one sin/cos per voxel-sample pair shared by BC
// coils, 4 packed fmas per coil and voxel pair.  Records: per sample, 2 + BC
// 16-byte entries, (kx kx ky ky), (kz kz 0 0), then (rMu_b rMu_b iMu_b iMu_b)
// for each coil: one broadcast LDS.128 per coil gives both of its weights as
// packed operands.  -sin is formed once per voxel pair and sample and shared
// by the coils.  The tile's partial sums are added into the outputs (or split
// partials) in global memory once per tile, so the register file holds only
// the partials of the tile.
// ---------------------------------------------------------------------------
#ifndef MRI_COIL_PAIRS
#define MRI_COIL_PAIRS 2
#endif
// samples per step of the sample loop (measured: two help the accurate
// path, 4,612 -> 4,687 Gpair-coils/s, and hurt the fast one, 6,360 -> 5,698)
#ifndef MRI_COIL_UNROLL_ACCURATE
#define MRI_COIL_UNROLL_ACCURATE 2
#endif
#ifndef MRI_COIL_UNROLL_FAST
#define MRI_COIL_UNROLL_FAST 1
#endif

template <int BC>
struct PairCoilRec {
    static constexpr int Q4 = 2 + BC;                 // 16-byte entries per sample
    static constexpr int TILE_FLOATS = kTile * 4 * Q4;
    static constexpr uint32_t TILE_BYTES = TILE_FLOATS * 4u;
};

template <int BC>
struct PairCoilShape {
    static constexpr int THREADS = 256;
    static constexpr int VP = MRI_COIL_PAIRS;        // voxel pairs per thread
    static constexpr int V = 2 * VP;
    static constexpr int MIN_BLOCKS = 2;
    static constexpr int VOXELS_PER_CTA = THREADS * V;
    // two CTAs per SM: eight coils (40 KB tiles) keep two stages
    static constexpr int STAGES = BC >= 8 ? 2 : kStages;
    static constexpr size_t SMEM = size_t(STAGES) * PairCoilRec<BC>::TILE_BYTES;
};

template <int BC>
__global__ void __launch_bounds__(256) prep_pair_coil_records_kernel(PrepParams p)
{
    using R = PairCoilRec<BC>;
    const int64_t total = p.ntiles * kTile;
    for (int64_t m = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; m < total;
         m += int64_t(gridDim.x) * blockDim.x) {
        float4 e[R::Q4];
#pragma unroll
        for (int i = 0; i < R::Q4; ++i) e[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < p.M) {
            const float kx = p.kx[m] * p.kscale, ky = p.ky[m] * p.kscale;
            const float kz = p.kz[m] * p.kscale;
            e[0] = make_float4(kx, kx, ky, ky);
            e[1] = make_float4(kz, kz, 0.f, 0.f);
            const float rp = p.rPhi[m], ip = p.iPhi[m];
#pragma unroll
            for (int b = 0; b < BC; ++b) {
                if (b < p.coils_valid) {
                    const float rd = p.rD[(p.b0 + b) * p.M + m];
                    const float id = p.iD[(p.b0 + b) * p.M + m];
                    const float rm = fmaf(ip, id, rp * rd);         // Re conj(Phi) D
                    const float im = fmaf(-ip, rd, rp * id);        // Im conj(Phi) D
                    e[2 + b] = make_float4(rm, rm, im, im);
                }
            }
        }
        float4* dst = reinterpret_cast<float4*>(p.rec) + m * R::Q4;   // tiles are contiguous
#pragma unroll
        for (int i = 0; i < R::Q4; ++i) dst[i] = e[i];
    }
}

template <int BC, int TRIG>
__global__ void __launch_bounds__(256, 2) gather_pair_coils_kernel(GatherParams p)
{
    using R = PairCoilRec<BC>;
    using S = PairCoilShape<BC>;
    constexpr int VP = S::VP;
    constexpr int T = S::THREADS;
    constexpr int KS = S::STAGES;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* const ring = reinterpret_cast<float*>(smem_raw);
    __shared__ __align__(8) uint64_t full_bar[KS];

    const int tid = threadIdx.x;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t n0 = int64_t(blockIdx.x) * S::VOXELS_PER_CTA + tid;

    f2 x2[VP], y2[VP], z2[VP];
#pragma unroll
    for (int i = 0; i < VP; ++i) {
        float c[2][3];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + int64_t(2 * i + h) * T;
            const bool in = n < p.N;
            c[h][0] = in ? p.x[n] : 0.0f;
            c[h][1] = in ? p.y[n] : 0.0f;
            c[h][2] = in ? p.z[n] : 0.0f;
        }
        x2[i] = f2_pack(c[0][0], c[1][0]);
        y2[i] = f2_pack(c[0][1], c[1][1]);
        z2[i] = f2_pack(c[0][2], c[1][2]);
    }
    float* const out_r = p.out_r + split * p.split_stride;
    float* const out_i = p.out_i + split * p.split_stride;

    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < KS; ++st) mbar_init(&full_bar[st], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int st = 0; st < KS && st < nt; ++st)
            tma_load_checked(ring + st * R::TILE_FLOATS, p.rec, t_begin + st, p.ntiles,
                             R::TILE_BYTES, &full_bar[st], p.err);
    }

    int failed_at = -1;
    for (int t = 0; t < nt; ++t) {
        const int st = t % KS;
        const bool ok = mbar_wait_bounded(&full_bar[st], uint32_t(t / KS) & 1u);
        const float* tile = ring + st * R::TILE_FLOATS;

        f2 pr[VP][BC], pi[VP][BC];
#pragma unroll
        for (int i = 0; i < VP; ++i)
#pragma unroll
            for (int b = 0; b < BC; ++b) pr[i][b] = pi[i][b] = f2_splat(0.0f);

        if (ok) {
            constexpr int kUnroll =
                TRIG == TRIG_ACCURATE ? MRI_COIL_UNROLL_ACCURATE : MRI_COIL_UNROLL_FAST;
#pragma unroll kUnroll
            for (int j = 0; j < kTile; ++j) {
                const ulonglong2* rec = reinterpret_cast<const ulonglong2*>(tile) + j * R::Q4;
                const ulonglong2 kxy = rec[0], kzz = rec[1];
                const f2 kx = kxy.x, ky = kxy.y, kz = kzz.x;
                f2 sn[VP], cs[VP], ns[VP];
#pragma unroll
                for (int i = 0; i < VP; ++i) {
                    const f2 ph = f2_fma(kz, z2[i], f2_fma(ky, y2[i], f2_mul(kx, x2[i])));
                    phase_sincos2<TRIG>(ph, sn[i], cs[i]);
                    ns[i] = f2_mul(sn[i], f2_splat(-1.0f));
                }
#pragma unroll
                for (int b = 0; b < BC; ++b) {
                    const ulonglong2 w = rec[2 + b];
                    const f2 rm = w.x, im = w.y;
#pragma unroll
                    for (int i = 0; i < VP; ++i) {
                        // (rMu + i iMu)(cos + i sin)
                        pr[i][b] = f2_fma(rm, cs[i], pr[i][b]);
                        pr[i][b] = f2_fma(im, ns[i], pr[i][b]);
                        pi[i][b] = f2_fma(im, cs[i], pi[i][b]);
                        pi[i][b] = f2_fma(rm, sn[i], pi[i][b]);
                    }
                }
            }
        }

        if (__syncthreads_or(!ok)) {
            failed_at = t;
            break;
        }

        // the tile's partial sums into the outputs
        const bool first = (t == 0) && !p.accumulate;
#pragma unroll
        for (int i = 0; i < VP; ++i) {
#pragma unroll
            for (int b = 0; b < BC; ++b) {
                float r[2], im[2];
                f2_unpack(pr[i][b], r[0], r[1]);
                f2_unpack(pi[i][b], im[0], im[1]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t n = n0 + int64_t(2 * i + h) * T;
                    if (n < p.N) {
                        float* rp = out_r + b * p.coil_stride + n;
                        float* ip = out_i + b * p.coil_stride + n;
                        if (first) {
                            *rp = r[h];
                            *ip = im[h];
                        } else {
                            *rp += r[h];
                            *ip += im[h];
                        }
                    }
                }
            }
        }

        if (tid == 0 && t + KS < nt) {
            fence_proxy_async_smem();
            tma_load_checked(ring + st * R::TILE_FLOATS, p.rec, t_begin + t + KS, p.ntiles,
                             R::TILE_BYTES, &full_bar[st], p.err);
        }
    }

    if (failed_at >= 0) {
        if (tid == 0) {
            unsigned int bits = DEVERR_TILE_WAIT_TIMEOUT;
            const int last = (failed_at + KS < nt) ? failed_at + KS : nt;
            for (int u = failed_at; u < last; ++u)
                if (!mbar_wait_bounded(&full_bar[u % KS], uint32_t(u / KS) & 1u))
                    bits |= DEVERR_DRAIN_TIMEOUT;
            atomicOr(p.err, bits);
        }
        __syncthreads();
    }
}

}  // namespace mri
