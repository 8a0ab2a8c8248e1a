// gather.cuh -- the F^H D / Q gather kernels for sm_103a.
//
// Method (pages on iterative non-Cartesian MRI reconstruction, section 17.3):
//   cmpMu (Fig. 17.7):      Mu[m] = conj(Phi[m]) * D[m]
//   cmpFhD gather (Figs. 17.10/17.11, register-promoted):
//       FhD[n] = sum_m Mu[m] * e^{+i 2 pi (kx[m] x[n] + ky[m] y[n] + kz[m] z[n])}
//   Q (section 17.2, "same core structure"): the same gather with weight |Phi|^2.
//
// GB300 design:
//   * A prep kernel writes the trajectory and weights into tile-major records
//     (kTile samples per tile, zero-padded to whole tiles; padded samples have
//     k = 0 and weight 0 and so add exactly +0).  It fuses cmpMu and folds the
//     trig path's phase scale into k.
//   * The gather kernel keeps V voxels per thread in registers (the register
//     promotion of Fig. 17.11, widened to V voxels as the chapter suggests for
//     large grids), and streams record tiles through a kStages-deep ring in
//     shared memory with 1-D TMA bulk copies completing on mbarriers.  Every
//     warp reads each sample as a broadcast (the access pattern that made the
//     chapter put k-space in constant memory).
//   * Partial sums restart at every tile and are folded into the running sum
//     at tile end (blocked summation), which keeps fp32 summation error well
//     under the trig and phase error at M ~ 1e6.
//   * A grid dimension splits the samples across CTAs when the voxel count
//     alone would leave SMs idle; a deterministic reduction kernel then adds
//     the splits in a fixed order.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "sincospi_coeffs.h"

namespace mri {

enum TrigMode : int {
    TRIG_ACCURATE = 0,  // minimax polynomials on the FP32 pipe, phase in quarter turns
    TRIG_FAST = 1,      // MUFU on the phase in radians; a fixed share of voxels on the FP32 pipe
    TRIG_FAST_RR = 2,   // MUFU after explicit reduction of the phase to [-1/2, 1/2] turn
};

// Voxels per thread whose fast-path trig runs on the FP32 pipe (see Shape).
#ifndef MRI_NP_FP32_FHD
#define MRI_NP_FP32_FHD 0
#endif
#ifndef MRI_NP_FP32_Q
#define MRI_NP_FP32_Q 1
#endif

constexpr int kTile = 256;   // samples per k-tile
constexpr int kStages = 3;   // tiles resident per CTA

// Record layout of one tile.
//   single weight (F^H D: BC = 1, Q: REALW): structure of arrays [F][kTile]
//       F^H D: kx ky kz rMu iMu     Q: kx ky kz w
//   coil groups (BC > 1): array of records [kTile][F4]
//       kx ky kz rMu_0..rMu_{BC-1} iMu_0..iMu_{BC-1} (zero padding to F4)
//   SOA forces the structure-of-arrays layout for coil groups too
//       kx ky kz rMu_0..rMu_{BC-1} iMu_0..iMu_{BC-1}, each [TILE]
template <int BC, bool REALW, int TILE = kTile, bool SOA = false>
struct Rec {
    static_assert(!REALW || BC == 1, "a real weight has one coil");
    static constexpr int F = REALW ? 4 : 3 + 2 * BC;
    static constexpr bool AOS = BC > 1 && !SOA;
    static constexpr int F4 = (F + 3) / 4 * 4;
    static constexpr int STRIDE = AOS ? F4 : F;
    static constexpr int TILE_FLOATS = TILE * STRIDE;
    static constexpr uint32_t TILE_BYTES = TILE_FLOATS * 4u;
};

// Launch shape of the coil-group kernels (BC >= 4), overridable for sweeps.
#ifndef MRI_COIL_V
#define MRI_COIL_V 2
#endif
#ifndef MRI_COIL_THREADS
#define MRI_COIL_THREADS 256
#endif
#ifndef MRI_COIL_UNROLL
#define MRI_COIL_UNROLL 1
#endif
constexpr int kCoilUnroll = MRI_COIL_UNROLL;

// Per-kernel launch shape.
template <int BC, bool REALW>
struct Shape {
    static constexpr int THREADS = (BC >= 4) ? MRI_COIL_THREADS : 256;
    static constexpr int V = (BC >= 4) ? MRI_COIL_V : 8;   // voxels per thread
    static constexpr int MIN_BLOCKS = 512 / THREADS;
    static constexpr int VOXELS_PER_CTA = THREADS * V;
    // Fast trig: of the V voxels a thread holds, the last NP_FP32 take their
    // sin/cos from the quarter-turn polynomial on the FP32 pipe instead of the
    // SFU.  The SFU delivers 16 results per SM per clock and binds F^H D and
    // Q, while issue slots are left over (59 % issue-active on F^H D).  On the
    // 128^3 workloads one voxel in 8 on the FP32 pipe makes Q 6 % faster and
    // F^H D 2 % slower (it spends 4 FFMA per pair on the multiply-accumulate
    // against Q's 2, so fewer slots are left); coil groups are FP32-bound and
    // keep every pair on the SFU.
    static constexpr int NP_FP32 = REALW ? MRI_NP_FP32_Q : (BC == 1 ? MRI_NP_FP32_FHD : 0);
    static constexpr size_t SMEM = size_t(kStages) * Rec<BC, REALW>::TILE_BYTES;
};

struct PrepParams {
    const float *kx, *ky, *kz;
    const float *rPhi, *iPhi;
    const float *rD, *iD;   // coil-major [B][M]; coil b0 .. b0+BC-1 used
    int64_t M;
    int64_t b0;
    int64_t ntiles;
    float kscale;           // 4 (quarter turns), 2*pi (radians) or 1 (turns)
    float* rec;
    // Optional: raised by atomicMax to the float bits of the largest
    // |w_r| + |w_i| over samples and coils; the caller zeroes it first.
    unsigned int* wbound = nullptr;
    // Coils b0 .. b0 + coils_valid - 1 exist; the rest of a group get weight 0.
    int coils_valid = 1 << 30;
    // Phi == 1 (rPhi, iPhi unused): the weight is D itself (the forward model)
    bool unit_phi = false;
};

struct GatherParams {
    const float* rec;
    int64_t ntiles;
    int splits;
    const float *x, *y, *z;
    int64_t N;
    // Output of coil b of split s: out_r + s*split_stride + b*coil_stride (+n),
    // likewise out_i.  With one split these are the caller's arrays.
    float* out_r;
    float* out_i;
    int64_t coil_stride;
    int64_t split_stride;
    int accumulate;         // add into the existing outputs (one split only)
    unsigned int* err;      // device error word
};

// ---------------------------------------------------------------------------
// prep: cmpMu fused with the tile-record layout
// ---------------------------------------------------------------------------
template <int BC, bool REALW, int TILE = kTile, bool SOA = false>
__global__ void __launch_bounds__(256) prep_records_kernel(PrepParams p)
{
    using R = Rec<BC, REALW, TILE, SOA>;
    const int64_t total = p.ntiles * TILE;
    float wmax = 0.0f;
    for (int64_t m = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; m < total;
         m += int64_t(gridDim.x) * blockDim.x) {
        const int64_t tile = m / TILE;
        const int j = int(m - tile * TILE);
        float* base = p.rec + tile * R::TILE_FLOATS;
        float f[R::F4];
#pragma unroll
        for (int i = 0; i < R::F4; ++i) f[i] = 0.0f;
        if (m < p.M) {
            f[0] = p.kx[m] * p.kscale;
            f[1] = p.ky[m] * p.kscale;
            f[2] = p.kz[m] * p.kscale;
            const float rp = p.unit_phi ? 1.0f : p.rPhi[m];
            const float ip = p.unit_phi ? 0.0f : p.iPhi[m];
            if (REALW) {
                f[3] = fmaf(ip, ip, rp * rp);                       // |Phi|^2
            } else {
#pragma unroll
                for (int b = 0; b < BC; ++b) {
                    if (b < p.coils_valid) {
                        const float rd = p.rD[(p.b0 + b) * p.M + m];
                        const float id = p.iD[(p.b0 + b) * p.M + m];
                        f[3 + b] = fmaf(ip, id, rp * rd);           // Re conj(Phi) D
                        f[3 + BC + b] = fmaf(-ip, rd, rp * id);     // Im conj(Phi) D
                    }
                }
            }
            if constexpr (REALW) {
                wmax = fmaxf(wmax, fabsf(f[3]));
            } else {
#pragma unroll
                for (int b = 0; b < BC; ++b) wmax = fmaxf(wmax, fabsf(f[3 + b]) + fabsf(f[3 + BC + b]));
            }
        }
        if (R::AOS) {
            float4* dst = reinterpret_cast<float4*>(base + j * R::F4);
#pragma unroll
            for (int i = 0; i < R::F4 / 4; ++i)
                dst[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < R::F; ++i) base[i * TILE + j] = f[i];
        }
    }
    if (p.wbound != nullptr) {
        // non-negative floats order like their bit patterns (a NaN sorts last)
        const unsigned int w = __reduce_max_sync(0xffffffffu, __float_as_uint(wmax));
        if ((threadIdx.x & 31) == 0 && w != 0u) atomicMax(p.wbound, w);
    }
}

// ---------------------------------------------------------------------------
// trig on one phase value
// ---------------------------------------------------------------------------

// sin and cos of (pi/2) u for u in quarter turns (|u| < 2^22), on the FP32
// pipe: exact reduction q = rint(u), f = u - q in [-1/2, 1/2] (adding and
// removing 1.5 * 2^23 rounds to an integer and leaves q in the low mantissa
// bits of the sum), minimax polynomials for sin and cos of (pi/2) f
// (coefficients from gen_sincospi.py), then a rotation by q quarter turns:
// odd q swaps sin and cos; sin changes sign when bit 1 of q is set, cos when
// bit 1 of q + 1 is.
__device__ __forceinline__ void sincos_quarter_turns(float u, float& s, float& c)
{
    using Coef = SinCosQuarter;
    const float v = u + 12582912.0f;
    const float f = u - (v - 12582912.0f);
    const float f2 = f * f;
    float p = Coef::P(Coef::P_TERMS - 1);
#pragma unroll
    for (int i = Coef::P_TERMS - 2; i >= 0; --i) p = fmaf(p, f2, Coef::P(i));
    float q = Coef::Q(Coef::Q_TERMS - 1);
#pragma unroll
    for (int i = Coef::Q_TERMS - 2; i >= 0; --i) q = fmaf(q, f2, Coef::Q(i));
    const float sf = f * p;
    const unsigned qi = __float_as_uint(v);
    const bool odd = (qi & 1u) != 0u;
    const float s_sel = odd ? q : sf;
    const float c_sel = odd ? sf : q;
    const unsigned m1 = qi << 30;   // bit 31 = bit 1 of q
    const unsigned m0 = qi << 31;   // bit 31 = bit 0 of q
    s = __uint_as_float(__float_as_uint(s_sel) ^ (m1 & 0x80000000u));
    c = __uint_as_float(__float_as_uint(c_sel) ^ ((m1 ^ m0) & 0x80000000u));
}

// `on_fp32` is a compile-time constant after unrolling (the voxel slot).
template <int TRIG>
__device__ __forceinline__ void phase_sincos(float ph, bool on_fp32, float& s, float& c)
{
    if (TRIG == TRIG_ACCURATE) {
        // records hold 4k, so ph is the phase in quarter turns
        sincos_quarter_turns(ph, s, c);
    } else if (TRIG == TRIG_FAST) {
        // records hold 2 pi k, so ph is the phase in radians
        if (on_fp32)
            sincos_quarter_turns(ph * 0.636619772367581343076f, s, c);
        else
            __sincosf(ph, &s, &c);
    } else {
        // records hold k in turns; subtract the nearest integer exactly
        const float rn = (ph + 12582912.0f) - 12582912.0f;
        const float r = ph - rn;
        __sincosf(r * 6.28318530717958647692f, &s, &c);
    }
}

// ---------------------------------------------------------------------------
// the gather
// ---------------------------------------------------------------------------
template <int BC, bool REALW, int TRIG>
__global__ void __launch_bounds__(Shape<BC, REALW>::THREADS, Shape<BC, REALW>::MIN_BLOCKS)
    gather_kernel(GatherParams p)
{
    using R = Rec<BC, REALW>;
    using S = Shape<BC, REALW>;
    constexpr int V = S::V;
    constexpr int T = S::THREADS;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    float* const ring = reinterpret_cast<float*>(smem_raw);
    __shared__ __align__(8) uint64_t full_bar[kStages];

    const int tid = threadIdx.x;
    const int split = blockIdx.y;
    const int64_t t_begin = (p.ntiles * split) / p.splits;
    const int64_t t_end = (p.ntiles * (split + 1)) / p.splits;
    const int nt = int(t_end - t_begin);
    const int64_t n0 = int64_t(blockIdx.x) * S::VOXELS_PER_CTA + tid;

    // register-promoted voxel coordinates (Fig. 17.11), V per thread
    float xv[V], yv[V], zv[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int64_t n = n0 + int64_t(v) * T;
        const bool in = n < p.N;
        xv[v] = in ? p.x[n] : 0.0f;
        yv[v] = in ? p.y[n] : 0.0f;
        zv[v] = in ? p.z[n] : 0.0f;
    }

    float* const out_r = p.out_r + split * p.split_stride;
    float* const out_i = p.out_i + split * p.split_stride;

    // running sums: in registers for a single weight, in the outputs for coil groups
    float run_r[BC == 1 ? V : 1], run_i[BC == 1 ? V : 1];
#pragma unroll
    for (int v = 0; v < (BC == 1 ? V : 1); ++v) run_r[v] = run_i[v] = 0.0f;

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

        float pr[V][BC], pi[V][BC];
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int b = 0; b < BC; ++b) pr[v][b] = pi[v][b] = 0.0f;

        if (ok) {
            if (!R::AOS) {
                // four samples per step: one broadcast 16-byte load per field
#pragma unroll 1
                for (int j = 0; j < kTile; j += 4) {
                    const float4 kx4 = *reinterpret_cast<const float4*>(tile + 0 * kTile + j);
                    const float4 ky4 = *reinterpret_cast<const float4*>(tile + 1 * kTile + j);
                    const float4 kz4 = *reinterpret_cast<const float4*>(tile + 2 * kTile + j);
                    const float4 w04 = *reinterpret_cast<const float4*>(tile + 3 * kTile + j);
                    float4 w14 = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (!REALW) w14 = *reinterpret_cast<const float4*>(tile + 4 * kTile + j);
                    const float kxs[4] = {kx4.x, kx4.y, kx4.z, kx4.w};
                    const float kys[4] = {ky4.x, ky4.y, ky4.z, ky4.w};
                    const float kzs[4] = {kz4.x, kz4.y, kz4.z, kz4.w};
                    const float w0s[4] = {w04.x, w04.y, w04.z, w04.w};
                    const float w1s[4] = {w14.x, w14.y, w14.z, w14.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const float ph =
                                fmaf(kzs[q], zv[v], fmaf(kys[q], yv[v], kxs[q] * xv[v]));
                            float sn, cs;
                            phase_sincos<TRIG>(ph, v >= V - S::NP_FP32, sn, cs);
                            if (REALW) {
                                pr[v][0] = fmaf(w0s[q], cs, pr[v][0]);
                                pi[v][0] = fmaf(w0s[q], sn, pi[v][0]);
                            } else {
                                // (rMu + i iMu)(cos + i sin)
                                pr[v][0] = fmaf(w0s[q], cs, pr[v][0]);
                                pr[v][0] = fmaf(-w1s[q], sn, pr[v][0]);
                                pi[v][0] = fmaf(w1s[q], cs, pi[v][0]);
                                pi[v][0] = fmaf(w0s[q], sn, pi[v][0]);
                            }
                        }
                    }
                }
            } else {
                // coil groups: one record per step, one sin/cos per voxel for all coils
#pragma unroll kCoilUnroll
                for (int j = 0; j < kTile; ++j) {
                    const float4* rec4 = reinterpret_cast<const float4*>(tile + j * R::F4);
                    float f[R::F4];
#pragma unroll
                    for (int i = 0; i < R::F4 / 4; ++i) {
                        const float4 r4 = rec4[i];
                        f[4 * i] = r4.x;
                        f[4 * i + 1] = r4.y;
                        f[4 * i + 2] = r4.z;
                        f[4 * i + 3] = r4.w;
                    }
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const float ph = fmaf(f[2], zv[v], fmaf(f[1], yv[v], f[0] * xv[v]));
                        float sn, cs;
                        phase_sincos<TRIG>(ph, v >= V - S::NP_FP32, sn, cs);
#pragma unroll
                        for (int b = 0; b < BC; ++b) {
                            const float rm = f[3 + b], im = f[3 + BC + b];
                            pr[v][b] = fmaf(rm, cs, pr[v][b]);
                            pr[v][b] = fmaf(-im, sn, pr[v][b]);
                            pi[v][b] = fmaf(im, cs, pi[v][b]);
                            pi[v][b] = fmaf(rm, sn, pi[v][b]);
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
        if (BC == 1) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                run_r[BC == 1 ? v : 0] += pr[v][0];
                run_i[BC == 1 ? v : 0] += pi[v][0];
            }
        } else {
            const bool first = (t == 0) && !p.accumulate;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int64_t n = n0 + int64_t(v) * T;
                if (n < p.N) {
#pragma unroll
                    for (int b = 0; b < BC; ++b) {
                        float* rp = out_r + b * p.coil_stride + n;
                        float* ip = out_i + b * p.coil_stride + n;
                        if (first) {
                            *rp = pr[v][b];
                            *ip = pi[v][b];
                        } else {
                            *rp += pr[v][b];
                            *ip += pi[v][b];
                        }
                    }
                }
            }
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

    if (BC == 1) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int64_t n = n0 + int64_t(v) * T;
            if (n < p.N) {
                float r = run_r[BC == 1 ? v : 0], i = run_i[BC == 1 ? v : 0];
                if (p.accumulate) {
                    r = out_r[n] + r;
                    i = out_i[n] + i;
                }
                out_r[n] = r;
                out_i[n] = i;
            }
        }
    }
}

}  // namespace mri
