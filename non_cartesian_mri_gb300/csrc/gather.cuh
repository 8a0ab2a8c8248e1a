// gather.cuh -- shared pieces of the F^H D / Q gathers for sm_103a: trig
// modes, the tile-record layout and prep of the grid paths, the launch
// parameters, and the scalar quarter-turn polynomial trig.
//
// Method (pages on iterative non-Cartesian MRI reconstruction, section 17.3):
//   cmpMu (Fig. 17.7):      Mu[m] = conj(Phi[m]) * D[m]
//   cmpFhD gather (Figs. 17.10/17.11, register-promoted):
//       FhD[n] = sum_m Mu[m] * e^{+i 2 pi (kx[m] x[n] + ky[m] y[n] + kz[m] z[n])}
//   Q (section 17.2, "same core structure"): the same gather with weight |Phi|^2.
//
// The general gathers (arbitrary voxel coordinates) are in gather_pair.cuh;
// the grid paths in gather_grid_tc*.cuh.  Common design:
//   * A prep kernel writes the trajectory and weights into tile-major records
//     (zero-padded to whole tiles; padded samples have k = 0 and weight 0 and
//     so add exactly +0).  It fuses cmpMu and folds the trig path's phase
//     scale into k.
//   * Record tiles stream through a ring in shared memory filled by 1-D TMA
//     bulk copies completing on mbarriers; every warp reads each sample as a
//     broadcast (the access pattern that made the chapter put k-space in
//     constant memory).
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
    TRIG_ACCURATE = 0,  // minimax polynomials on the FP32 pipe
    TRIG_FAST = 1,      // MUFU on the phase in radians (Q: a share of voxels on the FP32 pipe)
    TRIG_FAST_RR = 2,   // MUFU after explicit reduction of the phase to [-1/2, 1/2] turn
};

constexpr int kTile = 256;   // samples per k-tile
constexpr int kStages = 3;   // tiles resident per CTA

// Record layout of one tile of the grid paths (gather_grid_tc*.cuh):
// structure of arrays [F][TILE],
//   F^H D and coil groups: kx ky kz rMu_0..rMu_{BC-1} iMu_0..iMu_{BC-1}
//   Q:                     kx ky kz w
template <int BC, bool REALW, int TILE>
struct Rec {
    static_assert(!REALW || BC == 1, "a real weight has one coil");
    static constexpr int F = REALW ? 4 : 3 + 2 * BC;
    static constexpr int TILE_FLOATS = TILE * F;
    static constexpr uint32_t TILE_BYTES = TILE_FLOATS * 4u;
};

struct PrepParams {
    const float *kx, *ky, *kz;
    const float *rPhi, *iPhi;
    const float *rD, *iD;   // coil-major [B][M]; coil b0 .. b0+BC-1 used
    int64_t M;
    int64_t b0;
    int64_t ntiles;
    float kscale;           // 2 (half turns), 2*pi (radians) or 1 (turns)
    float* rec;
    // Optional: raised by atomicMax to the float bits of the largest
    // |w_r| + |w_i| over samples and coils; the caller zeroes it first.
    unsigned int* wbound = nullptr;
    // With bound_per_coil, wbound holds one word per coil of the group and
    // coil b's bound goes to wbound[b] (the caller zeroes BC words).
    bool bound_per_coil = false;
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
template <int BC, bool REALW, int TILE>
__global__ void __launch_bounds__(256) prep_records_kernel(PrepParams p)
{
    using R = Rec<BC, REALW, TILE>;
    const int64_t total = p.ntiles * TILE;
    float wmax = 0.0f;
    float wcoil[BC];   // per coil (bound_per_coil)
#pragma unroll
    for (int b = 0; b < BC; ++b) wcoil[b] = 0.0f;
    for (int64_t m = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; m < total;
         m += int64_t(gridDim.x) * blockDim.x) {
        const int64_t tile = m / TILE;
        const int j = int(m - tile * TILE);
        float* base = p.rec + tile * R::TILE_FLOATS;
        float f[R::F];
#pragma unroll
        for (int i = 0; i < R::F; ++i) f[i] = 0.0f;
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
                for (int b = 0; b < BC; ++b) {
                    const float a = fabsf(f[3 + b]) + fabsf(f[3 + BC + b]);
                    wmax = fmaxf(wmax, a);
                    wcoil[b] = fmaxf(wcoil[b], a);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < R::F; ++i) base[i * TILE + j] = f[i];
    }
    // non-negative floats order like their bit patterns (a NaN sorts last)
    if (p.wbound != nullptr && !REALW && p.bound_per_coil) {
#pragma unroll
        for (int b = 0; b < BC; ++b) {
            const unsigned int w = __reduce_max_sync(0xffffffffu, __float_as_uint(wcoil[b]));
            if ((threadIdx.x & 31) == 0 && w != 0u) atomicMax(p.wbound + b, w);
        }
    } else if (p.wbound != nullptr) {
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

// sin and cos of pi u for u in half turns (|u| < 2^22), on the FP32 pipe:
// exact reduction q = rint(u), f = u - q in [-1/2, 1/2], minimax polynomials
// of pi f (SinCosHalf, gen_sincospi.py), then the sign (-1)^q from the low
// bit of q -- no quadrant swap.
__device__ __forceinline__ void sincos_half_turns(float u, float& s, float& c)
{
    using Coef = SinCosHalf;
    const float v = u + 12582912.0f;
    const float f = u - (v - 12582912.0f);
    const float f2 = f * f;
    float p = Coef::P(Coef::P_TERMS - 1);
#pragma unroll
    for (int i = Coef::P_TERMS - 2; i >= 0; --i) p = fmaf(p, f2, Coef::P(i));
    float q = Coef::Q(Coef::Q_TERMS - 1);
#pragma unroll
    for (int i = Coef::Q_TERMS - 2; i >= 0; --i) q = fmaf(q, f2, Coef::Q(i));
    const unsigned m = __float_as_uint(v) << 31;   // bit 31 = parity of q
    s = __uint_as_float(__float_as_uint(f * p) ^ m);
    c = __uint_as_float(__float_as_uint(q) ^ m);
}

// The same on a pair of phases (.f32x2 instructions; the sign flip per half).
__device__ __forceinline__ void f2_halves(f2 v, uint32_t& lo, uint32_t& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}

__device__ __forceinline__ f2 f2_from_halves(uint32_t lo, uint32_t hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}

// sin and cos of pi u for a pair of phases u in half turns (|u| < 2^22):
// f = u - rint(u) exactly (adding and removing 1.5 * 2^23 rounds to an
// integer q and leaves it in the low mantissa bits of the sum), the
// polynomials of pi f, and the sign (-1)^q.
__device__ __forceinline__ void sincos_half_turns2(f2 u, f2& s, f2& c)
{
    using Coef = SinCosHalf;
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
    uint32_t vl, vh, sl, sh, cl, ch;
    f2_halves(v, vl, vh);
    f2_halves(sf, sl, sh);
    f2_halves(q, cl, ch);
    const uint32_t ml = vl << 31, mh = vh << 31;   // bit 31 = parity of q
    s = f2_from_halves(sl ^ ml, sh ^ mh);
    c = f2_from_halves(cl ^ ml, ch ^ mh);
}

}  // namespace mri
