// kernels_single.cu -- F^H D (one weight vector) and Q instantiations, the
// prep, reduction and cmpMu kernels.
#include <type_traits>

#include "launch.h"

namespace mri {

// ---------------------------------------------------------------------------
// deterministic reduction of the sample splits: part is [S][BC][2][N]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ part,
                                                            int S, int BC, int64_t N,
                                                            float* out_r, float* out_i,
                                                            int64_t out_coil_stride,
                                                            int accumulate)
{
    const int64_t total = int64_t(BC) * 2 * N;
    const int64_t split_stride = total;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t bc = e / N;          // b * 2 + c
        const int64_t n = e - bc * N;
        const int64_t b = bc >> 1;
        const int c = int(bc & 1);
        float sum = part[e];
        for (int s = 1; s < S; ++s) sum += part[s * split_stride + e];
        float* o = (c == 0 ? out_r : out_i) + b * out_coil_stride + n;
        *o = accumulate ? (*o + sum) : sum;
    }
}

// zero n floats (outputs of a call with no samples)
__global__ void __launch_bounds__(256) zero_fill_kernel(float* a, int64_t n)
{
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n;
         e += int64_t(gridDim.x) * blockDim.x)
        a[e] = 0.0f;
}

// Mu = conj(Phi) * D, one sample per thread (cmpMu, Fig. 17.7)
__global__ void __launch_bounds__(256) mu_kernel(const float* __restrict__ rPhi,
                                                 const float* __restrict__ iPhi,
                                                 const float* __restrict__ rD,
                                                 const float* __restrict__ iD, float* rMu,
                                                 float* iMu, int64_t M)
{
    for (int64_t m = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; m < M;
         m += int64_t(gridDim.x) * blockDim.x) {
        const float rp = rPhi[m], ip = iPhi[m], rd = rD[m], id = iD[m];
        rMu[m] = fmaf(ip, id, rp * rd);
        iMu[m] = fmaf(-ip, rd, rp * id);
    }
}


namespace {
template <bool REALW, int TRIG>
cudaError_t run_gather(const GatherParams& p, dim3 grid, cudaStream_t s)
{
    constexpr size_t smem = PairShape::smem<REALW>();
    const cudaError_t attr = cudaFuncSetAttribute(
        gather_pair_kernel<REALW, TRIG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        int(smem));
    if (attr != cudaSuccess) return attr;
    gather_pair_kernel<REALW, TRIG><<<grid, PairShape::THREADS, smem, s>>>(p);
    return cudaGetLastError();
}
}  // namespace

// one weight vector (F^H D, Q, the forward model): the kernel on pairs of floats
cudaError_t launch_gather_single(bool realw, int trig, const GatherParams& p, dim3 grid,
                                 cudaStream_t s)
{
    if (realw) {
        switch (trig) {
            case TRIG_ACCURATE: return run_gather<true, TRIG_ACCURATE>(p, grid, s);
            case TRIG_FAST: return run_gather<true, TRIG_FAST>(p, grid, s);
            case TRIG_FAST_RR: return run_gather<true, TRIG_FAST_RR>(p, grid, s);
        }
    } else {
        switch (trig) {
            case TRIG_ACCURATE: return run_gather<false, TRIG_ACCURATE>(p, grid, s);
            case TRIG_FAST: return run_gather<false, TRIG_FAST>(p, grid, s);
            case TRIG_FAST_RR: return run_gather<false, TRIG_FAST_RR>(p, grid, s);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_prep(int bc, bool realw, const PrepParams& p, int grid, cudaStream_t s)
{
    if (realw) {
        prep_pair_records_kernel<true><<<grid, 256, 0, s>>>(p);
        return cudaGetLastError();
    }
    if (bc == 1) {
        prep_pair_records_kernel<false><<<grid, 256, 0, s>>>(p);
        return cudaGetLastError();
    }
    return launch_prep_coils(bc, p, grid, s);
}

float gather_kscale(int, int trig) { return pair_kscale(trig); }

cudaError_t launch_gather(int bc, bool realw, int trig, const GatherParams& p, dim3 grid,
                          cudaStream_t s)
{
    if (bc == 1) return launch_gather_single(realw, trig, p, grid, s);
    return launch_gather_coils(bc, trig, p, grid, s);
}

cudaError_t launch_reduce(const float* part, int splits, int bc, int64_t N, float* out_r,
                          float* out_i, int64_t out_coil_stride, int accumulate, int grid,
                          cudaStream_t s)
{
    reduce_splits_kernel<<<grid, 256, 0, s>>>(part, splits, bc, N, out_r, out_i,
                                               out_coil_stride, accumulate);
    return cudaGetLastError();
}

cudaError_t launch_mu(const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                      float* rMu, float* iMu, int64_t M, int grid, cudaStream_t s)
{
    mu_kernel<<<grid, 256, 0, s>>>(rPhi, iPhi, rD, iD, rMu, iMu, M);
    return cudaGetLastError();
}

cudaError_t launch_zero(float* a, int64_t n, int grid, cudaStream_t s)
{
    zero_fill_kernel<<<grid, 256, 0, s>>>(a, n);
    return cudaGetLastError();
}

KernelShape gather_shape(int bc, bool realw)
{
    KernelShape k{};
    auto fill_pair = [&](auto realw_tag) {
        constexpr bool RW = decltype(realw_tag)::value;
        k.threads = PairShape::THREADS;
        k.v = PairShape::V;
        k.voxels_per_cta = PairShape::VOXELS_PER_CTA;
        k.min_blocks = PairShape::MIN_BLOCKS;
        k.smem = PairShape::smem<RW>();
        k.tile_floats = PairRec<RW>::TILE_FLOATS;
        k.fast_fp32_voxels = 2 * PairShape::np_fp32<RW>();
    };
    auto fill_coils = [&](auto bc_tag) {
        constexpr int B = decltype(bc_tag)::value;
        using Sh = PairCoilShape<B>;
        k.threads = Sh::THREADS;
        k.v = Sh::V;
        k.voxels_per_cta = Sh::VOXELS_PER_CTA;
        k.min_blocks = Sh::MIN_BLOCKS;
        k.smem = Sh::SMEM;
        k.tile_floats = PairCoilRec<B>::TILE_FLOATS;
    };
    if (realw) fill_pair(std::true_type{});
    else if (bc == 1) fill_pair(std::false_type{});
    else if (bc == 2) fill_coils(std::integral_constant<int, 2>{});
    else if (bc == 4) fill_coils(std::integral_constant<int, 4>{});
    else fill_coils(std::integral_constant<int, 8>{});
    return k;
}

}  // namespace mri
