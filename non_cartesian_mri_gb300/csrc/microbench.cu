// microbench.cu -- MUFU / FFMA / tensor-core throughput probes (see include/mri_microbench.h).
#include <cstdint>

#include <cuda_runtime.h>

#include "mri.h"
#include "mri_microbench.h"
#include "ptx.cuh"

namespace mri {
unsigned int* error_word_address(int dev);   // mri_abi.cu; symbol lookup only
}

namespace {

template <int WHICH>
__global__ void probe_kernel(int64_t iters, unsigned long long* cycles, float* sink)
{
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.001f * float(threadIdx.x + 37 * i) + 0.25f;
    __syncthreads();
    const unsigned long long t0 = clock64();
    for (int64_t it = 0; it < iters; ++it) {
        if (WHICH == 4) {
            // four chains of packed pairs: 4 FFMA2 instructions, 8 results
            const mri::f2 m = mri::f2_splat(0.999f), c = mri::f2_splat(0.0001f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mri::f2 v = mri::f2_pack(a[2 * i], a[2 * i + 1]);
                v = mri::f2_fma(v, m, c);
                mri::f2_unpack(v, a[2 * i], a[2 * i + 1]);
            }
            continue;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (WHICH == 0) a[i] = __sinf(a[i]);
            else if (WHICH == 1) a[i] = __cosf(a[i]);
            else if (WHICH == 2) a[i] = fmaf(a[i], 0.999f, 0.0001f);
            else a[i] = exp2f(-a[i]);
        }
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc += a[i];
    sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    extern __shared__ float occupancy_limiter[];   // sized by the launch, never read
    (void)occupancy_limiter;
}

template <int WHICH>
cudaError_t launch_probe(dim3 grid, int threads, int smem, cudaStream_t s, int64_t iters,
                         unsigned long long* cycles, float* sink)
{
    cudaError_t e = cudaFuncSetAttribute(probe_kernel<WHICH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    probe_kernel<WHICH><<<grid, threads, smem, s>>>(iters, cycles, sink);
    return cudaGetLastError();
}

// One CTA waits, bounded, on an mbarrier of arrival count 1 with the wait
// helper every kernel uses.  arrive = 0: nothing ever arrives, the wait must
// give up after its time limit and report through the device error word;
// arrive = 1: thread 0 arrives first and the wait completes at once.
__global__ void wait_selftest_kernel(int arrive, unsigned int* err)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mri::mbar_init(&bar, 1);
        mri::fence_barrier_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) mri::mbar_arrive(&bar);
    const bool ok = mri::mbar_wait_bounded(&bar, 0u);
    if (!ok && threadIdx.x == 0) atomicOr(err, mri::DEVERR_TILE_WAIT_TIMEOUT);
}

// Tensor-core issue-rate probe: one thread issues, per tile, the 12
// tcgen05.mma (kind::f16, 128 x 256 x 16) of a 32-sample tile of the
// tensor-core grid kernel, with no operand generation and no CTA barrier.
// MODE 0: A and B in shared memory (zeroed); MODE 1: A from tensor memory,
// B in shared memory; MODE 2: A from tensor memory, B brought per tile by
// one 48 KB TMA bulk copy from a table in global memory into a 4-stage ring
// (copies issued two tiles ahead, as the grid kernel does); MODE 3: as MODE 1
// with every product split into two N = 128 halves (24 MMAs of 128 x 128 x
// 16 per tile, the same work, alternating between two accumulators); MODE 4:
// as MODE 3 with every MMA into the same accumulator.  One commit per tile.  One CTA per SM (at least 128 KB of shared memory, all 512 TMEM
// columns).
constexpr int kProbePart = 128 * 32 * 2;          // 128 rows x 32 K of f16: 8 KB
constexpr int kProbeS = 3 * kProbePart;           // 384 B rows: 24 KB (hi; lo follows)
constexpr int kProbeStage = 2 * kProbeS;          // one B tile: 48 KB
constexpr int kProbeA = kProbeStage;              // A parts (MODE 0) after one B tile
constexpr int kProbeRing = 4;                     // MODE 2 B stages

__host__ __device__ constexpr int probe_smem(int mode)
{
    return mode == 2 ? kProbeRing * kProbeStage : 128 * 1024;
}

template <int MODE>
__global__ void __launch_bounds__(128, 1) mma_probe_kernel(int tiles, const unsigned char* b_tab,
                                                           int64_t b_tiles,
                                                           unsigned long long* cycles,
                                                           unsigned int* err)
{
    constexpr int SMEM = probe_smem(MODE);
    constexpr int NB = MODE == 2 ? kProbeRing : 2;    // commit barriers
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t done[NB];
    __shared__ __align__(8) uint64_t full[kProbeRing];
    __shared__ uint32_t tmem_sh;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    for (int i = tid; i < SMEM / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (warp == 0) mri::tmem_alloc(&tmem_sh, 512);
    if (tid == 0) {
        for (int i = 0; i < NB; ++i) mri::mbar_init(&done[i], 1);
        for (int i = 0; i < kProbeRing; ++i) mri::mbar_init(&full[i], 1);
        mri::fence_barrier_init();
    }
    mri::fence_proxy_async_smem();
    mri::tc_fence_before_sync();
    __syncthreads();
    mri::tc_fence_after_sync();
    const uint32_t tmem = tmem_sh;
    {
        // zero this warp's lane quarter of every column
        uint32_t z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0u;
        for (int c = 0; c < 512; c += 32)
            mri::tmem_st32u(tmem + (uint32_t(32 * warp) << 16) + uint32_t(c), z);
        mri::tmem_wait_st();
    }
    mri::tc_fence_before_sync();
    __syncthreads();
    mri::tc_fence_after_sync();

    if (tid == 0) {
        constexpr uint32_t ID = mri::umma_idesc_f16(128, 256);
        constexpr uint32_t ID128 = mri::umma_idesc_f16(128, 128);
        auto load = [&](int u) {
            uint64_t* bar = &full[u % kProbeRing];
            mri::mbar_arrive_expect_tx(bar, uint32_t(kProbeStage));
            mri::tma_bulk_g2s(smem + (u % kProbeRing) * kProbeStage,
                              b_tab + (u % b_tiles) * int64_t(kProbeStage),
                              uint32_t(kProbeStage), bar);
        };
        bool ok = true;
        int loaded = 0;
        if (MODE == 2)
            for (; loaded < kProbeRing && loaded < tiles; ++loaded) load(loaded);
        const unsigned long long t0 = clock64();
        int t = 0;
        for (; t < tiles && ok; ++t) {
            const unsigned char* stage = smem;
            if (MODE == 2) {
                stage = smem + (t % kProbeRing) * kProbeStage;
                ok = mri::mbar_wait_bounded(&full[t % kProbeRing],
                                            uint32_t(t / kProbeRing) & 1u);
            } else if (t >= 2) {
                ok = mri::mbar_wait_bounded(&done[t & 1], uint32_t((t - 2) >> 1) & 1u);
            }
            if (!ok) break;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
                auto sdesc = [&](int half, int r0) {
                    return mri::umma_desc_kmajor(stage + half * kProbeS + (r0 / 128) * kProbePart +
                                                     kb * 256,
                                                 128, 512);
                };
                auto mma = [&](int part, uint64_t b, uint32_t acc) {
                    if (MODE == 4) {
                        // the same 24 MMAs, all into one accumulator
                        const uint32_t a = tmem + 256u + uint32_t(part * 16 + 8 * kb);
                        mri::umma_f16_ta(tmem, a, b, ID128, acc);
                        mri::umma_f16_ta(tmem, a, b + uint64_t((16 * 512) >> 4), ID128, 1u);
                    } else if (MODE == 3) {
                        // the same product as two N = 128 halves (rows 0-127 and
                        // 128-255 of the window, D columns 0-127 and 128-255)
                        const uint32_t a = tmem + 256u + uint32_t(part * 16 + 8 * kb);
                        mri::umma_f16_ta(tmem, a, b, ID128, acc);
                        mri::umma_f16_ta(tmem + 128u, a, b + uint64_t((16 * 512) >> 4), ID128, acc);
                    } else if (MODE >= 1) {
                        mri::umma_f16_ta(tmem, tmem + 256u + uint32_t(part * 16 + 8 * kb), b, ID,
                                         acc);
                    } else {
                        const uint64_t a = mri::umma_desc_kmajor(
                            smem + kProbeA + part * kProbePart + kb * 256, 128, 512);
                        mri::umma_f16(tmem, a, b, ID, acc);
                    }
                };
                const uint32_t acc0 = (t == 0 && kb == 0) ? 0u : 1u;
                mma(0, sdesc(0, 128), acc0);
                mma(0, sdesc(1, 128), 1u);
                mma(1, sdesc(0, 128), 1u);
                mma(2, sdesc(0, 0), 1u);
                mma(2, sdesc(1, 0), 1u);
                mma(3, sdesc(0, 0), 1u);
            }
            mri::umma_commit(&done[t % NB]);
            if (MODE == 2) {
                // refill: tile t + 2 into the stage tile t - 2 used
                const int u = t + 2;
                if (u >= kProbeRing && u < tiles && loaded == u) {
                    ok = mri::mbar_wait_bounded(&done[u % kProbeRing],
                                                uint32_t((u - kProbeRing) / kProbeRing) & 1u);
                    if (ok) {
                        load(u);
                        ++loaded;
                    }
                }
            }
        }
        // the last commit covers every MMA issued before it
        if (t > 0 && !mri::mbar_wait_bounded(&done[(t - 1) % NB], uint32_t((t - 1) / NB) & 1u))
            ok = false;
        // copies still in flight (issued, never waited for) land before exit
        if (MODE == 2)
            for (int u = t; u < loaded; ++u)
                if (!mri::mbar_wait_bounded(&full[u % kProbeRing], uint32_t(u / kProbeRing) & 1u))
                    ok = false;
        const unsigned long long t1 = clock64();
        cycles[blockIdx.x] = t1 - t0;
        if (!ok) atomicOr(err, mri::DEVERR_TILE_WAIT_TIMEOUT);
    }
    mri::tc_fence_before_sync();
    __syncthreads();
    mri::tc_fence_after_sync();
    if (warp == 0) mri::tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" mri_status mri_mma_probe(int mode, int tiles, const void* b_tab, int64_t b_tiles,
                                    unsigned long long* cycles, void* stream)
{
    if (mode < 0 || mode > 4) return MRI_ERR_MODE;
    if (cycles == nullptr || (mode == 2 && b_tab == nullptr)) return MRI_ERR_NULL;
    if (tiles < 1 || tiles > (1 << 22)) return MRI_ERR_SIZE;
    if (mode == 2 && b_tiles < 1) return MRI_ERR_SIZE;
    if (mode == 2 && (reinterpret_cast<uintptr_t>(b_tab) & 15u) != 0) return MRI_ERR_SIZE;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MRI_ERR_UNSUPPORTED_DEVICE;
    unsigned int* err = mri::error_word_address(dev);
    if (err == nullptr) return MRI_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const unsigned char* tab = static_cast<const unsigned char*>(b_tab);
    auto go = [&](auto kernel, int smem) -> cudaError_t {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        kernel<<<sms, 128, smem, s>>>(tiles, tab, b_tiles, cycles, err);
        return cudaGetLastError();
    };
    cudaError_t e = cudaSuccess;
    switch (mode) {
        case 0: e = go(mma_probe_kernel<0>, probe_smem(0)); break;
        case 1: e = go(mma_probe_kernel<1>, probe_smem(1)); break;
        case 3: e = go(mma_probe_kernel<3>, probe_smem(3)); break;
        case 4: e = go(mma_probe_kernel<4>, probe_smem(4)); break;
        default: e = go(mma_probe_kernel<2>, probe_smem(2)); break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    return MRI_OK;
}

extern "C" mri_status mri_wait_selftest(int arrive, void* stream)
{
    if (arrive != 0 && arrive != 1) return MRI_ERR_MODE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MRI_ERR_UNSUPPORTED_DEVICE;
    unsigned int* err = mri::error_word_address(dev);
    if (err == nullptr) return MRI_ERR_CUDA;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(arrive, err);
    if (cudaGetLastError() != cudaSuccess) return MRI_ERR_CUDA;
    return MRI_OK;
}

extern "C" mri_status mri_microbench(int which, int ctas_per_sm, int threads, int64_t iters,
                                     unsigned long long* cycles, float* sink, void* stream)
{
    if (which < 0 || which > 4) return MRI_ERR_MODE;
    if (cycles == nullptr || sink == nullptr) return MRI_ERR_NULL;
    if (ctas_per_sm < 1 || threads < 32 || threads > 1024 || iters < 1) return MRI_ERR_SIZE;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MRI_ERR_UNSUPPORTED_DEVICE;
    int smem_sm = 0;
    if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    // Dynamic shared memory sized so that exactly ctas_per_sm CTAs fit on an
    // SM: the grid of sms * ctas_per_sm CTAs is then one even wave.
    const int smem = (smem_sm / ctas_per_sm) - 2048;
    if (smem < 1024) return MRI_ERR_SIZE;
    const dim3 grid(unsigned(sms * ctas_per_sm));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (which) {
        case 0: e = launch_probe<0>(grid, threads, smem, s, iters, cycles, sink); break;
        case 1: e = launch_probe<1>(grid, threads, smem, s, iters, cycles, sink); break;
        case 2: e = launch_probe<2>(grid, threads, smem, s, iters, cycles, sink); break;
        case 3: e = launch_probe<3>(grid, threads, smem, s, iters, cycles, sink); break;
        default: e = launch_probe<4>(grid, threads, smem, s, iters, cycles, sink); break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return MRI_ERR_CUDA;
    return MRI_OK;
}
