// microbench.cu -- MUFU / FFMA throughput probes (see include/mri_microbench.h).
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

}  // namespace

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
    if (which < 0 || which > 3) return MRI_ERR_MODE;
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
        default: e = launch_probe<3>(grid, threads, smem, s, iters, cycles, sink); break;
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return MRI_ERR_CUDA;
    return MRI_OK;
}
