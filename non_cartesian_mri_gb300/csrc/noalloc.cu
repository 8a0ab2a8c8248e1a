// noalloc.cu -- mri_fhd_noalloc: F^H D with no memory allocation at all.
//
// Some callers cannot allocate GPU memory while they run: a process whose
// memory budget is fixed and fully reserved up front, a real-time
// reconstruction loop that must not stall in the driver's allocator, or a
// host framework that owns every allocation and forbids libraries from
// making their own.  mri_fhd takes its scratch from a stream-ordered pool;
// this entry point instead uses a fixed array compiled into the library, so
// a call makes no cudaMalloc, cudaFree, pool or other allocating call.
//
// The array costs every GPU that loads the library kNoallocScratchBytes of
// device memory until the process exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "launch.h"
#include "mri.h"

namespace mri {
unsigned int* error_word_address(int dev);   // mri_abi.cu; symbol lookup only
// mri_abi.cu; the residency check every entry point makes (no allocation)
mri_status check_device_ptrs(const void* const* ptrs, int n, int dev);
}

namespace {

constexpr int64_t kNoallocScratchBytes = MRI_FHD_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself: tile records first, then the per-split partial sums.
// On the host this name only stands for the symbol; its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocDevice {
    bool ready = false;
    int dev = -1;
    mri_status status = MRI_OK;
    int sms = 0;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
    unsigned int* err = nullptr;
};

std::mutex g_noalloc_mutex;
NoallocDevice g_noalloc_dev[kMaxDevices];

mri_status fail_cuda()
{
    (void)cudaGetLastError();
    return MRI_ERR_CUDA;
}

// Once per device, with that device current: capability check, SM count and
// the device addresses of the scratch array and of the error word.  Nothing
// here allocates.
mri_status noalloc_device(NoallocDevice** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail_cuda();
    if (dev < 0 || dev >= kMaxDevices) return MRI_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocDevice& d = g_noalloc_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail_cuda();
        if (major != 10 || minor != 3) {
            d.status = MRI_ERR_UNSUPPORTED_DEVICE;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return fail_cuda();
            unsigned int* err = mri::error_word_address(dev);
            if (err == nullptr) return fail_cuda();
            d.dev = dev;
            d.sms = sms;
            d.scratch = static_cast<unsigned char*>(p);
            d.err = err;
        }
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

int grid_cap(int64_t elements, int sms)
{
    int64_t g = (elements + 255) / 256;
    const int64_t cap = int64_t(sms) * 8;
    if (g > cap) g = cap;
    return g < 1 ? 1 : int(g);
}

}  // namespace

extern "C" mri_status mri_fhd_noalloc(const float* kx, const float* ky, const float* kz,
                                      const float* x, const float* y, const float* z,
                                      const float* rPhi, const float* iPhi, const float* rD,
                                      const float* iD, int64_t M, int64_t N, float* rFhD,
                                      float* iFhD, mri_trig trig, int accumulate, void* stream)
{
    const int tr = int(trig);
    if (tr != MRI_TRIG_ACCURATE && tr != MRI_TRIG_FAST && tr != MRI_TRIG_FAST_RR)
        return MRI_ERR_MODE;
    if (accumulate != 0 && accumulate != 1) return MRI_ERR_MODE;
    if (M < 0 || N < 0 || N > (int64_t(1) << 40)) return MRI_ERR_SIZE;
    const int64_t ntiles = (M + mri::kTile - 1) / mri::kTile;
    const int64_t rec_bytes = round256(ntiles * int64_t(mri::PairRec<false>::TILE_BYTES));
    if (rec_bytes > kNoallocScratchBytes) return MRI_ERR_SIZE;   // M above the fixed maximum
    if (N == 0) return MRI_OK;

    const void* voxel_ptrs[5] = {x, y, z, rFhD, iFhD};
    const void* sample_ptrs[7] = {kx, ky, kz, rPhi, iPhi, rD, iD};
    for (const void* p : voxel_ptrs)
        if (p == nullptr) return MRI_ERR_NULL;
    if (M > 0)
        for (const void* p : sample_ptrs)
            if (p == nullptr) return MRI_ERR_NULL;
    for (const void* p : voxel_ptrs)
        if (!aligned4(p)) return MRI_ERR_ALIGN;
    if (M > 0)
        for (const void* p : sample_ptrs)
            if (!aligned4(p)) return MRI_ERR_ALIGN;

    NoallocDevice* d = nullptr;
    mri_status st = noalloc_device(&d);
    if (st != MRI_OK) return st;
    // as in mri_fhd: every array must be memory of the current device
    if ((st = mri::check_device_ptrs(voxel_ptrs, 5, d->dev)) != MRI_OK) return st;
    if (M > 0 && (st = mri::check_device_ptrs(sample_ptrs, 7, d->dev)) != MRI_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (M == 0) {
        if (!accumulate) {
            if (mri::launch_zero(rFhD, N, grid_cap(N, d->sms), s) != cudaSuccess ||
                mri::launch_zero(iFhD, N, grid_cap(N, d->sms), s) != cudaSuccess)
                return fail_cuda();
        }
        return MRI_OK;
    }

    // The same launch plan as mri_fhd, with the sample splits capped to the
    // partial sums that fit in the array after the records.
    mri_plan plan;
    st = mri_plan_gather(MRI_KIND_FHD, 1, M, N, d->sms, &plan);
    if (st != MRI_OK) return st;
    const int64_t part_room = kNoallocScratchBytes - rec_bytes;
    int64_t splits = plan.splits;
    const int64_t fit = part_room / (2 * N * int64_t(sizeof(float)));
    if (splits > fit) splits = fit;
    if (splits < 1) splits = 1;

    float* rec = reinterpret_cast<float*>(d->scratch);
    float* part = reinterpret_cast<float*>(d->scratch + rec_bytes);

    mri::PrepParams pp{kx, ky, kz, rPhi, iPhi, rD, iD, M, 0, ntiles, mri::gather_kscale(1, tr),
                       rec};
    if (mri::launch_prep(1, false, pp, grid_cap(ntiles * mri::kTile, d->sms), s) != cudaSuccess)
        return fail_cuda();

    mri::GatherParams gp{};
    gp.rec = rec;
    gp.ntiles = ntiles;
    gp.splits = int(splits);
    gp.x = x;
    gp.y = y;
    gp.z = z;
    gp.N = N;
    gp.err = d->err;
    if (splits == 1) {
        gp.out_r = rFhD;
        gp.out_i = iFhD;
        gp.coil_stride = N;
        gp.split_stride = 0;
        gp.accumulate = accumulate;
    } else {
        gp.out_r = part;
        gp.out_i = part + N;
        gp.coil_stride = 2 * N;
        gp.split_stride = 2 * N;
        gp.accumulate = 0;
    }
    const dim3 grid(unsigned(plan.voxel_ctas), unsigned(splits), 1);
    if (mri::launch_gather(1, false, tr, gp, grid, s) != cudaSuccess) return fail_cuda();
    if (splits > 1) {
        if (mri::launch_reduce(part, int(splits), 1, N, rFhD, iFhD, N, accumulate,
                               grid_cap(2 * N, d->sms), s) != cudaSuccess)
            return fail_cuda();
    }
    return MRI_OK;
}
