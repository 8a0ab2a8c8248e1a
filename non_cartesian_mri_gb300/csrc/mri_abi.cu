// mri_abi.cu -- the extern "C" entry points of libmri.so (declared in
// include/mri.h): argument checks, launch planning, scratch, launches.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>
#include <algorithm>

#include <cuda_runtime.h>

#include "gather_coils_tc.cuh"
#include "launch.h"
#include "mri.h"

namespace {

using mri::KernelShape;
using mri::kTile;

// OR-ed by kernels whose bounded waits gave up (see ptx.cuh).
__device__ unsigned int g_device_error_word;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxM = int64_t(1) << 38;
constexpr int64_t kMaxN = int64_t(1) << 40;
constexpr int64_t kMaxB = int64_t(1) << 20;
constexpr int64_t kMaxBN = int64_t(1) << 42;

constexpr int kMaxTimed = 4096;

struct DeviceState {
    bool ready = false;
    mri_status status = MRI_OK;
    int sms = 0;
    cudaMemPool_t pool = nullptr;
    unsigned int* err = nullptr;
    float2* fft_tw = nullptr;   // FFT twiddle table (fft.cuh), built with the state
    // gather-kernel timing window (mri_timing_begin / mri_timing_end)
    bool timing = false;
    int timed = 0;
    int events_made = 0;
    cudaEvent_t ev[2 * kMaxTimed];
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
std::mutex g_timing_mutex;

mri_status cuda_fail()
{
    (void)cudaGetLastError();   // clear a sticky non-fatal error
    return MRI_ERR_CUDA;
}

// Per-device set-up on first use: capability check, SM count, the scratch
// pool and the address of the device error word.
mri_status device_state(DeviceState** out, int* dev_out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
    if (dev < 0 || dev >= kMaxDevices) return MRI_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_fail();
        d.sms = sms;
        if (major != 10 || minor != 3) {
            d.status = MRI_ERR_UNSUPPORTED_DEVICE;
        } else {
            cudaMemPoolProps props;
            std::memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) return cuda_fail();
            uint64_t keep = UINT64_MAX;   // keep freed scratch for the next call
            if (cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep) !=
                cudaSuccess)
                return cuda_fail();
            void* err = nullptr;
            if (cudaGetSymbolAddress(&err, g_device_error_word) != cudaSuccess)
                return cuda_fail();
            d.err = static_cast<unsigned int*>(err);
            // FFT twiddles: one small table per device, written once
            if (cudaMalloc(reinterpret_cast<void**>(&d.fft_tw),
                           sizeof(float2) * (mri::kFftMaxLen / 2)) != cudaSuccess ||
                mri::launch_fft_twiddles(d.fft_tw, 0) != cudaSuccess ||
                cudaStreamSynchronize(0) != cudaSuccess)
                return cuda_fail();
        }
        d.ready = true;
    }
    *out = &d;
    if (dev_out) *dev_out = dev;
    return d.status;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

mri_status check_device_ptr(const void* p, int dev)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return MRI_ERR_NOT_DEVICE;
    }
    if (a.type == cudaMemoryTypeManaged) return MRI_OK;
    if (a.type == cudaMemoryTypeDevice && a.device == dev) return MRI_OK;
    return MRI_ERR_NOT_DEVICE;
}

// Checks a list of pointers: NULL, alignment, then (device known) residency.
mri_status check_ptrs(const void* const* ptrs, int n, int dev)
{
    for (int i = 0; i < n; ++i)
        if (ptrs[i] == nullptr) return MRI_ERR_NULL;
    for (int i = 0; i < n; ++i)
        if (!aligned4(ptrs[i])) return MRI_ERR_ALIGN;
    if (dev < 0) return MRI_OK;
    for (int i = 0; i < n; ++i) {
        mri_status s = check_device_ptr(ptrs[i], dev);
        if (s != MRI_OK) return s;
    }
    return MRI_OK;
}

// ---------------------------------------------------------------------------
// launch planning (host only)
// ---------------------------------------------------------------------------
struct GroupPlan {
    int bc;
    bool realw;
    KernelShape shape;
    int64_t ntiles;
    int64_t vblocks;
    int splits;
    int64_t rec_bytes;
    int64_t part_bytes;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Samples are split across CTAs when that finishes sooner: every CTA of the
// gather costs the same, so the run time is (waves of CTAs) x (tiles per CTA),
// plus a per-CTA fixed cost and the reduction of the splits.  Costs are in
// units of one tile of gather work.
// tile_us: rough time of one tile of one CTA; overhead_tiles: a CTA's fixed
// cost (prologue, first copy, epilogue) in tiles.
int choose_splits(int64_t ntiles, int64_t vblocks, int64_t slots, int bc, int64_t N,
                  double tile_us = 70.0, double overhead_tiles = 0.1)
{
    const double launch_tiles = 5.0 / tile_us;             // one extra kernel launch, ~5 us
    const double bytes_per_tile = 5e6 * tile_us;           // HBM bytes in one tile's time
    int best = 1;
    double best_cost = 0.0;
    const int64_t max_s = ntiles < 1024 ? ntiles : 1024;
    for (int64_t s = 1; s <= max_s; ++s) {
        const int64_t units = vblocks * s;
        const double waves = double(ceil_div(units, slots));
        double cost = waves * (double(ceil_div(ntiles, s)) + overhead_tiles);
        if (s > 1)
            cost += launch_tiles + double(s + 1) * double(bc) * 2.0 * 4.0 * double(N) /
                                       bytes_per_tile;
        if (s == 1 || cost < best_cost * (1.0 - 1e-9)) {
            best_cost = cost;
            best = int(s);
        }
    }
    return best;
}

GroupPlan plan_group(int bc, bool realw, int64_t M, int64_t N, int sms)
{
    GroupPlan g{};
    g.bc = bc;
    g.realw = realw;
    g.shape = mri::gather_shape(bc, realw);
    g.ntiles = ceil_div(M, kTile);
    g.vblocks = ceil_div(N, g.shape.voxels_per_cta);
    const int64_t slots = int64_t(sms) * g.shape.min_blocks;
    g.splits = (g.ntiles > 0 && g.vblocks > 0)
                   ? choose_splits(g.ntiles, g.vblocks, slots > 0 ? slots : 1, bc, N)
                   : 1;
    g.rec_bytes = g.ntiles * int64_t(g.shape.tile_floats) * 4;
    g.part_bytes = g.splits > 1 ? int64_t(g.splits) * bc * 2 * N * 4 : 0;
    return g;
}

// Coil groups of a batched call: as many 8s as fit, then at most one each of
// 4, 2, 1.  Index into the per-size plan table.
int group_index(int64_t left) { return left >= 8 ? 0 : left >= 4 ? 1 : left >= 2 ? 2 : 3; }
constexpr int kGroupSizes[4] = {8, 4, 2, 1};

int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

int grid_for(int64_t elements, int sms)
{
    int64_t g = ceil_div(elements, 256);
    const int64_t cap = int64_t(sms) * 8;
    if (g > cap) g = cap;
    return g < 1 ? 1 : int(g);
}

mri_status check_mode(int trig, int accumulate)
{
    if (trig != MRI_TRIG_ACCURATE && trig != MRI_TRIG_FAST && trig != MRI_TRIG_FAST_RR)
        return MRI_ERR_MODE;
    if (accumulate != 0 && accumulate != 1) return MRI_ERR_MODE;
    return MRI_OK;
}

float kscale_for(int trig)
{
    if (trig == MRI_TRIG_ACCURATE) return 2.0f;                  // half turns
    if (trig == MRI_TRIG_FAST) return 6.28318530717958647692f;   // radians
    return 1.0f;                                                 // turns
}

// The next event pair of an open timing window, or nullptr.
cudaEvent_t* timing_slot(DeviceState* d)
{
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    if (!d->timing || d->timed >= kMaxTimed) return nullptr;
    const int i = d->timed;
    while (d->events_made < 2 * (i + 1)) {
        if (cudaEventCreate(&d->ev[d->events_made]) != cudaSuccess) return nullptr;
        ++d->events_made;
    }
    ++d->timed;
    return &d->ev[2 * i];
}

// scratch slot of the weight bounds the tensor-core kernels scale by (a
// word per coil of a group; the grid calls' fold word and row offsets after)
constexpr int64_t kBoundBytes = 256;
static_assert((12 + mri::kTcCols / mri::kTcMinCols) * 4 <= kBoundBytes, "bound slot");

#ifndef MRI_COILS_TC_MIN
#define MRI_COILS_TC_MIN 3
#endif
// Batched F^H D: coil groups of at least this many coils (up to 8) run on the
// tensor cores (coils_tc_kernel), smaller ones on the per-pair coil kernels.
constexpr int kTcCoilsMin = MRI_COILS_TC_MIN;

// Coils of a batched call that the per-pair kernels take: all of them without
// tensor-core groups, else what is left after groups of 8 and one group of
// the remainder when it has at least kTcCoilsMin coils.
int64_t pair_coils(bool tc, int64_t B)
{
    if (!tc) return B;
    const int64_t r = B % mri::kCtCoils;
    return r >= kTcCoilsMin ? 0 : r;
}

bool use_coils_tc(bool realw, bool forward, int64_t B)
{
    return !realw && !forward && B >= kTcCoilsMin;
}

struct CoilTcPlan {
    int64_t ntiles;
    int64_t vblocks;
    int splits;
    int64_t rec_bytes;
    int64_t s_bytes;
    int64_t part_bytes;
    int64_t scratch() const
    {
        return align256(rec_bytes) + kBoundBytes + align256(s_bytes) + part_bytes;
    }
};

// nb: coils of the largest group (the partial sums of a split are per coil)
CoilTcPlan plan_coils_tc(int64_t M, int64_t N, int sms, int nb)
{
    CoilTcPlan g{};
    g.ntiles = ceil_div(M, mri::kTcTile);
    g.vblocks = ceil_div(N, mri::kCtRows);
    // a tile is ~0.5 us of a CTA (two per SM); filling and draining the
    // operand pipeline costs a few tiles
    g.splits = (g.ntiles > 0 && g.vblocks > 0)
                   ? choose_splits(g.ntiles, g.vblocks, int64_t(sms > 0 ? sms : 1) * 2, nb, N,
                                   0.5, 3.0)
                   : 1;
    g.rec_bytes = g.ntiles * int64_t(mri::kCtRecBytes);
    g.s_bytes = g.ntiles * int64_t(mri::kCtBBytes);
    g.part_bytes = g.splits > 1 ? int64_t(g.splits) * nb * 2 * N * 4 : 0;
    return g;
}

// One tensor-core coil group (coils b0 .. b0 + nb - 1, nb <= 8): records of 8
// coils (absent ones weight 0) and a weight bound per coil, the weight tiles
// (each coil scaled by its power of two), the gather, the reduction of the
// splits.
mri_status run_coils_tc_group(DeviceState* d, const CoilTcPlan& g, const float* kx,
                              const float* ky, const float* kz, const float* x, const float* y,
                              const float* z, const float* rPhi, const float* iPhi,
                              const float* rD, const float* iD, int64_t b0, int nb, int64_t M,
                              int64_t N, float* out_r, float* out_i, int trig, int accumulate,
                              char* scratch, cudaStream_t s)
{
    float* rec = reinterpret_cast<float*>(scratch);
    unsigned int* wbound = reinterpret_cast<unsigned int*>(scratch + align256(g.rec_bytes));
    unsigned char* s_tab =
        reinterpret_cast<unsigned char*>(scratch + align256(g.rec_bytes) + kBoundBytes);
    float* part = reinterpret_cast<float*>(scratch + align256(g.rec_bytes) + kBoundBytes +
                                           align256(g.s_bytes));
    mri::PrepParams pp{kx, ky, kz, rPhi, iPhi, rD, iD, M, b0, g.ntiles, kscale_for(trig), rec};
    pp.wbound = wbound;
    pp.bound_per_coil = true;
    pp.coils_valid = nb;
    if (cudaMemsetAsync(wbound, 0, mri::kCtCoils * sizeof(unsigned int), s) != cudaSuccess ||
        mri::launch_prep_grid_tc(false, mri::kCtCoils, pp,
                                 grid_for(g.ntiles * mri::kTcTile, d->sms), s) != cudaSuccess ||
        mri::launch_build_mu_tiles(rec, g.ntiles, wbound, s_tab,
                                   grid_for(g.ntiles * mri::kCtCoils * (mri::kTcTile / 8), d->sms),
                                   s) != cudaSuccess)
        return cuda_fail();

    mri::CoilTcParams cp{};
    cp.rec = rec;
    cp.s_tab = s_tab;
    cp.bounds = wbound;
    cp.ntiles = g.ntiles;
    cp.splits = g.splits;
    cp.x = x;
    cp.y = y;
    cp.z = z;
    cp.N = N;
    cp.coils = nb;
    cp.err = d->err;
    if (g.splits == 1) {
        cp.out_r = out_r + b0 * N;
        cp.out_i = out_i + b0 * N;
        cp.coil_stride = N;
        cp.split_stride = 0;
        cp.accumulate = accumulate;
    } else {
        // partials [split][coil][r / i][N], the reduction's layout
        cp.out_r = part;
        cp.out_i = part + N;
        cp.coil_stride = 2 * N;
        cp.split_stride = int64_t(nb) * 2 * N;
        cp.accumulate = 0;
    }
    const dim3 grid(unsigned(g.vblocks), unsigned(g.splits), 1);
    cudaEvent_t* ev = timing_slot(d);
    if (ev && cudaEventRecord(ev[0], s) != cudaSuccess) return cuda_fail();
    if (mri::launch_gather_coils_tc(trig, cp, grid, s) != cudaSuccess) return cuda_fail();
    if (ev && cudaEventRecord(ev[1], s) != cudaSuccess) return cuda_fail();
    if (g.splits > 1 &&
        mri::launch_reduce(part, g.splits, nb, N, out_r + b0 * N, out_i + b0 * N, N, accumulate,
                           grid_for(int64_t(nb) * 2 * N, d->sms), s) != cudaSuccess)
        return cuda_fail();
    return MRI_OK;
}

// One gather (one coil group): prep records, gather, reduce splits.
mri_status run_group(DeviceState* d, const GroupPlan& g, int sms, const float* kx, const float* ky,
                     const float* kz, const float* x, const float* y, const float* z,
                     const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                     int64_t b0, int64_t M, int64_t N, float* out_r, float* out_i, int trig,
                     int accumulate, char* scratch, unsigned int* err, cudaStream_t s,
                     bool forward)
{
    float* rec = reinterpret_cast<float*>(scratch);
    float* part = reinterpret_cast<float*>(scratch + align256(g.rec_bytes));

    mri::PrepParams pp{kx, ky, kz, rPhi, iPhi, rD, iD, M, b0, g.ntiles,
                       mri::gather_kscale(g.bc, trig), rec};
    if (forward) {
        // e^{-i2pi k.x}: the sign goes into the record scale; weight = rho
        pp.kscale = -pp.kscale;
        pp.unit_phi = true;
    }
    if (mri::launch_prep(g.bc, g.realw, pp, grid_for(g.ntiles * kTile, sms), s) != cudaSuccess)
        return cuda_fail();

    mri::GatherParams gp{};
    gp.rec = rec;
    gp.ntiles = g.ntiles;
    gp.splits = g.splits;
    gp.x = x;
    gp.y = y;
    gp.z = z;
    gp.N = N;
    gp.err = err;
    if (g.splits == 1) {
        gp.out_r = out_r + b0 * N;
        gp.out_i = out_i + b0 * N;
        gp.coil_stride = N;
        gp.split_stride = 0;
        gp.accumulate = accumulate;
    } else {
        gp.out_r = part;
        gp.out_i = part + N;
        gp.coil_stride = 2 * N;
        gp.split_stride = int64_t(g.bc) * 2 * N;
        gp.accumulate = 0;
    }
    dim3 grid(unsigned(g.vblocks), unsigned(g.splits), 1);
    cudaEvent_t* ev = timing_slot(d);
    if (ev && cudaEventRecord(ev[0], s) != cudaSuccess) return cuda_fail();
    if (mri::launch_gather(g.bc, g.realw, trig, gp, grid, s) != cudaSuccess) return cuda_fail();
    if (ev && cudaEventRecord(ev[1], s) != cudaSuccess) return cuda_fail();

    if (g.splits > 1) {
        if (mri::launch_reduce(part, g.splits, g.bc, N, out_r + b0 * N, out_i + b0 * N, N,
                               accumulate, grid_for(int64_t(g.bc) * 2 * N, sms),
                               s) != cudaSuccess)
            return cuda_fail();
    }
    return MRI_OK;
}

// One plan per coil-group size (Q: only the single-weight plan, index 3).
void group_plans(bool realw, int64_t B, int64_t M, int64_t N, int sms, GroupPlan plans[4],
                 bool used[4])
{
    for (int i = 0; i < 4; ++i) used[i] = false;
    if (realw) {
        plans[3] = plan_group(1, true, M, N, sms);
        used[3] = true;
        return;
    }
    if (B >= 8) used[0] = true;
    const int64_t rest = B % 8;
    if (rest >= 4) used[1] = true;
    if (rest % 4 >= 2) used[2] = true;
    if (rest % 2 == 1) used[3] = true;
    for (int i = 0; i < 4; ++i)
        if (used[i]) plans[i] = plan_group(kGroupSizes[i], false, M, N, sms);
}

// Shared driver of mri_fhd / mri_q / mri_fhd_batched after argument checks.
mri_status run_gather_call(bool realw, int64_t B, const float* kx, const float* ky,
                           const float* kz, const float* x, const float* y, const float* z,
                           const float* rPhi, const float* iPhi, const float* rD,
                           const float* iD, int64_t M, int64_t N, float* out_r, float* out_i,
                           int trig, int accumulate, DeviceState* d, cudaStream_t s,
                           bool forward = false)
{
    if (M == 0) {
        if (!accumulate) {
            if (mri::launch_zero(out_r, B * N, grid_for(B * N, d->sms), s) != cudaSuccess ||
                mri::launch_zero(out_i, B * N, grid_for(B * N, d->sms), s) != cudaSuccess)
                return cuda_fail();
        }
        return MRI_OK;
    }
    // tensor-core coil groups first (coils 0 .. B - rest - 1), then the
    // per-pair groups of the rest
    const bool tc = use_coils_tc(realw, forward, B);
    const int64_t rest = pair_coils(tc, B);
    CoilTcPlan tcp{};
    if (tc) tcp = plan_coils_tc(M, N, d->sms, int(std::min<int64_t>(B - rest, mri::kCtCoils)));
    GroupPlan plans[4];
    bool used[4];
    group_plans(realw, rest, M, N, d->sms, plans, used);
    int64_t scratch_bytes = tc ? tcp.scratch() : 0;
    for (int i = 0; i < 4; ++i) {
        const int64_t b = used[i] ? align256(plans[i].rec_bytes) + plans[i].part_bytes : 0;
        if (b > scratch_bytes) scratch_bytes = b;
    }
    char* scratch = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), size_t(scratch_bytes),
                                d->pool, s) != cudaSuccess)
        return cuda_fail();

    mri_status st = MRI_OK;
    for (int64_t b0 = 0; b0 < B && st == MRI_OK;) {
        if (b0 < B - rest) {
            const int nb = int(std::min<int64_t>(B - rest - b0, mri::kCtCoils));
            st = run_coils_tc_group(d, tcp, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, b0, nb, M,
                                    N, out_r, out_i, trig, accumulate, scratch, s);
            b0 += nb;
            continue;
        }
        const int i = realw ? 3 : group_index(B - b0);
        st = run_group(d, plans[i], d->sms, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, b0, M, N,
                       out_r, out_i, trig, accumulate, scratch, d->err, s, forward);
        b0 += plans[i].bc;
    }
    if (cudaFreeAsync(scratch, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

// ---------------------------------------------------------------------------
// separable grids
// ---------------------------------------------------------------------------
struct GridPlan {
    bool tensor_cores;      // nx >= 8: the tcgen05 kernel; else coordinates
                            // expanded and the general kernel
    int bc;                 // coils per CTA
    int ncb;                // column blocks of 128
    int64_t ntiles;
    int64_t vblocks;
    int rows_per_cta;
    int splits;
    int64_t rec_bytes;
    int64_t part_bytes;
    int64_t s_bytes;        // the B operand tiles
    int fold;               // grid rows folded into one block's columns (nx <= 64), else 1
    int64_t vblocks_launch; // CTAs along the rows launched: the unfolded count when
                            // fold > 1 (the device-side check may refuse the fold)
};

// A group of coils of a tensor-core grid call: coils b0 .. b0 + nb - 1 run in
// one launch whose CTAs hold bc coils each (bc >= nb; the rest carry weight 0).
struct TcGroup {
    int64_t b0;
    int nb;
    int bc;
};

// Groups of 8 coils; a remainder of 2..4 runs as one padded group of 4, 5..7
// as a padded group of 8 (the MMA work of a launch does not depend on how
// many of its coils are real), a single coil alone.
std::vector<TcGroup> tc_groups(int64_t B)
{
    std::vector<TcGroup> g;
    int64_t b0 = 0;
    for (; B - b0 >= 8; b0 += 8) g.push_back({b0, 8, 8});
    const int r = int(B - b0);
    if (r == 1) g.push_back({b0, 1, 1});
    else if (r >= 2 && r <= 4) g.push_back({b0, r, 4});
    else if (r >= 5) g.push_back({b0, r, 8});
    return g;
}

GridPlan plan_grid(bool realw, int64_t M, int nx, int ny, int nz, int sms, int bc = 1, int nb = 1)
{
    GridPlan g{};
    g.tensor_cores = mri::grid_tc_fits(nx);
    if (!g.tensor_cores) return g;
    const int64_t N = int64_t(nx) * ny * nz;
    g.bc = bc;
    g.ncb = mri::grid_tc_col_blocks(nx);
    g.rows_per_cta = mri::kTcRows / bc;
    g.ntiles = ceil_div(M, mri::kTcTile);
    g.fold = mri::grid_tc_fold(nx, ny);
    // planned for the folded rows (the y axes of images are evenly spaced)
    g.vblocks = ceil_div(int64_t(ny / g.fold) * nz, g.rows_per_cta);
    g.vblocks_launch = ceil_div(int64_t(ny) * nz, g.rows_per_cta);
    g.splits = (g.ntiles > 0 && g.vblocks > 0)
                   ? choose_splits(g.ntiles, g.vblocks * g.ncb, sms > 0 ? sms : 1, nb, N, 1.0, 3.0)
                   : 1;
    g.rec_bytes = g.ntiles * int64_t(realw ? 4 : 3 + 2 * bc) * mri::kTcTile * 4;
    g.part_bytes = g.splits > 1 ? int64_t(g.splits) * nb * 2 * N * 4 : 0;
    g.s_bytes = g.ntiles * g.ncb * int64_t(mri::kTcStageBytes);
    return g;
}

// One launch of the tensor-core grid kernel (timing events around it).
mri_status launch_grid_gather(const GridPlan& g, bool realw, int trig,
                              const mri::GridParams& gp, DeviceState* d, cudaStream_t s)
{
    mri_status st = MRI_OK;
    cudaEvent_t* ev = timing_slot(d);
    if (ev && cudaEventRecord(ev[0], s) != cudaSuccess) st = cuda_fail();
    const dim3 grid(unsigned(g.vblocks_launch), unsigned(g.splits), unsigned(g.ncb));
    if (st == MRI_OK && mri::launch_grid_tc(realw, trig, g.bc, gp, grid, s) != cudaSuccess)
        st = cuda_fail();
    if (st == MRI_OK && ev && cudaEventRecord(ev[1], s) != cudaSuccess) st = cuda_fail();
    return st;
}

mri::GridParams grid_params(const GridPlan& g, const float* rec, const float* xs, int nx,
                            const float* ys, int ny, const float* zs, int nz, DeviceState* d)
{
    mri::GridParams gp{};
    gp.rec = rec;
    gp.ntiles = g.ntiles;
    gp.splits = g.splits;
    gp.xs = xs;
    gp.ys = ys;
    gp.zs = zs;
    gp.nx = nx;
    gp.ny = ny;
    gp.nz = nz;
    gp.rows_per_cta = g.rows_per_cta;
    gp.err = d->err;
    gp.coils = 1;
    return gp;
}

// F^H D over B coils (coil-major rD / iD [B][M], outputs [B][N]) or Q (B = 1)
// on a separable grid.
mri_status run_grid_call(bool realw, int64_t B, const float* kx, const float* ky, const float* kz,
                         const float* xs, int nx, const float* ys, int ny, const float* zs,
                         int nz, const float* rPhi, const float* iPhi, const float* rD,
                         const float* iD, int64_t M, float* out_r, float* out_i, int trig,
                         int accumulate, DeviceState* d, cudaStream_t s)
{
    const int64_t N = int64_t(nx) * ny * nz;
    if (M == 0) {
        if (!accumulate) {
            if (mri::launch_zero(out_r, B * N, grid_for(B * N, d->sms), s) != cudaSuccess ||
                mri::launch_zero(out_i, B * N, grid_for(B * N, d->sms), s) != cudaSuccess)
                return cuda_fail();
        }
        return MRI_OK;
    }
    if (!mri::grid_tc_fits(nx)) {
        // expand the coordinates and take the general kernel
        float* xyz = nullptr;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&xyz), size_t(3 * N) * 4, d->pool,
                                    s) != cudaSuccess)
            return cuda_fail();
        mri_status st = MRI_OK;
        if (mri::launch_expand_grid(xs, ys, zs, nx, ny, N, xyz, xyz + N, xyz + 2 * N,
                                    grid_for(N, d->sms), s) != cudaSuccess)
            st = cuda_fail();
        if (st == MRI_OK)
            st = run_gather_call(realw, B, kx, ky, kz, xyz, xyz + N, xyz + 2 * N, rPhi, iPhi, rD,
                                 iD, M, N, out_r, out_i, trig, accumulate, d, s);
        if (cudaFreeAsync(xyz, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
        return st;
    }
    // tensor cores: coil groups sharing one table of B operand tiles
    const std::vector<TcGroup> groups = realw ? std::vector<TcGroup>{{0, 1, 1}} : tc_groups(B);
    std::vector<GridPlan> plans;
    int64_t rec_max = 0, part_max = 0;
    for (const TcGroup& grp : groups) {
        plans.push_back(plan_grid(realw, M, nx, ny, nz, d->sms, grp.bc, grp.nb));
        rec_max = std::max(rec_max, plans.back().rec_bytes);
        part_max = std::max(part_max, plans.back().part_bytes);
    }
    const int64_t s_bytes = plans[0].s_bytes;
    char* scratch = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch),
                                size_t(align256(rec_max) + kBoundBytes + align256(part_max) +
                                       align256(s_bytes)),
                                d->pool, s) != cudaSuccess)
        return cuda_fail();
    float* rec = reinterpret_cast<float*>(scratch);
    // the bound slot: a weight bound word per coil of a group (8), the fold
    // check's word, its row offsets (up to 16)
    unsigned int* wbound = reinterpret_cast<unsigned int*>(scratch + align256(rec_max));
    unsigned int* fold_ok = wbound + 8;
    float* fold_dy = reinterpret_cast<float*>(wbound + 12);
    float* part = reinterpret_cast<float*>(scratch + align256(rec_max) + kBoundBytes);
    unsigned char* s_tab = reinterpret_cast<unsigned char*>(scratch + align256(rec_max) +
                                                            kBoundBytes + align256(part_max));
    mri_status st = MRI_OK;
    // narrow grids: whether ys allows folding G rows into a block's columns
    const int fold = plans[0].fold;
    if (fold > 1 &&
        mri::launch_grid_fold_check(ys, ny, fold, fold_ok, fold_dy, s) != cudaSuccess)
        st = cuda_fail();
    for (size_t i = 0; i < groups.size() && st == MRI_OK; ++i) {
        const TcGroup& grp = groups[i];
        const GridPlan& g = plans[i];
        const int fields = realw ? 4 : 3 + 2 * grp.bc;
        mri::PrepParams pp{kx, ky, kz, rPhi, iPhi, rD, iD, M, grp.b0, g.ntiles, kscale_for(trig),
                           rec};
        pp.wbound = wbound;
        pp.bound_per_coil = true;   // each coil of a group scaled by its own power of two
        pp.coils_valid = grp.nb;
        if (cudaMemsetAsync(wbound, 0, grp.bc * sizeof(unsigned int), s) != cudaSuccess ||
            mri::launch_prep_grid_tc(realw, grp.bc, pp,
                                     grid_for(g.ntiles * mri::kTcTile, d->sms), s) != cudaSuccess ||
            mri::launch_scale_records(rec, fields, g.ntiles, wbound, realw ? 1 : grp.bc,
                                      grid_for(g.ntiles * (fields - 3) * mri::kTcTile, d->sms),
                                      s) != cudaSuccess)
            st = cuda_fail();
        // the B tiles of a coil group depend on kx and the columns only: built
        // once and shared; a single-coil launch carries its weight in B, so
        // its table is built from its own records (in place: the launches
        // before it on this stream are done with the old one)
        if (st == MRI_OK && (i == 0 || grp.bc == 1) &&
            mri::launch_build_ex_tiles(trig, grp.bc == 1, rec, fields, g.ntiles, xs, nx, s_tab,
                                       grid_for(g.ntiles * mri::grid_tc_col_blocks(nx) * 512,
                                                d->sms),
                                       s, fold, fold_ok, fold_dy) != cudaSuccess)
            st = cuda_fail();
        mri::GridParams gp = grid_params(g, rec, xs, nx, ys, ny, zs, nz, d);
        gp.wbound = wbound;
        gp.s_tab = s_tab;
        gp.coils = grp.nb;
        gp.ncb = mri::grid_tc_col_blocks(nx);
        gp.fold = fold;
        gp.log2_fw = mri::grid_tc_fold_log2_width(fold);
        gp.fold_ok = fold_ok;
        if (g.splits == 1) {
            gp.out_r = out_r + grp.b0 * N;
            gp.out_i = out_i + grp.b0 * N;
            gp.coil_stride = N;
            gp.split_stride = 0;
            gp.accumulate = accumulate;
        } else {
            // partials [split][coil][r / i][N], the reduction's layout
            gp.out_r = part;
            gp.out_i = part + N;
            gp.coil_stride = 2 * N;
            gp.split_stride = int64_t(grp.nb) * 2 * N;
            gp.accumulate = 0;
        }
        if (st == MRI_OK) st = launch_grid_gather(g, realw, trig, gp, d, s);
        if (st == MRI_OK && g.splits > 1 &&
            mri::launch_reduce(part, g.splits, grp.nb, N, out_r + grp.b0 * N, out_i + grp.b0 * N,
                               N, accumulate, grid_for(int64_t(grp.nb) * 2 * N, d->sms),
                               s) != cudaSuccess)
            st = cuda_fail();
    }
    if (cudaFreeAsync(scratch, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

mri_status check_grid_dims(int nx, int ny, int nz, int64_t M)
{
    if (nx < 0 || ny < 0 || nz < 0 || M < 0 || M > kMaxM) return MRI_ERR_SIZE;
    if (int64_t(nx) * ny * nz > kMaxN) return MRI_ERR_SIZE;
    return MRI_OK;
}

mri_status check_sizes(int64_t B, int64_t M, int64_t N)
{
    if (B < 1 || M < 0 || N < 0) return MRI_ERR_SIZE;
    if (B > kMaxB || M > kMaxM || N > kMaxN) return MRI_ERR_SIZE;
    if (N > 0 && B > kMaxBN / N) return MRI_ERR_SIZE;
    return MRI_OK;
}

// Full argument check shared by the gather entry points.
mri_status prepare(int trig, int accumulate, int64_t B, int64_t M, int64_t N,
                   const void* const* sample_ptrs, int n_sample, const void* const* voxel_ptrs,
                   int n_voxel, DeviceState** d)
{
    mri_status st = check_mode(trig, accumulate);
    if (st != MRI_OK) return st;
    if ((st = check_sizes(B, M, N)) != MRI_OK) return st;
    if (N == 0) return MRI_OK;
    if ((st = check_ptrs(voxel_ptrs, n_voxel, -1)) != MRI_OK) return st;
    if (M > 0 && (st = check_ptrs(sample_ptrs, n_sample, -1)) != MRI_OK) return st;
    int dev = -1;
    if ((st = device_state(d, &dev)) != MRI_OK) return st;
    if ((st = check_ptrs(voxel_ptrs, n_voxel, dev)) != MRI_OK) return st;
    if (M > 0 && (st = check_ptrs(sample_ptrs, n_sample, dev)) != MRI_OK) return st;
    return MRI_OK;
}

}  // namespace

namespace mri {

// Device address of the error word on device `dev` (which must be current):
// a symbol lookup, cached per device, that creates no pool and allocates
// nothing.  Used by the allocation-free entry point.
unsigned int* error_word_address(int dev)
{
    static std::mutex m;
    static unsigned int* addr[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(m);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        addr[dev] = static_cast<unsigned int*>(p);
    }
    return addr[dev];
}

// Residency of caller pointers on device `dev` (cudaPointerGetAttributes per
// pointer; no allocation): MRI_OK, or MRI_ERR_NOT_DEVICE for host, page-locked
// host or another device's memory.  Used by the allocation-free entry point.
mri_status check_device_ptrs(const void* const* ptrs, int n, int dev)
{
    return check_ptrs(ptrs, n, dev);
}

}  // namespace mri

extern "C" {

mri_status mri_mu(const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                  float* rMu, float* iMu, int64_t M, void* stream)
{
    if (M < 0 || M > kMaxM) return MRI_ERR_SIZE;
    if (M == 0) return MRI_OK;
    const void* ptrs[6] = {rPhi, iPhi, rD, iD, rMu, iMu};
    mri_status st = check_ptrs(ptrs, 6, -1);
    if (st != MRI_OK) return st;
    DeviceState* d = nullptr;
    int dev = -1;
    if ((st = device_state(&d, &dev)) != MRI_OK) return st;
    if ((st = check_ptrs(ptrs, 6, dev)) != MRI_OK) return st;
    if (mri::launch_mu(rPhi, iPhi, rD, iD, rMu, iMu, M, grid_for(M, d->sms),
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return cuda_fail();
    return MRI_OK;
}

mri_status mri_fhd(const float* kx, const float* ky, const float* kz, const float* x,
                   const float* y, const float* z, const float* rPhi, const float* iPhi,
                   const float* rD, const float* iD, int64_t M, int64_t N, float* rFhD,
                   float* iFhD, mri_trig trig, int accumulate, void* stream)
{
    const void* sp[7] = {kx, ky, kz, rPhi, iPhi, rD, iD};
    const void* vp[5] = {x, y, z, rFhD, iFhD};
    DeviceState* d = nullptr;
    mri_status st = prepare(int(trig), accumulate, 1, M, N, sp, 7, vp, 5, &d);
    if (st != MRI_OK || N == 0) return st;
    return run_gather_call(false, 1, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, M, N, rFhD, iFhD,
                           int(trig), accumulate, d, static_cast<cudaStream_t>(stream));
}

mri_status mri_q(const float* kx, const float* ky, const float* kz, const float* x,
                 const float* y, const float* z, const float* rPhi, const float* iPhi,
                 int64_t M, int64_t N, float* rQ, float* iQ, mri_trig trig, int accumulate,
                 void* stream)
{
    const void* sp[5] = {kx, ky, kz, rPhi, iPhi};
    const void* vp[5] = {x, y, z, rQ, iQ};
    DeviceState* d = nullptr;
    mri_status st = prepare(int(trig), accumulate, 1, M, N, sp, 5, vp, 5, &d);
    if (st != MRI_OK || N == 0) return st;
    return run_gather_call(true, 1, kx, ky, kz, x, y, z, rPhi, iPhi, nullptr, nullptr, M, N, rQ,
                           iQ, int(trig), accumulate, d, static_cast<cudaStream_t>(stream));
}

mri_status mri_fhd_batched(const float* kx, const float* ky, const float* kz, const float* x,
                           const float* y, const float* z, const float* rPhi,
                           const float* iPhi, const float* rD, const float* iD, int64_t B,
                           int64_t M, int64_t N, float* rFhD, float* iFhD, mri_trig trig,
                           int accumulate, void* stream)
{
    const void* sp[7] = {kx, ky, kz, rPhi, iPhi, rD, iD};
    const void* vp[5] = {x, y, z, rFhD, iFhD};
    DeviceState* d = nullptr;
    mri_status st = prepare(int(trig), accumulate, B, M, N, sp, 7, vp, 5, &d);
    if (st != MRI_OK || N == 0) return st;
    return run_gather_call(false, B, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD, M, N, rFhD, iFhD,
                           int(trig), accumulate, d, static_cast<cudaStream_t>(stream));
}

mri_status mri_forward(const float* kx, const float* ky, const float* kz, const float* x,
                       const float* y, const float* z, const float* rRho, const float* iRho,
                       int64_t M, int64_t N, float* rD, float* iD, mri_trig trig, int accumulate,
                       void* stream)
{
    // the gather with roles exchanged: the N voxels are summed over, the M
    // k-space samples are the outputs
    const void* sp[5] = {x, y, z, rRho, iRho};
    const void* vp[5] = {kx, ky, kz, rD, iD};
    DeviceState* d = nullptr;
    mri_status st = prepare(int(trig), accumulate, 1, N, M, sp, 5, vp, 5, &d);
    if (st != MRI_OK || M == 0) return st;
    return run_gather_call(false, 1, x, y, z, kx, ky, kz, nullptr, nullptr, rRho, iRho, N, M, rD,
                           iD, int(trig), accumulate, d, static_cast<cudaStream_t>(stream),
                           /*forward=*/true);
}

mri_status mri_forward_grid(const float* kx, const float* ky, const float* kz, const float* xs,
                            int nx, const float* ys, int ny, const float* zs, int nz,
                            const float* rRho, const float* iRho, int64_t M, float* rD,
                            float* iD, mri_trig trig, int accumulate, void* stream)
{
    mri_status st = check_mode(int(trig), accumulate);
    if (st != MRI_OK) return st;
    if ((st = check_grid_dims(nx, ny, nz, M)) != MRI_OK) return st;
    const int64_t N = int64_t(nx) * ny * nz;
    // the voxels (rho and the axes) are summed over, the M samples are outputs
    const void* sp[5] = {xs, ys, zs, rRho, iRho};
    const void* vp[5] = {kx, ky, kz, rD, iD};
    DeviceState* d = nullptr;
    if ((st = prepare(int(trig), accumulate, 1, N, M, sp, 5, vp, 5, &d)) != MRI_OK || M == 0)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {
        if (!accumulate &&
            (mri::launch_zero(rD, M, grid_for(M, d->sms), s) != cudaSuccess ||
             mri::launch_zero(iD, M, grid_for(M, d->sms), s) != cudaSuccess))
            return cuda_fail();
        return MRI_OK;
    }
    if (!mri::grid_tc_fwd_fits(nx)) {
        // expand the coordinates and take the general gather
        float* xyz = nullptr;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&xyz), size_t(3 * N) * 4, d->pool,
                                    s) != cudaSuccess)
            return cuda_fail();
        if (mri::launch_expand_grid(xs, ys, zs, nx, ny, N, xyz, xyz + N, xyz + 2 * N,
                                    grid_for(N, d->sms), s) != cudaSuccess)
            st = cuda_fail();
        if (st == MRI_OK)
            st = run_gather_call(false, 1, xyz, xyz + N, xyz + 2 * N, kx, ky, kz, nullptr, nullptr,
                                 rRho, iRho, N, M, rD, iD, int(trig), accumulate, d, s,
                                 /*forward=*/true);
        if (cudaFreeAsync(xyz, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
        return st;
    }
    // tensor cores: a CTA per 128 samples, row blocks split when too few CTAs
    const int64_t rows = int64_t(ny) * nz;
    const int64_t row_blocks = ceil_div(rows, int64_t(mri::kFwRows));
    const int ncb = mri::grid_tc_col_blocks(nx);
    const int64_t sample_tiles = ceil_div(M, int64_t(mri::kFwSamples));
    // a row block of 64 rows and one column block: about half a microsecond
    const int splits = choose_splits(row_blocks, sample_tiles, d->sms > 0 ? d->sms : 1, 1, M,
                                     0.5 * ncb, 3.0);
    const int64_t tab_bytes =
        row_blocks * ncb * mri::kFwChunks * int64_t(mri::kFwChunkBytes);
    const int64_t yz_bytes = row_blocks * mri::kFwRows * 8 + row_blocks * (mri::kFwRows / 8) * 4;
    const int64_t part_bytes = splits > 1 ? int64_t(splits) * 2 * M * 4 : 0;
    char* scratch = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch),
                                size_t(align256(tab_bytes) + align256(yz_bytes) + kBoundBytes +
                                       part_bytes),
                                d->pool, s) != cudaSuccess)
        return cuda_fail();
    unsigned char* tab = reinterpret_cast<unsigned char*>(scratch);
    float2* yz_rows = reinterpret_cast<float2*>(scratch + align256(tab_bytes));
    float* row_step = reinterpret_cast<float*>(yz_rows + row_blocks * mri::kFwRows);
    unsigned int* bound =
        reinterpret_cast<unsigned int*>(scratch + align256(tab_bytes) + align256(yz_bytes));
    float* part = reinterpret_cast<float*>(scratch + align256(tab_bytes) + align256(yz_bytes) +
                                           kBoundBytes);
    if (mri::launch_forward_grid_prep(rRho, iRho, rows, nx, row_blocks, ys, ny, zs, bound, tab,
                                      yz_rows, row_step, grid_for(row_blocks * ncb * 2048, d->sms),
                                      s) != cudaSuccess)
        st = cuda_fail();
    mri::FwdParams fp{};
    fp.kx = kx;
    fp.ky = ky;
    fp.kz = kz;
    fp.M = M;
    fp.kscale = kscale_for(int(trig));
    fp.xs = xs;
    fp.nx = nx;
    fp.ncb = ncb;
    fp.yz_rows = yz_rows;
    fp.row_step = row_step;
    fp.row_blocks = row_blocks;
    fp.splits = splits;
    fp.rho_tab = tab;
    fp.bound = bound;
    fp.out_r = splits > 1 ? part : rD;
    fp.out_i = splits > 1 ? part + M : iD;
    fp.split_stride = splits > 1 ? 2 * M : 0;
    fp.accumulate = splits > 1 ? 0 : accumulate;
    fp.err = d->err;
    if (st == MRI_OK) {
        cudaEvent_t* ev = timing_slot(d);
        if (ev && cudaEventRecord(ev[0], s) != cudaSuccess) st = cuda_fail();
        const dim3 grid(unsigned(sample_tiles), unsigned(splits), 1);
        if (st == MRI_OK && mri::launch_forward_grid_tc(int(trig), fp, grid, s) != cudaSuccess)
            st = cuda_fail();
        if (st == MRI_OK && ev && cudaEventRecord(ev[1], s) != cudaSuccess) st = cuda_fail();
    }
    if (st == MRI_OK && splits > 1 &&
        mri::launch_reduce(part, splits, 1, M, rD, iD, M, accumulate, grid_for(2 * M, d->sms),
                           s) != cudaSuccess)
        st = cuda_fail();
    if (cudaFreeAsync(scratch, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

mri_status mri_fhd_grid(const float* kx, const float* ky, const float* kz, const float* xs,
                        int nx, const float* ys, int ny, const float* zs, int nz,
                        const float* rPhi, const float* iPhi, const float* rD, const float* iD,
                        int64_t M, float* rFhD, float* iFhD, mri_trig trig, int accumulate,
                        void* stream)
{
    mri_status st = check_mode(int(trig), accumulate);
    if (st != MRI_OK) return st;
    if ((st = check_grid_dims(nx, ny, nz, M)) != MRI_OK) return st;
    const int64_t N = int64_t(nx) * ny * nz;
    const void* sp[7] = {kx, ky, kz, rPhi, iPhi, rD, iD};
    const void* vp[5] = {xs, ys, zs, rFhD, iFhD};
    DeviceState* d = nullptr;
    if ((st = prepare(int(trig), accumulate, 1, M, N, sp, 7, vp, 5, &d)) != MRI_OK || N == 0)
        return st;
    return run_grid_call(false, 1, kx, ky, kz, xs, nx, ys, ny, zs, nz, rPhi, iPhi, rD, iD, M,
                         rFhD, iFhD, int(trig), accumulate, d, static_cast<cudaStream_t>(stream));
}

mri_status mri_fhd_batched_grid(const float* kx, const float* ky, const float* kz,
                                const float* xs, int nx, const float* ys, int ny, const float* zs,
                                int nz, const float* rPhi, const float* iPhi, const float* rD,
                                const float* iD, int64_t B, int64_t M, float* rFhD, float* iFhD,
                                mri_trig trig, int accumulate, void* stream)
{
    mri_status st = check_mode(int(trig), accumulate);
    if (st != MRI_OK) return st;
    if ((st = check_grid_dims(nx, ny, nz, M)) != MRI_OK) return st;
    const int64_t N = int64_t(nx) * ny * nz;
    const void* sp[7] = {kx, ky, kz, rPhi, iPhi, rD, iD};
    const void* vp[5] = {xs, ys, zs, rFhD, iFhD};
    DeviceState* d = nullptr;
    if ((st = prepare(int(trig), accumulate, B, M, N, sp, 7, vp, 5, &d)) != MRI_OK || N == 0)
        return st;
    return run_grid_call(false, B, kx, ky, kz, xs, nx, ys, ny, zs, nz, rPhi, iPhi, rD, iD, M,
                         rFhD, iFhD, int(trig), accumulate, d, static_cast<cudaStream_t>(stream));
}

mri_status mri_q_grid(const float* kx, const float* ky, const float* kz, const float* xs, int nx,
                      const float* ys, int ny, const float* zs, int nz, const float* rPhi,
                      const float* iPhi, int64_t M, float* rQ, float* iQ, mri_trig trig,
                      int accumulate, void* stream)
{
    mri_status st = check_mode(int(trig), accumulate);
    if (st != MRI_OK) return st;
    if ((st = check_grid_dims(nx, ny, nz, M)) != MRI_OK) return st;
    const int64_t N = int64_t(nx) * ny * nz;
    const void* sp[5] = {kx, ky, kz, rPhi, iPhi};
    const void* vp[5] = {xs, ys, zs, rQ, iQ};
    DeviceState* d = nullptr;
    if ((st = prepare(int(trig), accumulate, 1, M, N, sp, 5, vp, 5, &d)) != MRI_OK || N == 0)
        return st;
    return run_grid_call(true, 1, kx, ky, kz, xs, nx, ys, ny, zs, nz, rPhi, iPhi, nullptr,
                         nullptr, M, rQ, iQ, int(trig), accumulate, d,
                         static_cast<cudaStream_t>(stream));
}

namespace {
mri_status plan_grid_call(int kind, int64_t B, int64_t M, int nx, int ny, int nz, int num_sms,
                          mri_plan* plan)
{
    if (plan == nullptr) return MRI_ERR_NULL;
    if (kind != MRI_KIND_FHD && kind != MRI_KIND_Q && kind != MRI_KIND_FHD_BATCHED)
        return MRI_ERR_MODE;
    mri_status st = check_grid_dims(nx, ny, nz, M);
    if (st != MRI_OK) return st;
    if (num_sms < 0 || B < 1 || B > kMaxB) return MRI_ERR_SIZE;
    if (num_sms == 0) {
        DeviceState* d = nullptr;
        if ((st = device_state(&d, nullptr)) != MRI_OK && st != MRI_ERR_UNSUPPORTED_DEVICE)
            return st;
        num_sms = d->sms;
    }
    const bool realw = kind == MRI_KIND_Q;
    const int64_t N = int64_t(nx) * ny * nz;
    std::memset(plan, 0, sizeof(*plan));
    if (N == 0) return MRI_OK;
    if (M == 0) {
        plan->launches = 2;
        return MRI_OK;
    }
    const GridPlan g = plan_grid(realw, M, nx, ny, nz, num_sms);
    if (!g.tensor_cores) {
        // expanded coordinates, then the general plan
        st = mri_plan_gather(B > 1 ? MRI_KIND_FHD_BATCHED : kind, B, M, N, num_sms, plan);
        plan->launches += 1;
        plan->scratch_bytes += 3 * N * 4;
        return st;
    }
    plan->threads_per_cta = mri::grid_tc_threads();
    plan->samples_per_tile = mri::kTcTile;
    plan->tiles = g.ntiles;
    plan->tensor_cores = 1;
    // tensor cores: per coil group a prep, a scale, a gather and (split) a
    // reduction, plus one build of the B tiles (and one more for a trailing
    // single coil); the first group's shape is reported
    const std::vector<TcGroup> groups = realw ? std::vector<TcGroup>{{0, 1, 1}} : tc_groups(B);
    int64_t rec_max = 0, part_max = 0;
    plan->launches = 1 + (g.fold > 1 ? 1 : 0);   // the B tiles (and the fold check)
    for (size_t i = 0; i < groups.size(); ++i) {
        const GridPlan gi = plan_grid(realw, M, nx, ny, nz, num_sms, groups[i].bc, groups[i].nb);
        if (i == 0) {
            // voxels whose running sums one generating thread holds
            plan->voxels_per_thread = mri::kTcRows * mri::kTcCols / mri::kTcThreads;
            plan->voxels_per_cta = gi.rows_per_cta * mri::kTcCols;
            plan->splits = gi.splits;
            plan->voxel_ctas = gi.vblocks * gi.ncb;
            plan->grid_fold = gi.fold;
        }
        rec_max = std::max(rec_max, gi.rec_bytes);
        part_max = std::max(part_max, gi.part_bytes);
        plan->launches += 3 + (gi.splits > 1 ? 1 : 0);   // prep, scale, gather (+ reduce)
        if (i > 0 && groups[i].bc == 1) plan->launches += 1;   // its own B tiles
    }
    plan->coil_groups = int(groups.size());
    plan->scratch_bytes = align256(rec_max) + kBoundBytes + align256(part_max) + g.s_bytes;
    return MRI_OK;
}
}  // namespace

mri_status mri_plan_grid(int kind, int64_t M, int nx, int ny, int nz, int num_sms,
                         mri_plan* plan)
{
    if (kind == MRI_KIND_FHD_BATCHED) return MRI_ERR_MODE;
    return plan_grid_call(kind, 1, M, nx, ny, nz, num_sms, plan);
}

mri_status mri_plan_grid_batched(int64_t B, int64_t M, int nx, int ny, int nz, int num_sms,
                                 mri_plan* plan)
{
    return plan_grid_call(MRI_KIND_FHD_BATCHED, B, M, nx, ny, nz, num_sms, plan);
}

// ---------------------------------------------------------------------------
// the find-rho step on a grid: Toeplitz F^H F and conjugate gradients
// ---------------------------------------------------------------------------
namespace {
mri_status check_toeplitz_grid(int nx, int ny, int nz)
{
    const int m = mri::kFftMaxLen / 2;   // the doubled grid must be one FFT length
    auto ok = [&](int n) { return n >= 1 && n <= m && (n & (n - 1)) == 0; };
    return (ok(nx) && ok(ny) && ok(nz)) ? MRI_OK : MRI_ERR_SIZE;
}

bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
}  // namespace

mri_status mri_fft3(float* data, int Lx, int Ly, int Lz, int inverse, void* stream)
{
    if (inverse != 0 && inverse != 1) return MRI_ERR_MODE;
    if (!mri::fft_len_ok(Lx) || !mri::fft_len_ok(Ly) || !mri::fft_len_ok(Lz))
        return MRI_ERR_SIZE;
    if (data != nullptr && !aligned8(data)) return MRI_ERR_ALIGN;
    const void* vp[1] = {data};
    DeviceState* d = nullptr;
    mri_status st = prepare(0, 0, 1, 0, int64_t(Lx) * Ly * Lz, nullptr, 0, vp, 1, &d);
    if (st != MRI_OK) return st;
    if (mri::launch_fft3(reinterpret_cast<float2*>(data), Lx, Ly, Lz, inverse != 0, d->fft_tw,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return cuda_fail();
    return MRI_OK;
}

mri_status mri_toeplitz_kernel(const float* kx, const float* ky, const float* kz,
                               const float* rPhi, const float* iPhi, int64_t M, int nx, int ny,
                               int nz, float hx, float hy, float hz, float* K, mri_trig trig,
                               void* stream)
{
    mri_status st = check_mode(int(trig), 0);
    if (st != MRI_OK) return st;
    if ((st = check_toeplitz_grid(nx, ny, nz)) != MRI_OK) return st;
    if (!std::isfinite(hx) || !std::isfinite(hy) || !std::isfinite(hz)) return MRI_ERR_SIZE;
    if (M < 0 || M > kMaxM) return MRI_ERR_SIZE;
    if (K != nullptr && !aligned8(K)) return MRI_ERR_ALIGN;
    const int64_t N2 = int64_t(8) * nx * ny * nz;   // the doubled grid
    const void* sp[5] = {kx, ky, kz, rPhi, iPhi};
    const void* vp[1] = {K};
    DeviceState* d = nullptr;
    if ((st = prepare(int(trig), 0, 1, M, N2, sp, 5, vp, 1, &d)) != MRI_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // scratch: the difference axes, Q (real and imaginary parts) on the z
    // planes iz < nz (the others follow by conjugate symmetry), the complex
    // spectrum
    const int64_t axes_n = 2 * (int64_t(nx) + ny + nz);
    const int64_t Nq = N2 / 2;
    const int64_t q_bytes = align256(2 * Nq * 4);
    char* scratch = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch),
                                size_t(align256(axes_n * 4) + q_bytes + N2 * 8), d->pool,
                                s) != cudaSuccess)
        return cuda_fail();
    float* axes = reinterpret_cast<float*>(scratch);
    float* q_r = reinterpret_cast<float*>(scratch + align256(axes_n * 4));
    float* q_i = q_r + Nq;
    float2* spec = reinterpret_cast<float2*>(scratch + align256(axes_n * 4) + q_bytes);
    if (mri::launch_diff_axes(nx, ny, nz, hx, hy, hz, axes, s) != cudaSuccess) st = cuda_fail();
    // Q(d) = sum_m |Phi_m|^2 e^{+i 2 pi k_m . d} on the difference grid's z
    // planes 0 .. nz - 1: the grid Q path (tensor cores for 2 nx >= 8)
    if (st == MRI_OK)
        st = run_grid_call(true, 1, kx, ky, kz, axes, 2 * nx, axes + 2 * nx, 2 * ny,
                           axes + 2 * nx + 2 * ny, nz, rPhi, iPhi, nullptr, nullptr, M, q_r,
                           q_i, int(trig), 0, d, s);
    // the other planes by conjugate symmetry, the index-n planes zeroed
    // (unused by the product; without them the spectrum is real), FFT, real
    // part
    if (st == MRI_OK &&
        (mri::launch_spectrum_input(q_r, q_i, nx, ny, nz, spec, grid_for(N2, d->sms), s) !=
             cudaSuccess ||
         mri::launch_fft3(spec, 2 * nx, 2 * ny, 2 * nz, false, d->fft_tw, s) != cudaSuccess ||
         mri::launch_real_part(spec, N2, K, grid_for(N2, d->sms), s) != cudaSuccess))
        st = cuda_fail();
    if (cudaFreeAsync(scratch, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

mri_status mri_toeplitz_apply(const float* K, int nx, int ny, int nz, float lambda,
                              const float* rIn, const float* iIn, float* rOut, float* iOut,
                              int accumulate, void* stream)
{
    mri_status st = check_mode(0, accumulate);
    if (st != MRI_OK) return st;
    if ((st = check_toeplitz_grid(nx, ny, nz)) != MRI_OK) return st;
    if (!std::isfinite(lambda)) return MRI_ERR_SIZE;
    if (K != nullptr && !aligned8(K)) return MRI_ERR_ALIGN;
    const int64_t N = int64_t(nx) * ny * nz;
    const void* vp[5] = {K, rIn, iIn, rOut, iOut};
    DeviceState* d = nullptr;
    if ((st = prepare(0, accumulate, 1, 0, N, nullptr, 0, vp, 5, &d)) != MRI_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the FFT stages' work array: half the doubled grid, [nz][2 ny][2 nx]
    float2* work = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&work), size_t(4 * N) * sizeof(float2),
                                d->pool, s) != cudaSuccess)
        return cuda_fail();
    if (mri::launch_toeplitz_apply(K, nx, ny, nz, lambda, rIn,
                                   iIn, rOut, iOut, accumulate, work, d->fft_tw, s) != cudaSuccess)
        st = cuda_fail();
    if (cudaFreeAsync(work, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

mri_status mri_cg_solve(const float* K, int nx, int ny, int nz, float lambda, const float* rB,
                        const float* iB, float* rX, float* iX, int iters, double* rnorms,
                        void* stream)
{
    mri_status st = check_toeplitz_grid(nx, ny, nz);
    if (st != MRI_OK) return st;
    if (!std::isfinite(lambda) || iters < 0 || iters > (1 << 20)) return MRI_ERR_SIZE;
    if ((K != nullptr && !aligned8(K)) || (rnorms != nullptr && !aligned8(rnorms)))
        return MRI_ERR_ALIGN;
    const int64_t N = int64_t(nx) * ny * nz;
    const void* vp[6] = {K, rB, iB, rX, iX, rnorms};
    DeviceState* d = nullptr;
    if ((st = prepare(0, 0, 1, 0, N, nullptr, 0, vp, 6, &d)) != MRI_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // scratch: r, p, Ap (SoA), the FFT stages' work array (half the doubled
    // grid), the dot partials, p.Ap and two arrival counters
    const int dot_blocks = int(std::min<int64_t>(ceil_div(N, 256), int64_t(d->sms) * 4));
    const int64_t vec_bytes = align256(6 * N * 4);
    const int64_t work_bytes = align256(4 * N * int64_t(sizeof(float2)));
    const int64_t partials = std::max<int64_t>(dot_blocks, mri::toeplitz_dot_blocks(nx, ny, nz));
    char* scratch = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch),
                                size_t(vec_bytes + work_bytes + (partials + 2) * 8), d->pool,
                                s) != cudaSuccess)
        return cuda_fail();
    float* vec = reinterpret_cast<float*>(scratch);
    float2* work = reinterpret_cast<float2*>(scratch + vec_bytes);
    double* scal = reinterpret_cast<double*>(scratch + vec_bytes + work_bytes);
    if (mri::launch_cg(K, nx, ny, nz, lambda, rB, iB, rX, iX,
                       iters, rnorms, vec, work, scal, d->fft_tw, grid_for(N, d->sms),
                       dot_blocks, s) != cudaSuccess)
        st = cuda_fail();
    if (cudaFreeAsync(scratch, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

// ---------------------------------------------------------------------------
// the gridding reconstruction
// ---------------------------------------------------------------------------
mri_status mri_gridding(const float* kx, const float* ky, const float* kz, const float* rPhi,
                        const float* iPhi, const float* rD, const float* iD, int64_t M, int nx,
                        int ny, int nz, float* rOut, float* iOut, int accumulate, void* stream)
{
    mri_status st = check_mode(0, accumulate);
    if (st != MRI_OK) return st;
    if (!mri::fft_len_ok(nx) || !mri::fft_len_ok(ny) || !mri::fft_len_ok(nz)) return MRI_ERR_SIZE;
    if (M < 0 || M > kMaxM) return MRI_ERR_SIZE;
    const int64_t N = int64_t(nx) * ny * nz;
    const void* sp[7] = {kx, ky, kz, rPhi, iPhi, rD, iD};
    const void* vp[2] = {rOut, iOut};
    DeviceState* d = nullptr;
    if ((st = prepare(0, accumulate, 1, M, N, sp, 7, vp, 2, &d)) != MRI_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2* G = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&G), size_t(N) * sizeof(float2), d->pool,
                                s) != cudaSuccess)
        return cuda_fail();
    if (mri::launch_gridding(kx, ky, kz, rPhi, iPhi, rD, iD, M, nx, ny, nz, rOut, iOut,
                             accumulate, G, d->fft_tw, d->sms, s) != cudaSuccess)
        st = cuda_fail();
    if (cudaFreeAsync(G, s) != cudaSuccess && st == MRI_OK) st = cuda_fail();
    return st;
}

const char* mri_status_string(mri_status status)
{
    switch (status) {
        case MRI_OK: return "ok";
        case MRI_ERR_NULL: return "a required pointer is NULL";
        case MRI_ERR_SIZE: return "M, N or B is negative or too large";
        case MRI_ERR_ALIGN: return "a pointer is not 4-byte aligned";
        case MRI_ERR_NOT_DEVICE: return "a pointer is not device memory of the current device";
        case MRI_ERR_MODE: return "unknown trig mode or accumulate flag not 0/1";
        case MRI_ERR_CUDA: return "a CUDA runtime call failed";
        case MRI_ERR_UNSUPPORTED_DEVICE: return "the current device is not sm_103 (GB300)";
    }
    return "unknown status";
}

mri_status mri_plan_gather(int kind, int64_t B, int64_t M, int64_t N, int num_sms,
                           mri_plan* plan)
{
    if (plan == nullptr) return MRI_ERR_NULL;
    if (kind != MRI_KIND_FHD && kind != MRI_KIND_Q && kind != MRI_KIND_FHD_BATCHED)
        return MRI_ERR_MODE;
    if (kind != MRI_KIND_FHD_BATCHED) B = 1;
    mri_status st = check_sizes(B, M, N);
    if (st != MRI_OK) return st;
    if (num_sms < 0) return MRI_ERR_SIZE;
    if (num_sms == 0) {
        DeviceState* d = nullptr;
        if ((st = device_state(&d, nullptr)) != MRI_OK && st != MRI_ERR_UNSUPPORTED_DEVICE)
            return st;
        num_sms = d->sms;
    }
    const bool realw = kind == MRI_KIND_Q;
    std::memset(plan, 0, sizeof(*plan));
    if (N == 0) return MRI_OK;
    if (M == 0) {
        plan->launches = 2;   // zero fill of both outputs
        return MRI_OK;
    }
    const bool tc = use_coils_tc(realw, false, B);
    const int64_t rest = pair_coils(tc, B);
    GroupPlan plans[4];
    bool used[4];
    group_plans(realw, rest, M, N, num_sms, plans, used);
    int64_t scratch = 0;
    if (tc) {
        // the first group's shape: tensor cores, one voxel per tensor-memory
        // lane (its 2 x 8 running sums in one thread)
        const CoilTcPlan g = plan_coils_tc(M, N, num_sms, int(std::min<int64_t>(B - rest, 8)));
        plan->threads_per_cta = mri::kCtThreads;
        plan->voxels_per_thread = 1;
        plan->voxels_per_cta = mri::kCtRows;
        plan->samples_per_tile = mri::kTcTile;
        plan->splits = g.splits;
        plan->voxel_ctas = g.vblocks;
        plan->tiles = g.ntiles;
        plan->tensor_cores = 1;
        for (int64_t b0 = 0; b0 < B - rest; b0 += mri::kCtCoils) {
            plan->coil_groups += 1;
            plan->launches += 3 + (g.splits > 1 ? 1 : 0);   // prep, tiles, gather
        }
        scratch = g.scratch();
    } else {
        const GroupPlan& g0 = plans[realw ? 3 : group_index(B)];
        plan->threads_per_cta = g0.shape.threads;
        plan->voxels_per_thread = g0.shape.v;
        plan->voxels_per_cta = g0.shape.voxels_per_cta;
        plan->fast_fp32_voxels = g0.shape.fast_fp32_voxels;
        plan->samples_per_tile = kTile;
        plan->splits = g0.splits;
        plan->voxel_ctas = g0.vblocks;
        plan->tiles = g0.ntiles;
    }
    for (int64_t b0 = B - rest; b0 < B;) {
        const int i = realw ? 3 : group_index(B - b0);
        plan->coil_groups += 1;
        plan->launches += 2 + (plans[i].splits > 1 ? 1 : 0);
        const int64_t b = align256(plans[i].rec_bytes) + plans[i].part_bytes;
        if (b > scratch) scratch = b;
        b0 += plans[i].bc;
    }
    plan->scratch_bytes = scratch;
    return MRI_OK;
}

mri_status mri_device_errors(unsigned int* bits, int clear)
{
    if (bits == nullptr) return MRI_ERR_NULL;
    DeviceState* d = nullptr;
    mri_status st = device_state(&d, nullptr);
    if (st != MRI_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail();
    if (cudaMemcpy(bits, d->err, sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_fail();
    if (clear) {
        if (cudaMemset(d->err, 0, sizeof(unsigned int)) != cudaSuccess) return cuda_fail();
        if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail();
    }
    return MRI_OK;
}

mri_status mri_timing_begin(void)
{
    DeviceState* d = nullptr;
    mri_status st = device_state(&d, nullptr);
    if (st != MRI_OK) return st;
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    d->timing = true;
    d->timed = 0;
    return MRI_OK;
}

mri_status mri_timing_end(double* gather_ms, int64_t* launches)
{
    if (gather_ms == nullptr || launches == nullptr) return MRI_ERR_NULL;
    DeviceState* d = nullptr;
    mri_status st = device_state(&d, nullptr);
    if (st != MRI_OK) return st;
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    d->timing = false;
    double total = 0.0;
    for (int i = 0; i < d->timed; ++i) {
        if (cudaEventSynchronize(d->ev[2 * i + 1]) != cudaSuccess) return cuda_fail();
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, d->ev[2 * i], d->ev[2 * i + 1]) != cudaSuccess)
            return cuda_fail();
        total += ms;
    }
    *gather_ms = total;
    *launches = d->timed;
    d->timed = 0;
    return MRI_OK;
}

}  // extern "C"
