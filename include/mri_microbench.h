/*
 * mri_microbench.h -- throughput probes of the two units the gather is bound
 * by, for the roofline of the F^H D / Q kernels.
 *
 * The chapter "Iterative MRI reconstruction" (section 17.3) counts about 13
 * floating-point operations and 2 trig operations per voxel-sample pair and
 * moves sin/cos onto the SFUs (step 3, Fig. 17.17) because trig would
 * otherwise dominate.  How many MUFU and FFMA results an SM delivers per
 * clock on this GPU decides which unit binds; these probes measure it.
 *
 * mri_microbench launches ONE wave of CTAs (ctas_per_sm per SM, `threads`
 * threads each) on `stream`; each CTA takes 1/ctas_per_sm of the SM's shared
 * memory, so exactly ctas_per_sm CTAs share every SM.  Each thread runs `iters` iterations of 8
 * independent dependency chains of the probed instruction:
 *   which = 0: __sinf (MUFU sine),   which = 1: __cosf (MUFU cosine),
 *   which = 2: fmaf (FFMA),          which = 3: exp2f (MUFU base-2 exponential),
 *   which = 4: fma.rn.f32x2 (packed FFMA2 on pairs of floats; four chains of
 *              pairs, so again 8 results per iteration).
 * Each CTA writes its elapsed SM clock cycles (clock64) to cycles[cta] and a
 * value derived from its chains to sink[cta * threads + thread] (so the work
 * is not removed).  Rate per SM per clock =
 *   ctas_per_sm * threads * iters * 8 / cycles,
 * which holds for ctas_per_sm = 1: CTAs that share an SM need not start and
 * finish together, so their own elapsed cycles understate the SM's busy time
 * and the formula then overstates the rate (measured: up to 1.5x with four
 * CTAs of 256 threads).  Use one CTA of 1024 threads per SM for rates.
 * cycles: device array of (num_sms * ctas_per_sm) uint64; sink: device array
 * of (num_sms * ctas_per_sm * threads) floats.  num_sms is the current
 * device's SM count.  Returns MRI_ERR_MODE for an unknown probe.
 */
#ifndef MRI_MICROBENCH_H
#define MRI_MICROBENCH_H

#include <stdint.h>

#include "mri.h"

#ifdef __cplusplus
extern "C" {
#endif

mri_status mri_microbench(int which, int ctas_per_sm, int threads, int64_t iters,
                          unsigned long long* cycles, float* sink, void* stream);

/*
 * Tensor-core issue-rate probe: the ceiling of the MMA form the tensor-core
 * grid kernels use (mri_fhd_grid and friends), with nothing else running.
 * Launches one CTA per SM (128 threads; at least 128 KB of shared memory so
 * that no second CTA fits; all 512 tensor-memory columns) on `stream`.
 * Thread 0 issues `tiles` times the 12 tcgen05.mma.cta_group::1.kind::f16 of
 * 128 x 256 x 16 that one 32-sample tile of the grid kernel takes, one
 * tcgen05.commit per tile, every wait bounded (a wait that gives up sets bit
 * 0x1 of the device error word):
 *   mode 0: A and B from shared memory (zeros), at most two tiles in flight;
 *   mode 1: A from tensor memory, B from shared memory (zeros), likewise;
 *   mode 2: A from tensor memory, B brought per tile by one 48 KB TMA bulk
 *           copy (tile t from b_tab + (t mod b_tiles) * 49152, 16-byte
 *           aligned device memory) into a ring of 4 stages, copies issued two
 *           tiles ahead, as the grid kernel streams its B-operand table;
 *   mode 3: as mode 1 with each product split into two N = 128 halves
 *           (24 MMAs of 128 x 128 x 16 per tile, the same work), the halves
 *           alternating between two accumulators;
 *   mode 4: as mode 3 with all 24 MMAs into one accumulator (each depends
 *           on the one before).
 * b_tab / b_tiles are read in mode 2 only.  cycles[cta] (device, one uint64
 * per SM) receives the SM clock cycles from the first issue to the last
 * completion.  One tile is 32 samples x 128 x 128 voxels = 524,288
 * voxel-sample pairs, so the ceiling in pairs per SM per clock is
 * tiles * 524288 / cycles.  MRI_ERR_MODE for mode outside 0..4, MRI_ERR_NULL
 * for a missing array, MRI_ERR_SIZE for tiles outside 1 .. 2^22, b_tiles < 1
 * or an unaligned b_tab (mode 2), MRI_ERR_UNSUPPORTED_DEVICE off sm_103.
 */
mri_status mri_mma_probe(int mode, int tiles, const void* b_tab, int64_t b_tiles,
                         unsigned long long* cycles, void* stream);

/*
 * Failure-detection self-test (no counterpart on the pages).  Every wait in
 * the gather kernels (an mbarrier for a TMA copy or for the tensor core) is
 * bounded: after 1 s it gives up, sets a bit in the device error word that
 * mri_device_errors() returns, lets its own copies land and exits, so a copy
 * that never completes costs an error code, not a hung GPU.  This launches
 * one CTA that waits with the same helper on an mbarrier nothing arrives on
 * (arrive = 0: expect bit 0x1 after about a second) or on one it arrived on
 * first (arrive = 1: no bit).  Asynchronous on `stream`; MRI_ERR_MODE for
 * arrive not 0/1, MRI_ERR_UNSUPPORTED_DEVICE off sm_103.
 */
mri_status mri_wait_selftest(int arrive, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MRI_MICROBENCH_H */
