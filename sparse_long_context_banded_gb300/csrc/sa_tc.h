// sa_tc.h -- tensor-core (tcgen05 / TMEM / TMA) kernels: bf16 inputs
// (kind::f16, D 64 or 128) and fp32 inputs with tf32 products (SA_TF32:
// kind::tf32, D 64).
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "sa_kernels.h"

namespace sa {

// Tiling of the tensor-core family on a device with `sms` SMs.
Tiling tc_tiling(int D, int sms);

// Whether the tensor-core kernels take inputs of this type and head dimension.
bool tc_supports(sa_dtype dt, int D);

// Band tiles: one launch per group of at most 16 residue classes
// (group_begin from the schedule).  host_slots mirrors p.slots on the host.
// With g_ctas > 0 (a single group), the launch also runs the global-row items
// on g_ctas CTAs of its own beside band_ctas band CTAs.  The band tiles write
// every row, global rows too; the merge of the global-row partials, enqueued
// after them, overwrites those.  `precise`: P is split into two bf16 parts for
// the P V product (bf16 inputs).
cudaError_t launch_band_tc(const DevProblem &p, sa_dtype dt, bool precise, const Slot *host_slots,
                           int n_slots, const std::vector<int32_t> &group_begin, int BH, int sms,
                           int g_ctas, int band_ctas, cudaStream_t s);

// Failure-detection check: a kernel whose wait can never be satisfied gives
// up after limit_us microseconds and sets kErrWaitTimeout in *err.
cudaError_t launch_stalled_wait_check(int *err, uint32_t limit_us, cudaStream_t s);

// Global rows against all keys, split over key chunks (partials for merge),
// as a launch of its own on at most `sms` persistent CTAs.
cudaError_t launch_global_tc(const DevProblem &p, sa_dtype dt, bool precise, int BH, int sms,
                             cudaStream_t s);

}  // namespace sa
