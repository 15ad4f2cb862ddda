// sa_tc.h -- tensor-core (tcgen05 / TMEM / TMA) kernels for bf16 inputs.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "sa_kernels.h"

namespace sa {

Tiling tc_tiling(int D);

// Band tiles: one launch per group of at most 16 residue classes
// (group_begin from the schedule).  host_slots mirrors p.slots on the host.
cudaError_t launch_band_tc(const DevProblem &p, const Slot *host_slots, int n_slots,
                           const std::vector<int32_t> &group_begin, int BH, cudaStream_t s);

// Global rows against all keys, split over key chunks (partials for merge).
cudaError_t launch_global_tc(const DevProblem &p, int BH, cudaStream_t s);

}  // namespace sa
