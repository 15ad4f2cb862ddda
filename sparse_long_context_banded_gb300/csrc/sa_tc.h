// sa_tc.h -- tensor-core (tcgen05 / TMEM / TMA) kernels for bf16 inputs.
#pragma once

#include <cuda_runtime.h>

#include "sa_kernels.h"

namespace sa {

Tiling tc_tiling(int D);
cudaError_t launch_band_tc(const DevProblem &p, cudaStream_t s);
cudaError_t launch_global_tc(const DevProblem &p, cudaStream_t s);

}  // namespace sa
