// sa_tc.cu -- placeholder: routes bf16 to the CUDA-core kernels until the
// tensor-core kernels land.
#include "sa_tc.h"

namespace sa {

Tiling tc_tiling(int) { return kSimtTiling; }
cudaError_t launch_band_tc(const DevProblem &p, cudaStream_t s) {
  return launch_band_simt(p, SA_BF16, s);
}
cudaError_t launch_global_tc(const DevProblem &p, cudaStream_t s) {
  return launch_global_simt(p, SA_BF16, s);
}

}  // namespace sa
