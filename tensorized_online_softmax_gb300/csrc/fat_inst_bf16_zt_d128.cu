// Kernel instances: bf16 d128, X = 128, Z on the tensor pipe (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
int dispatch_bf16_zt_d128(const FwdParams& fp, bool l_tensor, int dev, int grid, int splits,
                         cudaStream_t stream) {
  return l_tensor ? launch_fwd<128, 128, true, kDtBf16, true>(fp, dev, grid, splits, stream)
                  : launch_fwd<128, 128, false, kDtBf16, true>(fp, dev, grid, splits, stream);
}
}  // namespace fat
