// Kernel instances: bf16 d128 lvec (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_bf16_d128_lvec, 128, false, kDtBf16)
}  // namespace fat
