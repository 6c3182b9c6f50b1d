// Kernel instances: fp16 d64 lvec (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_f16_d64_lvec, 64, false, kDtF16)
}  // namespace fat
