// Kernel instances: bf16 d64 lvec (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_bf16_d64_lvec, 64, false, kDtBf16)
}  // namespace fat
