// Kernel instances: bf16 d64 ltensor (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_bf16_d64_ltensor, 64, true, kDtBf16)
}  // namespace fat
