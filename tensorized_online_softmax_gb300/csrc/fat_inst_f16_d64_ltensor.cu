// Kernel instances: fp16 d64 ltensor (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_f16_d64_ltensor, 64, true, kDtF16)
}  // namespace fat
