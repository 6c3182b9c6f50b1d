// Kernel instances: bf16 d128 ltensor (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_bf16_d128_ltensor, 128, true, kDtBf16)
}  // namespace fat
