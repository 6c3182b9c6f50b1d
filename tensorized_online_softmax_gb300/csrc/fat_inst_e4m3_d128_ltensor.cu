// Kernel instances: e4m3 d128 ltensor (see fat_launch.cuh).
#include "fat_launch.cuh"

namespace fat {
FAT_DEFINE_DISPATCH(dispatch_e4m3_d128_ltensor, 128, true, kDtE4M3)
}  // namespace fat
