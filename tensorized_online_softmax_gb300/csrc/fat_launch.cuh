// Kernel launchers: one explicit instance per (head dim, X, row-sum mode,
// input type), grouped into dispatchers that live in separate translation
// units so they compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "fat_fwd_kernel.cuh"

namespace fat {

constexpr int kMaxDevices = 64;

// Returns 0 or the fat_status code FAT_ERR_LAUNCH (-4).
template <int D, int kX, bool kLTensor, int kDt, bool kZT = false>
int launch_fwd(const FwdParams& fp, int dev, int grid, int splits, cudaStream_t stream) {
  // per device, once, whichever host thread launches first: the attribute
  // check and set-up below (1 = done, -1 = refused)
  static std::once_flag once[kMaxDevices];
  static int ready[kMaxDevices];
  auto kern = fat_fwd_kernel<D, kX, kLTensor, kDt, kZT>;
  const int smem = Smem<D, kDt == kDtE4M3, kZT>::kAlloc;
  std::call_once(once[dev], [&] {
    // The warpgroup register split inside the kernel assumes exactly
    // kLaunchRegs registers per thread at launch; anything else could make
    // the register increase wait forever, so refuse to launch.
    cudaFuncAttributes fa;
    const bool ok =
        cudaFuncGetAttributes(&fa, kern) == cudaSuccess && fa.numRegs == kLaunchRegs &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
            cudaSuccess;
    ready[dev] = ok ? 1 : -1;
  });
  if (ready[dev] != 1) return -4;
  kern<<<dim3(grid, splits), kNumThreads, smem, stream>>>(fp);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Backward pass (fat_bwd.cu): D / LSE preparation, then the fused kernel.
// Returns 0, -1 for a d without an instance, -4 on a CUDA error.
struct BwdParams;
int launch_bwd(const BwdParams& bp, int d, const float* o, const void* dout, const float* lse,
               int dev, cudaStream_t stream);

// LSE-weighted merge of split-KV partial results (fat_splitkv_combine.cu).
int launch_splitkv_combine(const float* o_part, const float* lse_part, float* o, float* lse,
                           long long rows, int splits, int d, cudaStream_t stream);

// X = 0 selects the vector-softmax kernel (row-sum mode ignored); otherwise
// X in {16, 32, 64, 128}.  Returns -1 for an X without an instance.
#define FAT_DECLARE_DISPATCH(name) \
  int name(const FwdParams& fp, int X, int dev, int grid, int splits, cudaStream_t stream);
FAT_DECLARE_DISPATCH(dispatch_bf16_d128_lvec)
FAT_DECLARE_DISPATCH(dispatch_bf16_d128_ltensor)
FAT_DECLARE_DISPATCH(dispatch_bf16_d64_lvec)
FAT_DECLARE_DISPATCH(dispatch_bf16_d64_ltensor)
FAT_DECLARE_DISPATCH(dispatch_e4m3_d128_lvec)
FAT_DECLARE_DISPATCH(dispatch_e4m3_d128_ltensor)
FAT_DECLARE_DISPATCH(dispatch_f16_d128_lvec)
FAT_DECLARE_DISPATCH(dispatch_f16_d128_ltensor)
FAT_DECLARE_DISPATCH(dispatch_f16_d64_lvec)
FAT_DECLARE_DISPATCH(dispatch_f16_d64_ltensor)
#undef FAT_DECLARE_DISPATCH

// Z on the tensor pipe (bf16, X = 128): d in {64, 128}, either row-sum mode.
// Returns -1 for a d without an instance.
int dispatch_bf16_zt_d128(const FwdParams& fp, bool l_tensor, int dev, int grid, int splits,
                          cudaStream_t stream);
int dispatch_bf16_zt_d64(const FwdParams& fp, bool l_tensor, int dev, int grid, int splits,
                         cudaStream_t stream);

#define FAT_DEFINE_DISPATCH(name, D, LT, DT)                                  \
  int name(const FwdParams& fp, int X, int dev, int grid, int splits, cudaStream_t stream) { \
    switch (X) {                                                                 \
      case 0:                                                                    \
        if constexpr (!(LT)) return launch_fwd<D, 0, false, DT>(fp, dev, grid, splits, stream); \
        return -1;                                                               \
      case 16: return launch_fwd<D, 16, LT, DT>(fp, dev, grid, splits, stream);        \
      case 32: return launch_fwd<D, 32, LT, DT>(fp, dev, grid, splits, stream);        \
      case 64: return launch_fwd<D, 64, LT, DT>(fp, dev, grid, splits, stream);        \
      case 128: return launch_fwd<D, 128, LT, DT>(fp, dev, grid, splits, stream);      \
      default: return -1;                                                        \
    }                                                                            \
  }

}  // namespace fat
