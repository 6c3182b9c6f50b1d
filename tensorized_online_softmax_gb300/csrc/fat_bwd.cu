// Backward-pass launchers: the D / LSE preparation and the fused kernel:
// fat_bwd_kernel for d = 128, fat_bwd_q2_kernel (a second Q stage) for d = 64.
#include <cuda_runtime.h>

#include "fat_bwd_kernel.cuh"
#include "fat_bwd_q2_kernel.cuh"
#include "fat_launch.cuh"

namespace fat {

namespace {
template <int D>
int launch_bwd_d(const BwdParams& bp, const float* o, const void* dout, const float* lse, int dev,
                 cudaStream_t stream) {
  // per device, once, whichever host thread launches first (1 = set up)
  static std::once_flag once[kMaxDevices];
  static int ready[kMaxDevices];
  auto kern = [] {
    if constexpr (D == 64) return fat_bwd_q2_kernel<D>;
    else return fat_bwd_kernel<D>;
  }();
  const int smem = [] {
    if constexpr (D == 64) return BwdSmemQ2<D>::kAlloc;
    else return BwdSmem<D>::kAlloc;
  }();
  std::call_once(once[dev], [&] {
    ready[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
                         cudaSuccess
                     ? 1
                     : -1;
  });
  if (ready[dev] != 1) return -4;
  const long long rows = static_cast<long long>(bp.BH) * bp.Npad;
  constexpr int kRowsPerBlock = kPrepWarps * kPrepRows;
  const long long prep_blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (prep_blocks > 0x7fffffffll) return -1;  // (beyond any device memory; nothing launched)
  fat_bwd_prep_kernel<D><<<static_cast<unsigned>(prep_blocks),
                           kPrepWarps * 32, 0, stream>>>(
      o, static_cast<const __nv_bfloat16*>(dout), lse, const_cast<float*>(bp.lse2),
      const_cast<float*>(bp.dvec), bp.dq, bp.N, bp.Npad, rows, bp.scale);
  if (cudaGetLastError() != cudaSuccess) return -4;
  // d = 128: programmatic stream serialisation, so that the fused kernel's
  // blocks may start (barriers, TMEM, the K and V loads) while the
  // preparation kernel's last blocks run; they wait for it before loading
  // LSE / D or adding into dQ (+0.5 to +1.3 % on the d = 128 shapes; the
  // d = 64 kernel measured 1.6 % slower that way and launches plainly)
  if constexpr (D != 128) {
    kern<<<bp.BH * bp.n_blocks, kBwdThreads, smem, stream>>>(bp);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(bp.BH * bp.n_blocks));
  cfg.blockDim = dim3(kBwdThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, bp) != cudaSuccess) return -4;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
}  // namespace

int launch_bwd(const BwdParams& bp, int d, const float* o, const void* dout, const float* lse,
               int dev, cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128>(bp, o, dout, lse, dev, stream);
  if (d == 64) return launch_bwd_d<64>(bp, o, dout, lse, dev, stream);
  return -1;
}

}  // namespace fat
