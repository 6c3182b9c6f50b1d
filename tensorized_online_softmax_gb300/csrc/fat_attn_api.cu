// Host side of the C ABI declared in include/fat_attn.h: argument validation,
// TMA tensor-map encoding, kernel selection and launch.  Nothing here
// allocates device memory or synchronises (except fat_check_device_error).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fat_attn.h"
#include "fat_bwd_kernel.cuh"
#include "fat_launch.cuh"

namespace {

constexpr int kMaxDevices = fat::kMaxDevices;

// Device error word shared by every kernel of the library (their address is
// passed in the kernel parameters): bit 0 = a bounded wait ran out.
__device__ unsigned int g_fat_error_word = 0;

struct DeviceCache {
  std::once_flag once;
  int arch_ok = 0;                       // 1: sm_103
  unsigned int* error_word = nullptr;    // device address of g_fat_error_word
};
DeviceCache g_dev[kMaxDevices];

std::once_flag g_encoder_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encoder_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// [B*H, N, d] view of a contiguous [B, H, N, d] tensor, boxes of 128 rows x
// 128 bytes, 128-byte swizzle (the layout the tcgen05 descriptors expect).
// Rows past N read as zero.
bool encode_qkv_map(CUtensorMap* tm, const void* ptr, int d, int N, int BH, int elt_bytes,
                    CUtensorMapDataType dt) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elt_bytes,
                                 static_cast<cuuint64_t>(N) * d * elt_bytes};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elt_bytes), 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 O viewed as [rows, N, d]: 32-column x 128-row boxes, 128-byte
// swizzle (the layout the kernel stages O in).
bool encode_o_map(CUtensorMap* tm, float* ptr, int d, int N, long long rows) {
  auto enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_device(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FAT_ERR_LAUNCH;
  DeviceCache& c = g_dev[dev];
  std::call_once(c.once, [&] {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    c.arch_ok = (major == 10 && minor == 3) ? 1 : 0;
    void* addr = nullptr;
    if (c.arch_ok && cudaGetSymbolAddress(&addr, g_fat_error_word) == cudaSuccess)
      c.error_word = static_cast<unsigned int*>(addr);
  });
  *dev_out = dev;
  if (!c.arch_ok) return FAT_ERR_ARCH;
  return c.error_word ? FAT_OK : FAT_ERR_LAUNCH;
}

}  // namespace

extern "C" {

const char* fat_status_string(int status) {
  switch (status) {
    case FAT_OK: return "FAT_OK";
    case FAT_ERR_INVALID_ARG: return "FAT_ERR_INVALID_ARG";
    case FAT_ERR_UNSUPPORTED: return "FAT_ERR_UNSUPPORTED";
    case FAT_ERR_ALIGNMENT: return "FAT_ERR_ALIGNMENT";
    case FAT_ERR_LAUNCH: return "FAT_ERR_LAUNCH";
    case FAT_ERR_DEVICE_TIMEOUT: return "FAT_ERR_DEVICE_TIMEOUT";
    case FAT_ERR_ARCH: return "FAT_ERR_ARCH";
    default: return "FAT_ERR_UNKNOWN";
  }
}

}  // extern "C"

namespace {

constexpr int kMaxSplits = 64;

long long splitkv_bytes(long long BH, long long Nq, int d, int splits) {
  return static_cast<long long>(splits) * BH * Nq * (d + 1) * 4 + 256;
}

// Shared body of every entry point: Nq query rows against Nk keys, the key
// range cut into `splits` ranges (one thread-block row of the grid each) whose
// partial results go to `workspace` and are merged afterwards.
int run_fwd(const fat_params* p, int Nq, int Nk, int splits, void* workspace,
            size_t workspace_bytes) {
  if (!p) return FAT_ERR_INVALID_ARG;
  // ---- synchronous validation: nothing is launched on failure ----
  if (!p->q || !p->k || !p->v || !p->o || !p->lse) return FAT_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || Nq < 1 || Nk < 1) return FAT_ERR_INVALID_ARG;
  if (p->causal && Nk < Nq) return FAT_ERR_INVALID_ARG;  // early queries would see no key
  if (p->d != 64 && p->d != 128) return FAT_ERR_INVALID_ARG;
  if (p->X != 16 && p->X != 32 && p->X != 64 && p->X != 128) return FAT_ERR_INVALID_ARG;
  if (!(p->scale > 0.f) || !std::isfinite(p->scale)) return FAT_ERR_INVALID_ARG;
  if (p->variant != FAT_VARIANT_TENSOR && p->variant != FAT_VARIANT_VEC) return FAT_ERR_INVALID_ARG;
  if (p->dtype != FAT_DTYPE_BF16 && p->dtype != FAT_DTYPE_E4M3 && p->dtype != FAT_DTYPE_FP16)
    return FAT_ERR_INVALID_ARG;
  if (p->l_mode != FAT_LMODE_VECTOR && p->l_mode != FAT_LMODE_TENSOR) return FAT_ERR_INVALID_ARG;
  if (p->z_mode != FAT_ZMODE_VECTOR && p->z_mode != FAT_ZMODE_TENSOR) return FAT_ERR_INVALID_ARG;
  const bool z_tensor = p->z_mode == FAT_ZMODE_TENSOR;
  if (p->block_mode != FAT_BLOCKS_AUTO && p->block_mode != FAT_BLOCKS_PER_TILE)
    return FAT_ERR_INVALID_ARG;
  if (z_tensor &&
      (p->variant != FAT_VARIANT_TENSOR || p->X != 128 || p->dtype != FAT_DTYPE_BF16))
    return FAT_ERR_UNSUPPORTED;
  if (splits < 1 || splits > kMaxSplits) return FAT_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(p->B) * p->H;
  const long long n_mblocks = (Nq + fat::kRowsPerCta - 1) / fat::kRowsPerCta;
  if (BH > (1ll << 30) || BH * n_mblocks > 0x7fffffffll) return FAT_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->o) ||
      !aligned16(p->lse))
    return FAT_ERR_ALIGNMENT;
  if (p->trace && (reinterpret_cast<uintptr_t>(p->trace) & 7u)) return FAT_ERR_ALIGNMENT;
  const bool e4m3 = p->dtype == FAT_DTYPE_E4M3;
  if (e4m3) {
    for (float ds : {p->q_descale, p->k_descale, p->v_descale})
      if (!(ds > 0.f) || !std::isfinite(ds)) return FAT_ERR_INVALID_ARG;
    if (p->d != 128) return FAT_ERR_UNSUPPORTED;  // e4m3 rows must fill a 128-byte slab
  }
  // keys per split: a multiple of the 128-key tile; fewer splits may result
  const int n_kv_tiles = (Nk + fat::kBlockN - 1) / fat::kBlockN;
  const int tiles_per_split = (n_kv_tiles + splits - 1) / splits;
  const int kv_split_len = tiles_per_split * fat::kBlockN;
  const int n_splits = (Nk + kv_split_len - 1) / kv_split_len;
  float* o_part = nullptr;
  float* lse_part = nullptr;
  if (n_splits > 1) {
    if (!workspace) return FAT_ERR_INVALID_ARG;
    if (static_cast<long long>(workspace_bytes) < splitkv_bytes(BH, Nq, p->d, n_splits))
      return FAT_ERR_INVALID_ARG;
    const uintptr_t base = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255);
    o_part = reinterpret_cast<float*>(base);
    lse_part = o_part + static_cast<size_t>(n_splits) * BH * Nq * p->d;
  }

  int dev = 0;
  const int arch = check_device(&dev);
  if (arch != FAT_OK) return arch;

  fat::FwdParams fp;
  const bool f16 = p->dtype == FAT_DTYPE_FP16;
  const int elt = e4m3 ? 1 : 2;
  const CUtensorMapDataType tdt = e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  if (!encode_qkv_map(&fp.tm_q, p->q, p->d, Nq, static_cast<int>(BH), elt, tdt) ||
      !encode_qkv_map(&fp.tm_k, p->k, p->d, Nk, static_cast<int>(BH), elt, tdt) ||
      !encode_qkv_map(&fp.tm_v, p->v, p->d, Nk, static_cast<int>(BH), elt, tdt))
    return FAT_ERR_LAUNCH;
  if (!encode_o_map(&fp.tm_o, o_part ? o_part : p->o, p->d, Nq,
                    (o_part ? static_cast<long long>(n_splits) : 1ll) * BH))
    return FAT_ERR_LAUNCH;
  fp.o = p->o;
  fp.lse = p->lse;
  fp.fallback_rows = p->fallback_rows;
  fp.B = p->B;
  fp.H = p->H;
  fp.Nq = Nq;
  fp.Nk = Nk;
  fp.causal = p->causal ? 1 : 0;
  fp.X = p->X;
  fp.n_mblocks = static_cast<int>(n_mblocks);
  fp.n_items = static_cast<int>(BH * n_mblocks);
  // block order: groups of heads whose K and V (2 Nk d input bytes each)
  // fill about 48 MiB of L2
  {
    long long g = (48ll << 20) / (2ll * Nk * p->d * elt);
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    fp.group_heads = static_cast<int>(g);
  }
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // One block per SM taking items in turn, or one block per item (split-KV
  // launches, and on request); the latter prefetches for the block one wave
  // ahead, the former for its own next item.
  const int grid =
      fat::fwd_grid(fp.n_items, sms, p->block_mode == FAT_BLOCKS_PER_TILE || n_splits != 1);
  fp.prefetch_stride = (grid == fp.n_items && sms > 0) ? sms : 0;
  fp.kv_split_len = kv_split_len;
  fp.o_part = o_part;
  fp.lse_part = lse_part;
  fp.scale = p->scale;
  // logits are scale * (q_descale * q_code) . (k_descale * k_code)
  fp.c = e4m3 ? p->scale * p->q_descale * p->k_descale * fat::kLog2e : p->scale * fat::kLog2e;
  fp.v_scale = e4m3 ? p->v_descale : 1.f;
  // bf16 P~ keeps fp32's exponent range (2^-64 leaves 62 binades); e4m3 P~ =
  // 2^(Z+8) has its smallest normal at 2^-6, i.e. Z = -14; fp16 P~ = 2^(Z+15)
  // at 2^-14, i.e. Z = -29
  const float t_default = e4m3 ? 14.f : (f16 ? 29.f : 64.f);
  fp.underflow_thresh =
      p->underflow_log2_threshold > 0.f ? p->underflow_log2_threshold : t_default;
  fp.poll_limit = p->wait_poll_limit;
  fp.timeout_ns = p->wait_timeout_ns ? p->wait_timeout_ns : 4000000000ull;
  fp.trace = p->trace;
  fp.error_word = g_dev[dev].error_word;

  const bool tensor = p->variant == FAT_VARIANT_TENSOR;
  const bool l_tensor = tensor && p->l_mode == FAT_LMODE_TENSOR;
  const int X = tensor ? p->X : 0;  // X = 0: the vector-softmax kernel
  int st;
  if (z_tensor)
    st = p->d == 128 ? fat::dispatch_bf16_zt_d128(fp, l_tensor, dev, grid, n_splits, p->stream)
                     : fat::dispatch_bf16_zt_d64(fp, l_tensor, dev, grid, n_splits, p->stream);
  else if (e4m3)
    st = l_tensor ? fat::dispatch_e4m3_d128_ltensor(fp, X, dev, grid, n_splits, p->stream)
                  : fat::dispatch_e4m3_d128_lvec(fp, X, dev, grid, n_splits, p->stream);
  else if (f16 && p->d == 128)
    st = l_tensor ? fat::dispatch_f16_d128_ltensor(fp, X, dev, grid, n_splits, p->stream)
                  : fat::dispatch_f16_d128_lvec(fp, X, dev, grid, n_splits, p->stream);
  else if (f16)
    st = l_tensor ? fat::dispatch_f16_d64_ltensor(fp, X, dev, grid, n_splits, p->stream)
                  : fat::dispatch_f16_d64_lvec(fp, X, dev, grid, n_splits, p->stream);
  else if (p->d == 128)
    st = l_tensor ? fat::dispatch_bf16_d128_ltensor(fp, X, dev, grid, n_splits, p->stream)
                  : fat::dispatch_bf16_d128_lvec(fp, X, dev, grid, n_splits, p->stream);
  else
    st = l_tensor ? fat::dispatch_bf16_d64_ltensor(fp, X, dev, grid, n_splits, p->stream)
                  : fat::dispatch_bf16_d64_lvec(fp, X, dev, grid, n_splits, p->stream);
  if (st != 0) return st == -1 ? FAT_ERR_UNSUPPORTED : FAT_ERR_LAUNCH;
  if (n_splits > 1 &&
      fat::launch_splitkv_combine(o_part, lse_part, p->o, p->lse, BH * Nq, n_splits, p->d,
                                  p->stream) != 0)
    return FAT_ERR_LAUNCH;
  return FAT_OK;
}

}  // namespace

extern "C" {

int fat_attn_fwd_ex(const fat_params* p) {
  if (!p) return FAT_ERR_INVALID_ARG;
  return run_fwd(p, p->N, p->N, 1, nullptr, 0);
}

size_t fat_attn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128) || num_splits < 1 ||
      num_splits > kMaxSplits)
    return 0;
  return static_cast<size_t>(splitkv_bytes(static_cast<long long>(B) * H, Nq, d, num_splits));
}

int fat_attn_splitkv_default_splits(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 1;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items = static_cast<long long>(B) * H * ((Nq + fat::kRowsPerCta - 1) / fat::kRowsPerCta);
  // About eight thread blocks per SM (one is resident at a time): enough
  // waves that the last one is a small part of the run and that every SM
  // keeps K/V loads in flight; each split keeps at least four K/V tiles.
  long long s = (8ll * sms + items - 1) / items;
  const long long tiles = (Nk + fat::kBlockN - 1) / fat::kBlockN;
  if (s > tiles / 4) s = tiles / 4;
  if (s > kMaxSplits) s = kMaxSplits;
  return static_cast<int>(s < 1 ? 1 : s);
}

int fat_attn_fwd_splitkv(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                         int H, int Nq, int Nk, int d, int causal, float scale, int X,
                         int num_splits, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  fat_params p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.N = Nq;
  p.d = d;
  p.causal = causal;
  p.scale = scale;
  p.X = X;
  p.variant = FAT_VARIANT_TENSOR;
  p.dtype = FAT_DTYPE_BF16;
  p.stream = stream;
  return run_fwd(&p, Nq, Nk, num_splits, workspace, workspace_bytes);
}

static int fwd_common(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                      int H, int N, int d, int causal, float scale, int X, cudaStream_t stream,
                      int variant) {
  fat_params p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.causal = causal;
  p.scale = scale;
  p.X = X;
  p.variant = variant;
  p.dtype = FAT_DTYPE_BF16;
  p.stream = stream;
  return fat_attn_fwd_ex(&p);
}

int fat_attn_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, int X, cudaStream_t stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, causal, scale, X, stream, FAT_VARIANT_TENSOR);
}

int fat_attn_fwd_vec(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                     int H, int N, int d, int causal, float scale, int X, cudaStream_t stream) {
  return fwd_common(q, k, v, o, lse, B, H, N, d, causal, scale, X, stream, FAT_VARIANT_VEC);
}

int fat_attn_fwd_fp8(const void* q, const void* k, const void* v, float q_descale,
                     float k_descale, float v_descale, float* o, float* lse, int B, int H, int N,
                     int d, int causal, float scale, int X, cudaStream_t stream) {
  fat_params p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.causal = causal;
  p.scale = scale;
  p.X = X;
  p.variant = FAT_VARIANT_TENSOR;
  p.dtype = FAT_DTYPE_E4M3;
  p.q_descale = q_descale;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  p.stream = stream;
  return fat_attn_fwd_ex(&p);
}

// ---------------------------------------------------------------------------
// Split-KV without allocation.  Some callers cannot obtain device memory when
// they call us: their process hands all device memory to its own pool at
// start-up, or they may not call cudaMalloc / cudaFree on this path because
// those can block or synchronise the device.  For them the split-KV partial
// results live in a fixed array that is part of this library's device image
// (every GPU that loads the library holds it until the process exits).
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = FAT_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocScratch {
  std::mutex m;
  std::atomic<void*> ptr{nullptr};  // device address of g_noalloc_scratch on this device
};
NoAllocScratch g_noalloc[kMaxDevices];

}  // namespace

int fat_attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, float* o,
                                 float* lse, int B, int H, int Nq, int Nk, int d, int causal,
                                 float scale, int X, int num_splits, cudaStream_t stream) {
  const size_t need = fat_attn_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
  if (need == 0 || need > kNoAllocScratchBytes) return FAT_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FAT_ERR_LAUNCH;
  NoAllocScratch& c = g_noalloc[dev];
  // once per device, with that device current: the array's device address
  // (in host code its name is only a host-side stand-in).  Only a successful
  // lookup is kept; a failed one is tried again by the next call.
  void* ptr = c.ptr.load(std::memory_order_acquire);
  if (!ptr) {
    std::lock_guard<std::mutex> guard(c.m);
    ptr = c.ptr.load(std::memory_order_relaxed);
    if (!ptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) == cudaSuccess) {
        c.ptr.store(addr, std::memory_order_release);
        ptr = addr;
      }
    }
  }
  if (!ptr) return FAT_ERR_LAUNCH;
  return fat_attn_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, X, num_splits,
                              ptr, kNoAllocScratchBytes, stream);
}

int fat_check_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FAT_ERR_LAUNCH;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fat_error_word, sizeof(word)) != cudaSuccess)
    return FAT_ERR_LAUNCH;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fat_error_word, &zero, sizeof(zero)) != cudaSuccess)
      return FAT_ERR_LAUNCH;
    return FAT_ERR_DEVICE_TIMEOUT;
  }
  return FAT_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward pass
// ---------------------------------------------------------------------------
namespace {
long long bwd_npad(int N) { return (static_cast<long long>(N) + 127) / 128 * 128; }
}  // namespace

extern "C" {

size_t fat_attn_bwd_workspace_bytes(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return static_cast<size_t>(2ll * B * H * bwd_npad(N) * 4 + 256);
}

int fat_attn_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse,
                 const void* dout, float* dq, float* dk, float* dv, int B, int H, int N, int d,
                 int causal, float scale, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream) {
  // ---- synchronous validation: nothing is launched on failure ----
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace)
    return FAT_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FAT_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FAT_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FAT_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long npad = bwd_npad(N);
  if (BH > (1ll << 30) || BH * (npad / 128) > 0x7fffffffll) return FAT_ERR_INVALID_ARG;
  if (workspace_bytes < fat_attn_bwd_workspace_bytes(B, H, N)) return FAT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(o) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FAT_ERR_ALIGNMENT;

  int dev = 0;
  const int arch = check_device(&dev);
  if (arch != FAT_OK) return arch;

  fat::BwdParams bp;
  const int bh = static_cast<int>(BH);
  if (!encode_qkv_map(&bp.tm_q, q, d, N, bh, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
      !encode_qkv_map(&bp.tm_k, k, d, N, bh, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
      !encode_qkv_map(&bp.tm_v, v, d, N, bh, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
      !encode_qkv_map(&bp.tm_do, dout, d, N, bh, 2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
      !encode_o_map(&bp.tm_dq, dq, d, N, BH))
    return FAT_ERR_LAUNCH;
  const uintptr_t base = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255);
  bp.lse2 = reinterpret_cast<const float*>(base);
  bp.dvec = reinterpret_cast<const float*>(base) + BH * npad;
  bp.dq = dq;
  bp.dk = dk;
  bp.dv = dv;
  bp.BH = bh;
  bp.N = N;
  bp.Npad = static_cast<int>(npad);
  bp.causal = causal ? 1 : 0;
  bp.n_blocks = static_cast<int>(npad / 128);
  // causal block order: groups of heads whose Q, dO (bf16) and dQ (fp32),
  // 8 N d bytes each, fill about 48 MiB of L2
  {
    const long long per_head = 8ll * N * d;
    long long g = (48ll << 20) / per_head;
    if (g < 1) g = 1;
    if (g > BH) g = BH;
    if (d == 128) {
      // balanced groups (bwd_work_item)
      bp.group_heads = fat::bwd_group_heads(bh, static_cast<int>(g));
      bp.group_extra = fat::bwd_group_extra(bh, static_cast<int>(g));
    } else {
      // the d = 64 kernel's own order: groups of g heads, the last one smaller
      bp.group_heads = static_cast<int>(g);
      bp.group_extra = 0;
    }
  }
  bp.c = scale * fat::kLog2e;
  bp.scale = scale;
  bp.poll_limit = 0;
  bp.timeout_ns = 4000000000ull;
  bp.error_word = g_dev[dev].error_word;
  // (dQ is cleared by the preparation kernel, ahead of the fused kernel's adds)
  const int st = fat::launch_bwd(bp, d, o, dout, lse, dev, stream);
  if (st != 0) return st == -1 ? FAT_ERR_UNSUPPORTED : FAT_ERR_LAUNCH;
  return FAT_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Host-resident tensors: chunks of heads through kHostSlots device slots, the
// copies in, the kernel and the copies out on three streams of their own
// ---------------------------------------------------------------------------
namespace {

// (three slots: the copy in of a chunk need not wait for the copy out of the
// chunk two before it, which the shared link slows while both directions run)
constexpr int kHostSlots = 3;

struct HostPipe {
  std::once_flag once;
  bool ok = false;
  cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_ready[kHostSlots] = {}, run_done[kHostSlots] = {}, slot_free[kHostSlots] = {};
  std::mutex mu;
};
HostPipe g_pipe[kMaxDevices];

long long host_chunk_heads(long long BH, int heads_per_chunk) {
  long long c = heads_per_chunk > 0 ? heads_per_chunk : (BH + 7) / 8;
  if (c < 1) c = 1;
  return c < BH ? c : BH;
}

long long align256(long long x) { return (x + 255) / 256 * 256; }

// one slot: q, k, v (bf16), o (fp32), lse (fp32) of `hc` heads, each 256-byte aligned
long long host_slot_bytes(long long hc, int N, int d) {
  const long long rows = hc * N;
  return 3 * align256(rows * d * 2) + align256(rows * d * 4) + align256(rows * 4);
}

}  // namespace

extern "C" {

size_t fat_attn_fwd_host_workspace_bytes(int B, int H, int N, int d, int heads_per_chunk) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  const long long hc = host_chunk_heads(static_cast<long long>(B) * H, heads_per_chunk);
  return static_cast<size_t>(kHostSlots * host_slot_bytes(hc, N, d) + 256);
}

int fat_attn_fwd_host(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                      int H, int N, int d, int causal, float scale, int X, int heads_per_chunk,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  // ---- synchronous validation: nothing is queued on failure ----
  if (!q || !k || !v || !o || !lse || !workspace) return FAT_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FAT_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FAT_ERR_INVALID_ARG;
  if (X != 16 && X != 32 && X != 64 && X != 128) return FAT_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FAT_ERR_INVALID_ARG;
  if (workspace_bytes < fat_attn_fwd_host_workspace_bytes(B, H, N, d, heads_per_chunk))
    return FAT_ERR_INVALID_ARG;
  int dev = 0;
  const int arch = check_device(&dev);
  if (arch != FAT_OK) return arch;
  HostPipe& hp = g_pipe[dev];
  std::call_once(hp.once, [&] {
    bool ok = true;
    for (cudaStream_t* s : {&hp.s_in, &hp.s_run, &hp.s_out})
      ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&hp.end, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < kHostSlots; ++i)
      for (cudaEvent_t* e : {&hp.in_ready[i], &hp.run_done[i], &hp.slot_free[i]})
        ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    hp.ok = ok;
  });
  if (!hp.ok) return FAT_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(hp.mu);

  const long long BH = static_cast<long long>(B) * H;
  const long long hc = host_chunk_heads(BH, heads_per_chunk);
  const long long slot = host_slot_bytes(hc, N, d);
  const uintptr_t base = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255);
  struct Slot { void *q, *k, *v; float *o, *lse; } sl[kHostSlots];
  for (int s = 0; s < kHostSlots; ++s) {
    uint8_t* p = reinterpret_cast<uint8_t*>(base + s * slot);
    const long long in = align256(hc * N * d * 2);
    sl[s].q = p;
    sl[s].k = p + in;
    sl[s].v = p + 2 * in;
    sl[s].o = reinterpret_cast<float*>(p + 3 * in);
    sl[s].lse = reinterpret_cast<float*>(p + 3 * in + align256(hc * N * d * 4));
  }
  bool ok = cudaEventRecord(hp.start, stream) == cudaSuccess;
  for (cudaStream_t s : {hp.s_in, hp.s_run, hp.s_out})
    ok = ok && cudaStreamWaitEvent(s, hp.start, 0) == cudaSuccess;
  int st = FAT_OK;
  const auto* qh = static_cast<const uint8_t*>(q);
  const auto* kh = static_cast<const uint8_t*>(k);
  const auto* vh = static_cast<const uint8_t*>(v);
  for (long long h0 = 0, c = 0; ok && st == FAT_OK && h0 < BH; h0 += hc, ++c) {
    const int s = static_cast<int>(c % kHostSlots);
    const long long n = hc < BH - h0 ? hc : BH - h0;
    const size_t in_off = static_cast<size_t>(h0) * N * d * 2, in_bytes = n * N * d * 2;
    // the slot's previous chunk has been copied out
    if (c >= kHostSlots)
      ok = ok && cudaStreamWaitEvent(hp.s_in, hp.slot_free[s], 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(sl[s].q, qh + in_off, in_bytes, cudaMemcpyHostToDevice, hp.s_in) ==
                   cudaSuccess;
    ok = ok && cudaMemcpyAsync(sl[s].k, kh + in_off, in_bytes, cudaMemcpyHostToDevice, hp.s_in) ==
                   cudaSuccess;
    ok = ok && cudaMemcpyAsync(sl[s].v, vh + in_off, in_bytes, cudaMemcpyHostToDevice, hp.s_in) ==
                   cudaSuccess;
    ok = ok && cudaEventRecord(hp.in_ready[s], hp.s_in) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(hp.s_run, hp.in_ready[s], 0) == cudaSuccess;
    if (!ok) break;
    fat_params p = {};
    p.q = sl[s].q;
    p.k = sl[s].k;
    p.v = sl[s].v;
    p.o = sl[s].o;
    p.lse = sl[s].lse;
    p.B = 1;
    p.H = static_cast<int>(n);
    p.N = N;
    p.d = d;
    p.causal = causal;
    p.scale = scale;
    p.X = X;
    p.variant = FAT_VARIANT_TENSOR;
    p.dtype = FAT_DTYPE_BF16;
    p.stream = hp.s_run;
    st = fat_attn_fwd_ex(&p);
    ok = ok && cudaEventRecord(hp.run_done[s], hp.s_run) == cudaSuccess;
    ok = ok && cudaStreamWaitEvent(hp.s_out, hp.run_done[s], 0) == cudaSuccess;
    if (st != FAT_OK || !ok) break;
    ok = ok && cudaMemcpyAsync(o + static_cast<size_t>(h0) * N * d, sl[s].o, n * N * d * 4,
                               cudaMemcpyDeviceToHost, hp.s_out) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(lse + static_cast<size_t>(h0) * N, sl[s].lse, n * N * 4,
                               cudaMemcpyDeviceToHost, hp.s_out) == cudaSuccess;
    ok = ok && cudaEventRecord(hp.slot_free[s], hp.s_out) == cudaSuccess;
  }
  // `stream` continues after everything queued above (the copies out wait for
  // the kernels, which wait for the copies in)
  for (cudaStream_t s : {hp.s_in, hp.s_run}) {
    if (cudaEventRecord(hp.end, s) != cudaSuccess || cudaStreamWaitEvent(hp.s_out, hp.end, 0) != cudaSuccess)
      ok = false;
  }
  if (cudaEventRecord(hp.end, hp.s_out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, hp.end, 0) != cudaSuccess)
    ok = false;
  if (st != FAT_OK) return st;
  return ok ? FAT_OK : FAT_ERR_LAUNCH;
}

}  // extern "C"
