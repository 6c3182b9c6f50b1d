/*
 * fat_attn.h -- C ABI of the GB300 (sm_103a) fused attention forward pass with
 * the tensorized online softmax.
 *
 * Operation (every entry point): for each batch b, head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(scale * Q[b,h,i,:] . K[b,h,j,:])
 *
 * over keys j = 0..N-1, or j = 0..i with the causal mask.  This is the fused
 * attention flow of "FlashAttention-T: Towards Fully Tensorized Attention by
 * Exploiting Tensor-Vector Parallelism" (papercache.org summary, section A3,
 * Fig. 2: one output row block per worker, S and P kept on chip), with the
 * tensorized online softmax of its section A2 (surrogate maximum over X-row
 * tiles, the equation defining m_hat; Algorithm 1 steps 1-7).
 *
 * Conventions shared by all entry points
 *  - Pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or keeps them.  Tensors are contiguous row-major:
 *    q, k, v [B, H, N, d] (bf16, or e4m3 for the fp8 entry point); o fp32
 *    [B, H, N, d]; lse fp32 [B, H, N] (natural log, in units of the scaled
 *    logits).  q, k, v, o and lse must be 16-byte aligned.
 *  - d is 64 or 128; X (rows sharing one surrogate maximum) is 16, 32, 64 or
 *    128; B, H, N >= 1 (any N: a ragged last tile is masked).
 *  - Arguments are validated before anything is launched; on failure nothing
 *    runs and a negative fat_status is returned.
 *  - The work is enqueued asynchronously on `stream` (0 = legacy default
 *    stream).  The library never synchronises, except in
 *    fat_check_device_error().
 *  - Device-side waits are bounded.  A wait that runs out stops the kernel,
 *    leaves o/lse unspecified and records FAT_ERR_DEVICE_TIMEOUT in a device
 *    error word that fat_check_device_error() reports.
 *  - Calls are re-entrant; the only library state is a per-device cache of
 *    the driver's tensor-map encoder and kernel attributes.
 */
#ifndef FAT_ATTN_H_
#define FAT_ATTN_H_

#include <stddef.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FAT_OK = 0,
  FAT_ERR_INVALID_ARG = -1,    /* null pointer, bad size, bad d / X, bad scale */
  FAT_ERR_UNSUPPORTED = -2,    /* a valid request this build does not implement */
  FAT_ERR_ALIGNMENT = -3,      /* a tensor is not 16-byte aligned */
  FAT_ERR_LAUNCH = -4,         /* CUDA reported an error while setting up or launching */
  FAT_ERR_DEVICE_TIMEOUT = -5, /* a bounded device wait ran out (see fat_check_device_error) */
  FAT_ERR_ARCH = -6            /* the current device is not sm_103 */
} fat_status;

typedef enum { FAT_VARIANT_TENSOR = 0, FAT_VARIANT_VEC = 1 } fat_variant;
/* Input type of q, k, v (fat_attn_fwd_ex): bf16; e4m3 with per-tensor
 * descales (d = 128 only); fp16 (the FA-T summary's FP16-FP32 setting, A4).
 * P~ takes the input type for the O += P~ V MMA (fp16 P~ as 2^(Z+15), e4m3 as
 * 2^(Z+8), to use those formats' ranges; the factor is taken off LSE). */
typedef enum { FAT_DTYPE_BF16 = 0, FAT_DTYPE_E4M3 = 1, FAT_DTYPE_FP16 = 2 } fat_dtype;

/*
 * Where the row sum l of Algorithm 1 step 7 is formed in the tensorized
 * variant.  FAT_LMODE_VECTOR (default): fp32 sum of the unrounded P~ on the
 * vector units (packed f32x2 adds).  FAT_LMODE_TENSOR: on the tensor pipe as
 * the bf16-rounded P~ times a block of ones, plus a per-tile correction of
 * the dominant term's rounding; O stays consistent with l, but LSE can then
 * be off by up to ~2^-9 when a few comparable terms dominate a row.
 */
typedef enum { FAT_LMODE_VECTOR = 0, FAT_LMODE_TENSOR = 1 } fat_lmode;

/*
 * Where the subtraction of Algorithm 1 steps 4-5 (Z = log2(e) * scale * S -
 * m_hat) happens in the tensorized variant.  FAT_ZMODE_VECTOR (default): one
 * packed FMA per pair of scores on the vector units.  FAT_ZMODE_TENSOR (the
 * tensor-pipe half of the "AllTensor" variant of the page's ablation, Fig. 10):
 * S = Q K^T gets one more 16-deep K step, a bias tile against a tile of ones,
 * so the MMA itself writes S + b with b = -m_ref / (log2(e) * scale) rounded
 * to bf16, m_ref being the surrogate maximum settled three K/V tiles earlier
 * (the latest one known when that S is queued).  The multiply by
 * log2(e) * scale and the remaining offset log2(e) * scale * b + m_hat stay
 * one packed FMA per pair, so no vector instruction is saved, and the MMA does 1/8 (d = 128)
 * or 1/4 (d = 64) more work on S.  Requires the tensorized variant, X = 128
 * and bf16 inputs; anything else returns FAT_ERR_UNSUPPORTED.
 */
typedef enum { FAT_ZMODE_VECTOR = 0, FAT_ZMODE_TENSOR = 1 } fat_zmode;

/*
 * How query tiles (128 rows of one (b, h): the row blocks of the page's
 * section A3, one per worker) map to thread blocks.  FAT_BLOCKS_AUTO
 * (default): one thread block per SM takes tiles in turn, so the next tile's
 * Q and first K tiles load, and its first S tiles run on the tensor pipe,
 * while the last tile's output is normalised and stored; split-KV calls use
 * one block per tile.  FAT_BLOCKS_PER_TILE: one thread block per tile, in the
 * same order (for comparison).  The results are the same either way.
 */
typedef enum { FAT_BLOCKS_AUTO = 0, FAT_BLOCKS_PER_TILE = 1 } fat_block_mode;

/*
 * Tensorized online softmax (section A2 of the page above).
 *   - m_hat: per X-row tile, the maximum of the row maxima seen so far
 *     (Algorithm 1 step 1), kept as an integer number of binades so that the
 *     rescale factor exp(m_hat_old - m_hat) of steps 2-3 is an exact power of
 *     two shared by the tile;
 *   - Z = log2(e) * scale * S - m_hat, P~ = exp2(Z) (steps 4-6);
 *   - O is rescaled in tensor memory by the vector units, once per tile and
 *     only when m_hat grew (for X = 128 one factor for the whole tile);
 *   - the row sum l of step 7 is an fp32 sum on the vector units (see
 *     fat_lmode for the tensor-pipe alternative);
 *   - rows whose surrogate maximum exceeds their exact maximum by more than
 *     the underflow threshold (default 64 binades for bf16 P~, 29 for fp16,
 *     14 for e4m3),
 *     or whose sum is zero, are detected; their 128-row block is recomputed
 *     with one-row tiles (X = 1: each row's own maximum rounded up to a whole
 *     binade, so no row can underflow) -- the optional fallback of the
 *     all-underflow discussion -- after the thread block's other tiles,
 *     overwriting the block's O and LSE.
 * q, k, v: bf16.  Returns a fat_status.
 */
int fat_attn_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int H,
                 int N, int d, int causal, float scale, int X, cudaStream_t stream);

/*
 * Vector-softmax ablation baseline (the "FA2" arm of the page's Fig. 10
 * ablation): exact per-row maximum, per-row rescale of O whenever a row
 * maximum grows, row sum accumulated on the vector units.  Same pipeline,
 * tiling and signature as fat_attn_fwd; X is validated but unused.
 */
int fat_attn_fwd_vec(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                     int H, int N, int d, int causal, float scale, int X, cudaStream_t stream);

/*
 * FP8 (e4m3) inputs with per-tensor fp32 descales (real value = code * descale),
 * fp32 accumulation, the tensorized softmax of fat_attn_fwd.  (The page
 * evaluates FP8-FP32 attention in its section A4.)  d must be 128.  P~ is
 * stored as e4m3 scaled by 2^8 (largest term <= 256 < 448; the factor cancels
 * in O / l and is removed from LSE); O is rescaled on the vector side.
 * Descales must be finite and > 0.
 */
int fat_attn_fwd_fp8(const void* q, const void* k, const void* v, float q_descale,
                     float k_descale, float v_descale, float* o, float* lse, int B, int H, int N,
                     int d, int causal, float scale, int X, cudaStream_t stream);

/*
 * Split-KV forward (decode and long-key shapes): Nq query rows against Nk
 * keys per (b, h); q [B, H, Nq, d], k and v [B, H, Nk, d] (bf16), o fp32
 * [B, H, Nq, d], lse fp32 [B, H, Nq].  Causal keeps key j for query i iff
 * j <= i + Nk - Nq (the queries are the last Nq positions; requires
 * Nk >= Nq).  The key range is cut into up to num_splits ranges of whole
 * 128-key tiles (1 <= num_splits <= 64), each computed by its own thread
 * blocks with the tensorized online softmax of fat_attn_fwd; their partial
 * O and LSE go to `workspace` (device memory owned by the caller, at least
 * fat_attn_splitkv_workspace_bytes(B, H, Nq, d, num_splits) bytes; may be
 * NULL when a single range results) and are merged by LSE weights:
 * LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.  The merge is
 * the exact identity behind the page's online softmax (per-block maxima
 * and sums combined afterwards, section A3 / Fig. 2).  Calls sharing a
 * workspace must not overlap on the device.
 */
int fat_attn_fwd_splitkv(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                         int H, int Nq, int Nk, int d, int causal, float scale, int X,
                         int num_splits, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* Workspace size for fat_attn_fwd_splitkv (0 for invalid arguments). */
size_t fat_attn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/* A split count giving about eight thread blocks per SM of the current device
 * (at least four 128-key tiles per split). */
int fat_attn_splitkv_default_splits(int B, int H, int Nq, int Nk);

/*
 * fat_attn_fwd_splitkv without any device allocation, for callers that
 * cannot allocate device memory at the time of the call (their process gives
 * all device memory to its own pool at start-up, or they must not call
 * cudaMalloc / cudaFree, which can block or synchronise the device).  The
 * pages have no counterpart: this is a convenience of this library.
 *
 * Same arguments and results as fat_attn_fwd_splitkv, minus the workspace:
 * the partial results use a fixed array of FAT_NOALLOC_SCRATCH_BYTES that
 * belongs to the library's device image, so every GPU that loads the library
 * holds that memory until the process exits.  Requests whose workspace
 * (fat_attn_splitkv_workspace_bytes) exceeds it return FAT_ERR_INVALID_ARG
 * and launch nothing.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  If the lookup fails, that call returns FAT_ERR_LAUNCH and
 * the next call on the device tries again.  Nothing in the array needs to
 * start at zero (each call
 * writes every entry it reads), but all calls share it and it keeps the last
 * call's contents: calls whose work overlaps on the device race with each
 * other, so serialise them (for example on one stream).
 */
#define FAT_NOALLOC_SCRATCH_BYTES (16u << 20)
int fat_attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, float* o,
                                 float* lse, int B, int H, int Nq, int Nk, int d, int causal,
                                 float scale, int X, int num_splits, cudaStream_t stream);

/*
 * fat_attn_fwd on host-resident tensors: q, k, v bf16 [B, H, N, d] and o, lse
 * fp32 ([B, H, N, d], [B, H, N]) in page-locked host memory.  The problem is
 * streamed through the device in chunks of heads_per_chunk heads (heads are
 * independent and contiguous): the copy to the device of one chunk, the
 * kernel of the previous one and the copy back of the one before overlap on
 * three internal streams, through three chunk slots in `workspace` (device
 * memory owned by the caller, at least fat_attn_fwd_host_workspace_bytes(...)
 * bytes).  Every copy is one cudaMemcpyAsync.  The work starts after what is
 * already queued on `stream`, and `stream` waits for the last copy back, so
 * the results are on the host once `stream` has completed.  heads_per_chunk
 * <= 0 picks about eight chunks.  Calls sharing a workspace, or running on
 * the same device from several host threads, must not overlap.  No
 * counterpart on the pages.
 */
int fat_attn_fwd_host(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                      int H, int N, int d, int causal, float scale, int X, int heads_per_chunk,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace size for fat_attn_fwd_host (0 for invalid arguments). */
size_t fat_attn_fwd_host_workspace_bytes(int B, int H, int N, int d, int heads_per_chunk);

/* Every knob of the entry points above in one struct (tests and ablations). */
typedef struct fat_params {
  const void* q;
  const void* k;
  const void* v;
  float* o;
  float* lse;
  int B, H, N, d;
  int causal;
  float scale;
  int X;
  int variant;                        /* fat_variant */
  int dtype;                          /* fat_dtype */
  int l_mode;                         /* fat_lmode (tensorized variant only) */
  float q_descale, k_descale, v_descale; /* e4m3 only; ignored otherwise */
  float underflow_log2_threshold;     /* <= 0: default (64 binades for bf16 P~, 29 for fp16,
                                         14 for e4m3) */
  int* fallback_rows;                 /* nullable device int: += number of rows recomputed */
  unsigned long long wait_poll_limit; /* 0: no cap on polls of one device wait */
  unsigned long long wait_timeout_ns; /* 0: default of 4 s per device wait */
  cudaStream_t stream;
  /* nullable device buffer of FAT_TRACE_WORDS u64 (8-byte aligned): SM-clock
   * stamps of the first thread block's pipeline phases on its first query
   * tile, for measuring how long the tensor pipe waits for the softmax (see
   * the trace layout below) */
  unsigned long long* trace;
  int z_mode;                         /* fat_zmode (tensorized variant only) */
  int block_mode;                     /* fat_block_mode */
} fat_params;

/*
 * Trace layout (first thread block, first query tile, first pass): word
 * (e * 2 + t) * FAT_TRACE_ITERS + j holds the clock of event e at K/V tile j
 * (< FAT_TRACE_ITERS); t = the softmax set that takes tile j (j % 2) for the
 * softmax events, 0 for the MMA issuer's: e = 0 softmax received S_j; 1
 * softmax computed m_hat; 2 softmax published P_j; 3 MMA issuer saw P_j; 4
 * MMA issuer queued O += P_j V and S_{j+3}.  Word FAT_TRACE_WORDS-2: kernel
 * start; FAT_TRACE_WORDS-1: end of that tile's softmax epilogue.  Words of events
 * that did not happen are left untouched.
 */
#define FAT_TRACE_ITERS 128
#define FAT_TRACE_EVENTS 5
#define FAT_TRACE_WORDS (FAT_TRACE_EVENTS * 2 * FAT_TRACE_ITERS + 2)

int fat_attn_fwd_ex(const fat_params* p);

/*
 * Backward pass by recomputation (the v1 recap of the FA-T blog, "从融合到
 * 张量化：FlashAttention 演进脉络": only O and the softmax statistics are kept
 * from the forward pass).  For O = softmax(scale Q K^T [+ causal]) V and an
 * upstream gradient dout, writes the gradients of sum(O * dout):
 *   P = exp(scale S - LSE), D_i = sum_d dout_id O_id,
 *   dV = P^T dout, dS = P * (dout V^T - D), dQ = scale dS K, dK = scale dS^T Q.
 * q, k, v, dout: bf16 [B, H, N, d]; o, lse: the fp32 outputs of a forward
 * call on the same q, k, v (any variant: they are exact up to rounding);
 * dq, dk, dv: fp32 [B, H, N, d], overwritten (dq is cleared on `stream`
 * first and accumulated across key blocks with TMA reduce-adds in no fixed
 * order, so its low-order bits may differ from run to run).  d is 64 or 128.  P and dS enter their
 * MMAs as bf16, with fp32 accumulation.  workspace: device memory owned by
 * the caller, at least fat_attn_bwd_workspace_bytes(B, H, N) bytes (D and
 * log2(e) LSE per row); calls sharing it must not overlap on the device.
 * q, k, v, dout, o, dq, dk, dv must be 16-byte aligned, lse 4-byte aligned.
 * Returns a fat_status; nothing is launched when validation fails.
 */
int fat_attn_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse,
                 const void* dout, float* dq, float* dk, float* dv, int B, int H, int N, int d,
                 int causal, float scale, void* workspace, size_t workspace_bytes,
                 cudaStream_t stream);

/* Workspace size for fat_attn_bwd (0 for invalid arguments). */
size_t fat_attn_bwd_workspace_bytes(int B, int H, int N);

/* Human-readable name of a fat_status value (static string). */
const char* fat_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns FAT_ERR_DEVICE_TIMEOUT if a kernel of this library
 * stopped on a bounded wait since the last check, FAT_ERR_LAUNCH if the
 * synchronisation itself failed, FAT_OK otherwise.
 */
int fat_check_device_error(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FAT_ATTN_H_ */
