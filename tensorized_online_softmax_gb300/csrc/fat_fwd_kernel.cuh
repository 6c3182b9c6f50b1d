// Fused attention forward pass for sm_103a with the tensorized online softmax
// of "FlashAttention-T: Towards Fully Tensorized Attention by Exploiting
// Tensor-Vector Parallelism" (papercache.org summary, section A2, Algorithm 1)
// and its vector-softmax ablation (the FA2 arm of the page's Fig. 10).
//
// A work item is one 128-row query tile of one (batch, head), the fused flow
// of the page's section A3 / Fig. 2 (one output row block per worker, S and P
// on chip).  By default one CTA per SM takes items in turn (the next item's
// loads and first S tiles overlap the last one's epilogue); with one CTA per
// item the same code runs once.  Tensor-vector parallelism comes from a
// three-deep ring of score buffers in TMEM: while the softmax warps turn S_j
// into P_j, the tensor pipe already holds S_{j+1} and S_{j+2} and runs
// O += P_{j-1} V_{j-1}, so neither side waits for the other in the steady
// state.
//
//   warp 9      TMA producer of Q (once per item) and K_j, through an mbarrier ring;
//   warp 10     TMA producer of V_j, through its own ring, so neither stream
//               waits for a slot of the other (K runs three tiles ahead); it
//               also issues the TMA stores of each item's O, which the
//               softmax warps stage in the V ring.
//   warp 8      MMA issuer (the whole warp, one elected lane per MMA group):
//               S_j = Q K_j^T into buffer j % 3, O += P_j V_j, and (row sum on
//               the tensor pipe) l_j = P_j 1.  The tensor pipe queues only a
//               few MMAs, so this loop is kept short.  At d = 64 warp 8
//               issues only the S MMAs and warp 11 the P V MMAs (and row
//               sums), so that P V goes in as soon as P is ready.
//   warps 0-7   softmax in two sets of four: set w / 4 takes every other K/V
//               tile; warp w owns TMEM lanes 32 (w % 4) .. +31 (one row per
//               thread): row maximum, X-row tile maximum, O rescale,
//               P = exp2(Z); at the end of an item, O / l and LSE.
//
// TMEM (512 columns x 128 lanes, fp32): score buffers [0,128), [128,256),
// [256,384); O at [384, 384 + D).  P_j overwrites the scores it came from
// (bf16: columns 0-63 of the buffer, two keys per column; e4m3: 0-31, four
// keys per column); the tensor row sum lands in column 64 of the buffer.
#pragma once

#include <cuda.h>

#include "fat_schedule.h"
#include "sm103_ptx.cuh"

namespace fat {

constexpr int kBlockM = 128;  // query rows per item (= TMEM lanes)
constexpr int kBlockN = 128;  // keys per K/V tile
constexpr int kRowsPerCta = kBlockM;
constexpr int kSBufs = 3;     // score / P buffers in TMEM
constexpr int kOCol = kSBufs * kBlockN;  // first TMEM column of O
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;    // Q and K
constexpr int kLoadVWarp = 10;  // V; warp 11 completes the third warpgroup
constexpr int kPvWarp = 11;     // (d = 64) issues O += P V while warp 8 issues S = Q K^T
constexpr int kNumThreads = 384;
// Register budget: 384 threads launch with kLaunchRegs each; the MMA/TMA
// warpgroup drops to kCtrlRegs and the two softmax warpgroups rise to
// kSoftmaxRegs.  256 * kSoftmaxRegs + 128 * kCtrlRegs <= 384 * kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 56;
constexpr int kSoftmaxRegs = 224;
static_assert(256 * kSoftmaxRegs + 128 * kCtrlRegs <= kNumThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
// input types (template argument kDt)
constexpr int kDtBf16 = 0;
constexpr int kDtE4M3 = 1;
constexpr int kDtF16 = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// named barriers (0 is __syncthreads)
constexpr uint32_t kBarPair = 1;   // + quarter: the two warps (one per set) of 32 rows
constexpr uint32_t kBarSet = 5;    // + set: the set's four warps (X = 128)
constexpr uint32_t kBarGroup = 7;  // + 2 set + half: two warps of a set (X = 64)

struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;        // fp32 O (or the split partials) as [rows, N_q, d], 32 x 128 boxes
  float* o;
  float* lse;
  int* fallback_rows;
  int B, H;
  int Nq, Nk;              // query rows, keys per (b, h)
  int causal;              // key j allowed for query i iff j <= i + Nk - Nq
  int X;
  int n_mblocks;           // ceil(Nq / 128)
  int n_items;             // work items (query tiles) per split: B H n_mblocks
  int group_heads;         // heads whose query blocks are ordered together
  int prefetch_stride;     // > 0: prefetch into L2 the first tiles of block + this
  int kv_split_len;        // keys per split (a multiple of 128): blockIdx.y = split
  float* o_part;           // nullable: per-split partial O [splits][B*H][Nq][d] ...
  float* lse_part;         // ... and LSE [splits][B*H][Nq] instead of o / lse
  float scale;             // softmax scale as received
  float c;                 // log2(e) * scale (times q/k descales for e4m3)
  float underflow_thresh;  // binades between surrogate and exact row maximum
  float v_scale;           // applied to O in the epilogue (e4m3 V descale; 1 for bf16)
  unsigned long long poll_limit;
  unsigned long long timeout_ns;
  unsigned long long* trace;  // nullable: phase stamps of CTA 0 (kTraceWords)
  unsigned int* error_word;   // device error word: bit 0 = a bounded wait ran out
};

// Phase trace of CTA 0, SM clock (clock64) stamps, its first item's first
// pass only:
//   word (e * 2 + t) * kTraceIters + j for event e, K/V tile j, and t = the
//   softmax set that takes tile j (softmax events, written by warps 0 and
//   4) or 0 (MMA):
//   e = 0 softmax got S_j, 1 softmax has m_hat, 2 softmax publishes P_j,
//       3 MMA issuer sees P_j, 4 MMA issuer has queued O += P_j V, S_{j+3};
//   word kTraceWords - 2 / - 1: kernel start / softmax epilogue done.
constexpr int kTraceIters = 128;
constexpr int kTraceEvents = 5;
constexpr int kTraceWords = kTraceEvents * 2 * kTraceIters + 2;

__device__ __forceinline__ void trace_mark(const FwdParams& p, int e, int t, int j, bool on) {
  if (on && p.trace != nullptr && blockIdx.x == 0 && j < kTraceIters)
    p.trace[(e * 2 + t) * kTraceIters + j] = static_cast<unsigned long long>(clock64());
}

// The same once the caller has checked that this block traces this pass.
__device__ __forceinline__ void trace_at(const FwdParams& p, int e, int t, int j) {
  if (j < kTraceIters)
    p.trace[(e * 2 + t) * kTraceIters + j] = static_cast<unsigned long long>(clock64());
}

// Item idx -> (query block, head).  Heads run a few at a time, as many as
// keep their K and V in L2 while the query blocks re-read them; within a
// group, the heaviest causal blocks first.
__device__ __forceinline__ void fwd_work_item(const FwdParams& p, int idx, int& mblock, int& bh) {
  const int BH = p.B * p.H;
  const int per = p.group_heads * p.n_mblocks;
  const int g = idx / per;
  const int rem = idx - g * per;
  const int gh = min(p.group_heads, BH - g * p.group_heads);
  mblock = p.n_mblocks - 1 - rem / gh;
  bh = g * p.group_heads + rem % gh;
}

// The k-th item of this block, or -1 past the end (fat_schedule.h).
__device__ __forceinline__ int fwd_item_at(const FwdParams& p, int k) {
  return fwd_item_index(k, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                        p.n_items);
}

template <int D, bool kE4M3 = false, bool kZT = false>
struct Smem {
  static constexpr int kElt = kE4M3 ? 1 : 2;          // bytes per input element
  static constexpr int kTile = kBlockM * D * kElt;    // bytes of one 128 x D tile
  // K_{j+3} is loaded once S_j is done, V_j once O += P_{j-3} V is; 256-byte
  // rows fit two K and three V stages
  static constexpr int kKStages = (D * kElt == 256) ? 2 : 4;
  static constexpr int kVStages = (D * kElt == 256) ? 3 : 4;
  // With at most as many K stages as score buffers, the completion of S_it
  // also marks K stage it % kKStages free (K_{it + kKStages} is loaded after
  // it, and the buffer's next S needs a later K tile, so a waiter is never
  // two phases behind); deeper K rings keep their own "K free" barrier.
  static constexpr bool kKFreeOnS = kKStages <= kSBufs;
  static constexpr int kAtoms = D * kElt / 128;       // 128-byte-wide column slabs per tile
  static constexpr int kAtomCols = 128 / kElt;        // elements per slab row
  static constexpr int kMmaK = 32 / kElt;             // K of one MMA (bf16 16, e4m3 32)
  static constexpr int kPvStep = kMmaK * 128;         // bytes of V rows per PV K step
  static_assert(kAtoms >= 1, "rows must span at least one 128-byte slab");
  static constexpr int kQ = 0;
  static constexpr int kK = kTile;                     // K ring
  static constexpr int kV = kK + kKStages * kTile;     // V ring
  static constexpr int kOnes = kV + kVStages * kTile;  // 16 rows x 128 B of ones (2 KB)
  // Z on the tensor pipe (kZT): per score buffer a 128 x 16 bf16 bias tile
  // (the A of one more K step of S = Q K^T) and one 128 x 16 tile of ones
  // (its B); K-major without swizzle, 4 KB each
  static constexpr int kZBias = kOnes + 2048;
  static constexpr int kZOnes = kZBias + 3 * 4096;
  static constexpr int kBars = kZT ? kZOnes + 4096 : kOnes + 2048;
  // barrier slots
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;
  static constexpr int bKEmpty = bKFull + kKStages;
  static constexpr int bVFull = bKEmpty + kKStages;
  static constexpr int bVEmpty = bVFull + kVStages;
  static constexpr int bSFull = bVEmpty + kVStages;  // [kSBufs]
  static constexpr int bPFull = bSFull + kSBufs;     // [kSBufs], 4 arrivals (one set)
  static constexpr int bRsFull = bPFull + kSBufs;    // [kSBufs]
  static constexpr int bLFree = bRsFull + kSBufs;    // [kSBufs], 4 arrivals
  // [kSBufs]: O += P_it V landed, it % 3 (per buffer, so that a waiter is
  // never two phases behind: PV_{it-3} has completed once S_it has)
  static constexpr int bOReady = bLFree + kSBufs;
  static constexpr int bOFinal = bOReady + kSBufs;
  static constexpr int bDrain = bOFinal + 1;
  static constexpr int bMReady = bDrain + 1;         // [2 sets], 4 arrivals: offset published
  // a block runs several work items (query tiles) in turn:
  static constexpr int bQFree = bMReady + 2;         // every S MMA of an item has read Q
  static constexpr int bOFree = bQFree + 1;          // 8 arrivals: the epilogue has read O
  static constexpr int bDecided = bOFree + 1;        // 4 arrivals: set 0's detector done
  static constexpr int bStaged = bDecided + 1;       // 8 arrivals: a pass's O is staged
  static constexpr int bStageFree = bStaged + 1;     // its stores have read the staging
  static constexpr int bListReady = bStageFree + 1;  // once: every first pass detected
  // (d = 64: two MMA issuers) the P V issuer's drain after an abort
  static constexpr bool kTwoIssuers = D == 64;
  static constexpr int bDrainPv = bListReady + 1;
  static constexpr int kNumBars = bListReady + 1 + (kTwoIssuers ? 1 : 0);
  static constexpr int kRed = (kBars + 8 * kNumBars + 15) & ~15;  // float [2 sets][2 parity][4 warps]
  static constexpr int kMRow = kRed + 64;            // float [2 sets][128 rows]: offsets
  static constexpr int kFin = kMRow + 1024;          // float [2 epilogues][4][2 sets][128 rows]
  // u32: tmem base, abort, deferred count, last flagged item + 1, then (kZT)
  // as floats the bias held by each score buffer's bias tile [3]
  static constexpr int kMisc = kFin + 8192;
  static constexpr int kDefer = kMisc + 64;          // int [kMaxDeferred]: flagged items
  static constexpr int kBytes = kDefer + 4 * kMaxDeferred;
  static constexpr int kAlloc = kBytes + 1024;       // slack for 1024-byte alignment
  // The epilogue stages O (fp32, 128 x D) in the V ring, idle once O is
  // final, as 16 KB boxes of 32 columns x 128 rows (128-byte swizzled) for
  // the TMA tensor stores that the V producer issues.  Where the ring has
  // room, the boxes skip the stage of the next pass's first V tile, so that
  // tile loads while the last pass's O is still being written out.
  static constexpr int kBoxes = D / 32;
  static constexpr int kBoxesPerStage = kTile / 16384;
  static constexpr bool kStageSkipsFirst = (kVStages - 1) * kBoxesPerStage >= kBoxes;
  static_assert(kVStages * kTile >= kBlockM * D * 4, "O staging does not fit the V ring");
  // offset of box b when the next pass's first V tile goes to stage v0
  __device__ __forceinline__ static int box(int b, int v0) {
    if constexpr (kStageSkipsFirst)
      return kV + ((v0 + 1 + b / kBoxesPerStage) % kVStages) * kTile +
             (b % kBoxesPerStage) * 16384;
    return kV + b * 16384;
  }
  // whether V stage st holds part of that staging
  __device__ __forceinline__ static bool holds_o(int st, int v0) {
    if constexpr (kStageSkipsFirst)
      return st != v0 && ((st - v0 - 1 + kVStages) % kVStages) * kBoxesPerStage < kBoxes;
    return st * kBoxesPerStage < kBoxes;
  }
  static_assert(kK % 1024 == 0 && kV % 1024 == 0 && kOnes % 1024 == 0, "tiles 1 KB aligned");
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
// (P: any parameter block with poll_limit, timeout_ns and error_word)
template <class P>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const P& p,
                                             volatile uint32_t* abort_flag) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint64_t polls = 1;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    ++polls;
    if (*abort_flag) break;
    if (p.poll_limit != 0 && polls >= p.poll_limit) break;
    if ((polls & 63) == 0 && globaltimer_ns() - t0 > p.timeout_ns) break;
  }
  atomicOr(p.error_word, 1u);
  *abort_flag = 1u;
  return false;
}

// Waits used only to drain work already in flight after an abort: they never
// look at the abort flag and use a fixed one-second limit.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 1000000000ull) return;
  }
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float f16_round(float x) { return __half2float(__float2half_rn(x)); }

// ---------------------------------------------------------------------------
// softmax warps: two sets of four.  Set s = w / 4 takes the K/V tiles j with
// j % 2 == s, and warp w owns TMEM lanes 32 (w % 4) .. +31: one row per
// thread, all 128 keys of the tile.  The sets work on alternate tiles, so on
// each SM sub-partition one warp's TMEM loads and maxima run beside the
// other's exponentials.  The offset of the online softmax passes from tile
// to tile, i.e. from set to set, through shared memory (one value per row)
// and one mbarrier per set.
//   kX > 0   tensorized online softmax with the surrogate maximum over kX-row
//            tiles (X is a compile-time constant so no runtime branching sits
//            in the hot loop); kExact (the fallback pass) uses each row's own
//            maximum instead, rounded up to a whole binade.
//   kX == 0  the vector-softmax ablation: exact per-row maximum.
//
// One call covers one pass over one item (item idx, the seq-th of the
// block).  it0: the block's K/V tiles before this pass (all ring and buffer
// phases count from the block's start); epi: the block's passes before this
// one (phases of the once-per-pass barriers); mr_other: the other set's
// tiles before this pass (phases of its offset barrier); tr: stamp the phase
// trace.  In a first pass (not kExact) set 0 runs the detector and appends a
// flagged item to the block's deferred list, which gets its fallback pass
// after the block's last item.  Returns true when the block must stop (a
// bounded wait ran out somewhere); all eight warps return the same value.
// ---------------------------------------------------------------------------
constexpr uint32_t kBarSoftmax = 11;  // all eight softmax warps

template <int D, int kX, bool kLTensor, int kDt, bool kZT, bool kExact>
__device__ __forceinline__ bool softmax_role(const FwdParams& p, uint8_t* smem, uint32_t sb,
                                             uint32_t tmem, volatile uint32_t* misc, int warp,
                                             int lane, int idx, int seq, int m0, int bh, int n_kv,
                                             int it0, int split, int kv_begin, int kv_end,
                                             int kv_off, int epi, int mr_other, bool tr) {
  constexpr bool kE4M3 = kDt == kDtE4M3;
  using L = Smem<D, kE4M3, kZT>;
  constexpr bool kTensor = kX > 0;
  // e4m3 (fp16) P~ is formed as 2^(Z + kKappa) <= 2^8 < 448 (2^15 < 65504)
  // so that its terms use the format's range; the factor cancels in O / l and
  // is taken off LSE.  bf16 has fp32's exponent range and needs none.
  constexpr float kKappa = kE4M3 ? 8.f : (kDt == kDtF16 ? 15.f : 0.f);
  // Headroom of the surrogate offset (binades): it is raised only when a
  // tile's maximum exceeds it by more than this, so P~ <= 2^kHeadroom.  Once
  // an item's first tile has set it, Gaussian-like scores hardly ever climb
  // 8 binades further, so the uniform O rescale -- and its wait for the last
  // P V -- all but disappears.  bf16 P~ has fp32's exponent range to spare;
  // fp16 and e4m3 P~ use their range for kKappa, and the fallback pass keeps
  // each row's own maximum.
  constexpr float kHeadroom = (kTensor && !kExact && kDt == kDtBf16) ? 8.f : 0.f;
  constexpr int kHalfD = D / 2;  // O columns this set rescales and writes
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8 * i; };
  const int q = warp & 3;        // quarter of the tile (TMEM lanes 32 q ..)
  const int set = warp >> 2;     // K/V tiles j with j % 2 == set
  const int other = set ^ 1;
  const int r = q * 32 + lane;   // row within the tile
  const int row_g = m0 + r;
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  const uint32_t o_taddr = tmem + lane_base + kOCol;
  const float c = p.c;
  float* red = reinterpret_cast<float*>(smem + L::kRed);    // [2 sets][2 parity][4 warps]
  float* mrow = reinterpret_cast<float*>(smem + L::kMRow);  // [2 sets][128 rows]
  // [4][2 sets][128 rows], one copy per parity of epi (the other set may
  // still read the previous pass's values)
  float* fin = reinterpret_cast<float*>(smem + L::kFin) + (epi & 1) * (4 * 2 * kBlockM);
  // (kZT) the bias b held by each score buffer's bias tile, in raw score units
  volatile float* zvals = reinterpret_cast<volatile float*>(misc + 4);
  // Warps of the set that share a surrogate maximum: none besides this one
  // for X <= 32, the fallback pass and the vector variant; two for X = 64,
  // the set's four for X = 128.
  constexpr bool solo = kX <= 32 || kExact;
  const uint32_t gbar_id = kX == 64 ? kBarGroup + set * 2 + (q >> 1) : kBarSet + set;
  const uint32_t gbar_n = kX == 64 ? 64 : 128;

  float M = -INFINITY;    // offset of this set's latest tile (per row; uniform over
                          // the X-row group in the surrogate modes), binades
  float m_row = -INFINITY;  // exact maximum of this row over this set's tiles, logits
  float l = 0.f;          // this set's part of the row sum, relative to M
  float delta = 0.f;      // tensor row sum: rounding of each tile's dominant term
  bool dead = false;      // a bounded wait of this warp (or of its group) ran out
  int j = set;
  int k_local = 0;        // this set's tiles so far in this pass
  // Tensor row sum of this set's previous tile (read one tile late so the
  // read never waits); it refers to the offset M of that tile.
  int rs_pending = -1;
  auto take_row_sum = [&](int itp) -> bool {
    if (!__all_sync(0xffffffffu, wait_bounded(bar(L::bRsFull + itp % kSBufs),
                                              (itp / kSBufs) & 1, p, abort_flag)))
      return false;
    tc_fence_after();
    uint32_t lt;
    tmem_ld1(tmem + lane_base + (itp % kSBufs) * kBlockN + 64, lt);
    tmem_wait_ld1(lt);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bLFree + itp % kSBufs));
    l += __uint_as_float(lt);
    return true;
  };
  // offset of tile jj - 1 (the other set's), once that set has settled it
  auto prev_offset = [&](int jj) -> float {
    if (jj == 0) return -INFINITY;
    const int kk = (jj - 1) / 2;  // the other set's tile count
    if (!__all_sync(0xffffffffu, wait_bounded(bar(L::bMReady + other),
                                              (mr_other + kk) & 1, p, abort_flag))) {
      dead = true;
      return -INFINITY;
    }
    return mrow[other * kBlockM + r];
  };
  auto publish_offset = [&](float Mj) {
    mrow[set * kBlockM + r] = Mj;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bMReady + set));
  };

  for (; j < n_kv; j += 2, ++k_local) {
    const int it = it0 + j;
    const int buf = it % kSBufs;
    const uint32_t par = k_local & 1;
    const uint32_t s_taddr = tmem + lane_base + buf * kBlockN;
    dead = !__all_sync(0xffffffffu,
                       wait_bounded(bar(L::bSFull + buf), (it / kSBufs) & 1, p, abort_flag));
    if (q == 0 && lane == 0) trace_mark(p, 0, set, j, tr);
    uint32_t s[4][32];
    float rowmax = -INFINITY;
    int limit = kBlockN;  // keys of this K/V tile the row may see
    if (!dead) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_ld32(s_taddr + 32 * k, s[k]);
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_wait_ld(s[k]);
      // mask: keys >= N, keys after the query (causal), padding rows
      const int kv0 = kv_begin + j * kBlockN;
      limit = (row_g < p.Nq) ? (p.causal ? min(kv_end, row_g + kv_off + 1) : kv_end) - kv0 : 0;
      if (limit < kBlockN) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * k + i >= limit) s[k][i] = __float_as_uint(-INFINITY);
      }
      // row maximum as a tree of independent 3-input maxima
      float mx[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const int k = a >> 1, b = (a & 1) * 16;
        mx[a] = fmax3(__uint_as_float(s[k][b]), __uint_as_float(s[k][b + 1]),
                      __uint_as_float(s[k][b + 2]));
#pragma unroll
        for (int i = 3; i < 15; i += 2)
          mx[a] = fmax3(mx[a], __uint_as_float(s[k][b + i]), __uint_as_float(s[k][b + i + 1]));
        mx[a] = fmaxf(mx[a], __uint_as_float(s[k][b + 15]));
      }
      rowmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
      if constexpr (!kZT) m_row = fmaxf(m_row, rowmax);
    }
    // (kZT: these are maxima of S + b; b is taken off below, once known)
    const float rowmax_raw = rowmax;
    float zb = 0.f;  // (kZT) the bias in this tile's scores
    // Algorithm 1 step 1: maximum of the row maxima over the X-row tile: this
    // warp's part (its 32 rows, or 16-row groups for X = 16) ...
    float tmax = rowmax;
    if constexpr (kX == 16) {
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    } else if constexpr (kX >= 32) {
      tmax = warp_max(rowmax);
    }
    // ... and across the warps of the group (X = 64, 128) through shared
    // memory.  Every warp of a group joins the same group barriers, aborted
    // or not (see the drain loop below): one OR per tile, and the exchange
    // after it when the OR is set; an aborted warp posts NaN there, which
    // tells the others to stop.
    float* slot = red + (set * 2 + par) * 4;
    auto group_max = [&](float v) -> float {
      if (lane == 0) slot[q] = dead ? __uint_as_float(0x7fc00000u) : v;
      named_bar_sync(gbar_id, gbar_n);
      float m;
      if (kX == 64) {
        const float2 ab = *reinterpret_cast<const float2*>(slot + (q & 2));
        m = fmax_nan(ab.x, ab.y);
      } else {
        const float4 s4 = *reinterpret_cast<const float4*>(slot);
        m = fmax_nan(fmax_nan(s4.x, s4.y), fmax_nan(s4.z, s4.w));
      }
      if (isnan(m)) dead = true;
      return m;
    };

    // the offset of tile j - 1 (O refers to it until PV_j), then this tile's
    float M_prev, M_new;  // binades
    if (!solo) {
      // X = 64 / 128: the surrogate maximum is kept as a whole number of
      // binades (so the rescale factor is an exact power of two), and one OR
      // over the group's barrier settles whether any warp raises it -- rarely
      // once the running maximum has settled; only then are the warps'
      // maxima exchanged.  A warp that gave up votes yes and posts NaN.
      M_prev = prev_offset(j);
      if constexpr (kZT) {
        // written three tiles ago by the other set, before it published the
        // offset just read (or zero from the start of the pass)
        zb = zvals[buf];
        rowmax -= zb;
        tmax -= zb;
        m_row = fmaxf(m_row, rowmax);
      }
      const float Mc = (tmax == -INFINITY) ? -INFINITY : ceilf(tmax * c);
      const bool any = named_bar_or(gbar_id, gbar_n, dead || Mc > M_prev + kHeadroom);
      M_new = M_prev;
      if (any) {
        const float gmc = group_max(Mc);
        if (dead) break;
        M_new = fmaxf(M_prev, gmc);
      }
    } else {
      // X <= 32 within the warp; the fallback pass and the vector variant
      // each row's own maximum (the fallback pass rounded up to a binade)
      if (dead) break;
      M_prev = prev_offset(j);
      if (dead) break;
      if constexpr (kZT) {  // (the fallback pass: the bias tiles hold zero)
        zb = zvals[buf];
        rowmax -= zb;
        tmax -= zb;
        m_row = fmaxf(m_row, rowmax);
      }
      const float gm = (kExact || !kTensor) ? rowmax : tmax;
      if constexpr (kTensor) {
        const float Mc = (gm == -INFINITY) ? -INFINITY : ceilf(gm * c);
        M_new = Mc > M_prev + kHeadroom ? Mc : M_prev;
      } else {
        M_new = fmaxf(M_prev, (gm == -INFINITY) ? -INFINITY : gm * c);
      }
    }
    publish_offset(M_new);
    if constexpr (kZT) {
      // The bias of S_{j+3}, which the MMA issuer queues into this score
      // buffer once P~_j is published: -M_new in raw score units, as bf16
      // (zero in the fallback pass).  The tile is rewritten only when the
      // value changes; the set's four warps read the old value before the
      // group barrier above.
      const float bz = (!solo && M_new != -INFINITY)
                           ? __bfloat162float(__float2bfloat16_rn(-M_new / c))
                           : 0.f;
      if (bz != zb) {
        const uint32_t w = pack_bf16x2(bz * 0.0625f, bz * 0.0625f);  // 16 equal terms make b
        const uint32_t dst = sb + L::kZBias + buf * 4096 + r * 32;
        st_shared_v4u(dst, w, w, w, w);
        st_shared_v4u(dst + 16, w, w, w, w);
        fence_async_shared();
        if (q == 0 && lane == 0) zvals[buf] = bz;
      }
    }
    if (q == 0 && lane == 0) trace_mark(p, 1, set, j, tr);
    const float neg_E = (M_new == -INFINITY) ? 0.f : -M_new;
    // step 7 on the tensor pipe: the row sum of this set's previous tile
    // (relative to that tile's offset M), taken before the exponentials and
    // before any wait on the tensor pipe: the MMA issuer reuses that tile's
    // score buffer (and queues O += P_{j-1} V behind it) only after this read.
    if (kLTensor && rs_pending >= 0 && !dead) {
      if (!take_row_sum(rs_pending)) dead = true;
    }

    // steps 4-6: Z = c S - m_hat, P~ = exp2(Z), stored as bf16 (e4m3) over S
    // (kZT: c (S + b) - (c b + m_hat))
    const float nm = (kZT ? fmaf(-c, zb, neg_E) : neg_E) + kKappa;
    const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(nm, nm);
    uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float pf[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t z = f2_fma(f2_pack(__uint_as_float(s[k][2 * i]),
                                          __uint_as_float(s[k][2 * i + 1])), c2, nm2);
        float z0, z1;
        f2_unpack(z, z0, z1);
        pf[2 * i] = ex2_approx(z0);
        pf[2 * i + 1] = ex2_approx(z1);
        if (!kLTensor) acc2[i & 1] = f2_add(acc2[i & 1], f2_pack(pf[2 * i], pf[2 * i + 1]));
      }
      if constexpr (kE4M3) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = pack_e4m3x4(pf[4 * i], pf[4 * i + 1], pf[4 * i + 2], pf[4 * i + 3]);
        tmem_st8(s_taddr + 8 * k, pk);
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = kDt == kDtF16 ? pack_f16x2(pf[2 * i], pf[2 * i + 1])
                                : pack_bf16x2(pf[2 * i], pf[2 * i + 1]);
        tmem_st16(s_taddr + 16 * k, pk);
      }
    }
    float lt_vec;  // this tile's row sum (vector row sum only), relative to E
    {
      float r0, r1;
      f2_unpack(f2_add(acc2[0], acc2[1]), r0, r1);
      lt_vec = r0 + r1;
    }

    // steps 2-3: O (which refers to the offset of tile j - 1) takes the
    // factor exp(m_prev - m_new), from the vector side and only when the
    // offset grew -- for X = 128 one factor for the whole tile, a rare event
    // once the running maximum has settled -- once O += P_{j-1} V has landed
    // (PV_j waits for the P-full signal below).
    const bool grow = j > 0 && M_new > M_prev;
    const bool vec_rescale = grow;
    if (__any_sync(0xffffffffu, vec_rescale)) {
      const float alpha = grow ? ex2_approx(M_prev - M_new) : 1.f;
      if (!__all_sync(0xffffffffu, wait_bounded(bar(L::bOReady + (it - 1) % kSBufs),
                                                ((it - 1) / kSBufs) & 1, p, abort_flag))) {
        dead = true;
      } else {
        tc_fence_after();
        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          uint32_t ov[32];
          tmem_ld32(o_taddr + 32 * k, ov);
          tmem_wait_ld(ov);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float o0, o1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1])), a2), o0,
                      o1);
            ov[i] = __float_as_uint(o0);
            ov[i + 1] = __float_as_uint(o1);
          }
          tmem_st32(o_taddr + 32 * k, ov);
        }
      }
    }
    // step 7: this set's row sum, carried from its previous tile's offset to
    // this tile's
    if (M_new != -INFINITY && M != -INFINITY) {
      const float f = ex2_approx(M - M_new);
      l *= f;
      if (kLTensor) delta *= f;
    }
    if constexpr (kLTensor) {
      rs_pending = it;
      if (rowmax != -INFINITY) {
        // the dominant term exactly as the exponentials above formed it
        const float pm = ex2_approx(fmaf(rowmax_raw, c, nm));
        delta += pm - (kE4M3 ? e4m3_round(pm) : (kDt == kDtF16 ? f16_round(pm) : bf16_round(pm)));
      }
    } else {
      l += lt_vec;
    }
    M = M_new;
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (q == 0 && lane == 0) trace_mark(p, 2, set, j, tr);
    // a warp that gave up still signals; the MMA issuer sees the abort flag
    if (lane == 0) mbar_arrive(bar(L::bPFull + buf));
    if (dead) break;
  }
  if (dead && !solo) {
    // An aborted warp left the loop at tile j.  If it left at the group
    // barrier, every warp of its group left there too; otherwise (a wait of
    // its own ran out after the group barrier of tile j) the others meet it
    // at the next tile's barrier, where its NaN stops them.  From there on
    // all of them join the same barriers, tile by tile, until the end.
    for (j += 2, ++k_local; j < n_kv; j += 2, ++k_local) {
      named_bar_or(gbar_id, gbar_n, true);
      if (lane == 0) red[(set * 2 + (k_local & 1)) * 4 + q] = __uint_as_float(0x7fc00000u);
      named_bar_sync(gbar_id, gbar_n);
    }
  }

  bool ok = !dead;
  if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bOFinal), epi & 1, p, abort_flag));
  if (ok && kLTensor && rs_pending >= 0) ok = take_row_sum(rs_pending);
  // combine the two sets' parts of every row (both warps of a pair get here)
  fin[(0 * 2 + set) * kBlockM + r] = m_row;
  fin[(1 * 2 + set) * kBlockM + r] = l;
  fin[(2 * 2 + set) * kBlockM + r] = delta;
  fin[(3 * 2 + set) * kBlockM + r] = M;
  named_bar_sync(kBarPair + q, 64);
  const float m_o = fin[(0 * 2 + other) * kBlockM + r];
  const float l_o = fin[(1 * 2 + other) * kBlockM + r];
  const float d_o = fin[(2 * 2 + other) * kBlockM + r];
  const float M_o = fin[(3 * 2 + other) * kBlockM + r];
  const float m_full = fmaxf(m_row, m_o);
  const float M_fin = fmaxf(M, M_o);  // the offset of the last tile (offsets only grow)
  const float f_me = (M == -INFINITY) ? 0.f : ex2_approx(M - M_fin);
  const float f_o = (M_o == -INFINITY) ? 0.f : ex2_approx(M_o - M_fin);
  const float l_full = l * f_me + l_o * f_o;
  const float delta_full = delta * f_me + d_o * f_o;
  if (set == 0) {
    // Detector for the all-underflow case (first pass of the tensorized
    // softmax): surrogate far above the exact maximum, or nothing left of
    // the row sum; flagged rows counted once.  The first warp of set 0 to
    // flag a row puts the item on the block's deferred list (the atomic
    // maximum over seq + 1 lets exactly one warp per item through).  Then
    // each warp of set 0 arrives on the detector barrier, which every role
    // waits for before it reads the list, and (kZT) the MMA issuer before
    // the next S tiles -- so that is also where the bias tiles go back to
    // zero: every S MMA of this pass has completed (O final came after the
    // last one).
    bool flagged = false;
    if (kTensor && !kExact && ok) {
      // (a row with no key in this split's range is empty, not flagged)
      flagged = row_g < p.Nq && m_full != -INFINITY &&
                (!(l_full > 0.f) || (M_fin - m_full * c) > p.underflow_thresh);
    }
    const uint32_t ball = __ballot_sync(0xffffffffu, flagged);
    if (ball != 0 && lane == 0) {
      if (p.fallback_rows) atomicAdd(p.fallback_rows, __popc(ball));
      uint32_t* m = const_cast<uint32_t*>(misc);
      if (atomicMax(m + 3, static_cast<uint32_t>(seq + 1)) < static_cast<uint32_t>(seq + 1)) {
        const uint32_t k = atomicAdd(m + 2, 1u);
        if (k < kMaxDeferred) reinterpret_cast<volatile int*>(smem + L::kDefer)[k] = idx;
      }
    }
    if constexpr (kZT) {
      for (int i = r; i < 3 * 4096 / 16; i += kBlockM)
        st_shared_v4u(sb + L::kZBias + 16 * i, 0u, 0u, 0u, 0u);
      if (r < kSBufs) zvals[r] = 0.f;
      fence_async_shared();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bDecided));
  }
  // the last pass's stores must have read their staging before this pass
  // stages over it (long since, unless that pass was short)
  if (ok && epi > 0)
    ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bStageFree), (epi - 1) & 1, p, abort_flag));
  if (ok) {
    tc_fence_after();
    // epilogue: O / l, this set's half of the columns, staged in shared
    // memory as 128-byte-swizzled boxes of 32 columns x 128 rows for the TMA
    // store below
    const float inv_l = l_full > 0.f ? p.v_scale / l_full : 0.f;  // an empty row gets O = 0
    const int v0 = (it0 + n_kv) % L::kVStages;  // the next pass's first V stage
#pragma unroll
    for (int k = 0; k < kHalfD / 32; ++k) {
      uint32_t ov[32];
      tmem_ld32(o_taddr + set * kHalfD + 32 * k, ov);
      tmem_wait_ld(ov);
      const uint32_t box = sb + L::box(set * (kHalfD / 32) + k, v0) + r * 128;
      if (row_g < p.Nq) {  // (rows past N_q are clipped by the store anyway)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          st_shared_v4(box + ((cc ^ (r & 7)) << 4), __uint_as_float(ov[4 * cc]) * inv_l,
                       __uint_as_float(ov[4 * cc + 1]) * inv_l,
                       __uint_as_float(ov[4 * cc + 2]) * inv_l,
                       __uint_as_float(ov[4 * cc + 3]) * inv_l);
      }
    }
  }
  // O has been read: the next pass's (or item's) first O = P V may overwrite it
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar(L::bOFree));
  if (ok && row_g < p.Nq && set == 0) {
    const size_t out_row = (static_cast<size_t>(split) * (p.B * p.H) + bh) * p.Nq + row_g;
    const float lsum = kLTensor ? l_full + delta_full : l_full;
    (p.lse_part ? p.lse_part : p.lse)[out_row] =
        l_full > 0.f ? (M_fin - kKappa + __log2f(lsum)) * kLn2 : -INFINITY;
  }
  // The staged boxes go to the async proxy, whose stores the V producer
  // issues once all eight warps have arrived (every warp arrives, aborted or
  // not; the producer stores nothing after an abort).  The softmax warps go
  // straight on to the next pass.
  fence_async_shared();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar(L::bStaged));
  if (tr && r == 0 && set == 0 && p.trace != nullptr && blockIdx.x == 0)
    p.trace[kTraceWords - 1] = static_cast<unsigned long long>(clock64());
  tc_fence_before();
  // all eight warps take the same way on: stop if any warp (or any wait
  // anywhere in the block) gave up
  return named_bar_or(kBarSoftmax, kSoftmaxWarps * 32, !ok || *abort_flag != 0u);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// kX:       > 0: surrogate maximum over kX-row tiles (Algorithm 1);
//           0: the exact per-row maximum (vector-softmax ablation).
// kLTensor: (kTensor only) the row sum of step 7 on the tensor pipe as
//           P~ (bf16) times a block of ones; otherwise an fp32 sum of the
//           unrounded P~ on the vector units.
// kDt:      input type: kDtBf16 (kind::f16 MMAs, bf16 P~), kDtF16 (kind::f16,
//           fp16 P~) or kDtE4M3 (kind::f8f6f4, e4m3 P~).
// kZT:      (bf16, X = 128 only) the subtraction of Algorithm 1 steps 4-5 on
//           the tensor pipe: S = Q K^T gets one more 16-deep K step, a bias
//           tile (every entry b / 16, b = -m_ref / (log2(e) scale) rounded to
//           bf16) against a tile of ones, so the MMA writes S + b; m_ref is
//           the surrogate maximum settled three tiles earlier (the latest one
//           known when S is queued), and the vector side folds in the rest.
template <int D, int kX, bool kLTensor, int kDt, bool kZT = false>
__global__ void __launch_bounds__(kNumThreads, 1) fat_fwd_kernel(const __grid_constant__ FwdParams p) {
  static_assert(!kZT || (kX == 128 && kDt == kDtBf16), "Z on the tensor pipe: bf16, X = 128");
  constexpr bool kE4M3 = kDt == kDtE4M3;
  using L = Smem<D, kE4M3, kZT>;
  constexpr int SK = L::kKStages;
  constexpr int SV = L::kVStages;
  constexpr bool kTensor = kX > 0;
  constexpr bool kTwoIssuers = L::kTwoIssuers;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8 * i; };

  // This block's key range is the split's; a work item is one query tile
  // (mblock) of one head (bh), with the split's keys cut at the causal limit
  // of the tile's last row.
  const int BH = p.B * p.H;
  const int split = static_cast<int>(blockIdx.y);
  const int kv_begin = split * p.kv_split_len;
  const int kv_end = min(p.Nk, kv_begin + p.kv_split_len);
  const int kv_off = p.Nk - p.Nq;
  struct Item {
    int m0, bh, n_kv;
  };
  auto item = [&](int idx) -> Item {
    int mblock, bh;
    fwd_work_item(p, idx, mblock, bh);
    const int m0 = mblock * kRowsPerCta;
    const int kv_hi = p.causal ? min(kv_end, m0 + kRowsPerCta + kv_off) : kv_end;
    return {m0, bh, kv_hi > kv_begin ? (kv_hi - kv_begin + kBlockN - 1) / kBlockN : 0};
  };
  // (the launch never has more blocks than items; only a split can leave an
  // item without keys, and a split launch gives each block one item)
  const Item first = item(fwd_item_at(p, 0));
  const int m0 = first.m0, bh = first.bh, n_kv = first.n_kv;
  if (n_kv == 0) {
    // no key of this split reaches these rows (split-KV, causal): an empty
    // partial result that the combine step weighs by zero
    for (int i = threadIdx.x; i < kRowsPerCta; i += kNumThreads) {
      const int row = m0 + i;
      if (row >= p.Nq) continue;
      const size_t out_row = (static_cast<size_t>(split) * BH + bh) * p.Nq + row;
      float4* orow = reinterpret_cast<float4*>(p.o_part + out_row * D);
      for (int c4 = 0; c4 < D / 4; ++c4) orow[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.lse_part[out_row] = -INFINITY;
    }
    return;
  }

  // ---- set-up --------------------------------------------------------------
  // The Q/K producer's first thread initialises the barriers and at once
  // issues the loads of the first item's Q and first K tiles, which then
  // overlap the TMEM allocation and the block-wide sync.
  const bool init_thread = threadIdx.x == kLoadWarp * 32;
  int k_pre = 0;  // K tiles of pass 0 issued here (by init_thread)
  if (init_thread) {
    mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(bar(L::bKFull + s), 1);
      mbar_init(bar(L::bKEmpty + s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bar(L::bVFull + s), 1);
      mbar_init(bar(L::bVEmpty + s), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar(L::bSFull + b), 1);
      mbar_init(bar(L::bPFull + b), kSoftmaxWarps / 2);
      mbar_init(bar(L::bRsFull + b), 1);
      mbar_init(bar(L::bLFree + b), kSoftmaxWarps / 2);
      mbar_init(bar(L::bOReady + b), 1);
    }
    mbar_init(bar(L::bOFinal), 1);
    mbar_init(bar(L::bDrain), 1);
    if constexpr (L::kTwoIssuers) mbar_init(bar(L::bDrainPv), 1);
    mbar_init(bar(L::bMReady + 0), kSoftmaxWarps / 2);
    mbar_init(bar(L::bMReady + 1), kSoftmaxWarps / 2);
    mbar_init(bar(L::bQFree), 1);
    mbar_init(bar(L::bOFree), kSoftmaxWarps);
    mbar_init(bar(L::bDecided), kSoftmaxWarps / 2);
    mbar_init(bar(L::bStaged), kSoftmaxWarps);
    mbar_init(bar(L::bStageFree), 1);
    mbar_init(bar(L::bListReady), 1);
    misc[1] = 0;
    misc[2] = 0;
    misc[3] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    mbar_arrive_expect_tx(bar(L::bQFull), L::kTile);
    for (int a = 0; a < L::kAtoms; ++a)
      tma_load_3d(sb + L::kQ + a * 16384, &p.tm_q, bar(L::bQFull), a * L::kAtomCols, m0, bh);
    k_pre = min(SK, n_kv);
    for (int jj = 0; jj < k_pre; ++jj) {
      mbar_arrive_expect_tx(bar(L::bKFull + jj), L::kTile);
      for (int a = 0; a < L::kAtoms; ++a)
        tma_load_3d(sb + L::kK + jj * L::kTile + a * 16384, &p.tm_k, bar(L::bKFull + jj),
                    a * L::kAtomCols, kv_begin + jj * kBlockN, bh);
    }
  }
  if constexpr (kZT) {
    // zero bias tiles (12 KB, a bias of 0 for the first three S tiles) and the
    // ones tile (4 KB of bf16 1.0) right after them
    for (int i = threadIdx.x; i < 1024; i += kNumThreads) {
      const uint32_t w = i >= 768 ? 0x3F803F80u : 0u;
      st_shared_v4u(sb + L::kZBias + 16 * i, w, w, w, w);
    }
    if (threadIdx.x < 3) reinterpret_cast<volatile float*>(misc + 4)[threadIdx.x] = 0.f;
    fence_async_shared();
  }
  if (threadIdx.x < 256) {  // the ones tile used as B of the row-sum MMA
    // 1.0 in bf16 (0x3F80), fp16 (0x3C00) or e4m3 (0x38)
    const uint32_t one = kE4M3 ? 0x38383838u : (kDt == kDtF16 ? 0x3C003C00u : 0x3F803F80u);
    reinterpret_cast<uint2*>(smem + L::kOnes)[threadIdx.x] = make_uint2(one, one);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sb + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (threadIdx.x == 0 && p.trace != nullptr && blockIdx.x == 0)
    p.trace[kTraceWords - 2] = static_cast<unsigned long long>(clock64());

  // Registers: the control warpgroup (TMA, MMA) gives registers back and the
  // softmax warpgroups take them.  Each role runs its own loops so that no
  // code is shared between the two register budgets.  Every role walks the
  // same sequence: the block's items (first passes), then the items its
  // detector deferred (fallback passes); they count items (seq), tiles and
  // passes from the block's start, so ring slots and barrier phases carry on
  // from one item to the next.  Between items the roles meet only through
  // mbarriers: "Q read" (the last S MMA of an item has completed) before the
  // next Q, "O read" before the next first O = P V, "staging read" before the
  // ring that holds the staged O is refilled -- so the next item's Q, first K
  // tiles and first S tiles load and run while the softmax warps finish the
  // last item's epilogue -- and, once, "list ready" before the deferred
  // items.
  const volatile int* deferred = reinterpret_cast<const volatile int*>(smem + L::kDefer);
  if (warp >= kMmaWarp) {
    regs_dec<kCtrlRegs>();
    if (warp == kLoadWarp || warp == kLoadVWarp) {
      // =================== TMA producers ===================
      // warp 9: Q, then K_0, K_1, ... of each item; warp 10: V_0, V_1, ...
      if (lane == 0) {
        const bool is_k = warp == kLoadWarp;
        const int S = is_k ? SK : SV;
        const int full = is_k ? L::bKFull : L::bVFull;
        // with as many V stages as score buffers, "V stage free" and "O +=
        // P V landed" are the same event: one barrier serves both
        const int empty = is_k ? L::bKEmpty : (SV == kSBufs ? L::bOReady : L::bVEmpty);
        const int ring = is_k ? L::kK : L::kV;
        const CUtensorMap* tm = is_k ? &p.tm_k : &p.tm_v;
        // (V producer) the O of the last pass, staged in the V ring by the
        // softmax warps: it is stored from here -- so no softmax warp waits
        // for the store to read its staging -- and the ring stages that hold
        // it refill only once the stores have read them
        struct Pending {
          int m0, bh, v0;
          bool exact;
        } pend{0, 0, 0, false};
        bool has_pend = false;      // a pass whose O is yet to be stored
        bool read_pending = false;  // stores issued whose shared-memory reads are not waited for
        int staged_v0 = 0;          // first V stage of the pass after the stored one
        int stored = 0;             // passes whose staging has been taken
        auto store_staged = [&]() -> bool {
          if (!wait_bounded(bar(L::bStaged), stored & 1, p, abort_flag)) return false;
          ++stored;
          has_pend = false;
          if (*abort_flag) return false;
          // (a fallback pass rewrites a tile stored before: that store must
          // have landed first)
          if (pend.exact) bulk_wait_all();
          const int row_block = p.o_part ? split * BH + pend.bh : pend.bh;
#pragma unroll
          for (int b = 0; b < L::kBoxes; ++b)
            tma_store_3d(&p.tm_o, sb + L::box(b, pend.v0), b * 32, pend.m0, row_block);
          bulk_commit();
          read_pending = true;
          staged_v0 = pend.v0;
          return true;
        };
        // once the stores have read the staging: its stages may refill, and
        // the next pass may stage over it
        auto release_staging = [&]() {
          if (!read_pending) return;
          bulk_wait_read();
          read_pending = false;
          mbar_arrive(bar(L::bStageFree));
        };
        int issued = is_k ? k_pre : 0;  // tiles issued (the first K tiles during set-up)
        int q_issued = 1;               // Q tiles issued (the first during set-up)
        int seq = 0, it_base = 0;
        bool ok = true;
        if (!is_k) tma_prefetch_desc(&p.tm_v);
#pragma unroll 1
        for (int phase = 0; phase < 2 && ok; ++phase) {
          int count = 0;
          if (phase == 1) {
            if (!(ok = wait_bounded(bar(L::bListReady), 0, p, abort_flag))) break;
            count = min(static_cast<int>(misc[2]), kMaxDeferred);
          }
#pragma unroll 1
          for (int k = 0; ok; ++k, ++seq) {
            const int idx = phase == 0 ? fwd_item_at(p, k) : (k < count ? deferred[k] : -1);
            if (idx < 0) break;
            const Item w = item(idx);
            if (is_k && seq > 0) {
              // this item's Q, once every S MMA of the last item has read its Q
              if (!(ok = wait_bounded(bar(L::bQFree), (seq - 1) & 1, p, abort_flag))) break;
              mbar_arrive_expect_tx(bar(L::bQFull), L::kTile);
              for (int a = 0; a < L::kAtoms; ++a)
                tma_load_3d(sb + L::kQ + a * 16384, &p.tm_q, bar(L::bQFull), a * L::kAtomCols,
                            w.m0, w.bh);
              ++q_issued;
            }
            if (!is_k && phase == 0) {
              // into L2 ahead of time: the Q tile and first K tile of this
              // block's next item, or (one block per item) of the block about
              // one wave ahead
              int nxt = fwd_item_at(p, k + 1);
              if (nxt < 0 && k == 0 && p.prefetch_stride > 0 &&
                  static_cast<int>(blockIdx.x) + p.prefetch_stride < p.n_items)
                nxt = static_cast<int>(blockIdx.x) + p.prefetch_stride;
              if (nxt >= 0) {
                const Item n = item(nxt);
                for (int a = 0; a < L::kAtoms; ++a) {
                  tma_prefetch_l2_3d(&p.tm_q, a * L::kAtomCols, n.m0, n.bh);
                  tma_prefetch_l2_3d(&p.tm_k, a * L::kAtomCols, kv_begin, n.bh);
                }
              }
            }
            for (int jj = issued - it_base; jj < w.n_kv; ++jj) {
              const int it = it_base + jj, st = it % S;
              if (!is_k) {
                // the last pass's O is stored before its stages are reused
                // (after this pass's first V tile when the staging skips it)
                if (has_pend && (jj > 0 || !L::kStageSkipsFirst) && !(ok = store_staged())) break;
                if (read_pending && L::holds_o(st, staged_v0)) release_staging();
              }
              if (is_k && L::kKFreeOnS) {
                // K stage st is free once S_{it - S} has completed
                if (it >= S && !(ok = wait_bounded(bar(L::bSFull + (it - S) % kSBufs),
                                                   ((it - S) / kSBufs) & 1, p, abort_flag)))
                  break;
              } else if (!(ok = wait_bounded(bar(empty + st), ((it / S) & 1) ^ 1, p, abort_flag))) {
                break;
              }
              mbar_arrive_expect_tx(bar(full + st), L::kTile);
              for (int a = 0; a < L::kAtoms; ++a)
                tma_load_3d(sb + ring + st * L::kTile + a * 16384, tm, bar(full + st),
                            a * L::kAtomCols, kv_begin + jj * kBlockN, w.bh);
              issued = it + 1;
            }
            if (!ok) break;
            if (!is_k) {
              if (has_pend && !(ok = store_staged())) break;
              release_staging();
              pend = {w.m0, w.bh, (it_base + w.n_kv) % SV, phase == 1};
              has_pend = true;
            }
            it_base += w.n_kv;
          }
        }
        // the block's last pass; every store must have completed before exit
        if (!is_k && ok && has_pend) store_staged();
        if (!is_k) bulk_wait_all();
        if (*abort_flag) {
          // let every copy already issued land before the block can exit
          if (is_k) wait_drain(bar(L::bQFull), (q_issued - 1) & 1);
          for (int g = max(0, issued - S); g < issued; ++g)
            wait_drain(bar(full + g % S), (g / S) & 1);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp || (kTwoIssuers && warp == kPvWarp)) {
      if constexpr (kTwoIssuers) {
      // =================== MMA issuers ===================
      // Warp 8 issues S_it = Q K_it^T into buffer it % 3 once O += P_{it-3} V
      // (the buffer's last reader) has completed; warp 11 issues O += P_it V
      // once P~_it and V_it are there.  Two issuers, so that neither waits
      // behind the other's queue: the P V MMAs go in as soon as P~ is ready.
      // Each warp issues with one elected lane; each commit tracks only its
      // own warp's MMAs.
      const bool pv_role = warp == kPvWarp;
      constexpr uint32_t kFmt = kDt == kDtBf16 ? 1u : 0u;
      constexpr uint32_t idesc_s = idesc_f32acc<kFmt>(kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = idesc_f32acc<kFmt>(kBlockM, D, true);
      constexpr uint32_t idesc_rs = idesc_f32acc<kFmt>(kBlockM, 16, false);
      const uint64_t ones_desc = sdesc_sw128(sb + L::kOnes, 16, 1024);
      const uint64_t q_desc = sdesc_sw128(sb + L::kQ, 16, 1024);
      const uint64_t k_desc = sdesc_sw128(sb + L::kK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(sb + L::kV, 16384, 1024);
      const uint64_t zbias_desc = sdesc_plain(sb + L::kZBias, 128, 256);
      const uint64_t zones_desc = sdesc_plain(sb + L::kZOnes, 128, 256);
      struct Ring {  // a slot of an n-deep ring and the parity of its phase
        int slot = 0;
        uint32_t phase = 0;
        __device__ __forceinline__ void next(int n) {
          if (++slot == n) {
            slot = 0;
            phase ^= 1u;
          }
        }
      };
      auto issue_s = [&](int buf, int kst) {
        const uint64_t kd = k_desc + static_cast<uint32_t>((kst * L::kTile) >> 4);
        const uint32_t d_t = tmem + buf * kBlockN;
#pragma unroll
        for (int g = 0; g < D / L::kMmaK / 4; ++g)
          mma_ss_x4<kE4M3, 2>(d_t, q_desc + g * 1024, kd + g * 1024, idesc_s, g > 0);
        if constexpr (kZT)
          mma_ss<false>(d_t, zbias_desc + static_cast<uint32_t>((buf * 4096) >> 4), zones_desc,
                        idesc_s, 1u);
      };
      auto issue_pv = [&](int buf, int vst, bool acc) {
        const uint64_t vd = v_desc + static_cast<uint32_t>((vst * L::kTile) >> 4);
#pragma unroll
        for (int g = 0; g < kBlockN / L::kMmaK / 4; ++g)
          mma_ts_x4<kE4M3, 8, (L::kPvStep >> 4)>(
              tmem + kOCol, tmem + buf * kBlockN + g * 32,
              vd + static_cast<uint32_t>(g * 4 * (L::kPvStep >> 4)), idesc_pv, acc || g > 0);
      };
      auto issue_rs = [&](int buf) {
#pragma unroll
        for (int g = 0; g < kBlockN / L::kMmaK; ++g)
          mma_ts<kE4M3>(tmem + buf * kBlockN + 64, tmem + buf * kBlockN + g * 8, ones_desc,
                        idesc_rs, g > 0);
      };
      auto wait_all = [&](uint32_t b, uint32_t par) -> bool {
        return __all_sync(0xffffffffu, wait_bounded(b, par, p, abort_flag));
      };
      Ring buf_r, k_r, v_r;   // score buffer, K stage (S role), V stage (P V role)
      Ring free_r;            // (S role) the buffer's previous tile, three back
      int s_total = 0;        // (S role) S tiles issued so far
      bool ok = true;
      int seq = 0;
#pragma unroll 1
      for (int phase = 0; phase < 2 && ok; ++phase) {
        int count = 0;
        if (phase == 1) {
          if (!(ok = wait_all(bar(L::bListReady), 0))) break;
          count = min(static_cast<int>(misc[2]), kMaxDeferred);
        }
#pragma unroll 1
        for (int k = 0; ok; ++k, ++seq) {
          const int idx = phase == 0 ? fwd_item_at(p, k) : (k < count ? deferred[k] : -1);
          if (idx < 0) break;
          const int n_kv_t = item(idx).n_kv;
          const bool trc = seq == 0 && p.trace != nullptr && blockIdx.x == 0;
          if (!pv_role) {
            if (!(ok = wait_all(bar(L::bQFull), seq & 1))) break;
            // (kZT) the bias tiles are zero again once the last item's
            // detector has run
            if (kZT && seq > 0 && !(ok = wait_all(bar(L::bDecided), (seq - 1) & 1))) break;
#pragma unroll 1
            for (int jj = 0; jj < n_kv_t; ++jj) {
              if (s_total >= kSBufs) {
                // O += P~ V of the buffer's last tile has read it (and, with
                // the tensor row sum, its row sum has been read)
                if (!(ok = wait_all(bar(L::bOReady + free_r.slot), free_r.phase))) break;
                if (kLTensor &&
                    !(ok = wait_all(bar(L::bLFree + free_r.slot), free_r.phase))) break;
                free_r.next(kSBufs);
              }
              if (!(ok = wait_all(bar(L::bKFull + k_r.slot), k_r.phase))) break;
              tc_fence_after();
              issue_s(buf_r.slot, k_r.slot);
              mma_commit(bar(L::bSFull + buf_r.slot));
              if constexpr (!L::kKFreeOnS) mma_commit(bar(L::bKEmpty + k_r.slot));
              if (trc && lane == 0 && jj >= kSBufs) trace_at(p, 4, 0, jj - kSBufs);
              buf_r.next(kSBufs);
              k_r.next(SK);
              ++s_total;
            }
            if (!ok) break;
            // every S MMA of the item issued: Q is free once they have completed
            mma_commit(bar(L::bQFree));
          } else {
#pragma unroll 1
            for (int j = 0; j < n_kv_t; ++j) {
              const bool v_ok = mbar_test_wait(bar(L::bVFull + v_r.slot), v_r.phase);
              const bool p_ok = mbar_test_wait(bar(L::bPFull + buf_r.slot), buf_r.phase);
              if (__ballot_sync(0xffffffffu, v_ok && p_ok) != 0xffffffffu) {
                if (!(ok = wait_all(bar(L::bVFull + v_r.slot), v_r.phase))) break;
                if (!(ok = wait_all(bar(L::bPFull + buf_r.slot), buf_r.phase))) break;
              }
              // the first O = P V of an item overwrites O: the last epilogue
              // must have read it
              if (j == 0 && seq > 0 && !(ok = wait_all(bar(L::bOFree), (seq - 1) & 1))) break;
              if (trc && lane == 0) trace_at(p, 3, 0, j);
              tc_fence_after();
              if (kLTensor) {
                issue_rs(buf_r.slot);
                mma_commit(bar(L::bRsFull + buf_r.slot));
              }
              issue_pv(buf_r.slot, v_r.slot, j > 0);
              if (SV != kSBufs) mma_commit(bar(L::bVEmpty + v_r.slot));
              mma_commit(bar(L::bOReady + buf_r.slot));
              buf_r.next(kSBufs);
              v_r.next(SV);
            }
            if (!ok) break;
            mma_commit(bar(L::bOFinal));
          }
        }
      }
      if (ok) {
        // the last item's "Q read" is waited for by no one else
        if (!pv_role && seq > 0) wait_drain(bar(L::bQFree), (seq - 1) & 1);
      } else {
        // every MMA this warp issued must finish before TMEM can be released
        const uint32_t db = bar(pv_role ? L::bDrainPv : L::bDrain);
        mma_commit(db);
        wait_drain(db, 0);
      }
      __syncwarp();
      } else {
      // =================== MMA issuer ===================
      // The whole warp runs this code with warp-uniform values; one elected
      // lane issues each MMA and commit.
      // A/B format codes: bf16 1; fp16 0 (kind::f16); e4m3 0 (kind::f8f6f4)
      constexpr uint32_t kFmt = kDt == kDtBf16 ? 1u : 0u;
      constexpr uint32_t idesc_s = idesc_f32acc<kFmt>(kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = idesc_f32acc<kFmt>(kBlockM, D, true);
      constexpr uint32_t idesc_rs = idesc_f32acc<kFmt>(kBlockM, 16, false);
      const uint64_t ones_desc = sdesc_sw128(sb + L::kOnes, 16, 1024);
      // S_it = Q K^T into score buffer it % 3
      // Descriptors of the first K step of each operand; a step further
      // only adds its byte offset >> 4 to the start-address field (shared
      // memory stays below 256 KB, so the field never overflows).
      const uint64_t q_desc = sdesc_sw128(sb + L::kQ, 16, 1024);
      const uint64_t k_desc = sdesc_sw128(sb + L::kK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(sb + L::kV, 16384, 1024);
      // (kZT) bias and ones tiles: 16-byte core matrices 128 B apart along
      // K, 8-row groups 256 B apart; every entry of a tile is equal, so
      // only the tile's 4 KB extent matters
      const uint64_t zbias_desc = sdesc_plain(sb + L::kZBias, 128, 256);
      const uint64_t zones_desc = sdesc_plain(sb + L::kZOnes, 128, 256);
      // The tensor pipe queues only a handful of MMAs, so this warp's own
      // instruction count between MMA groups decides whether the pipe runs
      // dry: ring positions advance by counters (no divisions), the MMAs of
      // a GEMM go out four per elected issue, and the trace test is hoisted
      // out of the tile loop.
      struct Ring {  // a slot of an n-deep ring and the parity of its phase
        int slot = 0;
        uint32_t phase = 0;
        __device__ __forceinline__ void next(int n) {
          if (++slot == n) {
            slot = 0;
            phase ^= 1u;
          }
        }
      };
      Ring s_buf, s_k;  // score buffer and K stage of the next S MMA
      Ring p_buf, p_v;  // score buffer (P~) and V stage of the next P V MMA
      int s_count = 0;  // S tiles queued so far by this block
      // S = Q K^T: D / kMmaK K steps, four per 128-byte slab of the rows
      auto issue_s = [&](int buf, int kst) {
        const uint64_t kd = k_desc + static_cast<uint32_t>((kst * L::kTile) >> 4);
        const uint32_t d_t = tmem + buf * kBlockN;
#pragma unroll
        for (int g = 0; g < D / L::kMmaK / 4; ++g)
          mma_ss_x4<kE4M3, 2>(d_t, q_desc + g * 1024, kd + g * 1024, idesc_s, g > 0);
        if constexpr (kZT)
          mma_ss<false>(d_t, zbias_desc + static_cast<uint32_t>((buf * 4096) >> 4), zones_desc,
                        idesc_s, 1u);
      };
      // O (+)= P V: A = P~ in TMEM (8 columns per K step), B = V (MN-major)
      auto issue_pv = [&](int buf, int vst, bool acc) {
        const uint64_t vd = v_desc + static_cast<uint32_t>((vst * L::kTile) >> 4);
#pragma unroll
        for (int g = 0; g < kBlockN / L::kMmaK / 4; ++g)
          mma_ts_x4<kE4M3, 8, (L::kPvStep >> 4)>(
              tmem + kOCol, tmem + buf * kBlockN + g * 32,
              vd + static_cast<uint32_t>(g * 4 * (L::kPvStep >> 4)), idesc_pv, acc || g > 0);
      };
      auto issue_rs = [&](int buf) {
#pragma unroll
        for (int g = 0; g < kBlockN / L::kMmaK; ++g)
          mma_ts<kE4M3>(tmem + buf * kBlockN + 64, tmem + buf * kBlockN + g * 8, ones_desc,
                        idesc_rs, g > 0);
      };
      auto queue_s = [&](bool k_ready) -> bool {
        // a score buffer is written again only once the tensor row sum
        // that shared it has been read
        if (kLTensor && s_count >= kSBufs &&
            !__all_sync(0xffffffffu, wait_bounded(bar(L::bLFree + s_buf.slot), s_buf.phase ^ 1u,
                                                  p, abort_flag)))
          return false;
        if (!k_ready &&
            !__all_sync(0xffffffffu,
                        wait_bounded(bar(L::bKFull + s_k.slot), s_k.phase, p, abort_flag)))
          return false;
        tc_fence_after();
        issue_s(s_buf.slot, s_k.slot);
        // (with at most three K stages "S done" also frees the K stage)
        mma_commit(bar(L::bSFull + s_buf.slot));
        if constexpr (!L::kKFreeOnS) mma_commit(bar(L::bKEmpty + s_k.slot));
        s_buf.next(kSBufs);
        s_k.next(SK);
        ++s_count;
        return true;
      };

      bool ok = true;
      int seq = 0;
#pragma unroll 1
      for (int phase = 0; phase < 2 && ok; ++phase) {
        int count = 0;
        if (phase == 1) {
          if (!(ok = __all_sync(0xffffffffu,
                                wait_bounded(bar(L::bListReady), 0, p, abort_flag))))
            break;
          count = min(static_cast<int>(misc[2]), kMaxDeferred);
        }
#pragma unroll 1
        for (int k = 0; ok; ++k, ++seq) {
          const int idx = phase == 0 ? fwd_item_at(p, k) : (k < count ? deferred[k] : -1);
          if (idx < 0) break;
          const int n_kv_t = item(idx).n_kv;
          const bool trc = seq == 0 && p.trace != nullptr && blockIdx.x == 0;
          if (!(ok = __all_sync(0xffffffffu,
                                wait_bounded(bar(L::bQFull), seq & 1, p, abort_flag))))
            break;
          // (kZT) the bias tiles are zero again once the last item's detector
          // has run
          if (kZT && seq > 0 &&
              !(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bDecided), (seq - 1) & 1, p,
                                                          abort_flag))))
            break;
          for (int jj = 0; ok && jj < min(kSBufs, n_kv_t); ++jj) ok = queue_s(false);
          // every S MMA of the item issued: Q is free once they have completed
          if (ok && n_kv_t <= kSBufs) mma_commit(bar(L::bQFree));
#pragma unroll 1
          for (int j = 0; ok && j < n_kv_t; ++j) {
            const int buf = p_buf.slot;
            const bool more_s = j + kSBufs < n_kv_t;
            // V_j, P~_j and (when S_{j+3} follows) K_{j+3}: three independent
            // probes and one vote when all are there, the usual case, so that
            // nothing but a commit separates O += P_j V from S_{j+3}; the
            // bounded waits otherwise
            const bool v_ok = mbar_test_wait(bar(L::bVFull + p_v.slot), p_v.phase);
            const bool p_ok = mbar_test_wait(bar(L::bPFull + buf), p_buf.phase);
            const bool k_ok = !more_s || mbar_test_wait(bar(L::bKFull + s_k.slot), s_k.phase);
            const uint32_t all3 = __ballot_sync(0xffffffffu, v_ok && p_ok && k_ok);
            const bool k_ready = all3 == 0xffffffffu && more_s;
            if (all3 != 0xffffffffu) {
              if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bVFull + p_v.slot),
                                                              p_v.phase, p, abort_flag))))
                break;
              if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bPFull + buf),
                                                              p_buf.phase, p, abort_flag))))
                break;
            }
            // the first O = P V of an item overwrites O: the last epilogue
            // must have read it
            if (j == 0 && seq > 0 &&
                !(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bOFree), (seq - 1) & 1, p,
                                                            abort_flag))))
              break;
            if (trc && lane == 0) trace_at(p, 3, 0, j);
            tc_fence_after();
            if (kLTensor) {
              issue_rs(buf);
              mma_commit(bar(L::bRsFull + buf));
            }
            issue_pv(buf, p_v.slot, j > 0);
            if (SV != kSBufs) mma_commit(bar(L::bVEmpty + p_v.slot));
            mma_commit(bar(L::bOReady + buf));
            p_buf.next(kSBufs);
            p_v.next(SV);
            if (more_s) {
              if (!(ok = queue_s(k_ready))) break;
              if (j + kSBufs == n_kv_t - 1) mma_commit(bar(L::bQFree));
            }
            if (trc && lane == 0) trace_at(p, 4, 0, j);
          }
          if (!ok) break;
          mma_commit(bar(L::bOFinal));
        }
      }
      if (ok) {
        // the last item's "Q read" is waited for by no one else
        if (seq > 0) wait_drain(bar(L::bQFree), (seq - 1) & 1);
      } else {
        // every MMA issued so far must finish before TMEM can be released
        mma_commit(bar(L::bDrain));
        wait_drain(bar(L::bDrain), 0);
      }
      __syncwarp();
      }
    }
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  } else {
    regs_inc<kSoftmaxRegs>();
    // =================== softmax warps ===================
    int seq = 0, it_base = 0;
    int mr[2] = {0, 0};  // tiles each set has taken so far
    const int other = (warp >> 2) ^ 1;
    bool stop = false;
#pragma unroll 1
    for (int k = 0; !stop; ++k, ++seq) {
      const int idx = fwd_item_at(p, k);
      if (idx < 0) break;
      const Item w = item(idx);
      stop = softmax_role<D, kX, kLTensor, kDt, kZT, false>(
          p, smem, sb, tmem, misc, warp, lane, idx, seq, w.m0, w.bh, w.n_kv, it_base, split,
          kv_begin, kv_end, kv_off, /*epi=*/seq, mr[other], /*tr=*/seq == 0);
      it_base += w.n_kv;
      mr[0] += (w.n_kv + 1) / 2;
      mr[1] += w.n_kv / 2;
    }
    if constexpr (kTensor) {
      // The fallback pass of each deferred item (one-row tiles, X = 1: every
      // row's own maximum rounded up to a whole binade, so no row can
      // underflow -- the vector fallback of the page's all-underflow
      // discussion, on the same code path).  Set 0 appended to the list
      // before the last barrier of the loop above.
      if (!stop) {
        if (warp == 0 && lane == 0) mbar_arrive(bar(L::bListReady));
        const int count = min(static_cast<int>(misc[2]), kMaxDeferred);
#pragma unroll 1
        for (int k = 0; k < count && !stop; ++k, ++seq) {
          const int idx = deferred[k];
          const Item w = item(idx);
          stop = softmax_role<D, kX, kLTensor, kDt, kZT, true>(
              p, smem, sb, tmem, misc, warp, lane, idx, seq, w.m0, w.bh, w.n_kv, it_base, split,
              kv_begin, kv_end, kv_off, /*epi=*/seq, mr[other], /*tr=*/false);
          it_base += w.n_kv;
          mr[0] += (w.n_kv + 1) / 2;
          mr[1] += w.n_kv / 2;
        }
      }
    } else {
      if (!stop && warp == 0 && lane == 0) mbar_arrive(bar(L::bListReady));
    }
    __syncthreads();
  }
}

}  // namespace fat
