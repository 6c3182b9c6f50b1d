// Fused attention forward pass for sm_103a with the tensorized online softmax
// of "FlashAttention-T: Towards Fully Tensorized Attention by Exploiting
// Tensor-Vector Parallelism" (papercache.org summary, section A2, Algorithm 1)
// and its vector-softmax ablation (the FA2 arm of the page's Fig. 10).
//
// One CTA computes 256 query rows of one (batch, head) as two 128-row tiles
// (t = 0, 1) that ping-pong on the tensor pipe, the fused flow of the page's
// section A3 / Fig. 2 (one output row block per worker, S and P on chip):
//
//   warp 9      TMA producer: Q0, Q1 once; K_j, V_j through an mbarrier ring.
//   warp 8      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM,
//               O_t += P_t V_j from TMEM, and (tensorized) l_t = P_t 1.
//   warps 0-7   softmax, warpgroup t owns tile t, thread i owns row i
//               (TMEM lane i): row max, X-row tile max, O rescale, P = exp2(Z).
//
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+D), O_1 [256+D, 256+2D).  P_t is written as packed bf16 over
// S_t columns [0,64); the tensorized row sum lands in S_t column 64.
#pragma once

#include <cuda.h>

#include "sm103_ptx.cuh"

namespace fat {

constexpr int kBlockM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;  // keys per K/V tile
constexpr int kRowsPerCta = 2 * kBlockM;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;   // warps 10, 11 complete the third warpgroup
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
// Of the 16 element pairs in each 32-column chunk of a row, this many take
// 2^z from the FMA-pipe polynomial (f2_exp2_poly) and the rest from MUFU ex2:
// one MUFU ex2 costs a warp 8 issue cycles of its pipe (16 results per SM
// per cycle), the polynomial about 5 single-cycle instructions per element.
constexpr int kPolyPairs = 0;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;


struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  float* o;
  float* lse;
  int* fallback_rows;
  int B, H;
  int Nq, Nk;              // query rows, keys per (b, h)
  int causal;              // key j allowed for query i iff j <= i + Nk - Nq
  int X;
  int n_mblocks;           // ceil(Nq / 256)
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

// Phase trace of CTA 0, SM clock (clock64) stamps, pass 0 only:
//   word (e * 2 + t) * kTraceIters + j for event e, tile t, K/V tile j:
//   e = 0 softmax got S_j, 1 softmax has m_hat, 2 softmax publishes P_j,
//       3 MMA issuer sees P_j, 4 MMA issuer has queued O += P_j V, S_{j+1};
//   word kTraceWords - 2 / - 1: kernel start / softmax epilogue done.
constexpr int kTraceIters = 128;
constexpr int kTraceWords = 5 * 2 * kTraceIters + 2;

__device__ __forceinline__ void trace_mark(const FwdParams& p, int e, int t, int j, int pass) {
  if (p.trace != nullptr && blockIdx.x == 0 && pass == 0 && j < kTraceIters)
    p.trace[(e * 2 + t) * kTraceIters + j] = static_cast<unsigned long long>(clock64());
}

template <int D, bool kE4M3 = false>
struct Smem {
  static constexpr int kElt = kE4M3 ? 1 : 2;          // bytes per input element
  static constexpr int kStages = (D * kElt == 256) ? 2 : 4;
  static constexpr int kTile = kBlockM * D * kElt;    // bytes of one 128 x D tile
  static constexpr int kAtoms = D * kElt / 128;       // 128-byte-wide column slabs per tile
  static constexpr int kAtomCols = 128 / kElt;        // elements per slab row
  static constexpr int kMmaK = 32 / kElt;             // K of one MMA (bf16 16, e4m3 32)
  static constexpr int kPvStep = kMmaK * 128;         // bytes of V rows per PV K step
  static_assert(kAtoms >= 1, "rows must span at least one 128-byte slab");
  static constexpr int kQ = 0;                   // Q_t at kQ + t * kTile
  static constexpr int kK = 2 * kTile;           // K ring
  static constexpr int kV = kK + kStages * kTile;  // V ring
  static constexpr int kOnes = kV + kStages * kTile;  // 16 rows x 128 B of ones (2 KB)
  static constexpr int kBars = kOnes + 2048;
  // barrier slots
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;
  static constexpr int bKEmpty = bKFull + kStages;
  static constexpr int bVFull = bKEmpty + kStages;
  static constexpr int bVEmpty = bVFull + kStages;
  static constexpr int bSFull = bVEmpty + kStages;  // [2]
  static constexpr int bPFull = bSFull + 2;         // [2]
  static constexpr int bRsFull = bPFull + 2;        // [2]
  static constexpr int bLFree = bRsFull + 2;        // [2]
  static constexpr int bRed = bLFree + 2;           // [2] tile-max exchange
  static constexpr int bOFinal = bRed + 2;
  static constexpr int bDrain = bOFinal + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kRed = kBars + 8 * kNumBars;  // float [2 tiles][2 parity][4 warps]
  static constexpr int kMisc = kRed + 64;  // u32: tmem base, abort, redo, -, pv scale[2]
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;       // slack for 1024-byte alignment
  static_assert(kK % 1024 == 0 && kV % 1024 == 0 && kOnes % 1024 == 0, "tiles 1 KB aligned");
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const FwdParams& p,
                                             volatile uint32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
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

// ---------------------------------------------------------------------------
// softmax warpgroups: warpgroup t owns query tile t; thread i owns row i
// (TMEM lane i).
//   kX > 0   tensorized online softmax with the surrogate maximum over kX-row
//            tiles (X is a compile-time constant so no runtime branching sits
//            in the hot loop); `exact` (the fallback pass) uses each row's own
//            maximum instead, rounded up to a whole binade.
//   kX == 0  the vector-softmax ablation: exact per-row maximum.
// ---------------------------------------------------------------------------
template <int D, int kX, bool kLTensor, bool kE4M3>
__device__ __forceinline__ void softmax_role(const FwdParams& p, uint8_t* smem, uint32_t sb,
                                             uint32_t tmem, volatile uint32_t* misc, int warp,
                                             int lane, int m0, int bh, int n_kv, int it0,
                                             int pass, bool exact, int split, int kv_begin,
                                             int kv_end, int kv_off) {
  using L = Smem<D, kE4M3>;
  constexpr bool kTensor = kX > 0;
  constexpr bool kGroup = kX > 32;  // tile maximum spans several warps
  constexpr bool kMmaScale = kX == 128 && !kE4M3;
  // e4m3 P~ is formed as 2^(Z + kKappa) <= 2^8 < 448 so that its largest
  // terms use the format's range; the factor cancels in O / l and is taken
  // off LSE.
  constexpr float kKappa = kE4M3 ? 8.f : 0.f;
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8 * i; };
  const int t = warp >> 2;       // tile
  const int wq = warp & 3;       // quarter of the tile (TMEM lanes 32 wq ..)
  const int r = wq * 32 + lane;  // row within the tile
  const int row_g = m0 + t * kBlockM + r;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t s_taddr = tmem + lane_base + t * kBlockN;
  const uint32_t o_taddr = tmem + lane_base + 2 * kBlockN + t * D;
  const float c = p.c;
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  const uint32_t gbar_id = 1 + 4 * t + (kX == 64 ? (wq >> 1) : 0);
  constexpr uint32_t kGbarN = kX == 64 ? 64 : 128;
  const bool mma_scale = kMmaScale && !exact;

  float M = -INFINITY;      // offset of the exponent, binades (exact row max * c in vec mode)
  float m_row = -INFINITY;  // exact running row maximum, raw logits
  float l = 0.f;            // running row sum
  float delta = 0.f;        // tensorized row sum: rounding of each tile's dominant term
  int kscale_prev = 0;      // last value written to this tile's PV scale word
  bool dead = false;        // a bounded wait of this warp (or of its X-row group) ran out
  int j = 0;
  for (; j < n_kv; ++j) {
    const int it = it0 + j;
    const uint32_t par = it & 1;
    dead = !__all_sync(0xffffffffu, wait_bounded(bar(L::bSFull + t), par, p, abort_flag));
    if (wq == 0 && lane == 0) trace_mark(p, 0, t, j, pass);
    // X = 128 (bf16), from the second K/V tile on: steps 4-6 start from the
    // previous tile's surrogate maximum, and step 1 (the maximum over the four
    // warps of the tile) is settled afterwards.  Usually no warp raises the
    // maximum, which one OR over the group barrier establishes; a tile that
    // does raise it has its P~ scaled by the exact power of two
    // 2^(m_old - m_new).  The P~ that reaches the MMA is the same as when the
    // maximum is known first.  M is uniform over the 128-row tile, and so is
    // this choice.
    const bool spec = kMmaScale && !exact && M != -INFINITY;
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
      m_row = fmaxf(m_row, rowmax);
    }
    // Algorithm 1 step 1: maximum of the row maxima over the X-row tile
    float tmax = rowmax;
    if constexpr (kX == 16) {
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
    } else if constexpr (kX >= 32) {
      tmax = warp_max(rowmax);
    }
    // X = 64 / 128: the warps of the X-row group combine their maxima through
    // shared memory.  Every warp of the group joins the same sequence of group
    // barriers, aborted or not (one per K/V tile; two on a speculative tile
    // that raises the maximum or aborts; see the drain loop below), and the OR
    // spreads an abort to the whole group.
    float* slot = red + (t * 2 + par) * 4;
    auto group_max = [&]() {
      if constexpr (kGroup) {
        dead = named_bar_or(gbar_id, kGbarN, dead);
        if (!dead) {
          if constexpr (kX == 64) {
            tmax = fmaxf(slot[wq & 2], slot[(wq & 2) + 1]);
          } else {
            tmax = fmaxf(fmaxf(slot[0], slot[1]), fmaxf(slot[2], slot[3]));
          }
        }
      }
    };
    if (!spec) {
      if constexpr (kGroup) {
        if (lane == 0) slot[wq] = tmax;
      }
      group_max();
      if (dead) break;
    }

    // The new offset of step 2; the factor of steps 2-3 is exp(m_old - m_new),
    // one exact power of two per X-row tile (exact per-row factor in the
    // vector variant).  With X = 128 the whole 128-row tile shares the factor
    // 2^-k and the tensor pipe applies it inside the next O += P V
    // (scale-input-d); other cases rescale O in TMEM from the vector side.
    auto new_offset = [&]() -> float {
      if constexpr (kTensor) {
        // the surrogate maximum is kept as a whole number of binades so the
        // rescale factor is an exact power of two; the fallback pass uses
        // one-row tiles (each row's own maximum)
        const float tm = exact ? rowmax : tmax;
        const float Mc = (tm == -INFINITY) ? -INFINITY : ceilf(tm * c);
        return fmaxf(M, Mc);
      } else {
        return (m_row == -INFINITY) ? -INFINITY : m_row * c;
      }
    };
    float M_new = M, alpha = 1.f;
    bool vec_rescale = false;
    auto bookkeeping = [&]() {
      const bool grow = j > 0 && M_new > M;
      alpha = (M_new == -INFINITY) ? 1.f : ex2_approx(M - M_new);
      vec_rescale = grow;
      if constexpr (kMmaScale) {
        int kscale = 0;
        if (mma_scale && grow && M_new - M <= 15.f) {
          kscale = static_cast<int>(M_new - M);
          vec_rescale = false;
        }
        if (wq == 0 && lane == 0) misc[4 + t] = static_cast<uint32_t>(kscale);
        kscale_prev = kscale;
      }
    };
    if (!spec) {
      M_new = new_offset();
      bookkeeping();
      if (j > 0) {
        l *= alpha;
        if (kLTensor) delta *= alpha;
      }
      M = M_new;
      if (wq == 0 && lane == 0) trace_mark(p, 1, t, j, pass);
    }
    const float neg_M = (M == -INFINITY) ? 0.f : -M;

    // steps 4-6: Z = c S - m_hat, P~ = exp2(Z), stored as bf16 (e4m3) over S
    const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(neg_M + kKappa, neg_M + kKappa);
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
        if ((i * kPolyPairs) % 16 < kPolyPairs) {
          // the polynomial leaves a tiny positive value for a masked (-inf)
          // key: zero it in the tiles that have masked keys
          f2_unpack(f2_exp2_poly(z0, z1), pf[2 * i], pf[2 * i + 1]);
          if (limit < kBlockN) {
            if (32 * k + 2 * i >= limit) pf[2 * i] = 0.f;
            if (32 * k + 2 * i + 1 >= limit) pf[2 * i + 1] = 0.f;
          }
        } else {
          pf[2 * i] = ex2_approx(z0);
          pf[2 * i + 1] = ex2_approx(z1);
        }
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
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(pf[2 * i], pf[2 * i + 1]);
        tmem_st16(s_taddr + 16 * k, pk);
      }
    }
    float lt_vec;  // this tile's row sum (vector row sum only)
    {
      float r0, r1;
      f2_unpack(f2_add(acc2[0], acc2[1]), r0, r1);
      lt_vec = r0 + r1;
    }
    if (spec) {
      // step 1 completes: does any warp of the tile raise the maximum?
      const float Mc_w = (tmax == -INFINITY) ? -INFINITY : ceilf(tmax * c);
      const bool any = named_bar_or(gbar_id, kGbarN, dead || Mc_w > M);
      if (any) {
        // rare: exchange the raised maxima (or learn of an abort)
        if (lane == 0) slot[wq] = Mc_w;
        dead = named_bar_or(gbar_id, kGbarN, dead);
        if (dead) break;
        M_new = fmaxf(M, fmaxf(fmaxf(slot[0], slot[1]), fmaxf(slot[2], slot[3])));
        // M_new > M here: P~ was formed with the old offset.  Multiply it
        // (and its row sum) by 2^(m_old - m_new), exact in bf16; O takes the
        // same factor in the PV MMA (at most 15 binades) or from the vector
        // side.  A jump above 100 binades can only come from logits that far
        // apart; the block is then redone with per-row maxima (the fallback
        // pass).
        const int kb = min(static_cast<int>(M_new - M), 126);  // M, M_new whole binades
        alpha = __uint_as_float(static_cast<uint32_t>(127 - kb) << 23);  // 2^-kb
        vec_rescale = kb > 15;
        const int kscale = vec_rescale ? 0 : kb;
        if (wq == 0 && lane == 0) {
          misc[4 + t] = static_cast<uint32_t>(kscale);
          if (kb > 100) atomicOr(const_cast<uint32_t*>(misc + 2), 1u);
        }
        kscale_prev = kscale;
        const uint32_t a2 = pack_bf16x2(alpha, alpha);
        tmem_wait_st();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pv[32];
          tmem_ld32(s_taddr + 32 * h, pv);
          tmem_wait_ld(pv);
#pragma unroll
          for (int i = 0; i < 32; ++i) pv[i] = bf16x2_mul(pv[i], a2);
          tmem_st32(s_taddr + 32 * h, pv);
        }
        lt_vec *= alpha;
        l *= alpha;
        if (kLTensor) delta *= alpha;
        M = M_new;
      } else if (kscale_prev != 0) {
        // the previous tile's PV scale is spent
        if (wq == 0 && lane == 0) misc[4 + t] = 0u;
        kscale_prev = 0;
      }
      if (wq == 0 && lane == 0) trace_mark(p, 1, t, j, pass);
    }
    const float neg_Mn = (M == -INFINITY) ? 0.f : -M;
    // steps 2-3 on the vector side: O <- alpha O in TMEM.  PV_{j-1} has
    // completed (issued before S_j, whose completion was awaited) and PV_j
    // waits for this warpgroup's P-full signal below.
    if (__any_sync(0xffffffffu, vec_rescale)) {
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
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (wq == 0 && lane == 0) trace_mark(p, 2, t, j, pass);
    if (lane == 0) mbar_arrive(bar(L::bPFull + t));

    if constexpr (kLTensor) {
      // step 7 on the tensor pipe (P~ times ones, S column 64); the LSE also
      // gets back the rounding of the tile's dominant term
      if (rowmax != -INFINITY) {
        const float pm = ex2_approx(fmaf(rowmax, c, neg_Mn + kKappa));
        delta += pm - (kE4M3 ? e4m3_round(pm) : bf16_round(pm));
      }
      dead = !__all_sync(0xffffffffu, wait_bounded(bar(L::bRsFull + t), par, p, abort_flag));
      if (dead) break;
      tc_fence_after();
      uint32_t lt;
      tmem_ld1(s_taddr + 64, lt);
      tmem_wait_ld1(lt);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bLFree + t));
      l += __uint_as_float(lt);
    } else {
      l += lt_vec;
    }
  }
  if constexpr (kGroup) {
    // an aborted warp left the loop at K/V tile j after joining the group
    // barriers of tiles 0..j; it joins the remaining ones so the other warps
    // of the group are never left waiting there
    if (dead) {
      const bool spec = kMmaScale && !exact && M != -INFINITY;
      for (++j; j < n_kv; ++j) {
        named_bar_or(gbar_id, kGbarN, true);
        if (spec) named_bar_or(gbar_id, kGbarN, true);
      }
    }
  }

  bool ok = !dead;
  if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bOFinal), pass & 1, p, abort_flag));
  if (ok) {
    tc_fence_after();
    // detector for the all-underflow case: surrogate far above the exact
    // maximum, or nothing left of the row sum
    if (kTensor && pass == 0) {
      // (a row with no key in this split's range is empty, not flagged)
      const bool flagged = row_g < p.Nq && m_row != -INFINITY &&
                           (!(l > 0.f) || (M - m_row * c) > p.underflow_thresh);
      const uint32_t ball = __ballot_sync(0xffffffffu, flagged);
      if (ball != 0 && lane == 0) {
        atomicOr(const_cast<uint32_t*>(misc + 2), 1u);
        if (p.fallback_rows) atomicAdd(p.fallback_rows, __popc(ball));
      }
    }
    // epilogue: O / l and LSE
    const float inv_l = l > 0.f ? p.v_scale / l : 0.f;  // an empty row gets O = 0
    const size_t out_row = (static_cast<size_t>(split) * (p.B * p.H) + bh) * p.Nq + row_g;
    float* orow = (p.o_part ? p.o_part : p.o) + out_row * D;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
      uint32_t ov[32];
      tmem_ld32(o_taddr + 32 * k, ov);
      tmem_wait_ld(ov);
      if (row_g < p.Nq) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 v4 =
              make_float4(__uint_as_float(ov[i]) * inv_l, __uint_as_float(ov[i + 1]) * inv_l,
                          __uint_as_float(ov[i + 2]) * inv_l, __uint_as_float(ov[i + 3]) * inv_l);
          *reinterpret_cast<float4*>(orow + 32 * k + i) = v4;
        }
      }
    }
    if (r == 0 && t == 0 && pass == 0 && p.trace != nullptr && blockIdx.x == 0)
      p.trace[kTraceWords - 1] = static_cast<unsigned long long>(clock64());
    if (row_g < p.Nq) {
      const float lsum = kLTensor ? l + delta : l;
      (p.lse_part ? p.lse_part : p.lse)[out_row] =
          l > 0.f ? (M - kKappa + __log2f(lsum)) * kLn2 : -INFINITY;
    }
  }
  tc_fence_before();
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// kX:       > 0: surrogate maximum over kX-row tiles (Algorithm 1);
//           0: the exact per-row maximum (vector-softmax ablation).
// kLTensor: (kTensor only) the row sum of step 7 on the tensor pipe as
//           P~ (bf16) times a block of ones; otherwise an fp32 sum of the
//           unrounded P~ on the vector units.
// kE4M3:    e4m3 inputs, kind::f8f6f4 MMAs, e4m3 P~ (otherwise bf16).
template <int D, int kX, bool kLTensor, bool kE4M3>
__global__ void __launch_bounds__(kNumThreads, 1) fat_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = Smem<D, kE4M3>;
  constexpr int S = L::kStages;
  constexpr bool kTensor = kX > 0;
  // X = 128 (bf16): the uniform rescale of O rides in the PV MMA
  constexpr bool kMmaScale = kX == 128 && !kE4M3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8 * i; };

  // work item: heaviest query blocks first (causal), then (b, h)
  const int BH = p.B * p.H;
  const int mblock = p.n_mblocks - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int m0 = mblock * kRowsPerCta;
  // this block's key range: the split's range, cut at the causal limit of
  // its last row
  const int split = static_cast<int>(blockIdx.y);
  const int kv_begin = split * p.kv_split_len;
  const int kv_end = min(p.Nk, kv_begin + p.kv_split_len);
  const int kv_off = p.Nk - p.Nq;
  const int kv_hi = p.causal ? min(kv_end, m0 + kRowsPerCta + kv_off) : kv_end;
  const int n_kv = kv_hi > kv_begin ? (kv_hi - kv_begin + kBlockN - 1) / kBlockN : 0;
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
  if (threadIdx.x == 0) {
    mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(L::bKFull + s), 1);
      mbar_init(bar(L::bKEmpty + s), 1);
      mbar_init(bar(L::bVFull + s), 1);
      mbar_init(bar(L::bVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::bSFull + t), 1);
      mbar_init(bar(L::bPFull + t), 4);
      mbar_init(bar(L::bRsFull + t), 1);
      mbar_init(bar(L::bLFree + t), 4);
      mbar_init(bar(L::bRed + t), 4);
    }
    mbar_init(bar(L::bOFinal), 1);
    mbar_init(bar(L::bDrain), 1);
    misc[1] = 0;
    misc[2] = 0;
    misc[4] = 0;
    misc[5] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 256) {  // the ones tile used as B of the row-sum MMA
    // 1.0 in bf16 (0x3F80) or e4m3 (0x38)
    const uint32_t one = kE4M3 ? 0x38383838u : 0x3F803F80u;
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
  // softmax warpgroups take them.  Each role runs its own loop over the
  // passes so that no code is shared between the two register budgets.
  if (warp >= kMmaWarp) {
    regs_dec<kCtrlRegs>();
    for (int pass = 0; pass < 2; ++pass) {
      const bool tensor_pass = kTensor && pass == 0;
      const int it0 = pass * n_kv;
      if (warp == kLoadWarp) {
        // =================== TMA producer ===================
        if (lane == 0) {
          int k_issued = 0, v_issued = 0;
          if (pass == 0) {
            tma_prefetch_desc(&p.tm_q);
            tma_prefetch_desc(&p.tm_k);
            tma_prefetch_desc(&p.tm_v);
            mbar_arrive_expect_tx(bar(L::bQFull), 2 * L::kTile);
            for (int t = 0; t < 2; ++t)
              for (int a = 0; a < L::kAtoms; ++a)
                tma_load_3d(sb + L::kQ + t * L::kTile + a * 16384, &p.tm_q, bar(L::bQFull), a * L::kAtomCols,
                            m0 + t * kBlockM, bh);
          }
          for (int j = 0; j < n_kv; ++j) {
            const int it = it0 + j, st = it % S;
            const uint32_t ph = (it / S) & 1;
            if (!wait_bounded(bar(L::bKEmpty + st), ph ^ 1, p, abort_flag)) break;
            mbar_arrive_expect_tx(bar(L::bKFull + st), L::kTile);
            for (int a = 0; a < L::kAtoms; ++a)
              tma_load_3d(sb + L::kK + st * L::kTile + a * 16384, &p.tm_k, bar(L::bKFull + st),
                          a * L::kAtomCols, kv_begin + j * kBlockN, bh);
            k_issued = j + 1;
            if (!wait_bounded(bar(L::bVEmpty + st), ph ^ 1, p, abort_flag)) break;
            mbar_arrive_expect_tx(bar(L::bVFull + st), L::kTile);
            for (int a = 0; a < L::kAtoms; ++a)
              tma_load_3d(sb + L::kV + st * L::kTile + a * 16384, &p.tm_v, bar(L::bVFull + st),
                          a * L::kAtomCols, kv_begin + j * kBlockN, bh);
            v_issued = j + 1;
          }
          if (*abort_flag) {
            // let every copy already issued land before the CTA can exit
            if (pass == 0) wait_drain(bar(L::bQFull), 0);
            for (int j = max(0, k_issued - S); j < k_issued; ++j)
              wait_drain(bar(L::bKFull + (it0 + j) % S), ((it0 + j) / S) & 1);
            for (int j = max(0, v_issued - S); j < v_issued; ++j)
              wait_drain(bar(L::bVFull + (it0 + j) % S), ((it0 + j) / S) & 1);
          }
        }
        __syncwarp();
      } else if (warp == kMmaWarp) {
        // =================== MMA issuer ===================
        if (lane == 0) {
          constexpr uint32_t idesc_s = idesc_f32acc<kE4M3>(kBlockM, kBlockN, false);
          constexpr uint32_t idesc_pv = idesc_f32acc<kE4M3>(kBlockM, D, true);
          constexpr uint32_t idesc_rs = idesc_f32acc<kE4M3>(kBlockM, 16, false);
          const uint64_t ones_desc = sdesc_sw128(sb + L::kOnes, 16, 1024);
          bool ok = true;
          auto issue_s = [&](int t, int st) {
            const uint32_t qa = sb + L::kQ + t * L::kTile, ka = sb + L::kK + st * L::kTile;
  #pragma unroll
            for (int kk = 0; kk < D / L::kMmaK; ++kk) {
              // each 128-byte slab row holds four 32-byte K steps
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_ss<kE4M3>(tmem + t * kBlockN, sdesc_sw128(qa + off, 16, 1024),
                            sdesc_sw128(ka + off, 16, 1024), idesc_s, kk > 0);
            }
          };
          // O_t (+)= P_t V; with kscale > 0 the first K step also applies the
          // uniform rescale O_t <- 2^-kscale O_t of Algorithm 1 steps 2-3.
          auto issue_pv = [&](int t, int st, bool acc, int kscale) {
            const uint32_t va = sb + L::kV + st * L::kTile;
  #pragma unroll
            for (int kk = 0; kk < kBlockN / L::kMmaK; ++kk) {
              // P~ packs 2 (bf16) or 4 (e4m3) keys per TMEM column: 8 columns per K step
              const uint32_t d_t = tmem + 2 * kBlockN + t * D, a_t = tmem + t * kBlockN + kk * 8;
              const uint64_t bd = sdesc_sw128(va + kk * L::kPvStep, 16384, 1024);
              if (kMmaScale && kk == 0 && acc && kscale > 0)
                mma_ts_scale_rt(d_t, a_t, bd, idesc_pv, kscale);
              else
                mma_ts<kE4M3>(d_t, a_t, bd, idesc_pv, acc || kk > 0);
            }
          };
          volatile uint32_t* pv_scale = misc + 4;
          auto issue_rs = [&](int t) {
  #pragma unroll
            for (int kk = 0; kk < kBlockN / L::kMmaK; ++kk)
              mma_ts<kE4M3>(tmem + t * kBlockN + 64, tmem + t * kBlockN + kk * 8, ones_desc, idesc_rs,
                            kk > 0);
          };

          if (pass == 0) ok = wait_bounded(bar(L::bQFull), 0, p, abort_flag);
          if (ok) {
            const int st = it0 % S;
            ok = wait_bounded(bar(L::bKFull + st), (it0 / S) & 1, p, abort_flag);
            if (ok) {
              tc_fence_after();
              issue_s(0, st);
              mma_commit(bar(L::bSFull + 0));
              issue_s(1, st);
              mma_commit(bar(L::bSFull + 1));
              mma_commit(bar(L::bKEmpty + st));
            }
          }
          for (int j = 0; ok && j < n_kv; ++j) {
            const int it = it0 + j, st = it % S;
            const uint32_t ph = (it / S) & 1, par = it & 1;
            const bool more = j + 1 < n_kv;
            const int st1 = (it + 1) % S;
            const uint32_t ph1 = ((it + 1) / S) & 1;
            if (!(ok = wait_bounded(bar(L::bVFull + st), ph, p, abort_flag))) break;
            // tile 0
            if (!(ok = wait_bounded(bar(L::bPFull + 0), par, p, abort_flag))) break;
            trace_mark(p, 3, 0, j, pass);
            tc_fence_after();
            if (kLTensor) {
              issue_rs(0);
              mma_commit(bar(L::bRsFull + 0));
            }
            issue_pv(0, st, j > 0, (kMmaScale && pass == 0) ? static_cast<int>(pv_scale[0]) : 0);
            if (more) {
              if (!(ok = wait_bounded(bar(L::bKFull + st1), ph1, p, abort_flag))) break;
              if (kLTensor && !(ok = wait_bounded(bar(L::bLFree + 0), par, p, abort_flag)))
                break;
              tc_fence_after();
              issue_s(0, st1);
              mma_commit(bar(L::bSFull + 0));
            }
            trace_mark(p, 4, 0, j, pass);
            // tile 1
            if (!(ok = wait_bounded(bar(L::bPFull + 1), par, p, abort_flag))) break;
            trace_mark(p, 3, 1, j, pass);
            tc_fence_after();
            if (kLTensor) {
              issue_rs(1);
              mma_commit(bar(L::bRsFull + 1));
            }
            issue_pv(1, st, j > 0, (kMmaScale && pass == 0) ? static_cast<int>(pv_scale[1]) : 0);
            mma_commit(bar(L::bVEmpty + st));
            if (more) {
              if (kLTensor && !(ok = wait_bounded(bar(L::bLFree + 1), par, p, abort_flag)))
                break;
              tc_fence_after();
              issue_s(1, st1);
              mma_commit(bar(L::bSFull + 1));
              mma_commit(bar(L::bKEmpty + st1));
            }
            trace_mark(p, 4, 1, j, pass);
          }
          if (ok) {
            mma_commit(bar(L::bOFinal));
          } else {
            // every MMA issued so far must finish before TMEM can be released
            mma_commit(bar(L::bDrain));
            wait_drain(bar(L::bDrain), 0);
          }
        }
        __syncwarp();
      }
      __syncthreads();
      if (!kTensor || misc[2] == 0u || *abort_flag != 0u) break;
    }
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  } else {
    regs_inc<kSoftmaxRegs>();
    for (int pass = 0; pass < 2; ++pass) {
      const int it0 = pass * n_kv;
      // =================== softmax warpgroups ===================
      // Pass 1 (only after a flagged pass 0) reruns the block with one-row
      // tiles, X = 1: every row's own maximum rounded up to a whole binade,
      // so no row can underflow (the vector fallback of the page's
      // all-underflow discussion, on the same code path).
      softmax_role<D, kX, kLTensor, kE4M3>(p, smem, sb, tmem, misc, warp, lane, m0, bh, n_kv, it0,
                                           pass, /*exact=*/pass == 1, split, kv_begin, kv_end,
                                           kv_off);
      __syncthreads();
      if (!kTensor || misc[2] == 0u || *abort_flag != 0u) break;
    }
  }
}

}  // namespace fat
