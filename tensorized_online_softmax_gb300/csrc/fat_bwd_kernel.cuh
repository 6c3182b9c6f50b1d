// Fused attention backward pass for sm_103a: recomputes the attention
// weights from Q, K and the forward's LSE (the backward pass by
// recomputation that the v1 recap of "FlashAttention-T 完全张量化内核与内存布局
// 优化深度剖析" describes: only O and the softmax statistics are kept) and
// forms dQ, dK, dV with five tcgen05 MMAs per 128 x 128 tile:
//
//   S^T  = K Q^T           (TMEM)       P^T  = exp2(c S^T - log2(e) LSE)
//   dP^T = V dO^T          (TMEM)       dS^T = scale P^T * (dP^T - D)
//   dV  += P^T dO          (A = P^T from TMEM, bf16)
//   dK  += dS^T Q          (A = dS^T from shared memory, K-major)
//   dQ   = dS K            (A = the same tile read MN-major), staged in
//                           shared memory and added to global dQ with TMA
//                           tensor reduce-adds
//
// with D_i = sum_d dO_id O_id formed beforehand (fat_bwd_prep_kernel).
// This schedule serves d = 128; d = 64, whose tiles leave room for a second
// Q stage, runs fat_bwd_q2_kernel (fat_bwd_q2_kernel.cuh) instead.
// One CTA per 128-key block of one (b, h); it walks the query blocks that
// see those keys (all of them, or those at or after the diagonal when
// causal).  Warps: 0-7 form P^T and dS^T (warp w: key rows 32 (w % 4) ..,
// query columns 64 (w / 4) ..) and then stage the block's dQ partial from
// TMEM in shared memory; 8 issues the MMAs; 9 loads K and V once and Q, dO,
// -log2(e) LSE and -scale D per query block with TMA; 10 adds each staged dQ
// partial into global dQ with TMA reduce-adds.  Q and dO swap their two
// shared-memory slots every query block, so that the next Q loads as soon as
// dV has read dO rather than after dK, and dQ is issued before dK: the
// softmax warps wait for the dQ partial, the next dO for dK.
#pragma once

#include <climits>

#include "fat_fwd_kernel.cuh"

namespace fat {

struct BwdParams {
  CUtensorMap tm_q;   // bf16 [B*H, N, d], boxes of 64 columns x 128 rows, 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  CUtensorMap tm_dq;  // fp32 [B*H, N, d], boxes of 32 columns x 128 rows, 128-byte swizzle
  const float* lse2;  // [B*H][Npad] -log2(e) * LSE; -inf for rows >= N
  const float* dvec;  // [B*H][Npad] -scale * D; 0 for rows >= N
  float* dq;          // fp32 [B*H, N, d], cleared by the preparation kernel, then
                      // accumulated by TMA reduce-adds
  float* dk;          // fp32 [B*H, N, d]
  float* dv;          // fp32 [B*H, N, d]
  int BH, N, Npad, causal, n_blocks;
  int group_heads;    // causal: heads per group of blocks ordered together ...
  int group_extra;    // ... the first group_extra groups holding one more
                      // (d = 128; the d = 64 kernel takes groups of
                      // group_heads, the last one smaller)
  float c;            // log2(e) * scale
  float scale;
  unsigned long long poll_limit;
  unsigned long long timeout_ns;
  unsigned int* error_word;
};

constexpr int kBwdThreads = 352;
constexpr int kBwdMmaWarp = 8;
constexpr int kBwdLoadWarp = 9;
constexpr int kBwdReduceWarp = 10;
// TMEM columns: S^T / P^T; dP^T; dV; dK; the dQ partial in columns of its
// own when they fit (d = 64), else over dP^T once dS^T has been formed
constexpr int kBwdColS = 0;
constexpr int kBwdColDP = 128;
constexpr int kBwdColDV = 256;
template <int D>
struct BwdColDQ {
  static constexpr int value = 256 + 3 * D <= 512 ? 256 + 2 * D : kBwdColDP;
};

// Two fp32 pairs from shared memory (16-byte aligned address).
__device__ __forceinline__ void ld_shared_2xf2(uint32_t addr, uint64_t& a, uint64_t& b) {
  asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}

// P^T of one 32-column chunk of a thread's key row, in place over its scores
// s (fp32 bits): exp2(c S^T - log2(e) LSE) with -log2(e) LSE of the chunk's
// 32 queries at nlse (shared memory), one f32x2 FMA per pair of columns;
// pk receives the bf16 pairs for TMEM.  kMasked: columns below lim (causal)
// are zero; callers pass lim = INT_MAX for a key row past N.
template <bool kMasked>
__device__ __forceinline__ void bwd_p_chunk(uint32_t (&s)[32], uint32_t (&pk)[16], uint32_t nlse,
                                            uint64_t c2, int col0, int lim) {
#pragma unroll
  for (int i4 = 0; i4 < 8; ++i4) {
    uint64_t nl[2];
    ld_shared_2xf2(nlse + 16 * i4, nl[0], nl[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 4 * i4 + 2 * h;
      float z0, z1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(s[i]), __uint_as_float(s[i + 1])), c2, nl[h]), z0,
                z1);
      float p0 = ex2_approx(z0), p1 = ex2_approx(z1);
      if constexpr (kMasked) {
        p0 = col0 + i >= lim ? p0 : 0.f;
        p1 = col0 + i + 1 >= lim ? p1 : 0.f;
      }
      s[i] = __float_as_uint(p0);
      s[i + 1] = __float_as_uint(p1);
      pk[2 * i4 + h] = pack_bf16x2(p0, p1);
    }
  }
}

// dS^T of one 32-column chunk: P^T (fp32 bits, p) times
// scale dP^T - scale D, with -scale D of the chunk's queries at nsd (shared
// memory): one f32x2 FMA and one f32x2 multiply per pair of columns; dsk
// receives the bf16 pairs.
__device__ __forceinline__ void bwd_ds_chunk(const uint32_t (&p)[32], const uint32_t (&dp)[32],
                                             uint32_t (&dsk)[16], uint32_t nsd, uint64_t sc2) {
#pragma unroll
  for (int i4 = 0; i4 < 8; ++i4) {
    uint64_t nd[2];
    ld_shared_2xf2(nsd + 16 * i4, nd[0], nd[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 4 * i4 + 2 * h;
      const uint64_t u =
          f2_fma(f2_pack(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])), sc2, nd[h]);
      float d0, d1;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(p[i]), __uint_as_float(p[i + 1])), u), d0, d1);
      dsk[2 * i4 + h] = pack_bf16x2(d0, d1);
    }
  }
}

template <int D>
struct BwdSmem {
  static constexpr int kTile = 128 * D * 2;  // one 128 x D bf16 tile
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  // [2 slots] Q of query block t in slot t % 2, dO of block t in the other:
  // the next Q goes where dO was as soon as dV has read it, the next dO where
  // Q was once dK has read that
  static constexpr int kSlot = 2 * kTile;
  static constexpr int kDS = 4 * kTile;      // dS^T: 128 keys x 128 queries bf16 (32 KB)
  // the dQ partial of a query block: fp32, 128-byte-swizzled boxes of 32
  // columns x 128 rows (16 KB each), the layout of the dQ tensor map
  static constexpr int kDQ = kDS + 32768;
  // [2 slots by t % 2] -log2(e) LSE and -scale D of the query block (128
  // fp32 each): the next block's arrive with its Q while dS^T of this one
  // still reads D
  static constexpr int kLse = kDQ + 128 * D * 4;
  static constexpr int kDvec = kLse + 1024;
  static constexpr int kBars = kDvec + 1024;
  // bQFull / bQFree: Q with -log2(e) LSE and -scale D; bOFull / bOFree: dO;
  // bSFull, bDPFull: S^T, dP^T in TMEM; bPReady: P^T in TMEM, bDSReady: dS^T
  // in shared memory (8 arrivals each); bSHeld + w % 4: both warps of those
  // key rows hold their scores (2 arrivals); bStaged: the dQ partial is in
  // shared memory (8 arrivals); bStageFree: its reduce-adds have read it
  static constexpr int bKV = 0, bQFull = 1, bQFree = 2, bSFull = 3, bPReady = 4, bDQFull = 5,
                       bDQFree = 6, bFinal = 7, bDrain = 8, bSHeld = 9, bStaged = 13,
                       bStageFree = 14, bOFull = 15, bOFree = 16, bDPFull = 17, bDSReady = 18,
                       kNumBars = 19;
  static constexpr int kMisc = kBars + 8 * kNumBars;  // u32: tmem base, abort
  static constexpr int kBytes = kMisc + 16;
  // no room to align the base by hand: the dynamic shared memory must start
  // 1024-byte aligned (the kernel checks and stops with an error otherwise)
  static constexpr int kAlloc = kBytes;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) fat_bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdSmem<D>;
  constexpr int kAtoms = D / 64;  // 128-byte column slabs of a tile
  constexpr int kColDQ = BwdColDQ<D>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // (uniform over the block: no barrier has been used yet)
    if (threadIdx.x == 0) atomicOr(p.error_word, 1u);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8 * i; };

  // work item: key block jb of head bh.  The blocks of a head re-read its Q
  // and dO and add into its dQ, so heads run a few at a time, as many as keep
  // those in L2 (bwd_work_item in fat_schedule.h: balanced groups of heads
  // when causal, the first key blocks first within a group).
  int jb, bh;
  bwd_work_item(static_cast<int>(blockIdx.x), p.n_blocks, p.causal != 0, p.group_heads,
                p.group_extra, jb, bh);
  const int ib0 = p.causal ? jb : 0;
  const int n_q = p.n_blocks - ib0;
  // query block of step t: causal blocks start at their diagonal; the others
  // start at their own index and wrap, so that the key blocks of a head add
  // into different dQ rows at any one time
  auto q_block = [&](int t) -> int {
    return p.causal ? ib0 + t : (jb + t < p.n_blocks ? jb + t : jb + t - p.n_blocks);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::bKV), 1);
    mbar_init(bar(L::bQFull), 1);
    mbar_init(bar(L::bQFree), 1);
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bPReady), 8);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDQFree), 8);
    mbar_init(bar(L::bFinal), 1);
    mbar_init(bar(L::bDrain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(L::bSHeld + i), 2);
    mbar_init(bar(L::bStaged), 8);
    mbar_init(bar(L::bStageFree), 1);
    mbar_init(bar(L::bOFull), 1);
    mbar_init(bar(L::bOFree), 1);
    mbar_init(bar(L::bDPFull), 1);
    mbar_init(bar(L::bDSReady), 8);
    misc[1] = 0;
    fence_mbar_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(sb + L::kMisc, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == kBwdLoadWarp) {
    // =================== TMA producer ===================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(bar(L::bKV), 2 * L::kTile);
      for (int a = 0; a < kAtoms; ++a) {
        tma_load_3d(sb + L::kK + a * 16384, &p.tm_k, bar(L::bKV), a * 64, jb * 128, bh);
        tma_load_3d(sb + L::kV + a * 16384, &p.tm_v, bar(L::bKV), a * 64, jb * 128, bh);
      }
      // -log2(e) LSE and -scale D come from the preparation kernel, which may
      // still be running (programmatic dependent launch)
      grid_dep_wait();
      // Q of block t (with -log2(e) LSE and -scale D: D is read while dS^T
      // is formed, so it travels with Q) into slot t % 2 once dV of block
      // t - 1 has read dO of block t - 1 there; dO of block t into the other
      // slot once dK of block t - 1 has read Q of block t - 1 there
      int issued_o = 0, issued_q = 0;
      for (int t = 0; t < n_q; ++t) {
        const int ib = q_block(t);
        const int s = t & 1;
        if (t > 0 && !wait_bounded(bar(L::bOFree), (t - 1) & 1, p, abort_flag)) break;
        mbar_arrive_expect_tx(bar(L::bQFull), L::kTile + 1024);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sb + L::kSlot + s * L::kTile + a * 16384, &p.tm_q, bar(L::bQFull), a * 64,
                      ib * 128, bh);
        const size_t row0 = static_cast<size_t>(bh) * p.Npad + ib * 128;
        bulk_load(sb + L::kLse + s * 512, p.lse2 + row0, 512, bar(L::bQFull));
        bulk_load(sb + L::kDvec + s * 512, p.dvec + row0, 512, bar(L::bQFull));
        issued_q = t + 1;
        if (t > 0 && !wait_bounded(bar(L::bQFree), (t - 1) & 1, p, abort_flag)) break;
        mbar_arrive_expect_tx(bar(L::bOFull), L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sb + L::kSlot + (s ^ 1) * L::kTile + a * 16384, &p.tm_do, bar(L::bOFull),
                      a * 64, ib * 128, bh);
        issued_o = t + 1;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA can exit
        wait_drain(bar(L::bKV), 0);
        if (issued_o > 0) wait_drain(bar(L::bOFull), (issued_o - 1) & 1);
        if (issued_q > 0) wait_drain(bar(L::bQFull), (issued_q - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    // =================== MMA issuer (whole warp, elected lane) ===================
    constexpr uint32_t idesc_sq = idesc_f32acc<1u>(128, 128, false);       // K-major A, B
    constexpr uint32_t idesc_b_mn = idesc_f32acc<1u>(128, D, true);        // B MN-major
    constexpr uint32_t idesc_ab_mn = idesc_f32acc<1u>(128, D, true, true); // A, B MN-major
    const uint64_t k_kmaj = sdesc_sw128(sb + L::kK, 16, 1024);
    const uint64_t v_kmaj = sdesc_sw128(sb + L::kV, 16, 1024);
    const uint64_t slot_kmaj = sdesc_sw128(sb + L::kSlot, 16, 1024);
    const uint64_t ds_kmaj = sdesc_sw128(sb + L::kDS, 16, 1024);
    const uint64_t slot_mn = sdesc_sw128(sb + L::kSlot, 16384, 1024);
    const uint64_t k_mn = sdesc_sw128(sb + L::kK, 16384, 1024);
    const uint64_t ds_mn = sdesc_sw128(sb + L::kDS, 16384, 1024);
    // Q of block t in slot t % 2, dO in the other (descriptor units)
    constexpr uint32_t kSlot1 = static_cast<uint32_t>(L::kTile >> 4);
    // K step kk (16 elements) of a K-major operand: 128-byte slab kk / 4,
    // 32-byte step kk % 4 within its rows; of an MN-major one: 16 rows
    auto kstep = [](int kk) -> uint32_t { return ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4; };
    auto mnstep = [](int kk) -> uint32_t { return (kk * 2048) >> 4; };
    bool ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bKV), 0, p, abort_flag));
    auto wait_all = [&](int b, int phase) -> bool {
      return __all_sync(0xffffffffu, wait_bounded(bar(b), phase & 1, p, abort_flag));
    };
    for (int t = 0; ok && t < n_q; ++t) {
      const uint32_t q_slot = (t & 1) * kSlot1, do_slot = ((t & 1) ^ 1) * kSlot1;
      // S^T = K Q^T (its columns last held P^T of block t - 1, which the dV
      // MMAs issued before this one read)
      if (!(ok = wait_all(L::bQFull, t))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss<false>(tmem + kBwdColS, k_kmaj + kstep(kk), slot_kmaj + q_slot + kstep(kk),
                      idesc_sq, kk > 0);
      mma_commit(bar(L::bSFull));
      // dP^T = V dO^T (when the dQ partial shares its columns, once the
      // previous one has left them)
      if (!(ok = wait_all(L::bOFull, t))) break;
      if (kColDQ == kBwdColDP && t > 0 && !(ok = wait_all(L::bDQFree, t - 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss<false>(tmem + kBwdColDP, v_kmaj + kstep(kk), slot_kmaj + do_slot + kstep(kk),
                      idesc_sq, kk > 0);
      mma_commit(bar(L::bDPFull));
      // dV += P^T dO: P^T (bf16, two per column) from TMEM, 8 columns per K
      // step, while the softmax warps still form dS^T
      if (!(ok = wait_all(L::bPReady, t))) break;
      tc_fence_after();
#pragma unroll
      for (int g = 0; g < 8; ++g)
        mma_ts<false>(tmem + kBwdColDV, tmem + kBwdColS + g * 8, slot_mn + do_slot + mnstep(g),
                      idesc_b_mn, t > 0 || g > 0);
      // dO's slot takes the next Q once these have completed
      mma_commit(bar(L::bOFree));
      if (!(ok = wait_all(L::bDSReady, t))) break;
      // dQ partial = dS K (over dP^T, which the softmax warps have read, or in
      // its own columns once the previous partial has left them), before dK:
      // the softmax warps wait for it
      if (kColDQ != kBwdColDP && t > 0 && !(ok = wait_all(L::bDQFree, t - 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss<false>(tmem + kColDQ, ds_mn + mnstep(kk), k_mn + mnstep(kk), idesc_ab_mn, kk > 0);
      mma_commit(bar(L::bDQFull));
      // dK += dS^T Q
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss<false>(tmem + kBwdColDV + D, ds_kmaj + kstep(kk), slot_mn + q_slot + mnstep(kk),
                      idesc_b_mn, t > 0 || kk > 0);
      // Q's slot takes the next dO once these have completed
      mma_commit(bar(L::bQFree));
    }
    if (ok) {
      mma_commit(bar(L::bFinal));
    } else {
      mma_commit(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0);
    }
    __syncwarp();
  } else if (warp == kBwdReduceWarp) {
    // =================== dQ reduce-adds ===================
    grid_dep_wait();  // dQ is cleared by the preparation kernel
    for (int t = 0; t < n_q; ++t) {
      if (!__all_sync(0xffffffffu, wait_bounded(bar(L::bStaged), t & 1, p, abort_flag))) break;
      if (lane == 0) {
        // rows past N are clipped by the tensor map
        for (int b = 0; b < D / 32; ++b)
          tma_reduce_add_3d(&p.tm_dq, sb + L::kDQ + b * 16384, b * 32, q_block(t) * 128, bh);
        bulk_commit();
        bulk_wait_read();
        mbar_arrive(bar(L::bStageFree));
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    // ============ P^T, dS^T and the dQ partials (warps 0-7) ============
    const int qw = warp & 3;   // TMEM lanes 32 qw ..: key rows (S^T, dP^T), query rows (dQ)
    const int hf = warp >> 2;  // query columns 64 hf .. of S^T and dP^T
    const int r = qw * 32 + lane;
    const int key = jb * 128 + r;
    const bool row_ok = key < p.N;
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const uint64_t c2 = f2_pack(p.c, p.c);
    const uint64_t sc2 = f2_pack(p.scale, p.scale);
    bool ok = true;
    for (int t = 0; t < n_q; ++t) {
      const int ib = q_block(t);
      const uint32_t lse_s = sb + L::kLse + (t & 1) * 512;
      const uint32_t dvec_s = sb + L::kDvec + (t & 1) * 512;
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bSFull), t & 1, p, abort_flag))))
        break;
      tc_fence_after();
      uint32_t s[2][32];
      tmem_ld32(tmem + lane_base + kBwdColS + 64 * hf, s[0]);
      tmem_ld32(tmem + lane_base + kBwdColS + 64 * hf + 32, s[1]);
      tmem_wait_ld(s[0]);
      tmem_wait_ld(s[1]);
      // P^T goes over the scores in place (columns 0-63): both warps of these
      // rows must hold their scores first
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bSHeld + qw));
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bSHeld + qw), t & 1, p, abort_flag))))
        break;
      tc_fence_after();
      // causal: query ib * 128 + col sees this key iff col >= lim (none for
      // a key row past N)
      const int lim = !row_ok ? INT_MAX : p.causal ? key - ib * 128 : -1;
      // P^T = exp2(c S^T - log2(e) LSE), kept in fp32 (over the scores'
      // registers) for dS^T and stored as bf16 over the scores' columns
      // (columns 16 k .. for the 32-column chunk k); the mask only where
      // this thread's columns 64 hf .. need it
      const bool masked = lim > 64 * hf;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * hf + kk;  // 32-column chunk of the block's queries
        uint32_t pk[16];
        if (masked)
          bwd_p_chunk<true>(s[kk], pk, lse_s + 128 * k, c2, 32 * k, lim);
        else
          bwd_p_chunk<false>(s[kk], pk, lse_s + 128 * k, c2, 32 * k, lim);
        tmem_st16(tmem + lane_base + kBwdColS + 16 * k, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bPReady));

      // dS^T = scale P^T (dP^T - D) into row r of the swizzled tile (queries
      // 32 k .. 32 k + 31 are four 16-byte chunks), while the dV MMAs run
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bDPFull), t & 1, p, abort_flag))))
        break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * hf + kk;
        uint32_t dp[32];
        tmem_ld32(tmem + lane_base + kBwdColDP + 32 * k, dp);
        tmem_wait_ld(dp);
        uint32_t dk[16];
        bwd_ds_chunk(s[kk], dp, dk, dvec_s + 128 * k, sc2);
        const uint32_t row = sb + L::kDS + (k >> 1) * 16384 + r * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int chunk = (k & 1) * 4 + cc;
          st_shared_v4u(row + ((chunk ^ (r & 7)) << 4), dk[4 * cc], dk[4 * cc + 1],
                        dk[4 * cc + 2], dk[4 * cc + 3]);
        }
      }
      fence_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bDSReady));

      // this block's dQ partial (query rows 32 qw .., columns D/2 hf ..) into
      // the staging boxes, once the previous partial's reduce-adds read them
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bDQFull), t & 1, p, abort_flag))))
        break;
      if (t > 0 &&
          !(ok = __all_sync(0xffffffffu,
                            wait_bounded(bar(L::bStageFree), (t - 1) & 1, p, abort_flag))))
        break;
      tc_fence_after();
#pragma unroll
      for (int cg = 0; cg < D / 64; ++cg) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + kColDQ + hf * (D / 2) + 32 * cg, v);
        tmem_wait_ld(v);
        const uint32_t box = sb + L::kDQ + (hf * (D / 64) + cg) * 16384 + r * 128;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4u(box + ((c4 ^ (r & 7)) << 4), v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2],
                        v[4 * c4 + 3]);
      }
      fence_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(L::bDQFree));
        mbar_arrive(bar(L::bStaged));
      }
    }
    // epilogue: dV and dK rows of this block's keys (columns D/2 hf ..)
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bFinal), 0, p, abort_flag));
    if (ok) {
      tc_fence_after();
      const size_t base = (static_cast<size_t>(bh) * p.N + key) * D + hf * (D / 2);
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        float* out = which == 0 ? p.dv : p.dk;
#pragma unroll
        for (int cg = 0; cg < D / 64; ++cg) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + kBwdColDV + which * D + hf * (D / 2) + 32 * cg, v);
          tmem_wait_ld(v);
          if (row_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_global_v4(out + base + 32 * cg + 4 * i, __uint_as_float(v[4 * i]),
                           __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                           __uint_as_float(v[4 * i + 3]));
          }
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// -scale D_i (D_i = sum_d dO_id O_id) and -log2(e) LSE_i for every row,
// padded to whole 128-row blocks (0 and -inf past N, so those queries weigh
// nothing), in the forms the elementwise warps use: exp2(c S + (-log2(e)
// LSE)) and P (scale dP + (-scale D)), one f32x2 FMA per pair; and dQ's rows
// cleared for the reduce-adds that follow, in the same pass over the rows.
// Each warp takes kPrepRows consecutive rows and issues all of their loads
// before it reduces any, so that enough bytes are in flight to keep HBM busy.
constexpr int kPrepRows = 4;
constexpr int kPrepWarps = 8;
template <int D>
__global__ void __launch_bounds__(kPrepWarps * 32)
    fat_bwd_prep_kernel(const float* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                        const float* __restrict__ lse, float* __restrict__ lse2,
                        float* __restrict__ dvec, float* __restrict__ dq, int N, int Npad,
                        long long rows, float scale) {
  static_assert(D == 64 || D == 128, "head dimension");
  constexpr int kCols = D / 32;  // columns per lane: 2 or 4
  // the fused kernel may start its set-up (it waits for this grid before it
  // reads anything written here)
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const long long row0 =
      (static_cast<long long>(blockIdx.x) * kPrepWarps + (threadIdx.x >> 5)) * kPrepRows;
  float ov[kPrepRows][kCols];
  __nv_bfloat162 dv2[kPrepRows][kCols / 2];
  size_t base[kPrepRows];
  bool live[kPrepRows];
#pragma unroll
  for (int r = 0; r < kPrepRows; ++r) {
    const long long row = row0 + r;
    const long long bh = row / Npad;
    const int n = static_cast<int>(row - bh * Npad);
    live[r] = row < rows && n < N;
    base[r] = (static_cast<size_t>(bh) * N + n) * D + lane * kCols;
#pragma unroll
    for (int c = 0; c < kCols; ++c) ov[r][c] = 0.f;
#pragma unroll
    for (int c = 0; c < kCols / 2; ++c) dv2[r][c] = __floats2bfloat162_rn(0.f, 0.f);
    if (live[r]) {
      if constexpr (kCols == 4) {
        const float4 a = *reinterpret_cast<const float4*>(o + base[r]);
        ov[r][0] = a.x; ov[r][1] = a.y; ov[r][2] = a.z; ov[r][3] = a.w;
      } else {
        const float2 a = *reinterpret_cast<const float2*>(o + base[r]);
        ov[r][0] = a.x; ov[r][1] = a.y;
      }
#pragma unroll
      for (int c = 0; c < kCols / 2; ++c)
        dv2[r][c] = *reinterpret_cast<const __nv_bfloat162*>(dout + base[r] + 2 * c);
    }
  }
  float acc[kPrepRows];
#pragma unroll
  for (int r = 0; r < kPrepRows; ++r) {
    acc[r] = 0.f;
#pragma unroll
    for (int c = 0; c < kCols / 2; ++c)
      acc[r] += ov[r][2 * c] * __low2float(dv2[r][c]) + ov[r][2 * c + 1] * __high2float(dv2[r][c]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int r = 0; r < kPrepRows; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
#pragma unroll
  for (int r = 0; r < kPrepRows; ++r) {
    const long long row = row0 + r;
    if (live[r]) {
      if constexpr (kCols == 4)
        *reinterpret_cast<float4*>(dq + base[r]) = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        *reinterpret_cast<float2*>(dq + base[r]) = make_float2(0.f, 0.f);
    }
    if (lane == r && row < rows) {
      const long long bh = row / Npad;
      const int n = static_cast<int>(row - bh * Npad);
      dvec[row] = n < N ? -scale * acc[r] : 0.f;
      lse2[row] = n < N ? -(lse[bh * N + n] * kLog2e) : -INFINITY;
    }
  }
}

}  // namespace fat
