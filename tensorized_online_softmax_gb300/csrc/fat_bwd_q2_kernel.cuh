// The backward pass with a second Q stage, for d = 64: the same five
// tcgen05 MMAs per 128 x 128 tile and the same roles as fat_bwd_kernel, in
// another order.  Q (with its -log2(e) LSE and -scale D) is double-buffered, so Sᵀ of
// the next query block is issued right after dV of this one and runs while
// the softmax warps form dSᵀ; they find it ready once they have.  Between the
// two the softmax warps stage the last block's dQ partial, and the reduce
// warp adds it into global dQ with TMA tensor reduce-adds.  At d = 128 the
// shared memory holds the second Q stage only with the dQ staging split
// between an area of its own and the dSᵀ tile, whose reduce-adds then delay
// the next dSᵀ, so fat_bwd_kernel keeps d = 128 (the recap of "FlashAttention-T
// 完全张量化内核与内存布局优化深度剖析" describes the backward pass by
// recomputation that both follow).
#pragma once

#include "fat_bwd_kernel.cuh"

namespace fat {

template <int D>
struct BwdSmemQ2 {
  static constexpr int kTile = 128 * D * 2;  // one 128 x D bf16 tile
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;       // [2 slots] by the parity of the query block
  static constexpr int kDO = 4 * kTile;
  static constexpr int kDS = 5 * kTile;      // dS^T: 128 keys x 128 queries bf16 (32 KB)
  static constexpr int kLse = kDS + 32768;   // [2 slots] -log2(e) LSE of the query block (128 fp32)
  static constexpr int kDvec = kLse + 1024;  // [2 slots] -scale D of the query block (128 fp32)
  // the dQ partial: fp32 as 128-byte-swizzled boxes of 32 columns x 128
  // rows (16 KB each, the layout of the dQ tensor map)
  static constexpr int kBoxes = D / 32;
  static constexpr int kX = kDvec + 1024;
  static constexpr int kBars = kX + kBoxes * 16384;
  __device__ __forceinline__ static int box(int b) { return kX + b * 16384; }
  // bQFull / bQFree + slot: Q with -log2(e) LSE and -scale D; bOFull / bOFree: dO;
  // bSFull, bDPFull: S^T, dP^T in TMEM; bPReady: P^T in TMEM, bDSReady: dS^T
  // in shared memory (8 arrivals each); bSHeld + w % 4: both warps of those
  // key rows hold their scores (2 arrivals); bDQFull: the dQ partial in
  // TMEM, bDQFree: read by the softmax warps (8 arrivals); bStaged: the
  // partial is in shared memory (8 arrivals); bStageFree: its reduce-adds
  // have read it
  static constexpr int bKV = 0, bQFull = 1, bQFree = 3, bSFull = 5, bPReady = 6, bDQFull = 7,
                       bDQFree = 8, bFinal = 9, bDrain = 10, bSHeld = 11, bOFull = 15,
                       bOFree = 16, bDPFull = 17, bDSReady = 18, bStaged = 19, bStageFree = 20,
                       kNumBars = 21;
  static constexpr int kMisc = kBars + 8 * kNumBars;  // u32: tmem base, abort
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;       // slack for 1024-byte alignment
  static_assert(kAlloc <= 227 * 1024, "shared memory budget (d = 64)");
};

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1) fat_bwd_q2_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdSmemQ2<D>;
  constexpr int kAtoms = D / 64;  // 128-byte column slabs of a tile
  constexpr int kColDQ = BwdColDQ<D>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8 * i; };

  // work item: key block jb of head bh.  The blocks of a head re-read its Q
  // and dO and add into its dQ, so heads run a few at a time, as many as keep
  // those in L2: without a mask every block does the same work and a head's
  // blocks are simply consecutive; causal blocks go in groups of
  // group_heads heads, the first key blocks (which see the most query blocks)
  // first within a group.
  int jb, bh;
  {
    const int idx = static_cast<int>(blockIdx.x);
    if (p.causal) {
      const int per = p.group_heads * p.n_blocks;
      const int g = idx / per;
      const int rem = idx - g * per;
      const int gh = min(p.group_heads, p.BH - g * p.group_heads);
      jb = rem / gh;
      bh = g * p.group_heads + rem % gh;
    } else {
      jb = idx % p.n_blocks;
      bh = idx / p.n_blocks;
    }
  }
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::bQFull + s), 1);
      mbar_init(bar(L::bQFree + s), 1);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bPReady), 8);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDQFree), 8);
    mbar_init(bar(L::bFinal), 1);
    mbar_init(bar(L::bDrain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(L::bSHeld + i), 2);
    mbar_init(bar(L::bOFull), 1);
    mbar_init(bar(L::bOFree), 1);
    mbar_init(bar(L::bDPFull), 1);
    mbar_init(bar(L::bDSReady), 8);
    mbar_init(bar(L::bStaged), 8);
    mbar_init(bar(L::bStageFree), 1);
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
      // Q of block t (with -log2(e) LSE and -scale D) into slot t % 2 once dK of
      // block t - 2 has read that slot (D is read while dS^T is formed,
      // which dK waits for, so it travels with Q); dO of block t once dV of
      // block t - 1 has read the previous one
      int issued_o = 0, issued_q = 0;
      for (int t = 0; t < n_q; ++t) {
        const int ib = q_block(t);
        const int s = t & 1;
        if (t >= 2 && !wait_bounded(bar(L::bQFree + s), ((t - 2) >> 1) & 1, p, abort_flag)) break;
        mbar_arrive_expect_tx(bar(L::bQFull + s), L::kTile + 1024);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sb + L::kQ + s * L::kTile + a * 16384, &p.tm_q, bar(L::bQFull + s), a * 64,
                      ib * 128, bh);
        const size_t row0 = static_cast<size_t>(bh) * p.Npad + ib * 128;
        bulk_load(sb + L::kLse + s * 512, p.lse2 + row0, 512, bar(L::bQFull + s));
        bulk_load(sb + L::kDvec + s * 512, p.dvec + row0, 512, bar(L::bQFull + s));
        issued_q = t + 1;
        if (t > 0 && !wait_bounded(bar(L::bOFree), (t - 1) & 1, p, abort_flag)) break;
        mbar_arrive_expect_tx(bar(L::bOFull), L::kTile);
        for (int a = 0; a < kAtoms; ++a)
          tma_load_3d(sb + L::kDO + a * 16384, &p.tm_do, bar(L::bOFull), a * 64, ib * 128, bh);
        issued_o = t + 1;
      }
      if (*abort_flag) {
        // let the copies already issued land before the CTA can exit
        wait_drain(bar(L::bKV), 0);
        if (issued_o > 0) wait_drain(bar(L::bOFull), (issued_o - 1) & 1);
        for (int u = max(0, issued_q - 2); u < issued_q; ++u)
          wait_drain(bar(L::bQFull + (u & 1)), (u >> 1) & 1);
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
    const uint64_t q_kmaj = sdesc_sw128(sb + L::kQ, 16, 1024);
    const uint64_t do_kmaj = sdesc_sw128(sb + L::kDO, 16, 1024);
    const uint64_t ds_kmaj = sdesc_sw128(sb + L::kDS, 16, 1024);
    const uint64_t q_mn = sdesc_sw128(sb + L::kQ, 16384, 1024);
    const uint64_t do_mn = sdesc_sw128(sb + L::kDO, 16384, 1024);
    const uint64_t k_mn = sdesc_sw128(sb + L::kK, 16384, 1024);
    const uint64_t ds_mn = sdesc_sw128(sb + L::kDS, 16384, 1024);
    constexpr uint32_t kSlot = static_cast<uint32_t>(L::kTile >> 4);  // Q slot, descriptor units
    // K step kk (16 elements) of a K-major operand: 128-byte slab kk / 4,
    // 32-byte step kk % 4 within its rows; of an MN-major one: 16 rows
    auto kstep = [](int kk) -> uint32_t { return ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4; };
    auto mnstep = [](int kk) -> uint32_t { return (kk * 2048) >> 4; };
    auto wait_all = [&](int b, int phase) -> bool {
      return __all_sync(0xffffffffu, wait_bounded(bar(b), phase & 1, p, abort_flag));
    };
    // S^T = K Q^T of block t (its columns last held P^T of block t - 1, which
    // the dV MMAs issued before this one read)
    auto issue_s = [&](int t) -> bool {
      if (!wait_all(L::bQFull + (t & 1), t >> 1)) return false;
      tc_fence_after();
      const uint64_t qd = q_kmaj + (t & 1) * kSlot;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss<false>(tmem + kBwdColS, k_kmaj + kstep(kk), qd + kstep(kk), idesc_sq, kk > 0);
      mma_commit(bar(L::bSFull));
      return true;
    };
    // dP^T = V dO^T of block t (when the dQ partial shares its columns, once
    // the last one has been read out)
    auto issue_dp = [&](int t) -> bool {
      if (!wait_all(L::bOFull, t)) return false;
      if (kColDQ == kBwdColDP && t > 0 && !wait_all(L::bDQFree, t - 1)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss<false>(tmem + kBwdColDP, v_kmaj + kstep(kk), do_kmaj + kstep(kk), idesc_sq, kk > 0);
      mma_commit(bar(L::bDPFull));
      return true;
    };
    bool ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bKV), 0, p, abort_flag));
    if (ok && n_q > 0) ok = issue_s(0) && issue_dp(0);
    for (int t = 0; ok && t < n_q; ++t) {
      // dV += P^T dO: P^T (bf16, two per column) from TMEM, 8 columns per K
      // step, while the softmax warps form dS^T
      if (!(ok = wait_all(L::bPReady, t))) break;
      tc_fence_after();
#pragma unroll
      for (int g = 0; g < 8; ++g)
        mma_ts<false>(tmem + kBwdColDV, tmem + kBwdColS + g * 8, do_mn + mnstep(g), idesc_b_mn,
                      t > 0 || g > 0);
      mma_commit(bar(L::bOFree));
      // the next block's scores, ready for the softmax warps once they have
      // formed this block's dS^T
      if (t + 1 < n_q && !(ok = issue_s(t + 1))) break;
      // dK += dS^T Q
      if (!(ok = wait_all(L::bDSReady, t))) break;
      tc_fence_after();
      const uint64_t qmn = q_mn + (t & 1) * kSlot;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss<false>(tmem + kBwdColDV + D, ds_kmaj + kstep(kk), qmn + mnstep(kk), idesc_b_mn,
                      t > 0 || kk > 0);
      mma_commit(bar(L::bQFree + (t & 1)));
      // dQ partial = dS K (over dP^T, which the softmax warps have read, or in
      // its own columns once the last partial has been read out)
      if (kColDQ != kBwdColDP && t > 0 && !(ok = wait_all(L::bDQFree, t - 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss<false>(tmem + kColDQ, ds_mn + mnstep(kk), k_mn + mnstep(kk), idesc_ab_mn, kk > 0);
      mma_commit(bar(L::bDQFull));
      if (t + 1 < n_q && !(ok = issue_dp(t + 1))) break;
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
    for (int t = 0; t < n_q; ++t) {
      if (!__all_sync(0xffffffffu, wait_bounded(bar(L::bStaged), t & 1, p, abort_flag))) break;
      if (lane == 0) {
        // rows past N are clipped by the tensor map
        for (int b = 0; b < L::kBoxes; ++b)
          tma_reduce_add_3d(&p.tm_dq, sb + L::box(b), b * 32, q_block(t) * 128, bh);
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
    // the dQ partial of block u (query rows 32 qw .., columns D/2 hf ..) out
    // of TMEM and into its staging boxes, once the reduce-adds of block u - 1
    // have read them
    auto dq_out = [&](int u) -> bool {
      if (!__all_sync(0xffffffffu, wait_bounded(bar(L::bDQFull), u & 1, p, abort_flag)))
        return false;
      tc_fence_after();
      uint32_t v[D / 64][32];
#pragma unroll
      for (int cg = 0; cg < D / 64; ++cg)
        tmem_ld32(tmem + lane_base + kColDQ + hf * (D / 2) + 32 * cg, v[cg]);
#pragma unroll
      for (int cg = 0; cg < D / 64; ++cg) tmem_wait_ld(v[cg]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bDQFree));
      if (u > 0 &&
          !__all_sync(0xffffffffu,
                      wait_bounded(bar(L::bStageFree), (u - 1) & 1, p, abort_flag)))
        return false;
#pragma unroll
      for (int cg = 0; cg < D / 64; ++cg) {
        const uint32_t box = sb + L::box(hf * (D / 64) + cg) + r * 128;
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4u(box + ((c4 ^ (r & 7)) << 4), v[cg][4 * c4], v[cg][4 * c4 + 1],
                        v[cg][4 * c4 + 2], v[cg][4 * c4 + 3]);
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bStaged));
      return true;
    };
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

      // the last block's dQ partial, whose MMA has long completed: reading it
      // out lets dP^T of this block into its columns
      if (t > 0 && !(ok = dq_out(t - 1))) break;

      // dS^T = scale P^T (dP^T - D) into row r of the swizzled tile (queries
      // 32 k .. 32 k + 31 are four 16-byte chunks), while the dV MMAs run;
      // the last block's dK and dQ MMAs, which read the tile, have completed
      // (the dQ partial read above came after them)
      if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar(L::bDPFull), t & 1, p, abort_flag))))
        break;
      tc_fence_after();
      uint32_t dsk[2][16];
      uint32_t dp[2][32];
      tmem_ld32(tmem + lane_base + kBwdColDP + 64 * hf, dp[0]);
      tmem_ld32(tmem + lane_base + kBwdColDP + 64 * hf + 32, dp[1]);
      tmem_wait_ld(dp[0]);
      tmem_wait_ld(dp[1]);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * hf + kk;
        bwd_ds_chunk(s[kk], dp[kk], dsk[kk], dvec_s + 128 * k, sc2);
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int k = 2 * hf + kk;
        const uint32_t row = sb + L::kDS + (k >> 1) * 16384 + r * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int chunk = (k & 1) * 4 + cc;
          st_shared_v4u(row + ((chunk ^ (r & 7)) << 4), dsk[kk][4 * cc], dsk[kk][4 * cc + 1],
                        dsk[kk][4 * cc + 2], dsk[kk][4 * cc + 3]);
        }
      }
      fence_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::bDSReady));
    }
    if (ok && n_q > 0) ok = dq_out(n_q - 1);
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


}  // namespace fat
