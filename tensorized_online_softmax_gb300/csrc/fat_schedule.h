// Work schedules of the forward kernel (which query tile a block takes next)
// and of the backward kernels (which key block a CTA takes), shared by the
// host (grid size, tests) and the device.  A forward work item is one
// 128-row query tile of one (batch, head) -- one output row block per worker, the
// fused flow of "FlashAttention-T: Towards Fully Tensorized Attention by
// Exploiting Tensor-Vector Parallelism" (papercache.org summary, section A3,
// Fig. 2).  Plain C++ apart from the CUDA qualifiers, so a host compiler can
// build it for tests.
#pragma once

#ifndef __CUDACC__
#define __host__
#define __device__
#define __forceinline__ inline
#endif

namespace fat {

// A block takes at most this many items, which bounds its list of items
// deferred to the fallback pass.
constexpr int kMaxDeferred = 64;

// The k-th item of block b of a launch of G blocks over n_items items, or -1
// past the end.  Blocks take items in strides of G, in alternating direction
// (0 1 .. G-1, then 2G-1 .. G, ...), so that where costs fall along the item
// list a block with a heavy item in one stride gets a light one in the next.
// With G == n_items every block takes exactly its own index.
__host__ __device__ __forceinline__ int fwd_item_index(int k, int b, int G, int n_items) {
  const int idx = k * G + ((k & 1) ? G - 1 - b : b);
  return idx < n_items ? idx : -1;
}

// Blocks of a forward launch: one per item, or (tiles in turn) one per SM --
// more if that would give a block more than kMaxDeferred items.
__host__ __device__ __forceinline__ int fwd_grid(int n_items, int sms, bool one_per_item) {
  if (one_per_item || sms <= 0 || n_items <= sms) return n_items;
  const int need = (n_items + kMaxDeferred - 1) / kMaxDeferred;
  return need > sms ? need : sms;
}

// Backward pass, causal: heads run in groups whose Q, dO and dQ stay in L2
// together, at most max_heads heads each.  The groups are balanced: of the
// ceil(BH / max_heads) groups the first bwd_group_extra() hold one head more
// than the rest (bwd_group_heads()), so that no small group of heavy blocks
// is left for the end of the launch (with groups 6, 6, 6, 6, 6, 2 of 32 heads
// the last two heads' 64-query-block blocks would start after everything
// else).
__host__ __device__ __forceinline__ int bwd_group_count(int BH, int max_heads) {
  if (max_heads < 1) max_heads = 1;
  return (BH + max_heads - 1) / max_heads;
}
__host__ __device__ __forceinline__ int bwd_group_heads(int BH, int max_heads) {
  return BH / bwd_group_count(BH, max_heads);
}
__host__ __device__ __forceinline__ int bwd_group_extra(int BH, int max_heads) {
  return BH % bwd_group_count(BH, max_heads);
}

// CTA idx of a backward launch -> (key block jb, head bh).  Without a mask
// every block does the same work and a head's blocks are consecutive; causal
// blocks go by groups (the first group_extra of group_heads + 1 heads, then
// groups of group_heads), the first key blocks (which see the most query
// blocks) first within a group, heads in turn.
__host__ __device__ __forceinline__ void bwd_work_item(int idx, int n_blocks, bool causal,
                                                      int group_heads, int group_extra, int& jb,
                                                      int& bh) {
  if (!causal) {
    jb = idx % n_blocks;
    bh = idx / n_blocks;
    return;
  }
  const int big = (group_heads + 1) * n_blocks;  // CTAs of one larger group
  int gh, head0, rem;
  if (idx < group_extra * big) {
    const int g = idx / big;
    rem = idx - g * big;
    gh = group_heads + 1;
    head0 = g * gh;
  } else {
    const int i2 = idx - group_extra * big;
    const int per = group_heads * n_blocks;
    const int g = i2 / per;
    rem = i2 - g * per;
    gh = group_heads;
    head0 = group_extra * (group_heads + 1) + g * group_heads;
  }
  jb = rem / gh;
  bh = head0 + rem % gh;
}

}  // namespace fat
