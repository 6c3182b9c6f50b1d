// Work schedule of the forward kernel, shared by the host (grid size) and the
// device (which query tile a block takes next).  A work item is one 128-row
// query tile of one (batch, head) -- one output row block per worker, the
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

}  // namespace fat
