// page_walk.cuh -- which pages a warp of a partition kernel handles, and in what order.
//
// A CTA handles the partitions [p_begin, p_end) of one (sequence, kv head), one after the
// other; inside a partition (first page f, n pages of 16 tokens) warp w of W takes pages
// f + w, f + w + W, ... The copy side of a warp walks this list ahead of the compute side
// with IssueCursor, across partition boundaries, so the next partition's pages are already
// in flight while a partition is merged; the compute side walks the same list with the same
// counts (warp_pages).
#pragma once

#include "da_internal.cuh"

namespace da {

constexpr int kPageTokens = 16;

// Pages of a partition that warp w of W handles.
__device__ __forceinline__ int warp_pages(int npages, int w, int W) { return npages > w ? (npages - w + W - 1) / W : 0; }

// First page and page count of a non-empty token range.
__device__ __forceinline__ void range_pages(const Range& r, int& first, int& npages) {
  first = r.start / kPageTokens;
  npages = (r.end - 1) / kPageTokens - first + 1;
}

template <int W>
struct IssueCursor {
  int b, L, w, lane;
  int p, p_end;  // partition of the cursor, end of the CTA's partitions
  int i, n;      // index of the warp's next page in partition p, and the warp's page count there
  int first;     // first page of partition p
  int bid;       // lane l: physical block of the warp's page (i & ~31) + l of partition p (-1 if none)
  bool more;     // a page is left at the cursor

  __device__ __forceinline__ void load_bids(const Args& a) {
    const int k = (i & ~31) + lane;
    bid = k < n ? load_block(a, b, first + w + W * k) : -1;
  }
  // Moves to the next partition that has pages for this warp.
  __device__ __forceinline__ void next_partition(const Args& a) {
    more = false;
    while (++p < p_end) {
      int npages;
      range_pages(partition_range(L, a.T, p, a.window, a.psize, a.thresh), first, npages);
      n = warp_pages(npages, w, W);
      i = 0;
      if (n > 0) {
        more = true;
        load_bids(a);
        return;
      }
    }
  }
  __device__ __forceinline__ void init(const Args& a, int b_, int L_, int p_begin, int p_end_, int w_, int lane_) {
    b = b_;
    L = L_;
    w = w_;
    lane = lane_;
    p = p_begin - 1;
    p_end = p_end_;
    next_partition(a);
  }
  // Physical block (-1: bad block id, nothing to load) of the page at the cursor, the same
  // in every lane; advances the cursor. Requires `more`.
  __device__ __forceinline__ int take(const Args& a) {
    if (i > 0 && (i & 31) == 0) load_bids(a);
    const int phys = __shfl_sync(0xffffffffu, bid, i & 31);
    if (++i == n) next_partition(a);
    return phys;
  }
};

}  // namespace da
