// page_walk.cuh -- which pages a warp of a partition kernel handles, and in what order.
//
// A CTA handles partitions [p_begin, p_end) of one (sequence, kv head). Either its warps
// share each partition (warp w of W takes pages f + w, f + w + W, ... of a partition whose
// first page is f) and walk the partitions one after the other, or each warp owns whole
// partitions (p_begin + w, p_begin + w + W, ...). The copy side of a warp walks its page list
// ahead of the compute side with IssueCursor, across partition boundaries, so the next
// partition's pages are already in flight while a partition is finished; the compute side
// walks the same list with the same counts (warp_pages).
//
// When warps own partitions, odd partitions are walked from their last page down. A partition
// that does not start on a page boundary (a window start) shares its first page with the end
// of the partition before it; with alternating directions the two warps that need such a page
// reach it at about the same time (both at the start, or both at the end, of their partitions),
// so the second read is served by L2 instead of a second read from DRAM.
#pragma once

#include "da_internal.cuh"

namespace da {

constexpr int kPageTokens = 16;

// Pages of a partition that warp w of W handles.
__device__ __forceinline__ int warp_pages(int npages, int w, int W) { return npages > w ? (npages - w + W - 1) / W : 0; }

// Index, within a partition's pages, of the k-th page of the warp's walk (n: the warp's page
// count there): pages page_off, page_off + page_step, ..., in reverse order when `rev`.
__device__ __forceinline__ int walk_page(int k, int n, int page_off, int page_step, bool rev) {
  return page_off + page_step * (rev ? n - 1 - k : k);
}

// Whether a warp walks partition p from its last page down (odd partitions, owned schedule).
__device__ __forceinline__ bool walk_reversed(bool owner, int p) { return owner && (p & 1); }

// First page and page count of a non-empty token range.
__device__ __forceinline__ void range_pages(const Range& r, int& first, int& npages) {
  first = r.start / kPageTokens;
  npages = (r.end - 1) / kPageTokens - first + 1;
}

// Walks the pages a warp copies: partitions p0, p0 + p_step, ... below p_end; in each, the
// pages first + page_off, first + page_off + page_step, ... (page_step W, page_off w when the
// warps of a CTA share a partition; 1 and 0 when a warp owns whole partitions).
struct IssueCursor {
  int b, L, lane;
  int p, p_step, p_end;   // partition of the cursor, stride between the warp's partitions, end
  int page_off, page_step;
  int i, n;               // index of the warp's next page in partition p, and its page count there
  int first;              // first page of partition p
  int bid;                // lane l: physical block of the warp's page (i & ~31) + l of partition p (-1 if none)
  bool more;              // a page is left at the cursor
  bool owner, rev;        // warps own partitions; partition p is walked in reverse

  __device__ __forceinline__ void load_bids(const Args& a) {
    const int k = (i & ~31) + lane;
    bid = k < n ? load_block(a, b, first + walk_page(k, n, page_off, page_step, rev)) : -1;
  }
  // Moves to the next of the warp's partitions that has pages for it (the first one when
  // p < p0 on entry).
  __device__ __forceinline__ void next_partition(const Args& a) {
    more = false;
    for (p += p_step; p < p_end; p += p_step) {
      int npages;
      range_pages(partition_range(L, a.T, p, a.window, a.psize, a.thresh), first, npages);
      n = warp_pages(npages, page_off, page_step);
      i = 0;
      rev = walk_reversed(owner, p);
      if (n > 0) {
        more = true;
        load_bids(a);
        return;
      }
    }
  }
  __device__ __forceinline__ void init(const Args& a, int b_, int L_, int p0, int p_step_, int p_end_, int page_off_,
                                       int page_step_, int lane_) {
    b = b_;
    L = L_;
    lane = lane_;
    p_step = p_step_;
    p = p0 - p_step;
    p_end = p_end_;
    page_off = page_off_;
    page_step = page_step_;
    owner = page_step_ == 1;  // a warp that takes every page of its partitions owns them
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
