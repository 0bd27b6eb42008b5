// item_walk.cuh -- the flattened work list walked by a persistent partition kernel.
//
// The work of one call is a list of items, in this order: for every sequence b, every kv head
// g, every partition p of b's attended span, every column group cg (eight (query token, head)
// pairs each) and every sub-item s < ksub, one item. With ksub > 1 (batches with few
// partitions) the pages of a partition are dealt round-robin to its ksub sub-items, each of
// which writes a partial of its own; the reduce combines them with the partition's others.
// The warps claim items from a counter in the workspace (one atomic add per item, issued one
// item ahead so its latency is hidden), so a warp that finishes early takes more: the work is
// spread evenly whatever the spread of the context lengths, and warps that are free at the same
// time take consecutive partitions of one (sequence, kv head). The last warp of the grid to run
// out of items puts the counters back to zero for the next call.
//
// The copy side of a warp walks its items ahead of the compute side (ItemIssue); when it
// reaches an item that has pages for the warp it records the item in a small ring in shared
// memory, from which the compute side takes it when it gets there (same warp: no cross-warp
// synchronisation). Items without pages for the warp (a sub-item past the last page of a
// short partition) are skipped by both sides and ignored by the reduce.
//
// Partition rules: turboquant-rs 0.4.1, src/cache/cuda/attention.rs, fused_attention()
// (PARTITION_SIZE, num_partitions = ceil(kv_len / PARTITION_SIZE)); attention.rs README, the
// sentence under the KV Cache Formats table (split-K from 1024 tokens of context).
#pragma once

#include "da_internal.cuh"
#include "page_walk.cuh"

namespace da {

// Ring entries per warp. The copy side is at most kStages + 1 pages ahead of the page being
// computed, each item holds at least one page, and the current item's entry is read again at its
// end: kRing must exceed kStages + 2 (kStages <= 6).
constexpr int kRing = 16;

// Per-CTA table of the batch's sequences in shared memory, built once at the kernel's start
// when it fits: entry b holds (first item of sequence b, its clamped length), entry B holds
// (item count, 0). A warp then finds the sequence of an item by a binary search in shared
// memory instead of walking the context lengths in global memory one sequence at a time.
struct SeqTable {
  uint32_t addr;  // shared address of entry 0 (8 bytes per entry)
  bool on;        // the table holds the whole batch
};

// Builds the table (all threads of the CTA; ends with a barrier). scratch: 32 words of shared memory.
__device__ __forceinline__ void build_seq_table(const Args& a, const SeqTable& t, uint32_t scratch, int per_part,
                                                int tid, int nthreads) {
  const int B = a.B, chunk = (B + nthreads - 1) / nthreads;
  const int c0 = min(tid * chunk, B), c1 = min(c0 + chunk, B);
  int sum = 0;  // items of the thread's sequences [c0, c1)
  for (int b = c0; b < c1; ++b) {
    const int L = load_len(a, b, true);
    sum += a.Hkv * seq_partitions(L, a.T, a.window, a.psize, a.thresh) * per_part;
  }
  // exclusive prefix over the threads: within the warp by shuffles, across warps in scratch
  const int lane = tid & 31, wid = tid >> 5;
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) asm volatile("st.shared.b32 [%0], %1;" ::"r"(scratch + 4 * wid), "r"(incl) : "memory");
  __syncthreads();
  int before = 0;
  for (int ww = 0; ww < wid; ++ww) {
    int x;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x) : "r"(scratch + 4 * ww) : "memory");
    before += x;
  }
  int first = before + incl - sum;
  for (int b = c0; b < c1; ++b) {
    const int L = load_len(a, b, false);
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(t.addr + 8 * b), "r"(first), "r"(L) : "memory");
    first += a.Hkv * seq_partitions(L, a.T, a.window, a.psize, a.thresh) * per_part;
  }
  if (c1 == B && c0 < c1 || (B == 0 && tid == 0))
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(t.addr + 8 * B), "r"(first), "r"(0) : "memory");
  __syncthreads();
}

// The sequence that holds a given item; items are only ever looked up in increasing order.
struct SeqCursor {
  int b;      // current sequence (-1 before the first)
  int base;   // its first item
  int count;  // its item count: Hkv * np * items_per_partition
  int L, np;  // its (clamped) length and partition count

  __device__ __forceinline__ void reset() {
    b = -1;
    base = count = L = np = 0;
  }
  // Moves to the sequence that holds item i; false when i is past the last item.
  __device__ __forceinline__ bool seek(const Args& a, const SeqTable& t, int i, int per_part) {
    if (i - base < count) return true;
    if (t.on) {  // binary search for the last sequence whose first item is <= i, among b+1 .. B-1
      int lo = b + 1, hi = a.B;  // the answer lies in [lo, hi); hi = B: past the last item
      uint32_t total;
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(total) : "r"(t.addr + 8 * a.B) : "memory");
      if (i >= (int)total) return false;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        int f;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(f) : "r"(t.addr + 8 * mid) : "memory");
        if (f <= i) lo = mid; else hi = mid;
      }
      int nf;
      asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(base), "=r"(L) : "r"(t.addr + 8 * lo) : "memory");
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(nf) : "r"(t.addr + 8 * (lo + 1)) : "memory");
      b = lo;
      count = nf - base;
      np = seq_partitions(L, a.T, a.window, a.psize, a.thresh);
      return true;
    }
    while (i - base >= count) {
      base += count;
      if (++b >= a.B) return false;
      L = load_len(a, b, true);
      np = seq_partitions(L, a.T, a.window, a.psize, a.thresh);
      count = a.Hkv * np * per_part;
    }
    return true;
  }
};

// One item: sequence, kv head, partition, column group, sub-item, the sequence's length and
// partition count.
struct Item {
  int b, g, p, cg, sub, L, np;
};

// Descriptor of an item in the ring (16 bytes).
__device__ __forceinline__ uint4 pack_item(const Item& it) {
  return make_uint4((uint32_t)it.b | ((uint32_t)it.g << 16), (uint32_t)it.p | ((uint32_t)it.cg << 16) |
                    ((uint32_t)it.sub << 20), (uint32_t)it.L, (uint32_t)it.np);
}
__device__ __forceinline__ Item unpack_item(const uint4& d) {
  return Item{(int)(d.x & 0xffffu), (int)(d.x >> 16), (int)(d.y & 0xffffu), (int)((d.y >> 16) & 15u),
              (int)(d.y >> 20), (int)d.z, (int)d.w};
}

// Pages of an item for its warp: the partition's first page, the warp's page count there and
// whether it walks them in reverse (odd partitions, when a partition is one item, so that the
// page two neighbouring partitions share is read by both warps at about the same time).
struct ItemPages {
  Range r;   // the partition's token range
  int first; // the partition's first page
  int n;     // pages of this sub-item: first + walk_page(k, n, sub, ksub, rev), k < n
  bool rev;
};
__device__ __forceinline__ ItemPages item_pages(const Args& a, const Item& it) {
  ItemPages ip;
  ip.r = partition_range_np(it.L, a.T, it.p, a.window, a.psize, it.np);
  int npages;
  range_pages(ip.r, ip.first, npages);
  ip.n = warp_pages(npages, it.sub, a.ksub);
  ip.rev = a.ksub == 1 && (it.p & 1);
  return ip;
}

// The copy side's walk over the warp's items and their pages. The hot state (the item's page
// walk) is held in registers, the same in every lane; the walk's position among the sequences
// (SeqCursor and the next item index) is kept in shared memory next to the ring, since it is
// only needed once per item. Lane 0 writes the ring and that state.
struct ItemIssue {
  int claimed;    // lane 0: the item index claimed for the warp's next item
  int b, g;       // sequence and kv head of the item at the cursor
  int pg0, pstep; // page index of the k-th page of its walk: pg0 + pstep * k
  int n, k;       // the walk's page count, index of the next page
  int bid;        // lane l: physical block of page (k & ~31) + l of the walk (-1 if none)
  bool more;      // a page is left at the cursor
  unsigned pushed;

  // Shared memory of a warp's walk: kRing descriptors, then SeqCursor.
  static constexpr int kStateBytes = kRing * 16 + 16;

  __device__ __forceinline__ void load_bids(const Args& a, int lane) {
    const int kk = (k & ~31) + lane;
    bid = kk < n ? load_block(a, b, pg0 + pstep * kk) : -1;
  }
  // Moves to the warp's next item that has pages for it and records it in the ring.
  __device__ __forceinline__ void next_item(const Args& a, const SeqTable& t, uint32_t ring, int lane) {
    __syncwarp();  // the state lane 0 wrote last time is visible to the warp
    const uint32_t st = ring + kRing * 16;
    SeqCursor seq;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(seq.b), "=r"(seq.base), "=r"(seq.L), "=r"(seq.np)
                 : "r"(st)
                 : "memory");
    const int per_part = a.ncg * a.ksub;
    seq.count = a.Hkv * seq.np * per_part;
    more = false;
    for (int next = __shfl_sync(0xffffffffu, claimed, 0); seq.seek(a, t, next, per_part);
         next = __shfl_sync(0xffffffffu, claimed, 0)) {
      if (lane == 0) claimed = (int)atomicAdd(a.claim, 1u);  // the item after this one
      Item it;
      int r = next - seq.base;
      const int per_head = seq.np * per_part;
      it.b = seq.b;
      it.L = seq.L;
      it.np = seq.np;
      it.g = r / per_head;
      r -= it.g * per_head;
      it.p = r / per_part;
      r -= it.p * per_part;
      it.cg = r / a.ksub;
      it.sub = r - it.cg * a.ksub;
      const ItemPages ip = item_pages(a, it);
      if (ip.n > 0) {
        b = it.b;
        g = it.g;
        n = ip.n;
        k = 0;
        pg0 = ip.first + it.sub + (ip.rev ? a.ksub * (ip.n - 1) : 0);
        pstep = ip.rev ? -a.ksub : a.ksub;
        if (lane == 0) {
          const uint4 d = pack_item(it);
          const uint32_t addr = ring + (pushed % kRing) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(d.x), "r"(d.y), "r"(d.z),
                       "r"(d.w)
                       : "memory");
        }
        ++pushed;
        load_bids(a, lane);
        more = true;
        break;
      }
    }
    if (lane == 0) {
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(st), "r"(seq.b), "r"(seq.base), "r"(seq.L),
                   "r"(seq.np)
                   : "memory");
    }
  }
  __device__ __forceinline__ void init(const Args& a, const SeqTable& t, uint32_t ring, int lane) {
    if (lane == 0) {  // no sequence yet; claim the first item
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ring + kRing * 16), "r"(-1), "r"(0), "r"(0),
                   "r"(0)
                   : "memory");
      claimed = (int)atomicAdd(a.claim, 1u);
    }
    pushed = 0;
    next_item(a, t, ring, lane);
  }
  // Physical block (-1: bad block id, nothing to load) of the page at the cursor, the same in
  // every lane; advances the cursor. Requires `more`.
  __device__ __forceinline__ int take(const Args& a, const SeqTable& t, uint32_t ring, int lane) {
    if (k > 0 && (k & 31) == 0) load_bids(a, lane);
    const int phys = __shfl_sync(0xffffffffu, bid, k & 31);
    if (++k == n) next_item(a, t, ring, lane);
    return phys;
  }
};

// A warp that has no items left counts itself out; the last warp of a grid of `warps` resets the
// item counter and the count for the next call (every warp claims its last item before it counts
// itself out, so no claim can follow the reset).
__device__ __forceinline__ void count_warp_out(const Args& a, unsigned warps, int lane) {
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(a.claim + 1, 1u) == warps - 1) {
      atomicExch(a.claim, 0u);
      atomicExch(a.claim + 1, 0u);
    }
  }
}

// The compute side's view of the ring: the descriptor of the warp's next item.
__device__ __forceinline__ Item ring_item(uint32_t ring, unsigned index) {
  uint4 d;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
               : "r"(ring + (index % kRing) * 16)
               : "memory");
  return unpack_item(d);
}

}  // namespace da
