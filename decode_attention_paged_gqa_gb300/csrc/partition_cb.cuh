// partition_cb.cuh -- split-K partition kernel for the formats whose values are stored as
// 4-bit codebook indices on the random-sign Walsh-Hadamard basis: 4-bit K and V, FP8 K +
// 4-bit V, 3-bit K + 4-bit V. Tensor-core MMAs on operands dequantised through a shared-
// memory lookup table.
//
// A persistent kernel: one CTA per SM (16 warps at D = 128 with up to four columns, else 8)
// builds the lookup tables once, then every warp claims items of the call's flattened item
// list (item_walk.cuh: one item per (sequence, kv head, partition, column group, sub-item)) one
// after the other from a counter until none is left, so the load is balanced whatever the
// context lengths and no warp ever waits for another. Each warp runs its own pipeline of shared-memory stages
// filled by TMA / bulk copies (a page's K codes, V codes and their per-token norms) and
// signalled on an mbarrier; it continues across its items, and a stage is refilled as soon as
// the page in it has been read into registers. Per page a warp computes, in the rotated basis
// (the keys' and values' own basis, no dequantisation to the original one):
//   S^T[16 tokens x 8 cols] = K_rot[16 x D] . Q_rot^T     then  s_t *= ||k_t||
//   O^T[D x 8 cols]        += V_rot^T[D x 16] . (P ||v||)^T
// with mma.m16n8k16 on f16 operands and fp32 accumulators, and at the end of an item writes
// its partial (output, max, sum) straight from registers; the reduce kernel combines the
// partials and un-rotates the output.
//
// A codebook operand is built from its codes with one byte permute and one shared-memory load
// per byte: a 256-entry table maps a byte (two 4-bit codes) to the f16 pair (cb[lo], cb[hi]) --
// for 3-bit keys a 64-entry table maps a 6-bit pair of codes. Entry e sits at byte 256 e and is
// replicated 32 times there, copy l in bank l, so the lanes of a warp never conflict whatever
// codes they look up. The table starts on a 64 KB boundary of the shared window, so the permute
// that extracts a byte (bits 8..15) and joins it with the lane's copy offset (4 l, bits 0..7)
// and the table's base (bits 16..31) gives the whole load address in one instruction.
//
// Columns: with up to four (query token, head) pairs the 8 MMA columns are pairs: column 2h
// carries pair h with the query's (and the probabilities') hi part, column 2h + 1 the lo part,
// so the thread that owns a pair's scores owns both halves (adding them is one register add)
// and each thread runs the online softmax of one pair over two tokens. With more pairs (8 per
// item) the lo parts take a second MMA / second column tile.
//
// The dot product's coordinate order is free, so each thread takes the coordinates that sit in
// a contiguous run of its key rows: thread (gid, tig) reads D/8 bytes of K rows gid and gid + 8,
// which hold the k-columns its A fragments need; Q^T's B fragments use the same coordinate
// order. For V^T (coordinates as the MMA's M) an m-tile's rows gid and gid + 8 are the two
// coordinates of one byte, and byte-wise logic pairs the codes of two tokens into one index.
//
// Precision: the rotated query is split q = q_hi + q_lo (both f16, after scaling by a power of
// two), so the scores carry only the rounding of the codebook values to f16 (2^-12 relative);
// P * ||v|| is split hi + lo the same way.
//
// (attention.rs README, KV Cache Formats table: the 4-bit Walsh-Hadamard codebook format and
// split-K decode for it; turboquant-rs 0.4.1, src/cache/cuda/attention.rs: the fused kernel
// reads the compressed cache as stored, with codebook and sign_pattern inputs, and writes
// partial output, max and sum per partition.)
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <mutex>

#include "da_internal.cuh"
#include "item_walk.cuh"
#include "kv_formats.cuh"
#include "page_softmax.cuh"
#include "page_walk.cuh"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kPage = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kSmemLimit = 227 * 1024;  // dynamic shared memory a CTA may use
// Shared address at which the dynamic shared memory of a kernel without static shared memory
// starts: the part of the CTA's window the system reserves (cudaDevAttrReservedSharedMemoryPerBlock,
// checked by the launcher).
constexpr int kDynStart = 1024;
constexpr int kLutAlign = 65536;  // the lookup tables start on a 64 KB boundary

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// KS: the key side (kSideCB4, kSideFP8, kSideCB3); values are 4-bit codes. NV: the CTA's
// columns, i.e. the group's (query token, head) pairs ("virtual heads" v = jq * G + h) padded
// to a power of two <= 8 (8 when more than 8 pairs are split into column groups).
template <int KS, int D, int NV>
struct Cb {
  static constexpr bool kPaired = NV <= 4;  // column 2h / 2h + 1: hi / lo part of pair h
  // 16 warps where 128 registers per thread suffice (D = 128, up to four pairs), else 8
  static constexpr int kWarps = (D == 128 && NV <= 4) ? 16 : 8;
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kKRow = row_bytes(KS, D);  // bytes of one key row
  static constexpr int kVRow = D / 2;             // bytes of one value row
  static constexpr int kKBytes = kPage * kKRow;
  static constexpr int kVBytes = kPage * kVRow;
  static constexpr bool kKNorms = KS != kSideFP8;  // per-token key norms
  // values by TMA: 64-byte rows with the 64-byte swizzle (D = 128), 128-byte rows with the
  // 128-byte swizzle (D = 256). Keys by TMA: FP8 in 128-byte swizzled slabs (read with
  // ldmatrix), 4-bit with the values' swizzle (one copy can then fetch both, the values right
  // behind the keys); 3-bit keys by a plain bulk copy (rows read unswizzled)
  static constexpr int kVAlign = D == 256 ? 1024 : 512;
  static constexpr int kKAlign = KS == kSideFP8 ? 1024 : KS == kSideCB4 ? kVAlign : 128;
  static constexpr int kAlign = kKAlign > kVAlign ? kKAlign : kVAlign;
  static constexpr int kOffV = align_up(kKBytes, kVAlign);          // V codes within a code stage
  static constexpr int kCodeBytes = align_up(kOffV + kVBytes, kAlign);
  static constexpr int kNormBytes = 128;                            // per stage: K norms, V norms
  static constexpr int kTxBytes = kKBytes + kVBytes + (kKNorms ? 64 : 0) + 64;
  // lookup tables: entry e at byte 256 e, the copy of lane l at + 4 l; the value table at the
  // first 64 KB boundary of the window, the 3-bit key table right behind it
  static constexpr int kLutV = 256 * 256;
  static constexpr int kLutK = KS == kSideCB3 ? 64 * 256 : 0;
  // Pages per stage (one mbarrier, one wait, one copy issue): two consecutive pages of the warp's
  // stream for 4-bit keys (measured faster), one for the other key sides (3-bit keys: measured
  // faster with one; FP8 keys, which the MMAs read from the stage, refill it after the MMAs).
  static constexpr int kSlots = KS == kSideCB4 ? 2 : 1;
  // Each warp's block: its pages' code and norm slots, walk state (ring) and mbarriers. The
  // blocks fill the space before the tables (region A) and after them (region B).
  static constexpr int block_bytes(int s) {
    return align_up(s * (kCodeBytes + kNormBytes) + ItemIssue::kStateBytes + 8 * (s / kSlots), kAlign);
  }
  static constexpr int kRegionA = kLutAlign - align_up(kDynStart, kAlign);
  static constexpr int kRegionB = kDynStart + kSmemLimit - kLutAlign - kLutV - kLutK;
  static constexpr bool fits(int s) {
    return s % kSlots == 0 && kRegionA / block_bytes(s) + kRegionB / block_bytes(s) >= kWarps;
  }
  static constexpr int kStages = fits(6) ? 6 : fits(5) ? 5 : fits(4) ? 4 : fits(3) ? 3 : 2;  // pages per warp
  static_assert(fits(kStages), "shared memory holds fewer than two pages per warp");
  static constexpr int kNStages = kStages / kSlots;  // stages (mbarriers) per warp
  static constexpr int kBlock = block_bytes(kStages);
  static constexpr int kOffNorms = kStages * kCodeBytes;  // within a block
  static constexpr int kOffRing = kOffNorms + kStages * kNormBytes;
  static constexpr int kOffBars = kOffRing + ItemIssue::kStateBytes;
  static constexpr int kSmem = kSmemLimit;
  static constexpr int kNT = kPaired ? 1 : 2;  // P.V column tiles (the second: lo parts)
  static constexpr int kMT = D / 16;           // O^T row tiles
  static constexpr int kKS = D / 16;           // k-steps of S^T
};

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float hi_f16(float p) { return __half2float(__float2half_rn(p)); }
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float ldsf(uint32_t addr) { return __uint_as_float(lds32(addr)); }
// The same at a constant byte offset from addr (the offset is the instruction's immediate).
template <int OFF>
__device__ __forceinline__ uint4 lds128_at(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64_at(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(addr), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds32_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ float ldsf_at(uint32_t addr) {
  return __uint_as_float(lds32_at<OFF>(addr));
}
// A load from the lookup tables, which no thread writes after the CTA's first barrier: not
// volatile, so the compiler may interleave the lookups with the work around them.
__device__ __forceinline__ uint32_t lds32_table(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// A lookup table as seen by one lane: the table's base (a multiple of 64 KB) joined with the
// lane's copy offset 4 * lane.
struct Lut {
  uint32_t lanebase;
};
// Entry (byte J of w) of the lane's copy: the permute takes bits 0..7 (lane offset) and 16..31
// (table base) from lanebase and puts the byte at bits 8..15.
template <int J>
__device__ __forceinline__ uint32_t lut_byte(const Lut& t, uint32_t w) {
  return lds32_table(__byte_perm(w, t.lanebase, 0x7604 | (J << 4)));
}
// byte J of a little-endian word array
template <int J>
__device__ __forceinline__ uint32_t lut_byte_of(const Lut& t, const uint32_t* w) {
  return lut_byte<J & 3>(t, w[J >> 2]);
}
// Entry (6-bit field J, bits 6J .. 6J + 5 of a little-endian word array) of the lane's copy:
// the field is moved to bits 8..13 by one shift, then masked and joined with lanebase.
template <int J>
__device__ __forceinline__ uint32_t lut_field6(const Lut& t, const uint32_t* w) {
  constexpr int bit = 6 * J, wi = bit >> 5, sh = bit & 31;
  uint32_t x;
  if constexpr (sh < 8)
    x = w[wi] << (8 - sh);
  else if constexpr (sh <= 26)
    x = w[wi] >> (sh - 8);
  else
    x = __funnelshift_r(w[wi], w[wi + 1], sh - 8);  // the field crosses into the next word
  return lds32_table((x & 0x3f00u) | t.lanebase);
}

// A fragments of S^T for k-step S from the thread's key bytes (rows gid: k0, gid + 8: k1).
template <int KS, int S>
__device__ __forceinline__ void key_frag(uint32_t (&af)[4], const uint32_t* k0, const uint32_t* k1, const Lut& lutk) {
  if constexpr (KS == kSideCB4) {
    af[0] = lut_byte_of<2 * S>(lutk, k0);
    af[1] = lut_byte_of<2 * S>(lutk, k1);
    af[2] = lut_byte_of<2 * S + 1>(lutk, k0);
    af[3] = lut_byte_of<2 * S + 1>(lutk, k1);
  } else {
    af[0] = lut_field6<2 * S>(lutk, k0);
    af[1] = lut_field6<2 * S>(lutk, k1);
    af[2] = lut_field6<2 * S + 1>(lutk, k0);
    af[3] = lut_field6<2 * S + 1>(lutk, k1);
  }
}

template <int S, int N, int KS, int NV>
struct KeySteps {
  // S^T += A(k-step S) . Q^T for S = S .. N-1 (compile-time unrolled so byte offsets are
  // constants), odd k-steps into sc1 so that the two dependent MMA chains are half as long
  __device__ static __forceinline__ void run(float (&sc0)[4], float (&sc1)[4], const uint32_t* k0, const uint32_t* k1,
                                             const Lut& lutk, const uint32_t (*qf)[2], const uint32_t (*ql)[2]) {
    if constexpr (S < N) {
      uint32_t af[4];
      key_frag<KS, S>(af, k0, k1, lutk);
      float(&sc)[4] = (S & 1) ? sc1 : sc0;
      ptx::mma_f16(sc, af, qf[S][0], qf[S][1]);
      if constexpr (NV == 8) ptx::mma_f16(sc, af, ql[S][0], ql[S][1]);
      KeySteps<S + 1, N, KS, NV>::run(sc0, sc1, k0, k1, lutk, qf, ql);
    }
  }
};

template <int M, int N, int D, int NT>
struct ValueTiles {
  // O^T[m-tile M] += V^T(m-tile M) . P^T for M = M .. N-1. vx[r]: table indices, byte M of
  // word array r: r = 0 / 1: the low / high nibbles of tokens (2 tig, 2 tig + 1) paired, r =
  // 2 / 3 the same for tokens (2 tig + 8, 2 tig + 9); one lookup gives an A register.
  __device__ static __forceinline__ void run(float (&o)[NT][D / 16][4], const uint32_t (*vx)[D / 64], const Lut& lutv,
                                             const uint32_t (&pb)[NT][2]) {
    if constexpr (M < N) {
      const uint32_t af[4] = {lut_byte_of<M>(lutv, vx[0]), lut_byte_of<M>(lutv, vx[1]), lut_byte_of<M>(lutv, vx[2]),
                              lut_byte_of<M>(lutv, vx[3])};
#pragma unroll
      for (int t = 0; t < NT; ++t) ptx::mma_f16(o[t][M], af, pb[t][0], pb[t][1]);
      ValueTiles<M + 1, N, D, NT>::run(o, vx, lutv, pb);
    }
  }
};

// The thread's score columns of an item: the (query token, head) pair of each, its query
// position, and the positions it attends within the partition, [lo, hi) (causal limit and
// window). Paired layout: one pair (columns 2 tig, 2 tig + 1); else two (2 tig + j).
struct Cols {
  int lo[2], hi[2], pos[2], vh[2];
};
template <int NV>
__device__ __forceinline__ Cols item_cols(const Args& a, const Item& it, const Range& r, int tig, int G) {
  const int vbase = 8 * it.cg, V = min(NV, a.T * G - vbase);
  Cols c;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    c.vh[j] = vbase + (NV <= 4 ? tig % V : (2 * tig + j) % V);
    c.pos[j] = it.L - a.T + (c.vh[j] >> a.g_shift);
    c.lo[j] = max(window_start(c.pos[j], a.window), r.start);
    c.hi[j] = min(c.pos[j] + 1, r.end);
  }
  return c;
}

// CAP: softcap on (a separate instantiation, so the plain kernel carries no tanh). PAIR: the
// launcher found one 3-D map for the K and V codes (4-bit keys) and one for the two norm arrays
// (codebook keys), so the copy issue has no runtime branch on them.
template <int KS, int D, int NV, bool CAP, bool PAIR>
__global__ void __launch_bounds__(Cb<KS, D, NV>::kThreads, 1)
    partition_cb_kernel(const Args a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap nmap) {
  using C = Cb<KS, D, NV>;
  constexpr int kWarps = C::kWarps, kThreads = C::kThreads;
  constexpr bool kPaired = C::kPaired;
  // the warp index through a shuffle from lane 0, which the compiler then treats as uniform
  const int tid = threadIdx.x, lane = tid & 31, w = __shfl_sync(kFull, tid >> 5, 0);
  const int gid = lane >> 2, tig = lane & 3;
  const int G = a.Hq / a.Hkv;
  ptx::grid_dependency_wait();    // what the kernel before this one writes (q, the rotated q, ...)
  ptx::grid_dependents_launch();  // the reduce may be scheduled once every CTA has started

  // ---- shared memory: the lookup tables at the first 64 KB boundary of the window, the warps'
  //      blocks before them (region A) and after them (region B)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t start = ptx::smem_u32(smem_raw);
  const uint32_t tbl = (start + (kLutAlign - 1)) & ~uint32_t(kLutAlign - 1);
  const uint32_t a0 = (start + (C::kAlign - 1)) & ~uint32_t(C::kAlign - 1);
  const int in_a = tbl > a0 ? (int)((tbl - a0) / C::kBlock) : 0;
  const uint32_t blk = w < in_a ? a0 + w * C::kBlock : tbl + C::kLutV + C::kLutK + (w - in_a) * C::kBlock;
  if (blk + C::kBlock > start + C::kSmem || tbl + C::kLutV + C::kLutK > start + C::kSmem) {
    if (tid == 0) atomicOr(a.err, DA_DEVERR_SMEM_LAYOUT);  // the launcher checks this never happens
    count_warp_out(a, gridDim.x * kWarps, lane);
    return;
  }
  const uint32_t code0 = blk, norm0 = blk + C::kOffNorms, ring = blk + C::kOffRing, bar0 = blk + C::kOffBars;
  // the batch's sequence table, in the space after the last block of region B when it fits
  SeqTable seqs;
  {
    const int in_b = kWarps - (in_a < kWarps ? in_a : kWarps);
    const uint32_t scratch = tbl + C::kLutV + C::kLutK + in_b * C::kBlock;
    seqs.addr = scratch + 128;
    seqs.on = (long long)seqs.addr + 8ll * (a.B + 1) <= (long long)start + C::kSmem;
    if (seqs.on) build_seq_table(a, seqs, scratch, a.ncg * a.ksub, tid, kThreads);
  }

  if (lane == 0) {
    ptx::prefetch_tensor_map(&kmap);
    if (!(PAIR || a.kv_pair)) ptx::prefetch_tensor_map(&vmap);
    if (PAIR || a.kn_pair) ptx::prefetch_tensor_map(&nmap);
    for (int s = 0; s < C::kNStages; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  // offsets within a code stage of the 4-bit K and V codes, and within a norm slot of the two
  // norm vectors (the side with the lower address first when one map spans both)
  const uint32_t koff = (KS == kSideCB4 && a.kv_zk) ? C::kOffV : 0;
  const uint32_t voff = KS == kSideCB4 ? C::kOffV - koff : C::kOffV;
  const uint32_t knoff = a.kn_zk ? 64 : 0;
  const uint32_t vnoff = C::kKNorms ? 64 - knoff : 0;

  // ---- the warp's items and their pages, copied kStages pages ahead of the compute
  ItemIssue cur;
  cur.init(a, seqs, ring, lane);
  unsigned issued = 0;  // stages issued
  int is = 0;           // stage of the next copies (issued % kNStages)
  auto issue_next = [&]() {  // all lanes; lane 0 issues the copies of the next kSlots pages
    int gk[C::kSlots], phys[C::kSlots], n = 0;
#pragma unroll
    for (int j = 0; j < C::kSlots; ++j)
      if (j == 0 || cur.more) {
        gk[j] = cur.g;
        phys[j] = cur.take(a, seqs, ring, lane);
        n = j + 1;
      }
    const int s = is;
    is = is + 1 == C::kNStages ? 0 : is + 1;
    ++issued;
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * s;
      ptx::fence_proxy_async();
      ptx::mbar_arrive_expect_tx(bar, n * C::kTxBytes);
#pragma unroll
      for (int j = 0; j < C::kSlots; ++j) {
        if (j >= n) break;
        const uint32_t dst = code0 + (s * C::kSlots + j) * C::kCodeBytes;
        const uint32_t ndst = norm0 + (s * C::kSlots + j) * C::kNormBytes;
        // a bad block id (flagged by the walk) reads block 0 in its place: the affected outputs
        // are unspecified, as the interface states
        const size_t unit = (size_t)(phys[j] < 0 ? 0 : phys[j]) * a.Hkv + gk[j];  // (block, kv head): 16 rows
        const int y = (int)unit * kPage;
        if constexpr (KS == kSideCB4) {  // codes of K and V: one copy when one map spans both
          if (PAIR || a.kv_pair) {
            ptx::tma_load_3d(dst, &kmap, 0, y, 0, bar);
          } else {
            ptx::tma_load_2d(dst + koff, &kmap, 0, y, bar);
            ptx::tma_load_2d(dst + voff, &vmap, 0, y, bar);
          }
        } else {
          if constexpr (KS == kSideFP8) {
#pragma unroll
            for (int u = 0; u < D / 128; ++u) ptx::tma_load_2d(dst + u * 2048, &kmap, u * 128, y, bar);
          } else {
            ptx::bulk_load(dst, static_cast<const uint8_t*>(a.k_cache) + unit * C::kKBytes, C::kKBytes, bar);
          }
          ptx::tma_load_2d(dst + C::kOffV, &vmap, 0, y, bar);
        }
        if constexpr (C::kKNorms) {  // per-token norms of K and V: one copy when one map spans both
          if (PAIR || a.kn_pair) {
            ptx::tma_load_3d(ndst, &nmap, 0, (int)unit, 0, bar);
          } else {
            ptx::bulk_load(ndst + knoff, a.k_scales + unit * kPage, 64, bar);
            ptx::bulk_load(ndst + vnoff, a.v_scales + unit * kPage, 64, bar);
          }
        } else {
          ptx::bulk_load(ndst, a.v_scales + unit * kPage, 64, bar);
        }
      }
    }
  };
  for (int k = 0; k < C::kNStages && cur.more; ++k) issue_next();

  // ---- lookup tables: byte -> (cb[lo], cb[hi]) for values (and 4-bit keys), 6-bit pair ->
  //      (cbk[lo], cbk[hi]) for 3-bit keys; entry e at word 64 e, 32 copies (word 64 e + l)
  {
    const float* cbv = a.codebook + (KS == kSideCB3 ? 8 : 0);
    uint32_t* lv = reinterpret_cast<uint32_t*>(smem_raw + (tbl - start));
    for (int i = tid; i < 256 * 8; i += kThreads) {
      const int e = i >> 3;
      const uint32_t x = pack_f16(__ldg(cbv + (e & 15)), __ldg(cbv + (e >> 4)));
      *reinterpret_cast<uint4*>(lv + e * 64 + (i & 7) * 4) = make_uint4(x, x, x, x);
    }
    if constexpr (KS == kSideCB3) {
      uint32_t* lk = lv + C::kLutV / 4;
      for (int i = tid; i < 64 * 8; i += kThreads) {
        const int e = i >> 3;
        const uint32_t x = pack_f16(__ldg(a.codebook + (e & 7)), __ldg(a.codebook + (e >> 3)));
        *reinterpret_cast<uint4*>(lk + e * 64 + (i & 7) * 4) = make_uint4(x, x, x, x);
      }
    }
  }
  const Lut lutv{tbl | (4u * lane)};
  const Lut lutk{(KS == kSideCB3 ? tbl + C::kLutV : tbl) | (4u * lane)};
  __syncthreads();  // lookup tables written; from here on no warp waits for another

  const float cap = a.softcap;
  const float cap_pre = CAP ? 1.0f / (cap * kLog2e) : 0.0f;  // log2-domain score -> s_nat / cap
  const float cap_post = cap * kLog2e;
  const bool alibi = a.alibi != nullptr;
  const int PK = a.P * a.ksub;  // partial slots per output row
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix (FP8 keys): matrix index and row of this lane's address
  unsigned consumed = 0, stall_from = 0, popped = 0;  // pages computed; stage of a stall
  // the page in registers: this lane's byte offsets within a code slot and a norm slot (the
  // rest of each load's address is an immediate). 4-bit keys at D = 128 (64-byte rows, 64-byte
  // swizzle: chunk c of row r at c ^ ((r >> 1) & 3)): row gid, chunk tig, and row gid + 8 at
  // +512, whose swizzle is the same. Values at D = 128: rows 2 tig + {0, 1, 8, 9} at + {0, 64,
  // 512, 576}, all with the swizzle term (row >> 1) & 3 = tig, the 8 bytes at 8 (gid & 1) of
  // chunk (gid >> 1) ^ tig. 3-bit keys: the row's 3D/32 bytes at (3D/32) tig, row gid + 8 at
  // + 8 kKRow. Norms: tokens gid and gid + 8 (+ 32) of each vector.
  const uint32_t lane_k = KS == kSideCB4 ? koff + gid * 64 + ((tig ^ ((gid >> 1) & 3)) << 4)
                                         : gid * C::kKRow + (3 * D / 32) * tig;
  const uint32_t lane_v = voff + 2 * tig * 64 + (((gid >> 1) ^ tig) << 4) + 8 * (gid & 1);
  const uint32_t lane_kn = knoff + 4 * gid, lane_vn = vnoff + 4 * gid;
  int cpage = 0;      // slot of the next page to compute among the warp's kStages (consumed % kStages)
  uint32_t cph = 0;   // the mbarrier phase parity of its stage
  bool stalled = false;  // a copy never arrived: no more waits, copies or compute
  int q_b = -1, q_g = -1, q_cg = -1;  // (sequence, kv head, column group) of the loaded query fragments
  uint32_t qf[C::kKS][2], ql[kPaired ? 1 : C::kKS][2];
  float score_scale = 0.0f;

  while (!stalled) {
    __syncwarp();  // the ring entry written by lane 0 is visible to the warp
    if (popped == cur.pushed) break;  // no item left for this warp
    const Item it = ring_item(ring, popped++);
    const ItemPages ip = item_pages(a, it);
    const int b = it.b, g = it.g;
    // the item's columns: virtual heads vbase .. vbase + V - 1
    const int vbase = 8 * it.cg, V = min(NV, a.T * G - vbase);

    // ---- query fragments (B operand of S^T). Paired: column n holds pair (n / 2) % V, its hi
    //      part for even n, its lo part for odd n; else column n holds pair n % V (hi part) and
    //      a second set of fragments the lo parts.
    if (b != q_b || g != q_g || it.cg != q_cg) {
      q_b = b, q_g = g, q_cg = it.cg;
      const int qv = vbase + (kPaired ? (gid >> 1) % V : gid % V);
      const size_t qrow = query_row(a, b, g, G, qv) * D;
      if constexpr (KS == kSideFP8) {
        // unrotated bf16 query, scaled by a power of two into the f16 range (exact)
        const uint16_t* qp = a.q + qrow;
        float x[C::kKS][4];
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[ks][e] = bf16_to_f32(qp[16 * ks + 4 * tig + e]);
            mx = fmaxf(mx, fabsf(x[ks][e]));
          }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        int ex = 0;
        frexpf(mx, &ex);
        const int e2 = ex > 14 ? 14 - ex : 0;
        const float qs = ldexpf(1.0f, e2);
        // bf16 values fit f16 exactly after the scaling: the lo parts are zero
        const bool lo_col = kPaired && (gid & 1);
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          qf[ks][0] = lo_col ? 0u : pack_f16(x[ks][0] * qs, x[ks][1] * qs);
          qf[ks][1] = lo_col ? 0u : pack_f16(x[ks][2] * qs, x[ks][3] * qs);
          if constexpr (!kPaired) ql[ks][0] = ql[ks][1] = 0u;
        }
        score_scale = a.scale * __ldg(a.k_scales) * ldexpf(1.0f, -e2) * kLog2e;
      } else {
        // rotated fp32 query: coordinates (D/4) tig + 4 ks + {0, 1} (b0) and + {2, 3} (b1),
        // scaled by 2^e2 (max below 2^15) and split into f16 hi + lo
        const float4* qp = reinterpret_cast<const float4*>(a.q_rot + qrow + (D / 4) * tig);
        float4 x[C::kKS];
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          x[ks] = qp[ks];
          mx = fmaxf(fmaxf(mx, fmaxf(fabsf(x[ks].x), fabsf(x[ks].y))), fmaxf(fabsf(x[ks].z), fabsf(x[ks].w)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        int ex = 0;
        frexpf(mx, &ex);
        const int e2 = 15 - ex;
        const float qs = ldexpf(1.0f, e2);
        const bool lo_col = kPaired && (gid & 1);
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
          const float y0 = x[ks].x * qs, y1 = x[ks].y * qs, y2 = x[ks].z * qs, y3 = x[ks].w * qs;
          const float h0 = hi_f16(y0), h1 = hi_f16(y1), h2 = hi_f16(y2), h3 = hi_f16(y3);
          if constexpr (kPaired) {
            qf[ks][0] = lo_col ? pack_f16(y0 - h0, y1 - h1) : pack_f16(h0, h1);
            qf[ks][1] = lo_col ? pack_f16(y2 - h2, y3 - h3) : pack_f16(h2, h3);
          } else {
            qf[ks][0] = pack_f16(h0, h1);
            qf[ks][1] = pack_f16(h2, h3);
            ql[ks][0] = pack_f16(y0 - h0, y1 - h1);
            ql[ks][1] = pack_f16(y2 - h2, y3 - h3);
          }
        }
        score_scale = a.scale * ldexpf(1.0f, -e2) * kLog2e;
      }
    }

    // the pages no column masks: tokens [lo_all, hi_all) (warp-uniform); first token of the
    // k-th page of the item's walk: tk0 + k * tkstep
    int lo_all, hi_all;
    {
      const Cols c = item_cols<NV>(a, it, ip.r, tig, G);
      lo_all = max(c.lo[0], c.lo[1]);
      hi_all = min(c.hi[0], c.hi[1]);
      lo_all = max(lo_all, __shfl_xor_sync(kFull, lo_all, 1));
      lo_all = max(lo_all, __shfl_xor_sync(kFull, lo_all, 2));
      hi_all = min(hi_all, __shfl_xor_sync(kFull, hi_all, 1));
      hi_all = min(hi_all, __shfl_xor_sync(kFull, hi_all, 2));
    }
    const int tk0 = (ip.first + it.sub + (ip.rev ? a.ksub * (ip.n - 1) : 0)) * kPage;
    const int tkstep = (ip.rev ? -a.ksub : a.ksub) * kPage;
    const int n_pages = ip.n;

    // ---- running state. Paired: one (m, l) per thread (its pair); else one per column j.
    //      O^T is kept in units of 2^(ev_run - 127): ev_run is the largest biased binary32
    //      exponent of the value norms seen so far, so P * ||v|| * 2^(127 - ev_run) <
    //      2^(kLazyLog2 + 1) fits f16.
    float m_run[2] = {kNoMax, kNoMax}, l_run[2] = {0.0f, 0.0f};
    if constexpr (!kPaired) m_run[0] = m_run[1] = -INFINITY;
    float o[C::kNT][C::kMT][4];
#pragma unroll
    for (int t = 0; t < C::kNT; ++t)
#pragma unroll
      for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[t][mt][e] = 0.0f;
    int ev_run = 0;
    float v_unit = 1.0f;  // 2^(127 - ev_run)

    for (int i = 0; i < n_pages; ++i, ++consumed) {
      // page `consumed` of the warp's stream: slot `slot` of stage s, whose mbarrier phase has
      // parity `parity`, page slot pg = s * kSlots + slot of the warp's block; at D = 128 from
      // counters kept alongside (cheaper than dividing), at D = 256 from `consumed` (the
      // 8-column kernels there have no registers to spare)
      const unsigned use = consumed / C::kSlots;
      const int slot = D == 128 ? cpage % C::kSlots : (int)(consumed % C::kSlots);
      const int s = D == 128 ? cpage / C::kSlots : (int)(use % C::kNStages);
      const int pg = D == 128 ? cpage : s * C::kSlots + slot;
      const uint32_t parity = D == 128 ? cph : (use / C::kNStages) & 1;
      if constexpr (D == 128) {
        if (++cpage == C::kStages) {
          cpage = 0;
          cph ^= 1u;
        }
      }
      if (slot == 0 && !ptx::mbar_wait(bar0 + 8 * s, parity)) {
        stalled = true;
        stall_from = consumed / C::kSlots;
        break;
      }
      const uint32_t cb0 = code0 + pg * C::kCodeBytes, kb = cb0 + koff, vb = cb0 + voff;
      const uint32_t nb = norm0 + pg * C::kNormBytes;
      const int tok0 = tk0 + i * tkstep;

      // -- the page into registers: key bytes (codebook keys), value bytes, norms
      constexpr int kWords = KS == kSideCB4 ? D / 32 : KS == kSideCB3 ? 3 * D / 128 : 1;
      uint32_t k0[kWords + 1], k1[kWords + 1];
      k0[kWords] = k1[kWords] = 0u;
      if constexpr (KS == kSideCB4 && D == 128) {
        const uint4 x0 = lds128_at<0>(cb0 + lane_k), x1 = lds128_at<512>(cb0 + lane_k);
        k0[0] = x0.x, k0[1] = x0.y, k0[2] = x0.z, k0[3] = x0.w;
        k1[0] = x1.x, k1[1] = x1.y, k1[2] = x1.z, k1[3] = x1.w;
      } else if constexpr (KS == kSideCB4) {  // D = 256, 128-byte swizzle: chunks 2 tig, 2 tig + 1
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int ch = 2 * tig + c;
          const uint4 x0 = lds128(kb + gid * 128 + ((ch ^ gid) << 4));
          const uint4 x1 = lds128(kb + (gid + 8) * 128 + ((ch ^ gid) << 4));  // (gid + 8) & 7 == gid
          k0[4 * c] = x0.x, k0[4 * c + 1] = x0.y, k0[4 * c + 2] = x0.z, k0[4 * c + 3] = x0.w;
          k1[4 * c] = x1.x, k1[4 * c + 1] = x1.y, k1[4 * c + 2] = x1.z, k1[4 * c + 3] = x1.w;
        }
      } else if constexpr (KS == kSideCB3) {  // 12 (D = 128) or 24 (D = 256) bytes per row at (3D/32) tig
        if constexpr (D == 128) {
          const uint32_t kl = kb + lane_k;
          k0[0] = lds32_at<0>(kl), k0[1] = lds32_at<4>(kl), k0[2] = lds32_at<8>(kl);
          k1[0] = lds32_at<8 * C::kKRow>(kl), k1[1] = lds32_at<8 * C::kKRow + 4>(kl);
          k1[2] = lds32_at<8 * C::kKRow + 8>(kl);
        } else {
#pragma unroll
          for (int c = 0; c < kWords; ++c) {
            k0[c] = lds32(kb + gid * C::kKRow + (3 * D / 32) * tig + 4 * c);
            k1[c] = lds32(kb + (gid + 8) * C::kKRow + (3 * D / 32) * tig + 4 * c);
          }
        }
      }
      // the thread's value bytes of tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9, D/16 bytes
      // each at byte (D/16) gid
      uint32_t vw[4][D / 64];
      if constexpr (D == 128) {  // 64-byte rows, 64-byte swizzle
        const uint32_t vl = cb0 + lane_v;
        const uint2 x0 = lds64_at<0>(vl), x1 = lds64_at<64>(vl), x2 = lds64_at<512>(vl), x3 = lds64_at<576>(vl);
        vw[0][0] = x0.x, vw[0][1] = x0.y, vw[1][0] = x1.x, vw[1][1] = x1.y;
        vw[2][0] = x2.x, vw[2][1] = x2.y, vw[3][0] = x3.x, vw[3][1] = x3.y;
      } else {
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {  // 128-byte rows, 128-byte swizzle
          const int row = 2 * tig + (i4 & 1) + 8 * (i4 >> 1);
          const uint4 x = lds128(vb + row * 128 + ((gid ^ (row & 7)) << 4));
          vw[i4][0] = x.x, vw[i4][1] = x.y, vw[i4][2] = x.z, vw[i4][3] = x.w;
        }
      }
      float kn0 = 1.0f, kn1 = 1.0f;
      float vn0, vn1;
      if constexpr (D == 128) {
        if constexpr (C::kKNorms) {
          kn0 = ldsf_at<0>(nb + lane_kn);
          kn1 = ldsf_at<32>(nb + lane_kn);
        }
        vn0 = ldsf_at<0>(nb + lane_vn), vn1 = ldsf_at<32>(nb + lane_vn);
      } else {  // (the 8-column kernels at D = 256 have no registers to spare for the offsets)
        if constexpr (C::kKNorms) {
          kn0 = ldsf(nb + knoff + 4 * gid);
          kn1 = ldsf(nb + knoff + 4 * (gid + 8));
        }
        vn0 = ldsf(nb + vnoff + 4 * gid), vn1 = ldsf(nb + vnoff + 4 * (gid + 8));
      }
      // FP8 keys are read with ldmatrix during the MMAs below, so their stage is refilled after
      if constexpr (KS != kSideFP8) {
        if (slot == C::kSlots - 1) {  // the stage's last page is in registers
          __syncwarp();                // every lane has read the stage
          if (cur.more) issue_next();
        }
      }

      {
        // -- S^T = K . Q^T, the k-steps alternating between two accumulators (two dependent MMA
        //    chains of half the length), added at the end
        float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (KS == kSideFP8) {
#pragma unroll
          for (int j2 = 0; j2 < C::kKS / 2; ++j2) {
            const int row = ri + 8 * (mi & 1), chunk = 2 * j2 + (mi >> 1);
            uint32_t rr[4];
            ptx::ldmatrix_x4(rr, kb + (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
            const uint32_t a0[4] = {e4m3x2_to_f16x2(rr[0]), e4m3x2_to_f16x2(rr[1]), e4m3x2_to_f16x2(rr[0] >> 16),
                                    e4m3x2_to_f16x2(rr[1] >> 16)};
            ptx::mma_f16(sc, a0, qf[2 * j2][0], qf[2 * j2][1]);
            const uint32_t a1[4] = {e4m3x2_to_f16x2(rr[2]), e4m3x2_to_f16x2(rr[3]), e4m3x2_to_f16x2(rr[2] >> 16),
                                    e4m3x2_to_f16x2(rr[3] >> 16)};
            ptx::mma_f16(sc2, a1, qf[2 * j2 + 1][0], qf[2 * j2 + 1][1]);
          }
        } else {
          KeySteps<0, C::kKS, KS, kPaired ? 1 : 8>::run(sc, sc2, k0, k1, lutk, qf, ql);
        }
        const float ss0 = score_scale * kn0, ss1 = score_scale * kn1;
        float alpha[2], pv[4];
        bool rescale;
        if constexpr (kPaired) {
          // -- the pair's scores of tokens gid and gid + 8: hi + lo columns, scale (and key
          //    norm), softcap, ALiBi, mask
          float sp[2] = {((sc[0] + sc2[0]) + (sc[1] + sc2[1])) * ss0, ((sc[2] + sc2[2]) + (sc[3] + sc2[3])) * ss1};
          if constexpr (CAP) {
#pragma unroll
            for (int e = 0; e < 2; ++e) sp[e] = cap_post * tanhf(sp[e] * cap_pre);
          }
          if (alibi || tok0 < lo_all || tok0 + kPage > hi_all) {
            // the column's limits and position again, from the item's ring entry (rare pages)
            const Item it2 = ring_item(ring, popped - 1);
            const Cols c = item_cols<NV>(a, it2, partition_range_np(it2.L, a.T, it2.p, a.window, a.psize, it2.np),
                                         tig, G);
            if (alibi) {  // + slope * (t - pos) for token t
              const float slope = __ldg(a.alibi + it2.g * G + (c.vh[0] & (G - 1))) * kLog2e;
#pragma unroll
              for (int e = 0; e < 2; ++e) sp[e] += slope * (float)(tok0 + gid + 8 * e - c.pos[0]);
            }
            if (tok0 < lo_all || tok0 + kPage > hi_all) mask_page_col(sp, tok0, gid, c.lo[0], c.hi[0]);
          }
          // -- online softmax of the pair (lazily moved reference max)
          float pr[2];
          rescale = page_softmax_col(sp, m_run[0], l_run[0], alpha[0], pr);
          alpha[1] = alpha[0];
          pv[0] = pr[0] * vn0;
          pv[1] = pr[1] * vn1;
        } else {
          // -- two columns per thread: hi + lo fragments were added by the MMAs
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[e] += sc2[e];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float y = sc[e] * ((e >> 1) ? ss1 : ss0);
            sc[e] = CAP ? cap_post * tanhf(y * cap_pre) : y;
          }
          if (alibi || tok0 < lo_all || tok0 + kPage > hi_all) {
            const Item it2 = ring_item(ring, popped - 1);
            const Cols c = item_cols<NV>(a, it2, partition_range_np(it2.L, a.T, it2.p, a.window, a.psize, it2.np),
                                         tig, G);
            if (alibi) {  // + slope * (t - pos) for token t of each element
#pragma unroll
              for (int e = 0; e < 4; ++e)
                sc[e] += __ldg(a.alibi + it2.g * G + (c.vh[e & 1] & (G - 1))) * kLog2e *
                         (float)(tok0 + gid + (e >> 1) * 8 - c.pos[e & 1]);
            }
            if (tok0 < lo_all || tok0 + kPage > hi_all) mask_page(sc, tok0, gid, c.lo, c.hi);
          }
          float pr[4];
          rescale = page_softmax(sc, m_run, l_run, alpha, pr);
#pragma unroll
          for (int e = 0; e < 4; ++e) pv[e] = pr[e] * ((e >> 1) ? vn1 : vn0);
        }
        // -- a larger value-norm exponent on this page rescales O^T by the same exact power of two
        int ev = (int)(__float_as_uint(fmaxf(fabsf(vn0), fabsf(vn1))) >> 23);
        if (__any_sync(kFull, ev > ev_run)) {  // the warp's max
          ev = max(ev, __shfl_xor_sync(kFull, ev, 4));
          ev = max(ev, __shfl_xor_sync(kFull, ev, 8));
          ev = max(ev, __shfl_xor_sync(kFull, ev, 16));
          const float f = ldexpf(1.0f, ev_run - ev);
          alpha[0] *= f;
          alpha[1] *= f;
          ev_run = ev;
          v_unit = ldexpf(1.0f, 127 - ev);
          rescale = true;
        }
        if (rescale) {
#pragma unroll
          for (int t = 0; t < C::kNT; ++t)
#pragma unroll
            for (int mt = 0; mt < C::kMT; ++mt) {
              o[t][mt][0] *= alpha[0];
              o[t][mt][1] *= alpha[1];
              o[t][mt][2] *= alpha[0];
              o[t][mt][3] *= alpha[1];
            }
        }
        // -- (P * value norms)^T as the B operand, split hi + lo, transposed with movmatrix
        uint32_t pb[C::kNT][2];
        if constexpr (kPaired) {
          // C layout (token gid: columns 2 tig, 2 tig + 1) = (hi, lo) of the pair's value
          const float x0 = pv[0] * v_unit, x1 = pv[1] * v_unit;
          const float h0 = hi_f16(x0), h1 = hi_f16(x1);
          pb[0][0] = ptx::movmatrix_trans(pack_f16(h0, x0 - h0));
          pb[0][1] = ptx::movmatrix_trans(pack_f16(h1, x1 - h1));
        } else {
          float hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x = pv[e] * v_unit;
            hi[e] = hi_f16(x);
            lo[e] = x - hi[e];
          }
          pb[0][0] = ptx::movmatrix_trans(pack_f16(hi[0], hi[1]));
          pb[0][1] = ptx::movmatrix_trans(pack_f16(hi[2], hi[3]));
          pb[C::kNT - 1][0] = ptx::movmatrix_trans(pack_f16(lo[0], lo[1]));
          pb[C::kNT - 1][1] = ptx::movmatrix_trans(pack_f16(lo[2], lo[3]));
        }
        // -- O^T += V^T . P^T: byte b of token t holds coordinates 2b (low nibble) and 2b + 1
        //    (high nibble); pair tokens t, t + 1 into the index (code_t | code_t+1 << 4) of the
        //    table, whose entry is then the A register (v_t, v_t+1) of one coordinate
        uint32_t vx[4][D / 64];
#pragma unroll
        for (int k = 0; k < D / 64; ++k) {
          vx[0][k] = (vw[0][k] & 0x0f0f0f0fu) | ((vw[1][k] << 4) & 0xf0f0f0f0u);
          vx[1][k] = ((vw[0][k] >> 4) & 0x0f0f0f0fu) | (vw[1][k] & 0xf0f0f0f0u);
          vx[2][k] = (vw[2][k] & 0x0f0f0f0fu) | ((vw[3][k] << 4) & 0xf0f0f0f0u);
          vx[3][k] = ((vw[2][k] >> 4) & 0x0f0f0f0fu) | (vw[3][k] & 0xf0f0f0f0u);
        }
        ValueTiles<0, C::kMT, D, C::kNT>::run(o, vx, lutv, pb);
      }
      if constexpr (KS == kSideFP8) {
        __syncwarp();  // every lane has read the stage
        if (cur.more) issue_next();
      }
    }
    if (stalled) break;

    // ---- item epilogue: the partial (output back to absolute units, running max and sum)
    //      straight from registers. Thread (gid, tig) holds, per column, the D/8 consecutive
    //      coordinates (D/8) gid .. (D/8) gid + D/8 - 1: O^T rows gid and gid + 8 of m-tile mt
    //      are coordinates 2 ((D/16) gid + mt) + {0, 1}.
    const float o_unit = ldexpf(1.0f, ev_run - 127);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      l_run[j] += __shfl_xor_sync(kFull, l_run[j], 4);
      l_run[j] += __shfl_xor_sync(kFull, l_run[j], 8);
      l_run[j] += __shfl_xor_sync(kFull, l_run[j], 16);
    }
    const Item it3 = ring_item(ring, popped - 1);
    const int slot = it3.p * a.ksub + it3.sub, vbase3 = 8 * it3.cg, V3 = min(NV, a.T * G - vbase3);
#pragma unroll
    for (int j = 0; j < (kPaired ? 1 : 2); ++j) {
      // paired: the thread's pair is tig (hi + lo columns added); else column 2 tig + j
      const int col = kPaired ? tig : 2 * tig + j;
      if (col < V3) {
        float ov[C::kMT][2];
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            ov[mt][h] = (kPaired ? o[0][mt][2 * h] + o[0][mt][2 * h + 1] : o[0][mt][2 * h + j] + o[1][mt][2 * h + j]) *
                        o_unit;
        const size_t row = query_row(a, it3.b, it3.g, G, vbase3 + col);
        float4* dst = reinterpret_cast<float4*>(a.part_o + (row * PK + slot) * D + (D / 8) * gid);
#pragma unroll
        for (int q4 = 0; q4 < C::kMT / 2; ++q4)
          dst[q4] = make_float4(ov[2 * q4][0], ov[2 * q4][1], ov[2 * q4 + 1][0], ov[2 * q4 + 1][1]);
        if (gid == 0) {
          a.part_m[row * PK + slot] = m_run[j];
          a.part_l[row * PK + slot] = l_run[j];
        }
      }
    }
  }  // items

  if (stalled) {
    if (lane == 0) atomicOr(a.err, DA_DEVERR_TIMEOUT);
    // give the copies still in flight into this warp's stages a bounded chance to land (one
    // time limit shared by all of them)
    uint64_t deadline = 0;
    for (unsigned k = stall_from; k < issued; ++k)
      ptx::mbar_wait_until(bar0 + 8 * (k % C::kNStages), (k / C::kNStages) & 1, deadline);
  }
  count_warp_out(a, gridDim.x * kWarps, lane);
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D byte view of a paged cache side: rows = (block, kv head, slot) of `row` bytes; boxes of
// 16 rows x `box` bytes with the given swizzle.
bool encode_map(CUtensorMap* map, const void* base, int row, int box, CUtensorMapSwizzle swz, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row};
  const cuuint32_t boxd[2] = {(cuuint32_t)box, (cuuint32_t)kPage};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, boxd, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One 3-D view of two equally shaped arrays (a K and a V side): (row element, row, side), the
// side stride being the distance between them, so one box fetches the same rows of both. The
// side with the lower address is side 0; *zk receives the side of the first array. Fails (the
// caller then uses one copy per side) when the arrays coincide or the distance is not a
// usable stride.
bool encode_pair(CUtensorMap* map, const void* k, const void* v, CUtensorMapDataType type, int elem_bytes, int row,
                 int box_rows, CUtensorMapSwizzle swz, long long rows, int* zk) {
  auto fn = encode_fn();
  if (!fn || k == v) return false;
  const uintptr_t ka = reinterpret_cast<uintptr_t>(k), va = reinterpret_cast<uintptr_t>(v);
  const uintptr_t lo = ka < va ? ka : va, diff = ka < va ? va - ka : ka - va;
  if (diff % 16 || diff >= (uintptr_t(1) << 40)) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)row, (cuuint64_t)rows, 2};
  const cuuint64_t strides[2] = {(cuuint64_t)row * elem_bytes, (cuuint64_t)diff};
  const cuuint32_t boxd[3] = {(cuuint32_t)row, (cuuint32_t)box_rows, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  *zk = ka > va;
  return fn(map, type, 3, reinterpret_cast<void*>(lo), dims, strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KS, int D, int NV, bool CAP, bool PAIR>
cudaError_t launch_kernel(const Args& b, const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& nm,
                          cudaStream_t s);

template <int KS, int D, int NV, bool CAP>
cudaError_t launch_fixed(const Args& a, cudaStream_t s) {
  using C = Cb<KS, D, NV>;
  CUtensorMap km{}, vm{}, nm{};
  const long long rows = (long long)a.num_blocks * a.Hkv * kPage;
  const CUtensorMapSwizzle vswz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  Args b = a;
  int zk = 0;
  // 4-bit keys and values have the same rows: one copy per page for both where possible
  b.kv_pair = KS == kSideCB4 &&
              encode_pair(&km, a.k_cache, a.v_cache, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, C::kVRow, kPage, vswz, rows, &zk);
  b.kv_zk = b.kv_pair ? zk : 0;
  if (!b.kv_pair) {
    if (KS == kSideFP8 && !encode_map(&km, a.k_cache, C::kKRow, 128, CU_TENSOR_MAP_SWIZZLE_128B, rows))
      return cudaErrorInvalidValue;
    if (KS == kSideCB4 && !encode_map(&km, a.k_cache, C::kKRow, C::kKRow, vswz, rows)) return cudaErrorInvalidValue;
    if (!encode_map(&vm, a.v_cache, C::kVRow, C::kVRow, vswz, rows)) return cudaErrorInvalidValue;
  }
  // the per-token norms of codebook keys and values: [num_blocks * Hkv] rows of 16 floats each
  b.kn_pair = C::kKNorms && encode_pair(&nm, a.k_scales, a.v_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, kPage, 1,
                                        CU_TENSOR_MAP_SWIZZLE_NONE, (long long)a.num_blocks * a.Hkv, &zk);
  b.kn_zk = b.kn_pair ? zk : 0;
  const bool pair = KS == kSideCB4 ? (b.kv_pair && b.kn_pair) : KS == kSideCB3 ? b.kn_pair != 0 : false;
  return pair ? launch_kernel<KS, D, NV, CAP, KS != kSideFP8>(b, km, vm, nm, s)
              : launch_kernel<KS, D, NV, CAP, false>(b, km, vm, nm, s);
}

template <int KS, int D, int NV, bool CAP, bool PAIR>
cudaError_t launch_kernel(const Args& b, const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& nm,
                          cudaStream_t s) {
  using C = Cb<KS, D, NV>;
  const Args& a = b;
  auto kern = partition_cb_kernel<KS, D, NV, CAP, PAIR>;
  static DeviceFlags attr;
  cudaError_t e = ensure_dynamic_smem(kern, C::kSmem, attr);
  if (e != cudaSuccess) return e;
  static int sms[64] = {}, reserved[64] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (sms[dev] == 0) {
    if ((e = cudaDeviceGetAttribute(&reserved[dev], cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
  }
  // the shared-memory layout (tables on a 64 KB boundary, warps' blocks around them) is laid out
  // for dynamic shared memory starting kDynStart bytes into the CTA's window
  if (reserved[dev] != kDynStart) return cudaErrorNotSupported;
  // one CTA per SM, fewer when the call has fewer items than the grid has warps
  const long long items = (long long)a.B * a.Hkv * a.P * a.ncg * a.ksub;
  const long long ctas = (items + C::kWarps - 1) / C::kWarps;
  const int grid = (int)(ctas < sms[dev] ? (ctas > 0 ? ctas : 1) : sms[dev]);
  // scheduled during the previous kernel's last CTAs (the query rotation, for codebook keys);
  // waits in-kernel before its first read
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmem, s, b, km, vm, nm);
}

template <int KS, int D, bool CAP>
cudaError_t launch_nv(const Args& a, cudaStream_t s) {
  const int v = a.T * (a.Hq / a.Hkv);  // virtual heads, padded to a power of two
  if (v <= 1) return launch_fixed<KS, D, 1, CAP>(a, s);
  if (v <= 2) return launch_fixed<KS, D, 2, CAP>(a, s);
  if (v <= 4) return launch_fixed<KS, D, 4, CAP>(a, s);
  if (v <= kMaxColumns) return launch_fixed<KS, D, 8, CAP>(a, s);  // 8 columns per item, a.ncg column groups
  return cudaErrorInvalidValue;
}

template <int KS, int D>
cudaError_t launch_cap(const Args& a, cudaStream_t s) {
  return a.softcap > 0.0f ? launch_nv<KS, D, true>(a, s) : launch_nv<KS, D, false>(a, s);
}

template <int KS>
cudaError_t launch_d(const Args& a, cudaStream_t s) {
  return a.D == 128 ? launch_cap<KS, 128>(a, s) : launch_cap<KS, 256>(a, s);
}

}  // namespace
}  // namespace da
