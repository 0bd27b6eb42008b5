// partition_tc.cu -- split-K partition kernel for the BF16 and FP8 E4M3 caches:
// TMA page staging + warp-level tensor-core MMA for the GQA group's tiles.
//
// A CTA of four warps takes `ppc` consecutive partitions of one (sequence, kv head). Either
// the warps share each partition (pages dealt round-robin, the warps' results merged at the
// partition's end) or each warp owns whole partitions; the launcher chooses per call. A small
// batch runs as one wave of CTAs (one per resident slot) that choose `ppc` themselves from the
// context lengths (spread_work). Every
// warp runs its own pipeline of kStages shared-memory stages, each holding one page (16
// tokens) of K and of V for the kv head, loaded by TMA (cp.async.bulk.tensor, 128-byte
// swizzle) and signalled on an mbarrier, continuing across partition boundaries. Per page a
// warp computes, on the tensor cores (mma.m16n8k16, fp32 accumulators):
//   S^T[16 tokens x 8 cols] = K[16 x D] . Q^T[D x 8]      (the group's query heads as columns)
//   O^T[D x 8 cols]       += V^T[D x 16]  . P^T[16 x 8]
// Tokens are the MMA's M dimension, so a group of G = 4 heads uses 4 of the 8 columns for
// its scores; the other 4 repeat the same heads and carry the low half of a hi/lo split of
// the probabilities (p = hi + lo, both in the MMA's 16-bit type), which keeps P.V accurate
// to ~2^-17 relative. The thread that owns a score column also owns that column of O^T, so
// the online-softmax rescale needs no data exchange. At a partition's end its partial is
// written (or, for an unsplit sequence, the normalised output directly).
//
// Multi-token decode (T query tokens per sequence at positions L-T .. L-1): the columns are
// the group's (query token, head) pairs, each masked at its own token's causal (and window)
// limit. Up to 8 pairs share one CTA's columns; more (T * G <= 32) are split into column
// groups of 8, one CTA each, adjacent in the grid so that the pages they all read are
// fetched from DRAM once and from L2 by the others. ALiBi slopes, when given, add
// slope_h * (t - pos) to each column's scores.
//
// (attention.rs README: split-K decode kernels per KV format and m16n8k16 tensor-core MMA
// with async copies on SM100-class GPUs; turboquant-rs 0.4.1, src/cache/cuda/attention.rs:
// a partition kernel writing partial output, max and sum.)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cmath>
#include <mutex>

#include "da_internal.cuh"
#include "page_softmax.cuh"
#include "page_walk.cuh"
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kPage = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// NV: the CTA's columns: the group's (query token, head) pairs ("virtual heads" v = jq * G + h)
// padded to a power of two <= 8 (8 when there are several column groups); with one query
// token NV = G.
template <int FMT, int D, int NV>
struct Tc {
  static constexpr int kElemBytes = FMT == DA_KV_BF16 ? 2 : 1;
  static constexpr int kSubs = D * kElemBytes / 128;       // 128-byte swizzled column slabs per row
  static constexpr int kSubBytes = kPage * 128;             // one slab of one page: 2 KB
  static constexpr int kPageBytes = kSubs * kSubBytes;      // one page of K (or V), one kv head
  static constexpr int kStageBytes = 2 * kPageBytes;        // K + V: slab u of K and of V side by side
  static constexpr int kStages = 16384 / kStageBytes > 0 ? 16384 / kStageBytes : 1;  // 64 KB of stages per CTA
  static constexpr int kNT = NV <= 4 ? 1 : 2;               // P.V column tiles (8 columns each)
  static constexpr int kMT = D / 16;                        // O^T row tiles
  static constexpr int kKS = D / 16;                        // k-steps of S^T
  static constexpr int kStageSmem = kWarps * kStages * kStageBytes;
  static constexpr int kDP = D + 4;  // padded row of the merge buffer
  // the epilogue stages at most 4 columns at a time (two passes at NV = 8), which keeps the
  // 8-column kernel within the shared memory of three CTAs per SM
  static constexpr int kEpCols = NV < 4 ? NV : 4;
  static constexpr int kEpPasses = NV / kEpCols;
  static constexpr int kMergeSmem = (kWarps * kEpCols * kDP + 2 * kWarps * 8) * 4;
  static constexpr int kSmem = kStageSmem + kMergeSmem + 1024;
};

__device__ __forceinline__ uint32_t swz(uint32_t slab, int row, int chunk) {
  return slab + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// p = hi + lo with hi, lo in the MMA's 16-bit type
template <int FMT>
__device__ __forceinline__ float hi_part(float p) {
  return FMT == DA_KV_BF16 ? __bfloat162float(__float2bfloat16_rn(p)) : __half2float(__float2half_rn(p));
}
template <int FMT>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  return FMT == DA_KV_BF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}
// two E4M3 codes (low 16 bits) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xffffu), __NV_E4M3);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int FMT>
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (FMT == DA_KV_BF16)
    ptx::mma_bf16(d, a, b0, b1);
  else
    ptx::mma_f16(d, a, b0, b1);
}

// A CTA's work: kv head g, column group cg of sequence b (L tokens, np partitions), its
// partitions [p_begin, p_end) (none when p_end <= p_begin).
struct CtaWork {
  int b, g, cg, L, np, p_begin, p_end;
};

// The launcher's fixed grid: x over (chunk of ppc partitions, column group), y over kv heads,
// z over sequences, so that the chunks of one (sequence, kv head) are neighbours in the
// schedule: a page two chunks share (a window start inside a page) is read while in L2.
__device__ __forceinline__ CtaWork fixed_work(const Args& a, int tid) {
  CtaWork c;
  c.cg = blockIdx.x % a.ncg;
  c.g = blockIdx.y, c.b = blockIdx.z;
  c.L = load_len(a, c.b, blockIdx.x == 0 && c.g == 0 && tid == 0);
  c.np = seq_partitions(c.L, a.T, a.window, a.psize, a.thresh);
  c.p_begin = (blockIdx.x / a.ncg) * a.ppc, c.p_end = min(c.p_begin + a.ppc, c.np);
  return c;
}

// Small batches (a.ppc == 0): a grid of one CTA per resident slot, all running at once. In each
// CTA warp 0 reads every context length and takes the smallest chunk size k <= 8 for which the
// batch's CTAs -- each sequence's partitions cut into chunks of k, times kv heads and column
// groups -- fit the grid (the launcher makes sure k = 8 does; the search starts from the bound
// that the total partition count gives), then the CTA of index blockIdx.x in (sequence, chunk,
// kv head, column group) order; CTAs past the count have no work. One wave of CTAs, each
// walking its chunk's partitions with one pipeline, avoids both the start-up gap of every
// further wave and a tail of whole partitions scheduled last.
constexpr int kMaxChunk = 8;
constexpr int kSpreadSeqs = 4;  // sequences per lane of warp 0: batches of up to 128
__device__ __forceinline__ CtaWork spread_work(const Args& a, int tid) {
  __shared__ int s_pick[4];  // sequence (-1: no work), CTA index within it, its length, chunk size
  if (tid < 32) {
    const int lane = tid;
    int lv[kSpreadSeqs], npv[kSpreadSeqs], total = 0;  // sequences b = lane + 32 i
#pragma unroll
    for (int i = 0; i < kSpreadSeqs; ++i) {
      const int bb = lane + 32 * i;
      lv[i] = bb < a.B ? load_len(a, bb, blockIdx.x == 0) : 0;
      npv[i] = seq_partitions(lv[i], a.T, a.window, a.psize, a.thresh);
      total += npv[i];
    }
    total = __reduce_add_sync(kFull, total);
    const int per_chunk = a.Hkv * a.ncg;         // CTAs per chunk of partitions
    const int fit = (int)gridDim.x / per_chunk;  // chunks the grid holds
    // the smallest chunk size whose chunk count fits, from the bound total / fit up
    int ppc = fit > 0 ? max(1, min((total + fit - 1) / fit, kMaxChunk)) : kMaxChunk;
    for (;; ++ppc) {
      int cnt = 0;
#pragma unroll
      for (int i = 0; i < kSpreadSeqs; ++i) cnt += (npv[i] + ppc - 1) / ppc;
      cnt = __reduce_add_sync(kFull, cnt);
      if (cnt <= fit || ppc == kMaxChunk) break;
    }
    // CTA j's sequence: an exclusive scan of the sequences' CTA counts in sequence order
    // (over the lanes for i = 0, then i = 1, ...)
    const int j = blockIdx.x;
    int base = 0, pick = -1, r = 0, L = 0;
#pragma unroll
    for (int i = 0; i < kSpreadSeqs; ++i) {
      if (32 * i >= a.B) break;
      const int n = (npv[i] + ppc - 1) / ppc * per_chunk;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const int first = base + incl - n;
      if (j >= first && j < first + n) pick = lane + 32 * i, r = j - first, L = lv[i];
      base += __shfl_sync(kFull, incl, 31);
    }
    const unsigned holder = __ballot_sync(kFull, pick >= 0);
    if (holder == 0 && lane == 0) s_pick[0] = -1;
    if (pick >= 0) s_pick[0] = pick, s_pick[1] = r, s_pick[2] = L, s_pick[3] = ppc;
  }
  __syncthreads();
  CtaWork c;
  c.b = s_pick[0];
  if (c.b < 0) {  // past the batch's CTAs
    c.b = c.g = c.cg = c.L = c.np = c.p_begin = c.p_end = 0;
    return c;
  }
  const int rr = s_pick[1], ppc = s_pick[3];
  c.cg = rr % a.ncg;
  c.g = (rr / a.ncg) % a.Hkv;
  c.L = s_pick[2];
  c.np = seq_partitions(c.L, a.T, a.window, a.psize, a.thresh);
  c.p_begin = rr / (a.Hkv * a.ncg) * ppc, c.p_end = min(c.p_begin + ppc, c.np);
  return c;
}

// CAP: softcap on (a separate instantiation, so the plain kernel carries no tanh)
template <int FMT, int D, int NV, bool CAP>
__global__ void __launch_bounds__(kThreads, D == 128 ? 3 : 2)
    partition_tc_kernel(const Args a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  using T = Tc<FMT, D, NV>;
  constexpr int DP = T::kDP;
  // the warp index through a shuffle from lane 0, which the compiler then treats as uniform
  const int tid = threadIdx.x, lane = tid & 31, w = __shfl_sync(kFull, tid >> 5, 0);
  const int gid = lane >> 2, tig = lane & 3;
  ptx::grid_dependency_wait();   // what the kernel before this one writes (q, the rotated q, ...)
  ptx::grid_dependents_launch();  // the reduce may be scheduled once every CTA has started
  const CtaWork cw = a.ppc > 0 ? fixed_work(a, tid) : spread_work(a, tid);
  if (cw.p_begin >= cw.p_end) return;
  const int b = cw.b, g = cw.g, L = cw.L, np = cw.np, p_begin = cw.p_begin, p_end = cw.p_end;
  // the CTA's columns: virtual heads (query token, head of the group) vbase .. vbase + V - 1
  const int G = a.Hq / a.Hkv, vbase = 8 * cw.cg, V = min(NV, a.T * G - vbase);

  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps * T::kStages];
  const uint32_t smem = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* smem_gen = smem_raw + (smem - ptx::smem_u32(smem_raw));
  const uint32_t bar0 = ptx::smem_u32(bars) + w * T::kStages * 8;
  const uint32_t stage0 = smem + w * T::kStages * T::kStageBytes;

  if (lane == 0) {
    ptx::prefetch_tensor_map(&kmap);
    ptx::prefetch_tensor_map(&vmap);
    for (int s = 0; s < T::kStages; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  // offsets of K and V within a slab pair of a stage (the side with the lower address first
  // when one map spans both caches)
  const uint32_t koff = a.kv_zk ? T::kSubBytes : 0, voff = T::kSubBytes - koff;
  // ---- the warp's partitions and pages, copied kStages ahead of the compute: with
  //      a.owner, partitions p_begin + w, p_begin + w + kWarps, ... and all their pages; else
  //      every partition of the CTA and pages w, w + kWarps, ... of each
  const bool owner = a.owner != 0;
  const int p_first = owner ? p_begin + w : p_begin, p_step = owner ? kWarps : 1;
  const int pg_off = owner ? 0 : w, pg_step = owner ? 1 : kWarps;
  IssueCursor cur;
  cur.init(a, b, L, p_first, p_step, p_end, pg_off, pg_step, lane);
  uint32_t valid_mask = 0;  // bit s: the page in stage s has a valid block (warp-uniform)
  unsigned issued = 0;
  int is = 0;  // stage of the next copy (issued % kStages)
  auto issue_next = [&]() {  // all lanes; lane 0 issues the copies of the page at the cursor
    const int phys = cur.take(a);
    const int s = is;
    is = is + 1 == T::kStages ? 0 : is + 1;
    ++issued;
    valid_mask = phys >= 0 ? (valid_mask | (1u << s)) : (valid_mask & ~(1u << s));
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * s, dst = stage0 + s * T::kStageBytes;
      if (phys < 0) {
        ptx::mbar_arrive(bar);  // completes the phase with nothing loaded
      } else {
        ptx::fence_proxy_async();
        ptx::mbar_arrive_expect_tx(bar, T::kStageBytes);
        const int y = (phys * a.Hkv + g) * kPage;
#pragma unroll
        for (int u = 0; u < T::kSubs; ++u) {
          // slab u of the page: K and V side by side (one copy when one map spans both caches)
          const uint32_t d = dst + u * 2 * T::kSubBytes;
          if (a.kv_pair) {
            ptx::tma_load_3d(d, &kmap, u * (128 / T::kElemBytes), y, 0, bar);
          } else {
            ptx::tma_load_2d(d + koff, &kmap, u * (128 / T::kElemBytes), y, bar);
            ptx::tma_load_2d(d + voff, &vmap, u * (128 / T::kElemBytes), y, bar);
          }
        }
      }
    }
  };
  for (int k = 0; k < T::kStages && cur.more; ++k) issue_next();

  // ---- query fragments (B operand of S^T): column n holds virtual head (n % NV) % V
  const int qv = vbase + (gid % NV) % V;
  const uint16_t* qrow = a.q + (((size_t)b * a.T + qv / G) * a.Hq + g * G + qv % G) * D;
  uint32_t qf[T::kKS][2];
  float score_scale = a.scale * kLog2e;  // applied to the MMA result (log2 domain)
  if constexpr (FMT == DA_KV_BF16) {
#pragma unroll
    for (int ks = 0; ks < T::kKS; ++ks) {
      qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tig);
      qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tig);
    }
  } else {
    // f16 operands: scale q by a power of two so that max|q| fits f16 (exact), undo in the score scale
    float qv[T::kKS][4];
    float mx = 0.0f;
#pragma unroll
    for (int ks = 0; ks < T::kKS; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qv[ks][e] = bf16_to_f32(qrow[16 * ks + 4 * tig + e]);
        mx = fmaxf(mx, fabsf(qv[ks][e]));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    int ex = 0;
    frexpf(mx, &ex);
    const int e2 = ex > 14 ? 14 - ex : 0;
    const float qs = ldexpf(1.0f, e2);
#pragma unroll
    for (int ks = 0; ks < T::kKS; ++ks) {
      qf[ks][0] = pack_f16(qv[ks][0] * qs, qv[ks][1] * qs);
      qf[ks][1] = pack_f16(qv[ks][2] * qs, qv[ks][3] * qs);
    }
    score_scale = a.scale * __ldg(a.k_scales) * ldexpf(1.0f, -e2) * kLog2e;
  }
  const float cap = a.softcap;
  const float cap_pre = CAP ? score_scale / (cap * kLog2e) : 0.0f;  // s_nat / cap
  const float cap_post = cap * kLog2e;

  // hi/lo role of this thread's two columns (NV <= 4: column c carries part c / NV), and the
  // positions its columns' query tokens attend: [lo_w, pos] (causal limit and window)
  int part[2], lo_w[2], pos_c[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    part[j] = NV <= 4 ? (2 * tig + j) / NV : 0;
    pos_c[j] = L - a.T + (vbase + ((2 * tig + j) % NV) % V) / G;
    lo_w[j] = window_start(pos_c[j], a.window);
  }
  // ALiBi: the slope of each column's query head, in the log2 domain of the scores
  const bool alibi = a.alibi != nullptr;
  float slope_c[2] = {0.0f, 0.0f};
  if (alibi) {
#pragma unroll
    for (int j = 0; j < 2; ++j) slope_c[j] = __ldg(a.alibi + g * G + (vbase + ((2 * tig + j) % NV) % V) % G) * kLog2e;
  }
  float* ep_o = reinterpret_cast<float*>(smem_gen + T::kStageSmem);  // [kWarps][kEpCols][DP]
  float* ep_m = ep_o + kWarps * T::kEpCols * DP;                      // [kWarps][8]
  float* ep_l = ep_m + kWarps * 8;                                    // [kWarps][8]
  const float out_scale = FMT == DA_KV_FP8_E4M3 ? __ldg(a.v_scales) : 1.0f;
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix index and row of this lane's address
  unsigned consumed = 0, stall_from = 0;
  int cs = 0;            // stage of the next page to compute (consumed % kStages)
  uint32_t cphase = 0;   // its mbarrier phase parity ((consumed / kStages) & 1)
  bool stalled = false;  // a copy never arrived: no more waits, copies or compute

  for (int p = p_first; p < p_end; p += p_step) {
  const Range r = partition_range(L, a.T, p, a.window, a.psize, a.thresh);
  int first_page, npages;
  range_pages(r, first_page, npages);
  const int nw = warp_pages(npages, pg_off, pg_step);
  const bool rev = walk_reversed(owner, p);  // odd owned partitions: last page first
  // tokens each column attends in this partition, and the pages that need no mask in any
  // column: [lo_all, hi_all) (warp-uniform)
  int lo_c[2], hi_c[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    lo_c[j] = max(lo_w[j], r.start);
    hi_c[j] = min(pos_c[j] + 1, r.end);
  }
  int lo_all = max(lo_c[0], lo_c[1]), hi_all = min(hi_c[0], hi_c[1]);
  lo_all = max(lo_all, __shfl_xor_sync(kFull, lo_all, 1));
  lo_all = max(lo_all, __shfl_xor_sync(kFull, lo_all, 2));
  hi_all = min(hi_all, __shfl_xor_sync(kFull, hi_all, 1));
  hi_all = min(hi_all, __shfl_xor_sync(kFull, hi_all, 2));
  // ---- running state: column c = 2*tig + j of S^T and of every O^T column tile
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
  float o[T::kNT][T::kMT][4];
#pragma unroll
  for (int t = 0; t < T::kNT; ++t)
#pragma unroll
    for (int mt = 0; mt < T::kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[t][mt][e] = 0.0f;

  for (int i = 0; i < nw; ++i, ++consumed) {
    const int s = cs;
    if (!stalled && !ptx::mbar_wait(bar0 + 8 * s, cphase)) {
      stalled = true;
      stall_from = consumed;
    }
    if (++cs == T::kStages) {
      cs = 0;
      cphase ^= 1u;
    }
    if (!stalled && (valid_mask & (1u << s))) {
      const uint32_t kb = stage0 + s * T::kStageBytes + koff, vb = stage0 + s * T::kStageBytes + voff;
      const int tok0 = (first_page + walk_page(i, nw, pg_off, pg_step, rev)) * kPage;
      // -- S^T = K . Q^T, the k-steps alternating between two accumulators (two dependent MMA
      //    chains of half the length), added at the end
      float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sc2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (FMT == DA_KV_BF16) {
#pragma unroll
        for (int ks = 0; ks < T::kKS; ++ks) {
          const int row = ri + 8 * (mi & 1), chunk = 2 * ks + (mi >> 1);
          uint32_t af[4];
          ptx::ldmatrix_x4(af, swz(kb + (chunk >> 3) * 2 * T::kSubBytes, row, chunk & 7));
          mma<FMT>((ks & 1) ? sc2 : sc, af, qf[ks][0], qf[ks][1]);
        }
      } else {
#pragma unroll
        for (int j2 = 0; j2 < T::kKS / 2; ++j2) {
          const int row = ri + 8 * (mi & 1), chunk = 2 * j2 + (mi >> 1);
          uint32_t rr[4];
          ptx::ldmatrix_x4(rr, swz(kb + (chunk >> 3) * 2 * T::kSubBytes, row, chunk & 7));
          const uint32_t a0[4] = {e4m3x2_to_f16x2(rr[0]), e4m3x2_to_f16x2(rr[1]), e4m3x2_to_f16x2(rr[0] >> 16),
                                  e4m3x2_to_f16x2(rr[1] >> 16)};
          mma<FMT>(sc, a0, qf[2 * j2][0], qf[2 * j2][1]);
          const uint32_t a1[4] = {e4m3x2_to_f16x2(rr[2]), e4m3x2_to_f16x2(rr[3]), e4m3x2_to_f16x2(rr[2] >> 16),
                                  e4m3x2_to_f16x2(rr[3] >> 16)};
          mma<FMT>(sc2, a1, qf[2 * j2 + 1][0], qf[2 * j2 + 1][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] += sc2[e];
      // -- scale (log2 domain), softcap, mask; sc[0], sc[1]: token gid; sc[2], sc[3]: token gid + 8
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] = CAP ? cap_post * tanhf(sc[e] * cap_pre) : sc[e] * score_scale;
      if (alibi) {  // + slope * (t - pos) for token t of each element
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sc[e] += slope_c[e & 1] * (float)(tok0 + gid + (e >> 1) * 8 - pos_c[e & 1]);
      }
      if (tok0 < lo_all || tok0 + kPage > hi_all) mask_page(sc, tok0, gid, lo_c, hi_c);
      // -- online softmax per column (lazily moved reference max)
      float alpha[2], pr[4];
      if (page_softmax(sc, m_run, l_run, alpha, pr)) {
#pragma unroll
        for (int t = 0; t < T::kNT; ++t)
#pragma unroll
          for (int mt = 0; mt < T::kMT; ++mt) {
            o[t][mt][0] *= alpha[0];
            o[t][mt][1] *= alpha[1];
            o[t][mt][2] *= alpha[0];
            o[t][mt][3] *= alpha[1];
          }
      }
      // -- P^T as the B operand: hi/lo parts in C layout, transposed with movmatrix
      uint32_t pb[T::kNT][2];
      if constexpr (NV <= 4) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pt = part[e & 1];
          const float h = hi_part<FMT>(pr[e]);
          x[e] = pt == 0 ? h : (pt == 1 ? pr[e] - h : 0.0f);
        }
        pb[0][0] = ptx::movmatrix_trans(pack16<FMT>(x[0], x[1]));
        pb[0][1] = ptx::movmatrix_trans(pack16<FMT>(x[2], x[3]));
      } else {
        float hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hi[e] = hi_part<FMT>(pr[e]);
          lo[e] = pr[e] - hi[e];
        }
        pb[0][0] = ptx::movmatrix_trans(pack16<FMT>(hi[0], hi[1]));
        pb[0][1] = ptx::movmatrix_trans(pack16<FMT>(hi[2], hi[3]));
        pb[T::kNT - 1][0] = ptx::movmatrix_trans(pack16<FMT>(lo[0], lo[1]));
        pb[T::kNT - 1][1] = ptx::movmatrix_trans(pack16<FMT>(lo[2], lo[3]));
      }
      // -- O^T += V^T . P^T
      if constexpr (FMT == DA_KV_BF16) {
#pragma unroll
        for (int mt = 0; mt < T::kMT; ++mt) {
          const int row = ri + 8 * (mi >> 1), chunk = 2 * mt + (mi & 1);
          uint32_t af[4];
          ptx::ldmatrix_x4_trans(af, swz(vb + (chunk >> 3) * 2 * T::kSubBytes, row, chunk & 7));
#pragma unroll
          for (int t = 0; t < T::kNT; ++t) mma<FMT>(o[t][mt], af, pb[t][0], pb[t][1]);
        }
      } else {
#pragma unroll
        for (int j2 = 0; j2 < T::kMT / 2; ++j2) {
          const int row = ri + 8 * (mi >> 1), chunk = 2 * j2 + (mi & 1);
          uint32_t rr[4];
          ptx::ldmatrix_x4_trans(rr, swz(vb + (chunk >> 3) * 2 * T::kSubBytes, row, chunk & 7));
          const uint32_t x0 = __byte_perm(rr[0], 0, 0x3120), x1 = __byte_perm(rr[1], 0, 0x3120);
          const uint32_t x2 = __byte_perm(rr[2], 0, 0x3120), x3 = __byte_perm(rr[3], 0, 0x3120);
          const uint32_t a0[4] = {e4m3x2_to_f16x2(x0), e4m3x2_to_f16x2(x0 >> 16), e4m3x2_to_f16x2(x2),
                                  e4m3x2_to_f16x2(x2 >> 16)};
          const uint32_t a1[4] = {e4m3x2_to_f16x2(x1), e4m3x2_to_f16x2(x1 >> 16), e4m3x2_to_f16x2(x3),
                                  e4m3x2_to_f16x2(x3 >> 16)};
#pragma unroll
          for (int t = 0; t < T::kNT; ++t) {
            mma<FMT>(o[t][2 * j2], a0, pb[t][0], pb[t][1]);
            mma<FMT>(o[t][2 * j2 + 1], a1, pb[t][0], pb[t][1]);
          }
        }
      }
    }
    __syncwarp();
    if (!stalled && cur.more) issue_next();
  }

  // ---- partition epilogue
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(kFull, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(kFull, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(kFull, l_run[j], 16);
  }
  const bool direct = np == 1;
  if (owner) {
    // the warp's (o, m, l) is the partition's result: O^T (hi and lo columns added; divided
    // by l for an unsplit sequence) through the warp's staging buffer, then 16-byte stores
    float* ep_w = ep_o + w * T::kEpCols * DP;
    if (!direct && gid == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 2 * tig + j;
        if (col < V) {
          const size_t pi = query_row(a, b, g, G, vbase + col) * a.P + p;
          a.part_m[pi] = m_run[j];
          a.part_l[pi] = l_run[j];
        }
      }
    }
#pragma unroll
    for (int pass = 0; pass < T::kEpPasses; ++pass) {
      const int c0 = pass * T::kEpCols;  // the pass's columns: c0 .. c0 + kEpCols - 1
#pragma unroll
      for (int mt = 0; mt < T::kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = o[0][mt][e];
          if constexpr (NV == 8) v += o[T::kNT - 1][mt][e];
          if constexpr (NV == 4) v += __shfl_xor_sync(kFull, v, 2);  // columns c, c + 4
          if constexpr (NV == 2) v += __shfl_xor_sync(kFull, v, 1);  // columns c, c + 2
          if constexpr (NV == 1) v += (e & 1) ? 0.0f : o[0][mt][e + 1];  // columns 0, 1
          const int col = 2 * tig + (e & 1);
          const float l = l_run[e & 1];
          if (direct) v = l > 0.0f ? v * out_scale / l : 0.0f;
          const int rowd = FMT == DA_KV_BF16 ? 16 * mt + gid + ((e >> 1) ? 8 : 0) : 16 * mt + 2 * gid + (e >> 1);
          if (col >= c0 && col < c0 + T::kEpCols && col < V) ep_w[(col - c0) * DP + rowd] = v;
        }
      __syncwarp();
      const int Vp = min(T::kEpCols, V - c0);
      for (int idx = lane; idx < Vp * D / 4; idx += 32) {
        const int v = idx / (D / 4), d = 4 * (idx % (D / 4));
        const size_t bh = query_row(a, b, g, G, vbase + c0 + v);
        const float4 x = *reinterpret_cast<const float4*>(ep_w + v * DP + d);
        if (direct) {  // the caller's output is only 4-byte aligned
          float* dst = a.out + bh * D + d;
          dst[0] = x.x, dst[1] = x.y, dst[2] = x.z, dst[3] = x.w;
        } else {
          *reinterpret_cast<float4*>(a.part_o + (bh * a.P + p) * D + d) = x;
        }
      }
      __syncwarp();  // the staging buffer is rewritten by the next pass or partition
    }
    continue;
  }
  // shared partition: each warp's (o, m, l) per virtual head into shared memory (hi and lo
  // columns added), then the warps merged into the partial (split sequence) or the
  // normalised output (unsplit), kEpCols columns per pass
  if (gid == 0) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      ep_m[w * 8 + 2 * tig + j] = m_run[j];
      ep_l[w * 8 + 2 * tig + j] = l_run[j];
    }
  }
#pragma unroll
  for (int pass = 0; pass < T::kEpPasses; ++pass) {
    const int c0 = pass * T::kEpCols;
#pragma unroll
    for (int mt = 0; mt < T::kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = o[0][mt][e];
        if constexpr (NV == 8) v += o[T::kNT - 1][mt][e];
        if constexpr (NV == 4) v += __shfl_xor_sync(kFull, v, 2);  // columns c, c + 4
        if constexpr (NV == 2) v += __shfl_xor_sync(kFull, v, 1);  // columns c, c + 2
        if constexpr (NV == 1) v += (e & 1) ? 0.0f : o[0][mt][e + 1];  // columns 0, 1
        const int col = 2 * tig + (e & 1);
        const int rowd = FMT == DA_KV_BF16 ? 16 * mt + gid + ((e >> 1) ? 8 : 0) : 16 * mt + 2 * gid + (e >> 1);
        if (col >= c0 && col < c0 + T::kEpCols && col < V) ep_o[(w * T::kEpCols + col - c0) * DP + rowd] = v;
      }
    __syncthreads();
    const int Vp = min(T::kEpCols, V - c0);
    for (int idx = tid; idx < Vp * D; idx += kThreads) {
      const int vp = idx / D, d = idx % D, v = c0 + vp;
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, ep_m[ww * 8 + v]);
      float acc = 0.0f, l = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float mw = ep_m[ww * 8 + v];
        const float wt = mw == -INFINITY ? 0.0f : exp2f(mw - M);
        acc += wt * ep_o[(ww * T::kEpCols + vp) * DP + d];
        l += wt * ep_l[ww * 8 + v];
      }
      const size_t bh = query_row(a, b, g, G, vbase + v);
      if (direct) {
        a.out[bh * D + d] = l > 0.0f ? acc * out_scale / l : 0.0f;
      } else {
        const size_t pi = bh * a.P + p;
        a.part_o[pi * D + d] = acc;
        if (d == 0) {
          a.part_m[pi] = M;
          a.part_l[pi] = l;
        }
      }
    }
    __syncthreads();  // the merge buffer is rewritten by the next pass or partition
  }
  }  // partitions

  if (stalled) {
    if (lane == 0) atomicOr(a.err, DA_DEVERR_TIMEOUT);
    // give the copies still in flight into this warp's stages a bounded chance to land (one
    // time limit shared by all of them)
    uint64_t deadline = 0;
    for (unsigned k = stall_from; k < issued; ++k)
      ptx::mbar_wait_until(bar0 + 8 * (k % T::kStages), (k / T::kStages) & 1, deadline);
  }
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

// 2-D view of a paged cache: rows = (block, kv head, slot), columns = the row's D elements;
// boxes of 16 rows x 128 bytes with the 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, int elem_bytes, int D, long long rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)kPage};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One 3-D view of both caches: (row element, row, side), the side stride being the distance
// between the two caches, so one box of 16 rows x 128 bytes x 2 sides fetches a page slab of
// K and of V. The side with the lower address is side 0; *zk receives the side of K. Fails
// (the caller then uses one map per cache) when the caches coincide or the distance is not a
// usable stride.
bool encode_pair_map(CUtensorMap* map, const void* k, const void* v, int elem_bytes, int D, long long rows, int* zk) {
  auto fn = encode_fn();
  if (!fn || k == v) return false;
  const uintptr_t ka = reinterpret_cast<uintptr_t>(k), va = reinterpret_cast<uintptr_t>(v);
  const uintptr_t lo = ka < va ? ka : va, diff = ka < va ? va - ka : ka - va;
  if (diff % 16 || diff >= (uintptr_t(1) << 40)) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, 2};
  const cuuint64_t strides[2] = {(cuuint64_t)D * elem_bytes, (cuuint64_t)diff};
  const cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)kPage, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  *zk = ka > va;
  return fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            reinterpret_cast<void*>(lo), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int D, int NV, bool CAP>
cudaError_t launch_fixed(const Args& a, cudaStream_t s) {
  using T = Tc<FMT, D, NV>;
  CUtensorMap km{}, vm{};
  const long long rows = (long long)a.num_blocks * a.Hkv * kPage;
  Args b = a;
  int zk = 0;
  b.kv_pair = encode_pair_map(&km, a.k_cache, a.v_cache, T::kElemBytes, D, rows, &zk);
  b.kv_zk = b.kv_pair ? zk : 0;
  if (!b.kv_pair && (!encode_cache_map(&km, a.k_cache, T::kElemBytes, D, rows) ||
                     !encode_cache_map(&vm, a.v_cache, T::kElemBytes, D, rows)))
    return cudaErrorInvalidValue;
  auto kern = partition_tc_kernel<FMT, D, NV, CAP>;
  static DeviceFlags attr;
  cudaError_t e = ensure_dynamic_smem(kern, T::kSmem, attr);
  if (e != cudaSuccess) return e;
  static int per_sm = 0, sms[64] = {};
  if (per_sm == 0 && (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, T::kSmem)) != cudaSuccess)
    return e;
  b.ppc = partitions_per_cta(a, per_sm, sms);
  b.owner = warps_own_partitions(a, per_sm, kWarps, 3, sms);  // from 1.5 partitions per resident warp
  if (b.owner) b.ppc = kWarps * ((b.ppc + kWarps - 1) / kWarps);
  // scheduled during the previous kernel's last CTAs (the query rotation, for codebook keys);
  // waits in-kernel before its first read
  // a small batch of at least two waves of single partitions (at the longest possible span):
  // one wave of CTAs, the chunk size chosen in-kernel from the lengths (below two waves the
  // fixed grid is as good and saves the choice's start-up time)
  const long long slots = resident_slots(per_sm, sms);
  const long long units = (long long)a.P * a.Hkv * a.B * a.ncg;
  if (!b.owner && a.ppc_req == 0 && a.schedule == 0 && slots > 0 && units >= 2 * slots &&
      a.B <= 32 * kSpreadSeqs &&
      (long long)a.B * a.Hkv * a.ncg * ((a.P + kMaxChunk - 1) / kMaxChunk) <= slots) {
    b.ppc = 0;
    return launch_pdl(kern, dim3((unsigned)slots), dim3(kThreads), T::kSmem, s, b, km, vm);
  }
  return launch_pdl(kern, dim3((a.P + b.ppc - 1) / b.ppc * a.ncg, a.Hkv, a.B), dim3(kThreads), T::kSmem, s, b, km, vm);
}

template <int FMT, int D, bool CAP>
cudaError_t launch_nv(const Args& a, cudaStream_t s) {
  const int v = a.T * (a.Hq / a.Hkv);  // virtual heads, padded to a power of two
  if (v <= 1) return launch_fixed<FMT, D, 1, CAP>(a, s);
  if (v <= 2) return launch_fixed<FMT, D, 2, CAP>(a, s);
  if (v <= 4) return launch_fixed<FMT, D, 4, CAP>(a, s);
  if (v <= kMaxColumns) return launch_fixed<FMT, D, 8, CAP>(a, s);  // 8 columns per CTA, a.ncg CTAs
  return cudaErrorInvalidValue;
}

template <int FMT, int D>
cudaError_t launch_g(const Args& a, cudaStream_t s) {
  return a.softcap > 0.0f ? launch_nv<FMT, D, true>(a, s) : launch_nv<FMT, D, false>(a, s);
}

}  // namespace

cudaError_t launch_partition_tc(const Args& a, cudaStream_t s) {
  if (a.fmt == DA_KV_BF16) return a.D == 128 ? launch_g<DA_KV_BF16, 128>(a, s) : launch_g<DA_KV_BF16, 256>(a, s);
  if (a.fmt == DA_KV_FP8_E4M3)
    return a.D == 128 ? launch_g<DA_KV_FP8_E4M3, 128>(a, s) : launch_g<DA_KV_FP8_E4M3, 256>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace da
