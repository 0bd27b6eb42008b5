// partition_tc.cu -- split-K partition kernel for the BF16 and FP8 E4M3 caches:
// TMA page staging + warp-level tensor-core MMA for the GQA group's tiles.
//
// Persistent CTAs of four warps walk the (sequence, kv head, partition) work units in a
// fixed round-robin order. A unit's pages are dealt round-robin to the warps; every warp
// runs its own pipeline of kStages shared-memory stages, each holding one page (16 tokens)
// of K and of V for the unit's kv head, loaded by TMA (cp.async.bulk.tensor, 128-byte
// swizzle) and signalled on an mbarrier. The warp's copies run kStages pages ahead of its
// computation, across unit boundaries, so HBM stays busy while a unit is finished. Per page
// a warp computes, on the tensor cores (mma.m16n8k16, fp32 accumulators):
//   S^T[16 tokens x 8 cols] = K[16 x D] . Q^T[D x 8]      (the group's query heads as columns)
//   O^T[D x 8 cols]       += V^T[D x 16]  . P^T[16 x 8]
// Tokens are the MMA's M dimension, so a group of G = 4 heads uses 4 of the 8 columns for
// its scores; the other 4 repeat the same heads and carry the low half of a hi/lo split of
// the probabilities (p = hi + lo, both in the MMA's 16-bit type), which keeps P.V accurate
// to ~2^-17 relative. The thread that owns a score column also owns that column of O^T, so
// the online-softmax rescale needs no data exchange. At the end of a unit the four warps'
// (m, l, o) are merged through shared memory and the partition's partial is written (or,
// for an unsplit sequence, the normalised output directly); the CTA that completes the last
// partition of a (sequence, kv head) -- counted with an atomic ticket, no CTA ever waits --
// combines the partials into the output (the float reduce).
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
#include "ptx.cuh"

namespace da {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kPage = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// NV: the group's (query token, head) pairs ("virtual heads" v = jq * G + h), padded to a
// power of two <= 8; with one query token NV = G.
template <int FMT, int D, int NV>
struct Tc {
  static constexpr int kElemBytes = FMT == DA_KV_BF16 ? 2 : 1;
  static constexpr int kSubs = D * kElemBytes / 128;       // 128-byte swizzled column slabs per row
  static constexpr int kSubBytes = kPage * 128;             // one slab of one page: 2 KB
  static constexpr int kPageBytes = kSubs * kSubBytes;      // one page of K (or V), one kv head
  static constexpr int kStageBytes = 2 * kPageBytes;        // K + V
  static constexpr int kStages = 16384 / kStageBytes > 0 ? 16384 / kStageBytes : 1;  // 64 KB of stages per CTA
  static constexpr int kNT = NV <= 4 ? 1 : 2;               // P.V column tiles (8 columns each)
  static constexpr int kMT = D / 16;                        // O^T row tiles
  static constexpr int kKS = D / 16;                        // k-steps of S^T
  static constexpr int kStageSmem = kWarps * kStages * kStageBytes;
  static constexpr int kEpiSmem = (kWarps * NV * (D + 4) + 2 * kWarps * 8) * 4;  // its own region
  static constexpr int kSmem = kStageSmem + kEpiSmem + 1024;
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

// One (sequence, kv head, partition) work unit.
struct Unit {
  int b, g, p, L, np, first_page, npages;
  Range r;
};

// Unit u of the p-major enumeration; false when the partition is empty.
__device__ __forceinline__ bool make_unit(const Args& a, long long u, Unit& x, bool report) {
  const int BH = a.B * a.Hkv;
  x.p = (int)(u / BH);
  const int rem = (int)(u % BH);
  x.b = rem / a.Hkv;
  x.g = rem % a.Hkv;
  x.L = load_len(a, x.b, report && x.p == 0 && x.g == 0);
  x.r = partition_range(x.L, a.T, x.p, a.window, a.psize, a.thresh);
  x.np = seq_partitions(x.L, a.T, a.window, a.psize, a.thresh);
  if (x.r.start >= x.r.end) return false;
  x.first_page = x.r.start / kPage;
  x.npages = (x.r.end - 1) / kPage - x.first_page + 1;
  return true;
}

__device__ __forceinline__ int warp_pages(int npages, int w) {
  return npages > w ? (npages - w + kWarps - 1) / kWarps : 0;
}

// Split-K completion ticket of one (sequence, kv head): the word holds (generation << 32)
// | count. Returns true for the caller that completes the np-th partition of this call.
__device__ __forceinline__ bool take_ticket(unsigned long long* t, unsigned gen, int np) {
  unsigned long long cur = atomicAdd(t, 0ull);
  for (;;) {
    const unsigned c1 = (unsigned)(cur >> 32) == gen ? (unsigned)cur + 1u : 1u;
    const unsigned long long nxt = ((unsigned long long)gen << 32) | c1;
    const unsigned long long prev = atomicCAS(t, cur, nxt);
    if (prev == cur) return c1 == (unsigned)np;
    cur = prev;
  }
}

// Persistent: gridDim.x CTAs walk the units u = blockIdx.x, blockIdx.x + gridDim.x, ...
template <int FMT, int D, int NV>
__global__ void __launch_bounds__(kThreads, (D == 128 ? 3 : 2))
    partition_tc_kernel(const Args a, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  using T = Tc<FMT, D, NV>;
  const int G = a.Hq / a.Hkv, V = a.T * G;  // group size, virtual heads in use (<= NV)
  constexpr int DP = D + 4;  // padded row of the epilogue buffer (spreads the banks)
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const long long total = (long long)a.P * a.B * a.Hkv, stride = gridDim.x;

  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps * T::kStages];
  __shared__ int ep_flag;
  const uint32_t smem = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  unsigned char* smem_gen = smem_raw + (smem - ptx::smem_u32(smem_raw));
  const uint32_t bar0 = ptx::smem_u32(bars) + w * T::kStages * 8;
  const uint32_t stage0 = smem + w * T::kStages * T::kStageBytes;
  float* ep_o = reinterpret_cast<float*>(smem_gen + T::kStageSmem);  // [kWarps][NV][DP]
  float* ep_m = ep_o + kWarps * NV * DP;                              // [kWarps][8]
  float* ep_l = ep_m + kWarps * 8;                                    // [kWarps][8]

  if (lane == 0) {
    ptx::prefetch_tensor_map(&kmap);
    ptx::prefetch_tensor_map(&vmap);
    for (int s = 0; s < T::kStages; ++s) ptx::mbar_init(bar0 + 8 * s, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  // ---- producer: this warp's pages of this CTA's units, issued kStages ahead of use
  long long pu = (long long)blockIdx.x - stride;  // producer's unit
  Unit pun{};
  int pk = 0, pn = 0, bid = -1;
  bool pdone = false;
  uint32_t issued = 0, valid_mask = 0;  // bit s: the page in stage s has a valid block
  auto load_bids = [&](int chunk) {  // lane l: physical block of local page 32 * chunk + l
    const int i = 32 * chunk + lane;
    bid = i < pn ? load_block(a, pun.b, pun.first_page + w + kWarps * i) : -1;
  };
  auto issue_one = [&]() {  // all lanes (warp-uniform); lane 0 issues the copies
    if (pdone) return;
    while (pk >= pn) {
      pu += stride;
      if (pu >= total) {
        pdone = true;
        return;
      }
      if (make_unit(a, pu, pun, false)) {
        pn = warp_pages(pun.npages, w);
        pk = 0;
        if (pn) load_bids(0);
      } else {
        pn = pk = 0;
      }
    }
    if (pk > 0 && (pk & 31) == 0) load_bids(pk >> 5);
    const int phys = __shfl_sync(kFull, bid, pk & 31);
    const int s = issued % T::kStages;
    valid_mask = phys >= 0 ? (valid_mask | (1u << s)) : (valid_mask & ~(1u << s));
    if (lane == 0) {
      const uint32_t bar = bar0 + 8 * s, dst = stage0 + s * T::kStageBytes;
      if (phys < 0) {
        ptx::mbar_arrive(bar);  // completes the phase with nothing loaded
      } else {
        ptx::fence_proxy_async();
        ptx::mbar_arrive_expect_tx(bar, T::kStageBytes);
        const int y = (phys * a.Hkv + pun.g) * kPage;
#pragma unroll
        for (int u = 0; u < T::kSubs; ++u) {
          ptx::tma_load_2d(dst + u * T::kSubBytes, &kmap, u * (128 / T::kElemBytes), y, bar);
          ptx::tma_load_2d(dst + T::kPageBytes + u * T::kSubBytes, &vmap, u * (128 / T::kElemBytes), y, bar);
        }
      }
    }
    ++pk;
    ++issued;
  };
  for (int k = 0; k < T::kStages; ++k) issue_one();

  // hi/lo role of this thread's two columns (NV <= 4: column c carries part c / NV) and the
  // virtual head each column scores (columns past V repeat earlier ones and are not stored)
  int part[2], vcol[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    part[j] = NV <= 4 ? (2 * tig + j) / NV : 0;
    vcol[j] = ((2 * tig + j) % NV) % V;
  }
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix index and row of this lane's address
  const float cap = a.softcap;
  const float out_scale = FMT == DA_KV_FP8_E4M3 ? __ldg(a.v_scales) : 1.0f;
  uint32_t consumed = 0;
  bool stalled = false;

  // ---- consumer: the same units in the same order
  for (long long cu = blockIdx.x; cu < total; cu += stride) {
    Unit un;
    if (!make_unit(a, cu, un, tid == 0)) {
      if (un.p == 0 && un.np == 0)  // an empty sequence: zero output rows
        for (int idx = tid; idx < V * D; idx += kThreads) {
          const int v = idx / D;
          a.out[(((size_t)un.b * a.T + v / G) * a.Hq + un.g * G + v % G) * D + idx % D] = 0.0f;
        }
      continue;
    }
    const int cn = warp_pages(un.npages, w);

    // -- query fragments (B operand of S^T): column n holds virtual head (n % NV) % V
    const int qv = (gid % NV) % V;
    const uint16_t* qrow = a.q + (((size_t)un.b * a.T + qv / G) * a.Hq + un.g * G + qv % G) * D;
    // tokens each of this thread's two columns attends in this unit: its query token's causal
    // (and window) limits, within the partition
    int lo_c[2], hi_c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int pos = un.L - a.T + vcol[j] / G, lo = window_start(pos, a.window);
      lo_c[j] = lo > un.r.start ? lo : un.r.start;
      hi_c[j] = pos + 1 < un.r.end ? pos + 1 : un.r.end;
    }
    uint32_t qf[T::kKS][2];
    float score_scale = a.scale * kLog2e;  // applied to the MMA result (log2 domain)
    if constexpr (FMT == DA_KV_BF16) {
#pragma unroll
      for (int ks = 0; ks < T::kKS; ++ks) {
        qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tig);
        qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tig);
      }
    } else {
      // f16 operands: scale q by a power of two so that max|q| fits f16 (exact); undone in the score scale
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
    const float cap_pre = cap > 0.0f ? score_scale / (cap * kLog2e) : 0.0f;  // s_nat / cap
    const float cap_post = cap * kLog2e;

    // -- running state: column c = 2 * tig + j of S^T and of every O^T column tile
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float o[T::kNT][T::kMT][4];
#pragma unroll
    for (int t = 0; t < T::kNT; ++t)
#pragma unroll
      for (int mt = 0; mt < T::kMT; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[t][mt][e] = 0.0f;

    for (int i = 0; i < cn; ++i) {
      const int s = consumed % T::kStages;
      if (!stalled && !ptx::mbar_wait(bar0 + 8 * s, (consumed / T::kStages) & 1)) {
        stalled = true;
        if (lane == 0) atomicOr(a.err, DA_DEVERR_TIMEOUT);
      }
      if (!stalled && (valid_mask & (1u << s))) {
        const uint32_t kb = stage0 + s * T::kStageBytes, vb = kb + T::kPageBytes;
        const int tok0 = (un.first_page + w + kWarps * i) * kPage;
        // -- S^T = K . Q^T
        float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (FMT == DA_KV_BF16) {
#pragma unroll
          for (int ks = 0; ks < T::kKS; ++ks) {
            const int row = ri + 8 * (mi & 1), chunk = 2 * ks + (mi >> 1);
            uint32_t af[4];
            ptx::ldmatrix_x4(af, swz(kb + (chunk >> 3) * T::kSubBytes, row, chunk & 7));
            mma<FMT>(sc, af, qf[ks][0], qf[ks][1]);
          }
        } else {
#pragma unroll
          for (int j2 = 0; j2 < T::kKS / 2; ++j2) {
            const int row = ri + 8 * (mi & 1), chunk = 2 * j2 + (mi >> 1);
            uint32_t rr[4];
            ptx::ldmatrix_x4(rr, swz(kb + (chunk >> 3) * T::kSubBytes, row, chunk & 7));
            const uint32_t a0[4] = {e4m3x2_to_f16x2(rr[0]), e4m3x2_to_f16x2(rr[1]), e4m3x2_to_f16x2(rr[0] >> 16),
                                    e4m3x2_to_f16x2(rr[1] >> 16)};
            mma<FMT>(sc, a0, qf[2 * j2][0], qf[2 * j2][1]);
            const uint32_t a1[4] = {e4m3x2_to_f16x2(rr[2]), e4m3x2_to_f16x2(rr[3]), e4m3x2_to_f16x2(rr[2] >> 16),
                                    e4m3x2_to_f16x2(rr[3] >> 16)};
            mma<FMT>(sc, a1, qf[2 * j2 + 1][0], qf[2 * j2 + 1][1]);
          }
        }
        // -- scale, softcap, mask; sc[0], sc[1]: token gid; sc[2], sc[3]: token gid + 8
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = tok0 + gid + (e >> 1) * 8, j = e & 1;
          const float x = cap > 0.0f ? cap_post * tanhf(sc[e] * cap_pre) : sc[e] * score_scale;
          sc[e] = (t >= lo_c[j] && t < hi_c[j]) ? x : -INFINITY;
        }
        // -- online softmax per column
        float alpha[2], pr[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float mx = fmaxf(sc[j], sc[j + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
          const float mn = fmaxf(m_run[j], mx);
          const bool none = mn == -INFINITY;
          alpha[j] = none ? 1.0f : exp2f(m_run[j] - mn);
          pr[j] = none ? 0.0f : exp2f(sc[j] - mn);
          pr[j + 2] = none ? 0.0f : exp2f(sc[j + 2] - mn);
          l_run[j] = l_run[j] * alpha[j] + pr[j] + pr[j + 2];
          m_run[j] = mn;
        }
        if (__any_sync(kFull, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
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
            ptx::ldmatrix_x4_trans(af, swz(vb + (chunk >> 3) * T::kSubBytes, row, chunk & 7));
#pragma unroll
            for (int t = 0; t < T::kNT; ++t) mma<FMT>(o[t][mt], af, pb[t][0], pb[t][1]);
          }
        } else {
#pragma unroll
          for (int j2 = 0; j2 < T::kMT / 2; ++j2) {
            const int row = ri + 8 * (mi >> 1), chunk = 2 * j2 + (mi & 1);
            uint32_t rr[4];
            ptx::ldmatrix_x4_trans(rr, swz(vb + (chunk >> 3) * T::kSubBytes, row, chunk & 7));
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
      if (!stalled) issue_one();  // after a copy that never arrived, issue nothing more
      ++consumed;
    }

    // -- unit epilogue: each warp's (o, m, l) per head into shared memory (hi + lo combined)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      l_run[j] += __shfl_xor_sync(kFull, l_run[j], 4);
      l_run[j] += __shfl_xor_sync(kFull, l_run[j], 8);
      l_run[j] += __shfl_xor_sync(kFull, l_run[j], 16);
    }
#pragma unroll
    for (int mt = 0; mt < T::kMT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = o[0][mt][e];
        if constexpr (NV == 8) v += o[T::kNT - 1][mt][e];
        if constexpr (NV == 4) v += __shfl_xor_sync(kFull, v, 2);
        if constexpr (NV == 2) v += __shfl_xor_sync(kFull, v, 1);
        if constexpr (NV == 1) v += (e & 1) ? 0.0f : o[0][mt][e + 1];
        const int col = 2 * tig + (e & 1);
        const int rowd = FMT == DA_KV_BF16 ? 16 * mt + gid + ((e >> 1) ? 8 : 0) : 16 * mt + 2 * gid + (e >> 1);
        if (col < V) ep_o[(w * NV + col) * DP + rowd] = v;
      }
    if (gid == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        ep_m[w * 8 + 2 * tig + j] = m_run[j];
        ep_l[w * 8 + 2 * tig + j] = l_run[j];
      }
    }
    __syncthreads();
    // -- merge the four warps: the unit's partial (split sequence) or its output (unsplit)
    const bool direct = un.np == 1;
    for (int idx = tid; idx < V * D; idx += kThreads) {
      const int v = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, ep_m[ww * 8 + v]);
      float acc = 0.0f, l = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float mw = ep_m[ww * 8 + v];
        const float wt = mw == -INFINITY ? 0.0f : exp2f(mw - M);
        acc += wt * ep_o[(ww * NV + v) * DP + d];
        l += wt * ep_l[ww * 8 + v];
      }
      const size_t bh = ((size_t)un.b * a.T + v / G) * a.Hq + un.g * G + v % G;
      if (direct) {
        a.out[bh * D + d] = l > 0.0f ? acc * out_scale / l : 0.0f;
      } else {
        const size_t pi = bh * a.P + un.p;
        a.part_o[pi * D + d] = acc;
        if (d == 0) {
          a.part_m[pi] = M;
          a.part_l[pi] = l;
        }
      }
    }
    if (!direct) {
      // -- the last partition of (sequence, kv head) to finish combines all of them:
      //    M = max_p m_p, w_p = 2^(m_p - M), out = sum_p w_p o_p / sum_p w_p l_p
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const bool last = take_ticket(a.tickets + (size_t)un.b * a.Hkv + un.g, a.gen, un.np);
        if (last) __threadfence();
        ep_flag = last;
      }
      __syncthreads();
      if (ep_flag) {
        // (1) per virtual head, warps over partitions: M = max_p m_p and the sum of l_p 2^(m_p - M)
        float* red_m = ep_m;  // [8] (the warps' per-column values are no longer needed)
        float* red_l = ep_l;  // [8]
        for (int v = w; v < V; v += kWarps) {
          const size_t base = (((size_t)un.b * a.T + v / G) * a.Hq + un.g * G + v % G) * a.P;
          float M = -INFINITY;
          for (int pp = lane; pp < un.np; pp += 32) M = fmaxf(M, __ldcg(a.part_m + base + pp));
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o2));
          float l = 0.0f;
          for (int pp = lane; pp < un.np; pp += 32) {
            const float mp = __ldcg(a.part_m + base + pp);
            l += mp == -INFINITY ? 0.0f : exp2f(mp - M) * __ldcg(a.part_l + base + pp);
          }
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) l += __shfl_xor_sync(kFull, l, o2);
          if (lane == 0) {
            red_m[v] = M;
            red_l[v] = l;
          }
        }
        __syncthreads();
        // (2) out = sum_p 2^(m_p - M) o_p / that sum, partitions in chunks of 32 whose weights
        //     sit in shared memory, the loads of a chunk independent of each other
        constexpr int kChunk = 32;
        float* wgt = ep_o;  // [V][kChunk], reusing the merge buffer
        constexpr int kOut = (NV * D + kThreads - 1) / kThreads;
        float acc[kOut];
#pragma unroll
        for (int k = 0; k < kOut; ++k) acc[k] = 0.0f;
        for (int p0 = 0; p0 < un.np; p0 += kChunk) {
          for (int i = tid; i < V * kChunk; i += kThreads) {
            const int v = i / kChunk, pp = p0 + i % kChunk;
            const size_t base = (((size_t)un.b * a.T + v / G) * a.Hq + un.g * G + v % G) * a.P;
            const float mp = pp < un.np ? __ldcg(a.part_m + base + pp) : -INFINITY;
            wgt[i] = mp == -INFINITY ? 0.0f : exp2f(mp - red_m[v]);
          }
          __syncthreads();
          const int n = un.np - p0 < kChunk ? un.np - p0 : kChunk;
#pragma unroll
          for (int k = 0; k < kOut; ++k) {
            const int idx = tid + k * kThreads;
            if (idx < V * D) {
              const int v = idx / D, d = idx % D;
              const float* src =
                  a.part_o + ((((size_t)un.b * a.T + v / G) * a.Hq + un.g * G + v % G) * a.P + p0) * D + d;
              float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
              int pp = 0;
              for (; pp + 4 <= n; pp += 4) {
                s0 += wgt[v * kChunk + pp] * __ldcg(src + (size_t)pp * D);
                s1 += wgt[v * kChunk + pp + 1] * __ldcg(src + (size_t)(pp + 1) * D);
                s2 += wgt[v * kChunk + pp + 2] * __ldcg(src + (size_t)(pp + 2) * D);
                s3 += wgt[v * kChunk + pp + 3] * __ldcg(src + (size_t)(pp + 3) * D);
              }
              for (; pp < n; ++pp) s0 += wgt[v * kChunk + pp] * __ldcg(src + (size_t)pp * D);
              acc[k] += (s0 + s1) + (s2 + s3);
            }
          }
          __syncthreads();
        }
#pragma unroll
        for (int k = 0; k < kOut; ++k) {
          const int idx = tid + k * kThreads;
          if (idx < V * D) {
            const int v = idx / D, d = idx % D;
            const size_t bh = ((size_t)un.b * a.T + v / G) * a.Hq + un.g * G + v % G;
            const float l = red_l[v];
            a.out[bh * D + d] = l > 0.0f ? acc[k] * out_scale / l : 0.0f;
          }
        }
      }
    }
    __syncthreads();  // the epilogue buffer is reused by the next unit
  }
  // every page issued has been consumed (producer and consumer walk the same pages)
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

template <int FMT, int D, int NV>
cudaError_t launch_fixed(const Args& a, cudaStream_t s) {
  using T = Tc<FMT, D, NV>;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.Hkv * kPage;
  if (!encode_cache_map(&km, a.k_cache, T::kElemBytes, D, rows) ||
      !encode_cache_map(&vm, a.v_cache, T::kElemBytes, D, rows))
    return cudaErrorInvalidValue;
  auto kern = partition_tc_kernel<FMT, D, NV>;
  static DeviceFlags attr;
  cudaError_t e = ensure_dynamic_smem(kern, T::kSmem, attr);
  if (e != cudaSuccess) return e;
  // one CTA per work unit: the unit loop of the kernel then runs once per CTA, and a
  // CTA's start-up loads overlap with other CTAs' streaming
  const long long units = (long long)a.P * a.B * a.Hkv;
  if (units > 0x7fffffffll) return cudaErrorInvalidValue;
  const int grid = (int)units;
  kern<<<grid, kThreads, T::kSmem, s>>>(a, km, vm);
  return cudaGetLastError();
}

template <int FMT, int D>
cudaError_t launch_g(const Args& a, cudaStream_t s) {
  const int v = a.T * (a.Hq / a.Hkv);  // virtual heads, padded to a power of two
  if (v <= 1) return launch_fixed<FMT, D, 1>(a, s);
  if (v <= 2) return launch_fixed<FMT, D, 2>(a, s);
  if (v <= 4) return launch_fixed<FMT, D, 4>(a, s);
  if (v <= 8) return launch_fixed<FMT, D, 8>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_partition_tc(const Args& a, cudaStream_t s) {
  if (a.fmt == DA_KV_BF16) return a.D == 128 ? launch_g<DA_KV_BF16, 128>(a, s) : launch_g<DA_KV_BF16, 256>(a, s);
  if (a.fmt == DA_KV_FP8_E4M3)
    return a.D == 128 ? launch_g<DA_KV_FP8_E4M3, 128>(a, s) : launch_g<DA_KV_FP8_E4M3, 256>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace da
