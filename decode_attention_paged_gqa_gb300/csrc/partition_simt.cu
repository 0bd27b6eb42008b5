// partition_simt.cu -- split-K partition kernel on the CUDA cores (fp32 throughout), used
// for the formats with a codebook side: 4-bit K and V, FP8 K + 4-bit V, 3-bit K + 4-bit V.
//
// One CTA per (partition p, kv head g, sequence b). It walks the partition's tokens in
// tiles of 32: the tile's K and V rows are gathered through the block table, dequantised
// to fp32 in shared memory, scored against the query heads of the group, folded into an
// online softmax (running max m, running sum l, unnormalised output o), and finally the
// partition's (o, m, l) are written to the workspace for the reduce kernel.
// (attention.rs README: split-K decode per KV format with a float-precision reduce;
// turboquant-rs 0.4.1, src/cache/cuda/attention.rs: partial output, max and sum buffers.)
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>

#include "da_internal.cuh"
#include "kv_formats.cuh"

namespace da {
namespace {

constexpr int kThreads = 128;
constexpr int kTile = 32;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// NV: the (query token, head) pairs of the group, padded to a power of two: "virtual
// heads" v = jq * G + h, each with its own causal limit (query token jq sits at position
// L - T + jq).
template <int FMT, int D, int NV>
__global__ void __launch_bounds__(kThreads) partition_simt_kernel(const Args a) {
  const int p = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.Hq / a.Hkv, V = a.T * G;
  const int L = load_len(a, b, p == 0 && g == 0 && tid == 0);
  const Range r = partition_range(L, a.T, p, a.window, a.psize, a.thresh);
  if (r.start >= r.end) return;

  extern __shared__ float smem[];
  float* q_s = smem;                        // [NV][D]
  float* k_s = q_s + NV * D;                // [kTile][D + 1]
  float* v_s = k_s + kTile * (D + 1);       // [kTile][D]
  float* p_s = v_s + kTile * D;             // [NV][kTile]
  float* alpha_s = p_s + NV * kTile;        // [NV]
  float* cbk_s = alpha_s + NV;              // [16] key codebook
  float* cbv_s = cbk_s + 16;                // [16] value codebook
  int* ok_s = reinterpret_cast<int*>(cbv_s + 16);  // [kTile]
  constexpr int KS = k_side(FMT), VS = v_side(FMT);

  // queries of the group's virtual heads (rotated ones when the keys are on the rotated basis)
  for (int i = tid; i < NV * D; i += kThreads) {
    const int v = i / D, d = i % D;
    float x = 0.0f;
    if (v < V) {
      const size_t qi = (((size_t)b * a.T + v / G) * a.Hq + g * G + v % G) * D + d;
      x = is_codebook(KS) ? a.q_rot[qi] : bf16_to_f32(a.q[qi]);
    }
    q_s[i] = x;
  }
  if (tid < 16) {
    if (is_codebook(KS)) cbk_s[tid] = tid < (KS == kSideCB3 ? 8 : 16) ? __ldg(a.codebook + tid) : 0.0f;
    if (is_codebook(VS)) cbv_s[tid] = __ldg(a.codebook + (KS == kSideCB3 ? 8 : 0) + tid);
  }

  constexpr int kHeadsPerWarp = (NV + 3) / 4;
  float m_run[kHeadsPerWarp], l_run[kHeadsPerWarp];
  int lo_v[kHeadsPerWarp], hi_v[kHeadsPerWarp];  // tokens virtual head w + 4i attends in this partition
#pragma unroll
  for (int i = 0; i < kHeadsPerWarp; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.0f;
    const int v = warp + 4 * i, pos = L - a.T + (v < V ? v / G : 0);
    const int lo = window_start(pos, a.window), hi = pos + 1;
    lo_v[i] = lo > r.start ? lo : r.start;
    hi_v[i] = hi < r.end ? hi : r.end;
  }
  constexpr int kDimsPerThread = D / kThreads;  // 1 or 2
  float o[NV][kDimsPerThread];
#pragma unroll
  for (int h = 0; h < NV; ++h)
#pragma unroll
    for (int j = 0; j < kDimsPerThread; ++j) o[h][j] = 0.0f;

  constexpr int kChunks = D / 8;  // 8-element chunks per row
  for (int t0 = r.start; t0 < r.end; t0 += kTile) {
    __syncthreads();  // previous tile fully consumed (and q_s / codebooks written on the first pass)
    for (int c = tid; c < kTile * kChunks; c += kThreads) {
      const int row = c / kChunks, col = (c % kChunks) * 8, t = t0 + row;
      float xk[8], xv[8];
      bool ok = false;
      if (t < r.end) {
        const int phys = load_block(a, b, t / a.bs);
        if (phys >= 0) {
          ok = true;
          const size_t crow = ((size_t)phys * a.Hkv + g) * a.bs + t % a.bs;
          SideFormat<KS>::load8(a.k_cache, crow, D, col, side_scale<KS>(a.k_scales, crow), cbk_s, xk);
          // an FP8 value side stays in code units; the reduce applies its scale once
          SideFormat<VS>::load8(a.v_cache, crow, D, col, VS == kSideFP8 ? 1.0f : side_scale<VS>(a.v_scales, crow),
                                cbv_s, xv);
        }
      }
      if (!ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) xk[i] = xv[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        k_s[row * (D + 1) + col + i] = xk[i];
        v_s[row * D + col + i] = xv[i];
      }
      if (col == 0) ok_s[row] = ok;
    }
    __syncthreads();

    // scores and online softmax: warp w owns virtual heads w, w + 4; lane = token of the tile
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
      const int hh = warp + 4 * i;
      if (hh < NV) {
        const int t = t0 + lane;
        float s = -INFINITY;
        if (hh < V && t >= lo_v[i] && t < hi_v[i] && ok_s[lane]) {
          float acc = 0.0f;
          const float* qh = q_s + hh * D;
          const float* kr = k_s + lane * (D + 1);
#pragma unroll 8
          for (int d = 0; d < D; ++d) acc = fmaf(qh[d], kr[d], acc);
          s = a.scale * acc;
          if (a.softcap > 0.0f) s = a.softcap * tanhf(s / a.softcap);
          s *= kLog2e;
        }
        const float m_new = fmaxf(m_run[i], warp_max(s));
        const float alpha = m_new == -INFINITY ? 1.0f : exp2f(m_run[i] - m_new);
        const float pr = s == -INFINITY ? 0.0f : exp2f(s - m_new);
        l_run[i] = l_run[i] * alpha + warp_sum(pr);
        m_run[i] = m_new;
        p_s[hh * kTile + lane] = pr;
        if (lane == 0) alpha_s[hh] = alpha;
      }
    }
    __syncthreads();

    // o[h][d] = alpha_h * o[h][d] + sum_t p[h][t] * v[t][d]; thread owns d = tid (+128)
#pragma unroll
    for (int h = 0; h < NV; ++h) {
      const float al = alpha_s[h];
#pragma unroll
      for (int j = 0; j < kDimsPerThread; ++j) {
        const int d = tid + j * kThreads;
        float acc = o[h][j] * al;
#pragma unroll 8
        for (int t = 0; t < kTile; ++t) acc = fmaf(p_s[h * kTile + t], v_s[t * D + d], acc);
        o[h][j] = acc;
      }
    }
  }

  // partials of this partition
#pragma unroll
  for (int h = 0; h < NV; ++h) {
    if (h >= V) break;
    const size_t base = (((size_t)b * a.T + h / G) * a.Hq + g * G + h % G) * a.P + p;
#pragma unroll
    for (int j = 0; j < kDimsPerThread; ++j) a.part_o[base * D + tid + j * kThreads] = o[h][j];
  }
#pragma unroll
  for (int i = 0; i < kHeadsPerWarp; ++i) {
    const int hh = warp + 4 * i;
    if (hh < V && lane == 0) {
      const size_t base = (((size_t)b * a.T + hh / G) * a.Hq + g * G + hh % G) * a.P + p;
      a.part_m[base] = m_run[i];
      a.part_l[base] = l_run[i];
    }
  }
}

template <int FMT, int D, int NV>
cudaError_t launch_fixed(const Args& a, cudaStream_t s) {
  const size_t smem =
      sizeof(float) * (NV * D + kTile * (D + 1) + kTile * D + NV * kTile + NV + 32) + sizeof(int) * kTile;
  auto kern = partition_simt_kernel<FMT, D, NV>;
  static DeviceFlags attr_set;
  cudaError_t e = ensure_dynamic_smem(kern, smem, attr_set);
  if (e != cudaSuccess) return e;
  dim3 grid(a.P, a.Hkv, a.B);
  kern<<<grid, kThreads, smem, s>>>(a);
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

template <int FMT>
cudaError_t launch_d(const Args& a, cudaStream_t s) {
  return a.D == 128 ? launch_g<FMT, 128>(a, s) : launch_g<FMT, 256>(a, s);
}

}  // namespace

cudaError_t launch_partition_simt(const Args& a, cudaStream_t s) {
  switch (a.fmt) {
    case DA_KV_CB4: return launch_d<DA_KV_CB4>(a, s);
    case DA_KV_FP8K_CB4V: return launch_d<DA_KV_FP8K_CB4V>(a, s);
    case DA_KV_CB3K_CB4V: return launch_d<DA_KV_CB3K_CB4V>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_partition(const Args& a, cudaStream_t s) {
  return a.fmt == DA_KV_BF16 || a.fmt == DA_KV_FP8_E4M3 ? launch_partition_tc(a, s) : launch_partition_simt(a, s);
}

}  // namespace da
