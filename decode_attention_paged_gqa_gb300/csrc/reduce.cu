// reduce.cu -- the float-precision reduce across split-K partitions (attention.rs README:
// one reduce kernel, in fp32, is shared by the split-K decode kernels of all formats;
// turboquant-rs 0.4.1, src/cache/cuda/attention.rs: partial output, max and sum buffers of
// [heads * partitions]).
//
// For sequence b, head h with partials (o_p, m_p, l_p), p < P_b (m in log2 units):
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
// When the partition kernel dealt each partition's pages to ksub sub-items, every sub-item
// that had pages wrote a partial of its own, and all of them are combined the same way
// (sub-item s of partition p has pages when s < the partition's page count).
// One CTA per (row, head); the partials' loads are issued together, with the partitions spread
// over thread groups (128 threads: 4 groups at D = 128, 2 at D = 256; 256 threads, for 32 or
// more partitions: 8 / 4): each thread's first m_p, l_p and float4 columns of o_p go out with
// the context length, the rest of m_p and l_p in one round and of o_p in one more.
// An empty sequence (or a query token that attends nothing) gets an all-zero row. An
// unsplit sequence of a format without a codebook value side was written by the partition
// kernel and is skipped here. When the values are stored on the rotated basis the result
// is un-rotated here: out <- diag(sign) H out / sqrt(D). For an FP8 value side the
// per-tensor V scale is applied once, here.
#include <cuda_runtime.h>

#include <cmath>

#include "da_internal.cuh"
#include "fwht.cuh"
#include "kv_formats.cuh"
#include "ptx.cuh"

namespace da {
namespace {

// Folds the partial (M, s) into (M, s): s <- s 2^(M - M') + s_o 2^(M_o - M'), M' = max(M, M_o);
// an empty side (M = -inf, s = 0) contributes nothing.
__device__ __forceinline__ void fold(float& M, float& s, float Mo, float so) {
  const float Mn = fmaxf(M, Mo);
  if (Mn == -INFINITY) return;
  s = s * exp2f(M - Mn) + so * exp2f(Mo - Mn);
  M = Mn;
}

template <int D, bool kUnrotate, int kThreads>
__global__ void __launch_bounds__(kThreads) reduce_kernel(const Args a) {
  constexpr int kCols = D / 4, kGroups = kThreads / kCols;  // float4 columns; partition groups
  const int h = blockIdx.x, row = blockIdx.y, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;  // row = b * T + query token
  const int b = row / a.T;
  ptx::grid_dependency_wait();  // the partials of the partition kernel before this one
  extern __shared__ float w_s[];  // [P]: m_p, then the weights 2^(m_p - M)
  __shared__ float4 red_o[kGroups][kCols];
  __shared__ float red_m[kThreads / 32], red_s[kThreads / 32];
  __shared__ float x_s[kUnrotate ? D : 1];
  const int PK = a.P * a.ksub;  // partial slots per row
  const size_t base = ((size_t)row * a.Hq + h) * PK;
  // The thread's first partials (max and sum of slot tid; kPre float4 columns of its group's
  // first slots), loaded together with the context length, before the row's partition count
  // is known: every row has PK slots, and a slot is used below only if it holds a partial of
  // this row. The three dependent rounds (length, then maxima and sums, then outputs) become
  // one for a row of up to kPre * kGroups partials.
  constexpr int kPre = 4;
  const int col = tid % kCols, group = tid / kCols;
  const float4* src = reinterpret_cast<const float4*>(a.part_o + base * D) + col;
  const float m_pre = tid < PK ? a.part_m[base + tid] : -INFINITY, l_pre = tid < PK ? a.part_l[base + tid] : 0.0f;
  float4 o_pre[kPre];
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int j = group + i * kGroups;
    o_pre[i] = j < PK ? src[(size_t)j * kCols] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  const int L = load_len(a, b, false);
  const int np = seq_partitions(L, a.T, a.window, a.psize, a.thresh);
  float* out = a.out + ((size_t)row * a.Hq + h) * D;
  if (np == 0) {
    for (int d = tid; d < D; d += kThreads) out[d] = 0.0f;
    return;
  }
  if (np == 1 && a.ksub == 1 && !kUnrotate) return;
  const int nk = np * a.ksub;  // partial slots of this row

  // M = max_p m_p and s = sum_p 2^(m_p - M) l_p, each thread folding its partials
  // j = tid, tid + kThreads, ... (m_p and l_p loaded together), then across the block
  float M = -INFINITY, s = 0.0f;
  for (int j = tid; j < nk; j += kThreads) {
    bool valid = true;
    if (a.ksub > 1) {  // sub-item j % ksub of partition j / ksub: written iff it had pages
      const Range r = partition_range(L, a.T, j / a.ksub, a.window, a.psize, a.thresh);
      valid = j % a.ksub < (r.end - 1) / kBlockSize - r.start / kBlockSize + 1;
    }
    float m = j == tid ? m_pre : a.part_m[base + j], l = j == tid ? l_pre : a.part_l[base + j];
    if (!valid) m = -INFINITY, l = 0.0f;
    w_s[j] = m;
    fold(M, s, m, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float Mo = __shfl_xor_sync(0xffffffffu, M, o), so = __shfl_xor_sync(0xffffffffu, s, o);
    fold(M, s, Mo, so);
  }
  if (lane == 0) {
    red_m[w] = M;
    red_s[w] = s;
  }
  __syncthreads();
  M = red_m[0];
  s = red_s[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) fold(M, s, red_m[i], red_s[i]);
  for (int j = tid; j < nk; j += kThreads) w_s[j] = M == -INFINITY ? 0.0f : exp2f(w_s[j] - M);
  __syncthreads();

  // sum_p w_p o_p: thread (group, column) takes float4 column `col` of partitions
  // group, group + kGroups, ... (the first kPre of them loaded above); the groups are then
  // added up
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < kPre; ++i) {
    const int j = group + i * kGroups;
    const float wp = j < nk ? w_s[j] : 0.0f;
    if (wp == 0.0f) continue;  // an empty partial, a slot never written, or past the row's partials
    acc.x = fmaf(wp, o_pre[i].x, acc.x);
    acc.y = fmaf(wp, o_pre[i].y, acc.y);
    acc.z = fmaf(wp, o_pre[i].z, acc.z);
    acc.w = fmaf(wp, o_pre[i].w, acc.w);
  }
#pragma unroll 8
  for (int j = group + kPre * kGroups; j < nk; j += kGroups) {
    const float wp = w_s[j];
    if (wp == 0.0f) continue;  // an empty partial, or a sub-item slot that was never written
    const float4 o = src[(size_t)j * kCols];
    acc.x = fmaf(wp, o.x, acc.x);
    acc.y = fmaf(wp, o.y, acc.y);
    acc.z = fmaf(wp, o.z, acc.z);
    acc.w = fmaf(wp, o.w, acc.w);
  }
  red_o[group][col] = acc;
  __syncthreads();
  const float inv_l = (s > 0.0f ? 1.0f / s : 0.0f) * (v_side(a.fmt) == kSideFP8 ? __ldg(a.v_scales) : 1.0f);
  const float* red = reinterpret_cast<const float*>(red_o);
  for (int d = tid; d < D; d += kThreads) {
    float v = red[d];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) v += red[g * D + d];
    if (kUnrotate)
      x_s[d] = v * inv_l;
    else
      out[d] = v * inv_l;
  }
  if (kUnrotate) {
    fwht_shared<D>(x_s);
    const float inv_sqrt_d = 1.0f / sqrtf((float)D);
    for (int d = tid; d < D; d += kThreads) out[d] = __ldg(a.sign + d) * x_s[d] * inv_sqrt_d;
  }
}

template <int D>
cudaError_t launch_d(const Args& a, cudaStream_t s) {
  dim3 grid(a.Hq, a.B * a.T);
  const size_t smem = sizeof(float) * (size_t)a.P * a.ksub;  // <= kMaxPartitions: within the default 48 KB
  // scheduled during the partition kernel's last CTAs; waits for its partials in-kernel. Many
  // partitions per row: 256 threads, so each thread's loads are one round; few: 128, so that a
  // large batch's rows stay within one wave of CTAs.
  const bool rot = is_codebook(v_side(a.fmt));
  if (a.P * a.ksub >= 32)
    return rot ? launch_pdl(reduce_kernel<D, true, 256>, grid, dim3(256), smem, s, a)
               : launch_pdl(reduce_kernel<D, false, 256>, grid, dim3(256), smem, s, a);
  return rot ? launch_pdl(reduce_kernel<D, true, 128>, grid, dim3(128), smem, s, a)
             : launch_pdl(reduce_kernel<D, false, 128>, grid, dim3(128), smem, s, a);
}

}  // namespace

cudaError_t launch_reduce(const Args& a, cudaStream_t s) {
  return a.D == 128 ? launch_d<128>(a, s) : launch_d<256>(a, s);
}

}  // namespace da
