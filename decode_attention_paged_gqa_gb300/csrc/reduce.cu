// reduce.cu -- the float-precision reduce across split-K partitions (attention.rs README:
// one reduce kernel, in fp32, is shared by the split-K decode kernels of all formats;
// turboquant-rs 0.4.1, src/cache/cuda/attention.rs: partial output, max and sum buffers of
// [heads * partitions]).
//
// For sequence b, head h with partials (o_p, m_p, l_p), p < P_b (m in log2 units):
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
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

namespace da {
namespace {

template <int D, bool kUnrotate>
__global__ void __launch_bounds__(128) reduce_kernel(const Args a) {
  const int h = blockIdx.x, row = blockIdx.y, tid = threadIdx.x, lane = tid & 31;  // row = b * T + query token
  const int b = row / a.T;
  extern __shared__ float w_s[];  // [P] weights
  __shared__ float x_s[D];
  __shared__ float inv_l_s;
  const int L = load_len(a, b, false);
  const int np = seq_partitions(L, a.T, a.window, a.psize, a.thresh);
  float* out = a.out + ((size_t)row * a.Hq + h) * D;
  if (np == 0) {
    for (int d = tid; d < D; d += blockDim.x) out[d] = 0.0f;
    return;
  }
  if (np == 1 && !kUnrotate) return;
  const size_t base = ((size_t)row * a.Hq + h) * a.P;
  if (tid < 32) {
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32) M = fmaxf(M, a.part_m[base + p]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float lsum = 0.0f;
    for (int p = lane; p < np; p += 32) {
      const float w = M == -INFINITY ? 0.0f : exp2f(a.part_m[base + p] - M);
      w_s[p] = w;
      lsum += w * a.part_l[base + p];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (lane == 0) inv_l_s = lsum > 0.0f ? 1.0f / lsum : 0.0f;
  }
  __syncthreads();
  const float inv_l = inv_l_s * (v_side(a.fmt) == kSideFP8 ? __ldg(a.v_scales) : 1.0f);
  for (int d = tid; d < D; d += blockDim.x) {
    float acc = 0.0f;
    for (int p = 0; p < np; ++p) acc = fmaf(w_s[p], a.part_o[(base + p) * D + d], acc);
    if (kUnrotate)
      x_s[d] = acc * inv_l;
    else
      out[d] = acc * inv_l;
  }
  if (kUnrotate) {
    fwht_shared<D>(x_s);
    const float inv_sqrt_d = 1.0f / sqrtf((float)D);
    for (int d = tid; d < D; d += blockDim.x) out[d] = __ldg(a.sign + d) * x_s[d] * inv_sqrt_d;
  }
}

template <int D>
cudaError_t launch_d(const Args& a, cudaStream_t s) {
  dim3 grid(a.Hq, a.B * a.T);
  const size_t smem = sizeof(float) * (size_t)a.P;  // P <= kMaxPartitions: within the default 48 KB
  if (is_codebook(v_side(a.fmt)))
    reduce_kernel<D, true><<<grid, 128, smem, s>>>(a);
  else
    reduce_kernel<D, false><<<grid, 128, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce(const Args& a, cudaStream_t s) {
  return a.D == 128 ? launch_d<128>(a, s) : launch_d<256>(a, s);
}

}  // namespace da
