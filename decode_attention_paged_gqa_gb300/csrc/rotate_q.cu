// rotate_q.cu -- query pre-rotation for the 4-bit codebook format:
//   q_rot = H diag(sign) q / sqrt(D),
// the rotation the cache's vectors were stored in, so that q_rot . k_rot = q . k and the
// partition kernel never leaves the rotated basis (turboquant-rs 0.4.1,
// src/cache/cuda/attention.rs: the fused kernel takes sign_pattern and reads the
// compressed cache directly, with no full dequantisation).
#include <cuda_runtime.h>

#include <cmath>

#include "da_internal.cuh"
#include "fwht.cuh"
#include "ptx.cuh"

namespace da {
namespace {

template <int D>
__global__ void __launch_bounds__(128) rotate_q_kernel(const Args a) {
  const int h = blockIdx.x, row = blockIdx.y;  // row = b * T + query token
  __shared__ float x[D];
  ptx::grid_dependents_launch();  // the partition kernel may be scheduled meanwhile
  const size_t base = ((size_t)row * a.Hq + h) * D;
  for (int d = threadIdx.x; d < D; d += blockDim.x) x[d] = bf16_to_f32(a.q[base + d]) * __ldg(a.sign + d);
  fwht_shared<D>(x);
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  for (int d = threadIdx.x; d < D; d += blockDim.x) a.q_rot[base + d] = x[d] * inv_sqrt_d;
}

}  // namespace

cudaError_t launch_rotate_q(const Args& a, cudaStream_t s) {
  dim3 grid(a.Hq, a.B * a.T);
  if (a.D == 128)
    rotate_q_kernel<128><<<grid, 128, 0, s>>>(a);
  else
    rotate_q_kernel<256><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace da
