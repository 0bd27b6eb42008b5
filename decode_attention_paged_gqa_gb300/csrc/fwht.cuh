// fwht.cuh -- in-place fast Walsh-Hadamard transform of D floats in shared memory.
//
// Computes y = H x for the D x D Sylvester Hadamard matrix H[i][j] = (-1)^popcount(i & j),
// one butterfly stage (u + v, u - v) per bit of the index. The codebook format rotates
// each cached vector by H diag(sign) / sqrt(D) (attention.rs README, KV Cache Formats
// table: 4-bit "Walsh-Hadamard" formats; turboquant-rs 0.4.1, src/cache/cuda/attention.rs:
// the sign_pattern input), so queries are rotated and outputs un-rotated with this.
#pragma once

namespace da {

// All threads of the block take part; x has D entries; ends with a __syncthreads().
template <int D>
__device__ __forceinline__ void fwht_shared(float* x) {
  static_assert((D & (D - 1)) == 0, "D must be a power of two");
#pragma unroll
  for (int len = 1; len < D; len <<= 1) {
    __syncthreads();
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
      const int lo = (i / len) * 2 * len + (i % len), hi = lo + len;
      const float u = x[lo], v = x[hi];
      x[lo] = u + v;
      x[hi] = u - v;
    }
  }
  __syncthreads();
}

}  // namespace da
