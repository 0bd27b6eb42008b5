// debug_exports.cu -- small kernels that run the partition kernel's own device code on
// request, so that tests can compare its integer work (partition bounds) and its
// dequantisation bit for bit with the CPU oracle.
#include <cuda_runtime.h>

#include "da_internal.cuh"
#include "kv_formats.cuh"

namespace da {
namespace {

__global__ void debug_bounds_kernel(const Args a, int32_t* bounds) {
  const int b = blockIdx.x;
  const int L = load_len(a, b, threadIdx.x == 0);
  for (int p = threadIdx.x; p < a.P; p += blockDim.x) {
    const Range r = partition_range(L, a.T, p, a.window, a.psize, a.thresh);
    const bool valid = r.start < r.end;
    bounds[((size_t)b * a.P + p) * 2 + 0] = valid ? r.start : -1;
    bounds[((size_t)b * a.P + p) * 2 + 1] = valid ? r.end : -1;
  }
}

// One CTA per listed block; each thread dequantises 8-element chunks of its rows.
template <int S>
__global__ void debug_dequant_kernel(const Args a, const void* cache, const float* scales, const int32_t* ids,
                                     const float* codebook, float* out) {
  __shared__ float cb_s[16];
  if (is_codebook(S) && threadIdx.x < (S == kSideCB3 ? 8 : 16)) cb_s[threadIdx.x] = codebook[threadIdx.x];
  __syncthreads();
  const int i = blockIdx.x;
  const int phys = ids[i];
  const int rows = a.Hkv * a.bs, chunks = a.D / 8;
  for (int c = threadIdx.x; c < rows * chunks; c += blockDim.x) {
    const int rr = c / chunks, col = (c % chunks) * 8;
    float x[8];
    if (phys >= 0 && phys < a.num_blocks) {
      const size_t crow = (size_t)phys * rows + rr;
      SideFormat<S>::load8(cache, crow, a.D, col, side_scale<S>(scales, crow), cb_s, x);
    } else {
      if (c == 0) atomicOr(a.err, DA_DEVERR_BLOCK_ID);
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) out[((size_t)i * rows + rr) * a.D + col + k] = x[k];
  }
}

}  // namespace

cudaError_t launch_debug_bounds(const Args& a, int32_t* bounds, cudaStream_t s) {
  if (a.B == 0) return cudaSuccess;
  debug_bounds_kernel<<<a.B, 128, 0, s>>>(a, bounds);
  return cudaGetLastError();
}

cudaError_t launch_debug_dequant(const Args& a, const void* cache, const float* scales, const int32_t* ids, int n,
                                 int which, float* out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int side = which ? v_side(a.fmt) : k_side(a.fmt);
  const float* cb = a.codebook + ((which && a.fmt == DA_KV_CB3K_CB4V) ? 8 : 0);
  switch (side) {
    case kSideBF16: debug_dequant_kernel<kSideBF16><<<n, 128, 0, s>>>(a, cache, scales, ids, cb, out); break;
    case kSideFP8: debug_dequant_kernel<kSideFP8><<<n, 128, 0, s>>>(a, cache, scales, ids, cb, out); break;
    case kSideCB3: debug_dequant_kernel<kSideCB3><<<n, 128, 0, s>>>(a, cache, scales, ids, cb, out); break;
    default: debug_dequant_kernel<kSideCB4><<<n, 128, 0, s>>>(a, cache, scales, ids, cb, out); break;
  }
  return cudaGetLastError();
}

}  // namespace da
