// kv_formats.cuh -- in-register dequantisation of one side (K or V) of a KV cache
// (attention.rs README, KV Cache Formats table: BF16, FP8 E4M3, and the 4-bit / 3-bit
// Walsh-Hadamard codebook formats, alone or mixed as FP8 K + 4-bit V and 3-bit K +
// 4-bit V). Codebook sides are dequantised in their rotated basis only: coordinate d is
// scale_t * codebook[idx_d] (turboquant-rs 0.4.1, src/cache/cuda/attention.rs: the fused
// kernel works on the compressed cache as stored and never dequantises it in full).
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "da_internal.cuh"

namespace da {

// storage of one side
enum Side { kSideBF16 = 0, kSideFP8 = 1, kSideCB3 = 2, kSideCB4 = 3 };

__host__ __device__ constexpr int k_side(int fmt) {
  return fmt == DA_KV_BF16 ? kSideBF16
         : fmt == DA_KV_FP8_E4M3 || fmt == DA_KV_FP8K_CB4V ? kSideFP8
         : fmt == DA_KV_CB3K_CB4V ? kSideCB3
                                  : kSideCB4;
}
__host__ __device__ constexpr int v_side(int fmt) {
  return fmt == DA_KV_BF16 ? kSideBF16 : fmt == DA_KV_FP8_E4M3 ? kSideFP8 : kSideCB4;
}
__host__ __device__ constexpr bool is_codebook(int side) { return side == kSideCB3 || side == kSideCB4; }
// bytes of one stored row (one token of one kv head)
__host__ __device__ constexpr int row_bytes(int side, int D) {
  return side == kSideBF16 ? 2 * D : side == kSideFP8 ? D : side == kSideCB3 ? 3 * D / 8 : D / 2;
}

template <int S>
struct SideFormat;

// bf16: the upper half of a binary32 word, converted exactly.
template <>
struct SideFormat<kSideBF16> {
  // 8 consecutive elements of cache row `row`, starting at column `col` (a multiple of 8).
  __device__ static __forceinline__ void load8(const void* cache, size_t row, int D, int col, float /*scale*/,
                                               const float* /*cb*/, float* x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(cache) + row * D + col));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// E4M3 -> f16 is exact (3 mantissa bits, exponents 2^-9 .. 2^8 fit f16); then one fp32
// multiply by `scale` (the caller passes 1 to keep the values in code units).
template <>
struct SideFormat<kSideFP8> {
  __device__ static __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
  }
  __device__ static __forceinline__ void load8(const void* cache, size_t row, int D, int col, float scale,
                                               const float* /*cb*/, float* x) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(cache) + row * D + col));
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 a = e4m3x2_to_float2(w[i]);
      const float2 b = e4m3x2_to_float2(w[i] >> 16);
      x[4 * i + 0] = scale * a.x;
      x[4 * i + 1] = scale * a.y;
      x[4 * i + 2] = scale * b.x;
      x[4 * i + 3] = scale * b.y;
    }
  }
};

// 4-bit codebook: byte k of a row holds coordinate 2k in its low nibble, 2k+1 in its high
// nibble; value = scale_t * codebook[idx] (rotated basis).
template <>
struct SideFormat<kSideCB4> {
  __device__ static __forceinline__ void load8(const void* cache, size_t row, int D, int col, float scale,
                                               const float* cb, float* x) {
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(cache) + row * (D / 2) +
                                                               col / 2));
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = scale * cb[(v >> (4 * i)) & 15u];
  }
};

// 3-bit codebook: the codes form a little-endian bit stream, coordinate d at stream bits
// [3d, 3d + 3); 8 coordinates starting at a multiple of 8 are the 3 bytes at 3 * col / 8.
template <>
struct SideFormat<kSideCB3> {
  __device__ static __forceinline__ void load8(const void* cache, size_t row, int D, int col, float scale,
                                               const float* cb, float* x) {
    const uint8_t* p = static_cast<const uint8_t*>(cache) + row * (3 * D / 8) + 3 * (col / 8);
    const uint32_t v = (uint32_t)__ldg(p) | ((uint32_t)__ldg(p + 1) << 8) | ((uint32_t)__ldg(p + 2) << 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = scale * cb[(v >> (3 * i)) & 7u];
  }
};

// Per-row scale: an FP8 side has one per tensor, a codebook side one per (block, kv head,
// slot), bf16 none.
template <int S>
__device__ __forceinline__ float side_scale(const float* scales, size_t row) {
  if constexpr (S == kSideFP8) return __ldg(scales);
  else if constexpr (S == kSideCB3 || S == kSideCB4) return __ldg(scales + row);
  else return 1.0f;
}

}  // namespace da
