// encode.cu -- cache writers for the quantised KV formats (the step before the hot path),
// and the Lloyd-Max codebook of the 4-bit format.
//
// FP8 E4M3 with one scale per tensor (attention.rs README, KV Cache Formats table, "FP8
// (E4M3)"): scale = amax|x| / 448 in binary32, code = round-to-nearest-even E4M3 of the
// binary32 quotient x / scale, saturating at +-448.
//
// 4-bit and 3-bit codebooks on a random-sign Walsh-Hadamard basis (same table, "Turbo4" /
// "Turbo3"; turboquant-rs 0.4.1, src/cache/cuda/attention.rs: codebook + sign_pattern):
//   r = H diag(sign) x / sqrt(D), scale = ||x||_2 (stored as binary32),
//   idx_d = nearest codebook value to r_d / scale (ties to the lower index),
//   codes packed as a little-endian bit stream (4 bits: coordinate 2k in the low nibble).
// Every code decision and scale is the one a plain sequential fp64 evaluation gives (the
// sums in index order); a fast path reaches them with less fp64 work (see the kernel).
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "da_internal.cuh"

namespace da {
namespace {

__global__ void amax_kernel(const float* __restrict__ x, long long n, unsigned* __restrict__ amax_bits) {
  float m = 0.0f;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // non-negative floats order like their bit patterns
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

__global__ void fp8_scale_kernel(float* scale) {
  const float amax = *scale;  // holds the amax bits written by amax_kernel
  *scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

__global__ void fp8_cast_kernel(const float* __restrict__ x, long long n, const float* __restrict__ scale,
                                uint8_t* __restrict__ codes) {
  const float s = *scale;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    codes[i] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[i], s), __NV_SATFINITE, __NV_E4M3);
}

// One warp per vector; lane l holds coordinates kPer * l .. kPer * l + kPer - 1 (kPer = D / 32).
//
// The codes must be the ones the plain definition gives: r = H diag(sign) x / sqrt(D) with each
// sum taken in index order in fp64, scale = binary32(sqrt(sum of x_k^2 in index order)), code =
// the first codebook value nearest to r / scale in fp64. A fast path computes the same decisions
// with less fp64 work and falls back to the definition wherever it could differ:
//   - r by the fast Walsh-Hadamard transform in fp64 (7 butterfly stages at D = 128: two in
//     registers, the rest across lanes by shuffles) instead of D index-ordered sums of D terms.
//     Its sums come in another order, so it differs from the definition's by at most
//     ~134 * 2^-53 * sum |x_k| (< 3e-13 relative to ||x||);
//   - the norm by a tree of partial sums; if the definition's sum, within its own bound of the
//     tree's, could round to another binary32 scale (checked by rounding the tree's root times
//     1 -+ 1e-9), lane 0 sums in index order instead;
//   - the code from the buckets between neighbouring levels of a strictly increasing codebook
//     (binary32 search, then a fp64 check): when u = r / scale lies more than 1e-6 away from
//     both of its bucket's boundaries (the midpoints of neighbouring levels), the definition's
//     u, within 1e-12 of it, has the same nearest level. Otherwise (or for a zero vector, or a
//     codebook that is not strictly increasing) that coordinate is recomputed by the
//     definition: the index-ordered sum, the division, the scan over every level.
template <int D>
__global__ void __launch_bounds__(128) codebook_encode_kernel(const float* __restrict__ x, long long nvec, int bits,
                                                              const float* __restrict__ sign,
                                                              const float* __restrict__ codebook,
                                                              uint8_t* __restrict__ packed,
                                                              float* __restrict__ scales) {
  constexpr int kPer = D / 32;
  constexpr double kDelta = 1e-6;  // margin around a bucket boundary (u is at most 1 in size)
  __shared__ double xs_all[4][D];
  __shared__ uint8_t codes_all[4][D];
  __shared__ float cb[16];
  __shared__ double mid_s[16];  // mid_s[j]: the midpoint of levels j and j + 1
  __shared__ int sorted_s;
  const int levels = 1 << bits;
  if (threadIdx.x < levels) cb[threadIdx.x] = codebook[threadIdx.x];
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    for (int j = 0; j + 1 < levels; ++j) {
      ok &= cb[j] < cb[j + 1];
      mid_s[j] = 0.5 * ((double)cb[j] + (double)cb[j + 1]);  // exact: binary32 sums fit binary64
    }
    sorted_s = ok;
  }
  __syncthreads();
  const bool sorted = sorted_s != 0;
  float mid32[15];  // binary32 copies of the midpoints, for the bucket search
#pragma unroll
  for (int j = 0; j < 15; ++j) mid32[j] = j + 1 < levels ? (float)mid_s[j] : INFINITY;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double* xs = xs_all[w];
  uint8_t* codes = codes_all[w];
  const int row_bytes = D * bits / 8;
  const double inv = 1.0 / sqrt((double)D);
  for (long long v = blockIdx.x * 4ll + w; v < nvec; v += gridDim.x * 4ll) {
    const float* xv = x + v * D + kPer * lane;
    // sign * x in fp64 (exact), kept in shared memory for the index-ordered fallbacks
    double y[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      y[i] = (double)__ldg(sign + kPer * lane + i) * (double)xv[i];
      xs[kPer * lane + i] = y[i];
    }
    // ||x||^2: a tree of partial sums, or lane 0's index-ordered sum near a rounding boundary
    double n2 = 0.0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) n2 = fma(y[i], y[i], n2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    double t = sqrt(n2);
    float scale = (float)t;
    __syncwarp();  // xs complete
    if ((float)(t * (1.0 - 1e-9)) != scale || (float)(t * (1.0 + 1e-9)) != scale) {
      double s2 = 0.0;
      if (lane == 0)
        for (int k = 0; k < D; ++k) s2 += xs[k] * xs[k];
      scale = (float)sqrt(__shfl_sync(0xffffffffu, s2, 0));
    }
    // r' = H (sign * x): butterflies within the lane's registers, then across lanes
#pragma unroll
    for (int d = 1; d < kPer; d <<= 1)
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (!(i & d)) {
          const double a = y[i], b = y[i + d];
          y[i] = a + b;
          y[i + d] = a - b;
        }
#pragma unroll
    for (int lo = 1; lo < 32; lo <<= 1) {  // index distance kPer * lo: lanes lo apart
      const bool upper = lane & lo;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const double o = __shfl_xor_sync(0xffffffffu, y[i], lo);
        y[i] = upper ? o - y[i] : y[i] + o;
      }
    }
    const double to_u = scale > 0.0f ? inv / (double)scale : __longlong_as_double(0x7ff8000000000000ll);  // NaN: fall back
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = kPer * lane + i;
      const double u = y[i] * to_u;
      const float u32 = (float)u;
      int b = 0;
#pragma unroll
      for (int j = 0; j < 15; ++j) b += u32 > mid32[j];
      bool fast = sorted && u == u;  // not NaN
      if (fast && b > 0) fast = u - mid_s[b - 1] > kDelta;
      if (fast && b < levels - 1) fast = mid_s[b] - u > kDelta;
      if (!fast) {  // the definition: index-ordered sum, division, scan over every level
        double acc = 0.0;
        for (int k = 0; k < D; ++k) acc += (__popc(c & k) & 1) ? -xs[k] : xs[k];  // H[c][k] sign[k] x[k]
        const double r = acc * inv;
        const double ue = scale > 0.0f ? r / (double)scale : 0.0;
        b = 0;
        double bd = fabs(ue - (double)cb[0]);
        for (int j = 1; j < levels; ++j) {
          const double dd = fabs(ue - (double)cb[j]);
          if (dd < bd) {
            bd = dd;
            b = j;
          }
        }
      }
      codes[c] = (uint8_t)b;
    }
    __syncwarp();
    for (int byte = lane; byte < row_bytes; byte += 32) {
      unsigned out = 0;
      for (int bit = 0; bit < 8; ++bit) {
        const int s = 8 * byte + bit;
        out |= ((codes[s / bits] >> (s % bits)) & 1u) << bit;
      }
      packed[v * row_bytes + byte] = (uint8_t)out;
    }
    if (lane == 0) scales[v] = scale;
    __syncwarp();
  }
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  return (int)(g < 4096 ? (g < 1 ? 1 : g) : 4096);
}

// ---------------------------------------------------------------- Lloyd-Max (host)
double phi(double z) { return exp(-0.5 * z * z) / sqrt(2.0 * M_PI); }
// standard normal mass of (a, b], from erfc so both tails keep their precision
double mass(double a, double b) {
  if (a >= 0.0) return 0.5 * (erfc(a / M_SQRT2) - erfc(b / M_SQRT2));
  if (b <= 0.0) return 0.5 * (erfc(-b / M_SQRT2) - erfc(-a / M_SQRT2));
  return 1.0 - 0.5 * erfc(-a / M_SQRT2) - 0.5 * erfc(b / M_SQRT2);
}

}  // namespace

cudaError_t launch_encode_fp8(const float* x, long long n, uint8_t* codes, float* scale, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (n > 0) amax_kernel<<<grid_for(n, 256), 256, 0, s>>>(x, n, reinterpret_cast<unsigned*>(scale));
  fp8_scale_kernel<<<1, 1, 0, s>>>(scale);
  if (n > 0) fp8_cast_kernel<<<grid_for(n, 256), 256, 0, s>>>(x, n, scale, codes);
  return cudaGetLastError();
}

cudaError_t launch_encode_codebook(const float* x, long long nvec, int D, int bits, const float* sign,
                                   const float* codebook, uint8_t* packed, float* scales, cudaStream_t s) {
  if (nvec == 0) return cudaSuccess;
  const int grid = (int)((nvec + 3) / 4 < 8192 ? (nvec + 3) / 4 : 8192);
  if (D == 128)
    codebook_encode_kernel<128><<<grid, 128, 0, s>>>(x, nvec, bits, sign, codebook, packed, scales);
  else
    codebook_encode_kernel<256><<<grid, 128, 0, s>>>(x, nvec, bits, sign, codebook, packed, scales);
  return cudaGetLastError();
}

// Lloyd-Max quantiser of `levels` output levels for N(0, sigma^2): thresholds at the
// midpoints of neighbouring levels, each level at the conditional mean of its cell,
// repeated from evenly spaced levels on [-3 sigma, 3 sigma] until no level moves by more
// than 1e-14 sigma; then made exactly symmetric and rounded to binary32.
int lloyd_max_codebook(int levels, double sigma, float* out) {
  if (levels < 2 || levels > 64 || !(sigma > 0.0)) return -1;
  double c[64], t[65];
  const int L = levels;
  for (int i = 0; i < L; ++i) c[i] = -3.0 + 6.0 * (i + 0.5) / L;
  int it = 0;
  for (; it < 1000000; ++it) {
    double moved = 0.0;
    t[0] = -INFINITY;
    t[L] = INFINITY;
    for (int i = 1; i < L; ++i) t[i] = 0.5 * (c[i - 1] + c[i]);
    for (int i = 0; i < L; ++i) {
      const double pa = std::isinf(t[i]) ? 0.0 : phi(t[i]), pb = std::isinf(t[i + 1]) ? 0.0 : phi(t[i + 1]);
      const double nc = (pa - pb) / mass(t[i], t[i + 1]);
      moved = fmax(moved, fabs(nc - c[i]));
      c[i] = nc;
    }
    if (moved < 1e-14) break;
  }
  if (it == 1000000) return -1;
  for (int i = 0; i < L / 2; ++i) {
    const double m = 0.5 * (c[L - 1 - i] - c[i]);
    c[i] = -m;
    c[L - 1 - i] = m;
  }
  if (L % 2) c[L / 2] = 0.0;
  for (int i = 0; i < L; ++i) out[i] = (float)(sigma * c[i]);
  return 0;
}

}  // namespace da
