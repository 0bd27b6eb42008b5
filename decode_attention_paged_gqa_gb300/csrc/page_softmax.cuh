// page_softmax.cuh -- the online-softmax step of the tensor-core partition kernels, per
// 16-token page, on the C-fragment layout of S^T[16 tokens x 8 columns] (mma.m16n8k16):
// thread (gid, tig) holds sc[0], sc[1] = token gid, columns 2 tig and 2 tig + 1, and sc[2],
// sc[3] = token gid + 8, same columns. Scores are in the log2 domain (x log2 e).
//
// The running state per column is (m, l): the reference max and the sum of 2^(s - m); the
// caller's unnormalised output O^T is scaled by alpha whenever m moves. The reference moves
// lazily: only when a page's max exceeds it by more than kLazyLog2, so most pages rescale
// nothing and the probabilities stay below 2^kLazyLog2 (well inside f16 / bf16 range). The
// final (m, l, o) is exact up to rounding whatever reference was used.
#pragma once

#include <cmath>

namespace da {

constexpr float kLazyLog2 = 8.0f;

// 2^x with the hardware approximation (ex2.approx: relative error ~2^-22; results below
// 2^-126 flush to zero, 2^-inf = 0), one instruction.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Tokens outside [lo_c[j], hi_c[j]) of column j get -inf (no weight). tok0: first token of
// the page.
__device__ __forceinline__ void mask_page(float (&sc)[4], int tok0, int gid, const int (&lo_c)[2],
                                          const int (&hi_c)[2]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int t = tok0 + gid + (e >> 1) * 8, j = e & 1;
    if (t < lo_c[j] || t >= hi_c[j]) sc[e] = -INFINITY;
  }
}

// One page: updates (m, l) of the thread's two columns and returns the page's
// probabilities pr (relative to the new reference) and the factor alpha[j] the column's
// running output must be multiplied by. Returns true if any column of the warp moved its
// reference (alpha != 1 somewhere). A column's page max is only needed when it exceeds the
// reference by more than kLazyLog2, which a warp vote on the threads' own scores decides: the
// usual page skips the max reduction altogether.
__device__ __forceinline__ bool page_softmax(const float (&sc)[4], float (&m)[2], float (&l)[2], float (&alpha)[2],
                                             float (&pr)[4]) {
  alpha[0] = alpha[1] = 1.0f;
  bool moved_any = false;
  // m = -inf (nothing seen yet): -inf + kLazyLog2 = -inf, so the first finite score counts as over
  const bool over = fmaxf(sc[0], sc[2]) > m[0] + kLazyLog2 || fmaxf(sc[1], sc[3]) > m[1] + kLazyLog2;
  if (__any_sync(0xffffffffu, over)) {
    bool moved = false;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mx = fmaxf(sc[j], sc[j + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const bool move = mx > m[j] + kLazyLog2;
      const float mn = move ? mx : m[j];
      alpha[j] = move ? exp2_fast(m[j] - mn) : 1.0f;  // 2^-inf = 0 clears the (zero) state
      moved |= move;
      m[j] = mn;
    }
    moved_any = __any_sync(0xffffffffu, moved);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    // with no finite score yet every score is -inf: any finite reference gives 2^-inf = 0
    const float ref = m[j] == -INFINITY ? 0.0f : m[j];
    pr[j] = exp2_fast(sc[j] - ref);
    pr[j + 2] = exp2_fast(sc[j + 2] - ref);
    l[j] = l[j] * alpha[j] + pr[j] + pr[j + 2];
  }
  return moved_any;
}

// ---- one column per thread: the thread holds the scores of tokens gid (s[0]) and gid + 8
//      (s[1]) of a single column (the layout in which a column pair carries one head's hi and
//      lo parts). The running max starts at kNoMax, a finite stand-in for "nothing seen yet":
//      the first finite score always moves it, masked (-inf) scores give 2^-inf = 0, and an
//      all-masked column keeps (kNoMax, 0), which a combine weighs with 2^(kNoMax - M) = 0.
constexpr float kNoMax = -3.4028234663852886e38f;  // -FLT_MAX

// Tokens outside [lo, hi) get -inf (no weight).
__device__ __forceinline__ void mask_page_col(float (&s)[2], int tok0, int gid, int lo, int hi) {
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int t = tok0 + gid + 8 * e;
    if (t < lo || t >= hi) s[e] = -INFINITY;
  }
}

// One page of one column: updates (m, l), returns the probabilities relative to the new
// reference and the factor alpha the column's running output must be multiplied by; true if
// any column of the warp moved its reference.
__device__ __forceinline__ bool page_softmax_col(const float (&s)[2], float& m, float& l, float& alpha,
                                                 float (&pr)[2]) {
  alpha = 1.0f;
  bool moved_any = false;
  if (__any_sync(0xffffffffu, fmaxf(s[0], s[1]) > m + kLazyLog2)) {
    float mx = fmaxf(s[0], s[1]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const bool move = mx > m + kLazyLog2;
    if (move) {
      alpha = exp2_fast(m - mx);  // 2^(kNoMax - mx) = 0 clears the (zero) state
      m = mx;
    }
    moved_any = __any_sync(0xffffffffu, move);
  }
  pr[0] = exp2_fast(s[0] - m);
  pr[1] = exp2_fast(s[1] - m);
  l = fmaf(l, alpha, pr[0] + pr[1]);
  return moved_any;
}

}  // namespace da
