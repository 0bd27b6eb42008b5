/*
 * oracle.c -- plain, slow fp64 CPU oracle for single-token (decode) GQA attention
 * over a paged KV cache, and for the three cache encodings it reads:
 * BF16, FP8 E4M3 with one fp32 scale per tensor, and a 4-bit codebook on a
 * random-sign Walsh-Hadamard-rotated basis.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this library. It shares no code, header, table or
 * constant generator with the CUDA library: every definition below is written out
 * from the method's description, in the order the description gives it.
 *
 * What it follows (page title, section):
 *   attention.rs README, "KV Cache Formats" table: the formats BF16/FP16,
 *     FP8 (E4M3) and the 4-bit Walsh-Hadamard codebook ("Turbo4"); the sentence
 *     under that table: split-K decode for contexts of 1024 tokens and more,
 *     partials combined by a float-precision reduce; "Features": softcapping,
 *     sliding window, GQA/MQA, paged block tables.
 *   turboquant-rs 0.4.1, src/cache/cuda/attention.rs, fused_attention():
 *     PARTITION_SIZE = 512, num_partitions = ceil(kv_len / 512), per-partition
 *     partial output + max + sum, an all-zero output when kv_len == 0, and the
 *     codebook / sign_pattern inputs of the codebook cache.
 *
 * Readings where the pages are silent are listed beside the code they shape.
 * Compile with -ffp-contract=off (no fused multiply-add contraction).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_FMT_BF16 0
#define OR_FMT_FP8 1
#define OR_FMT_CB4 2
#define OR_FMT_FP8K_CB4V 3  /* "Turbo8": FP8 keys, 4-bit codebook values */
#define OR_FMT_CB3K_CB4V 4  /* "Turbo3": 3-bit codebook keys, 4-bit codebook values */

/* How one side (K or V) of a cache format is stored. */
enum { OR_SIDE_BF16, OR_SIDE_FP8, OR_SIDE_CB3, OR_SIDE_CB4 };

static int or_side(int fmt, int which) {
  switch (fmt) {
    case OR_FMT_BF16: return OR_SIDE_BF16;
    case OR_FMT_FP8: return OR_SIDE_FP8;
    case OR_FMT_CB4: return OR_SIDE_CB4;
    case OR_FMT_FP8K_CB4V: return which ? OR_SIDE_CB4 : OR_SIDE_FP8;
    default: return which ? OR_SIDE_CB4 : OR_SIDE_CB3;
  }
}

/* Bytes of one stored row (one token of one kv head) of a side. */
static int64_t or_side_row_bytes(int side, int D) {
  switch (side) {
    case OR_SIDE_BF16: return 2 * (int64_t)D;
    case OR_SIDE_FP8: return D;
    case OR_SIDE_CB3: return 3 * (int64_t)D / 8;
    default: return D / 2;
  }
}

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_BLOCK -2  /* a block-table entry outside [0, num_blocks) */
#define OR_ERR_NOMEM -3

/* ------------------------------------------------------------------------- */
/* Element formats                                                           */
/* ------------------------------------------------------------------------- */

/* bfloat16 is the upper 16 bits of an IEEE-754 binary32 word. */
double or_bf16_decode(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* FP8 E4M3 ("E4M3FN" of the OCP 8-bit float format): 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9);
 * S.1111.111 is NaN; there is no infinity. Largest finite value 448. */
double or_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);          /* (m / 8) * 2^(1 - 7) */
  else
    v = ldexp((double)(8 + m), e - 10); /* (1 + m / 8) * 2^(e - 7) */
  return s ? -v : v;
}

/* Round-to-nearest-even cast of a binary32 value to E4M3, saturating to +-448
 * (values above 448 have no finite E4M3 neighbour above them). NaN -> 0x7F. */
uint8_t or_e4m3_encode(float xf) {
  double x = (double)xf, a, q, r, v;
  uint8_t s;
  int ex, E;
  if (isnan(x)) return 0x7F;
  s = signbit(x) ? 0x80 : 0x00;
  a = fabs(x);
  if (a == 0.0) return s;
  frexp(a, &ex);
  E = ex - 1;            /* 2^E <= a < 2^(E+1) */
  if (E < -6) E = -6;    /* below 2^-6 the grid is the subnormal one, step 2^-9 */
  q = ldexp(a, 3 - E);   /* a in units of the grid step 2^(E-3): exact */
  r = nearbyint(q);      /* default rounding mode: to nearest, ties to even */
  v = ldexp(r, E - 3);   /* the rounded value, exactly representable */
  if (v >= 448.0) return (uint8_t)(s | 0x7E);
  if (v < ldexp(1.0, -6)) /* subnormal: m * 2^-9, m in 0..7 */
    return (uint8_t)(s | (uint8_t)ldexp(v, 9));
  frexp(v, &ex);
  E = ex - 1;
  return (uint8_t)(s | (uint8_t)((E + 7) << 3) | (uint8_t)(ldexp(v, 3 - E) - 8.0));
}

void or_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_decode(c[i]);
}

void or_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Small thread pool: run fn(ctx, i) for i in [0, n) on `threads` threads.   */
/* ------------------------------------------------------------------------- */

typedef void (*or_task_fn)(void* ctx, int64_t i);
typedef struct {
  or_task_fn fn;
  void* ctx;
  int64_t n;
  int64_t next;
} or_pool;

static void* or_pool_worker(void* arg) {
  or_pool* p = (or_pool*)arg;
  for (;;) {
    int64_t i = __atomic_fetch_add(&p->next, 1, __ATOMIC_RELAXED);
    if (i >= p->n) break;
    p->fn(p->ctx, i);
  }
  return NULL;
}

int or_default_threads(void) {
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

/* Returns the number of threads actually used. */
static int or_parallel_for(or_task_fn fn, void* ctx, int64_t n, int threads) {
  or_pool p = {fn, ctx, n, 0};
  pthread_t tid[512];
  int t, used;
  if (threads <= 0) threads = or_default_threads();
  if (threads > 512) threads = 512;
  if ((int64_t)threads > n) threads = n > 0 ? (int)n : 1;
  used = threads;
  for (t = 1; t < threads; ++t)
    if (pthread_create(&tid[t], NULL, or_pool_worker, &p) != 0) {
      used = t;
      break;
    }
  or_pool_worker(&p);
  for (t = 1; t < used; ++t) pthread_join(tid[t], NULL);
  return used;
}

/* ------------------------------------------------------------------------- */
/* FP8 quantisation of one tensor (one scale per layer and per K or V)       */
/* ------------------------------------------------------------------------- */

typedef struct {
  const float* x;
  uint8_t* codes;
  int64_t n, chunk;
  float scale;
} or_fp8_job;

static void or_fp8_task(void* ctx, int64_t i) {
  or_fp8_job* j = (or_fp8_job*)ctx;
  int64_t lo = i * j->chunk, hi = lo + j->chunk, k;
  if (hi > j->n) hi = j->n;
  for (k = lo; k < hi; ++k) {
    float y = j->x[k] / j->scale; /* binary32 division, rounded to nearest */
    j->codes[k] = or_e4m3_encode(y);
  }
}

/* scale = amax / 448 in binary32 (amax over the binary32 source); code =
 * RNE-E4M3(x / scale). Reading: the division is a binary32 division and the cast
 * rounds its result once more, to nearest-even. A zero tensor gets scale 1. */
float or_fp8_quantize(const float* x, int64_t n, uint8_t* codes, int threads) {
  float amax = 0.0f;
  int64_t k;
  or_fp8_job j;
  for (k = 0; k < n; ++k) {
    float a = fabsf(x[k]);
    if (a > amax) amax = a;
  }
  j.x = x;
  j.codes = codes;
  j.n = n;
  j.chunk = 1 << 20;
  j.scale = amax > 0.0f ? amax / 448.0f : 1.0f;
  or_parallel_for(or_fp8_task, &j, (n + j.chunk - 1) / j.chunk, threads);
  return j.scale;
}

/* ------------------------------------------------------------------------- */
/* Walsh-Hadamard basis and the 4-bit codebook                               */
/* ------------------------------------------------------------------------- */

/* Sylvester's construction: H[i][j] = (-1)^popcount(i & j), D a power of two.
 * H is symmetric and H * H = D * I. */
void or_hadamard(int D, double* H) {
  for (int i = 0; i < D; ++i)
    for (int j = 0; j < D; ++j) H[(int64_t)i * D + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
}

static double or_phi(double z) { return exp(-0.5 * z * z) / sqrt(2.0 * M_PI); }
/* Phi(b) - Phi(a) for the standard normal, from erfc so that tails keep precision. */
static double or_mass(double a, double b) {
  if (a >= 0.0) return 0.5 * (erfc(a / M_SQRT2) - erfc(b / M_SQRT2));
  if (b <= 0.0) return 0.5 * (erfc(-b / M_SQRT2) - erfc(-a / M_SQRT2));
  return 1.0 - 0.5 * erfc(-a / M_SQRT2) - 0.5 * erfc(b / M_SQRT2);
}

/* Lloyd-Max quantiser of `levels` output levels for N(0, sigma^2): alternate
 * (i) thresholds at the midpoints of neighbouring levels and (ii) each level at
 * the conditional mean of its cell, sigma * (phi(a/sigma) - phi(b/sigma)) /
 * (Phi(b/sigma) - Phi(a/sigma)), until no level moves by more than tol*sigma.
 * Start: levels evenly spaced on [-3 sigma, 3 sigma] (any ordered start reaches
 * the same fixed point for a log-concave density). The result is made exactly
 * symmetric and written ascending to levels_out (fp64) and to codebook (fp32,
 * rounded to nearest). Returns the iteration count, or -1 if not converged. */
int or_lloyd_max(int levels, double sigma, double tol, int max_iter, double* levels_out, float* codebook) {
  double c[64], t[65];
  int L = levels, it, i;
  if (L < 2 || L > 64) return -1;
  for (i = 0; i < L; ++i) c[i] = -3.0 + 6.0 * (i + 0.5) / L; /* in units of sigma */
  for (it = 1; it <= max_iter; ++it) {
    double moved = 0.0;
    t[0] = -INFINITY;
    t[L] = INFINITY;
    for (i = 1; i < L; ++i) t[i] = 0.5 * (c[i - 1] + c[i]);
    for (i = 0; i < L; ++i) {
      double a = t[i], b = t[i + 1];
      double pa = isinf(a) ? 0.0 : or_phi(a), pb = isinf(b) ? 0.0 : or_phi(b);
      double nc = (pa - pb) / or_mass(a, b);
      double d = fabs(nc - c[i]);
      if (d > moved) moved = d;
      c[i] = nc;
    }
    if (moved < tol) break;
  }
  for (i = 0; i < L / 2; ++i) {
    double m = 0.5 * (c[L - 1 - i] - c[i]);
    c[i] = -m;
    c[L - 1 - i] = m;
  }
  if (L % 2) c[L / 2] = 0.0;
  for (i = 0; i < L; ++i) {
    levels_out[i] = sigma * c[i];
    codebook[i] = (float)(sigma * c[i]);
  }
  return it > max_iter ? -1 : it;
}

/* Index of the codebook value nearest to u; ties go to the lower index
 * (reading: the pages do not say how ties are broken). */
int or_cb_nearest(double u, const float* codebook, int levels) {
  int best = 0;
  double bd = fabs(u - (double)codebook[0]);
  for (int i = 1; i < levels; ++i) {
    double d = fabs(u - (double)codebook[i]);
    if (d < bd) {
      bd = d;
      best = i;
    }
  }
  return best;
}

/* b-bit codes are packed as a little-endian bit stream: the code of coordinate d occupies
 * stream bits [b*d, b*d + b), stream bit s being bit (s mod 8) of byte s / 8. For b = 4
 * this puts coordinate 2k in the low nibble of byte k and 2k + 1 in the high nibble (the
 * 4-bit config, step (4)). Reading for b = 3 (attention.rs README, "Turbo3": 3-bit K):
 * the pages give no packing; this is the plainest one. */
static int or_code_get(const uint8_t* vec, int bits, int d) {
  int v = 0;
  for (int i = 0; i < bits; ++i) {
    int s = bits * d + i;
    v |= ((vec[s >> 3] >> (s & 7)) & 1) << i;
  }
  return v;
}

static void or_code_put(uint8_t* vec, int bits, int d, int code) {
  for (int i = 0; i < bits; ++i) {
    int s = bits * d + i;
    if ((code >> i) & 1)
      vec[s >> 3] = (uint8_t)(vec[s >> 3] | (1u << (s & 7)));
    else
      vec[s >> 3] = (uint8_t)(vec[s >> 3] & ~(1u << (s & 7)));
  }
}

typedef struct {
  const float* x;
  const float* sign;
  const float* codebook;
  const double* H;
  uint8_t* packed;
  float* scales;
  int D, bits;
} or_cb_job;

/* One vector: (1) r = H * diag(sign) * x / sqrt(D); (2) scale = ||x||_2 stored as
 * binary32; (3) idx_d = nearest of the 2^bits codebook values to r_d / scale; (4) the
 * codes packed as a bit stream. A zero vector codes as r / scale = 0. */
static void or_cb_task(void* ctx, int64_t v) {
  or_cb_job* j = (or_cb_job*)ctx;
  int D = j->D, bits = j->bits, i, k;
  const float* x = j->x + v * D;
  double norm2 = 0.0, r[1024], inv = 1.0 / sqrt((double)D);
  float scale;
  for (k = 0; k < D; ++k) norm2 += (double)x[k] * (double)x[k];
  scale = (float)sqrt(norm2);
  for (i = 0; i < D; ++i) {
    double acc = 0.0;
    for (k = 0; k < D; ++k) acc += j->H[(int64_t)i * D + k] * (double)j->sign[k] * (double)x[k];
    r[i] = acc * inv;
  }
  for (i = 0; i < D; ++i) {
    double u = scale > 0.0f ? r[i] / (double)scale : 0.0;
    or_code_put(j->packed + v * (D * bits / 8), bits, i, or_cb_nearest(u, j->codebook, 1 << bits));
  }
  j->scales[v] = scale;
}

int or_cb_encode(int bits, const float* x, int64_t nvec, int D, const float* sign, const float* codebook,
                 uint8_t* packed, float* scales, int threads) {
  or_cb_job j;
  double* H;
  if (D <= 0 || D > 1024 || (D & (D - 1)) || D % 8 || bits < 1 || bits > 8) return OR_ERR_ARG;
  H = (double*)malloc(sizeof(double) * D * D);
  if (!H) return OR_ERR_NOMEM;
  or_hadamard(D, H);
  j.x = x;
  j.sign = sign;
  j.codebook = codebook;
  j.H = H;
  j.packed = packed;
  j.scales = scales;
  j.D = D;
  j.bits = bits;
  or_parallel_for(or_cb_task, &j, nvec, threads);
  free(H);
  return OR_OK;
}

int or_cb4_encode(const float* x, int64_t nvec, int D, const float* sign, const float* codebook, uint8_t* packed,
                  float* scales, int threads) {
  return or_cb_encode(4, x, nvec, D, sign, codebook, packed, scales, threads);
}

/* Rotated-basis value of coordinate d of a packed vector: scale * codebook[idx_d]. */
static double or_cb_rot_value(const uint8_t* packed_vec, int bits, int d, float scale, const float* codebook) {
  return (double)scale * (double)codebook[or_code_get(packed_vec, bits, d)];
}

/* Rotated-basis dequantisation of n packed vectors: out[v][d] = scale_v * cb[idx]. */
void or_cb_dequant_rotated(int bits, const uint8_t* packed, const float* scales, int64_t nvec, int D,
                           const float* codebook, double* out) {
  for (int64_t v = 0; v < nvec; ++v)
    for (int d = 0; d < D; ++d)
      out[v * D + d] = or_cb_rot_value(packed + v * (D * bits / 8), bits, d, scales[v], codebook);
}

void or_cb4_dequant_rotated(const uint8_t* packed, const float* scales, int64_t nvec, int D, const float* codebook,
                            double* out) {
  or_cb_dequant_rotated(4, packed, scales, nvec, D, codebook, out);
}

/* Back to the original basis: x = diag(sign) * H * r / sqrt(D) (H * H = D * I). */
static void or_unrotate(const double* r, int D, const double* H, const float* sign, double* x) {
  double inv = 1.0 / sqrt((double)D);
  for (int i = 0; i < D; ++i) {
    double acc = 0.0;
    for (int k = 0; k < D; ++k) acc += H[(int64_t)i * D + k] * r[k];
    x[i] = (double)sign[i] * acc * inv;
  }
}

void or_cb_dequant(int bits, const uint8_t* packed, const float* scales, int64_t nvec, int D, const float* codebook,
                   const float* sign, double* out) {
  double* H = (double*)malloc(sizeof(double) * D * D);
  double r[1024];
  if (!H) return;
  or_hadamard(D, H);
  for (int64_t v = 0; v < nvec; ++v) {
    for (int d = 0; d < D; ++d) r[d] = or_cb_rot_value(packed + v * (D * bits / 8), bits, d, scales[v], codebook);
    or_unrotate(r, D, H, sign, out + v * D);
  }
  free(H);
}

void or_cb4_dequant(const uint8_t* packed, const float* scales, int64_t nvec, int D, const float* codebook,
                    const float* sign, double* out) {
  or_cb_dequant(4, packed, scales, nvec, D, codebook, sign, out);
}

/* ------------------------------------------------------------------------- */
/* Partition bounds                                                          */
/* ------------------------------------------------------------------------- */

/* Partitions of the attended span [start, L): the span is split iff partition_size > 0
 * and its length n = L - start is at least split_threshold; then partition p covers
 * [start + p * partition_size, min(start + (p + 1) * partition_size, L)) and there are
 * ceil(n / partition_size) of them; otherwise one range [start, L). An empty span has no
 * range. Writes up to `cap` (start, end) pairs; returns the count. */
int or_partition_bounds_span(int start, int L, int partition_size, int split_threshold, int32_t* starts, int32_t* ends,
                             int cap) {
  int n = L - start, count, p;
  if (n <= 0) return 0;
  if (partition_size > 0 && n >= split_threshold) {
    count = (n + partition_size - 1) / partition_size;
    for (p = 0; p < count && p < cap; ++p) {
      starts[p] = start + p * partition_size;
      ends[p] = start + (p + 1) * partition_size < L ? start + (p + 1) * partition_size : L;
    }
    return count;
  }
  if (cap > 0) {
    starts[0] = start;
    ends[0] = L;
  }
  return 1;
}

/* First position attended by a query token at position `pos`: with a window of W tokens
 * only positions t with pos - W < t <= pos are attended (reading: the window is the W most
 * recent positions that query sees, its own included); else all t <= pos. */
static int or_window_start(int pos, int window) {
  int a = window > 0 ? pos + 1 - window : 0;
  return a > 0 ? a : 0;
}

/* Single query token (the last position, L - 1): attended positions [start, L) with
 * start = max(0, L - window) when a window is set, else 0; partitions counted from the
 * window start. */
int or_partition_bounds(int L, int window, int partition_size, int split_threshold, int32_t* starts, int32_t* ends,
                        int cap) {
  return or_partition_bounds_span(or_window_start(L - 1, window), L, partition_size, split_threshold, starts, ends,
                                  cap);
}

/* T query tokens (multi-token decode): the grid spans every position attended by any of
 * them, from the first query token's window start to L. */
int or_partition_bounds_multi(int L, int T, int window, int partition_size, int split_threshold, int32_t* starts,
                              int32_t* ends, int cap) {
  return or_partition_bounds_span(or_window_start(L - T, window), L, partition_size, split_threshold, starts, ends,
                                  cap);
}

/* ------------------------------------------------------------------------- */
/* Paged GQA decode attention                                                */
/* ------------------------------------------------------------------------- */

typedef struct {
  int B, T, Hq, Hkv, D, bs, fmt, num_blocks, max_blocks;
  const uint16_t* q;      /* bf16 bits [B][T][Hq][D] */
  const void* k_cache;    /* [num_blocks][Hkv][bs][row bytes of the side] */
  const void* v_cache;
  const float* k_scales;  /* fp8 side: [1]; codebook side: [num_blocks][Hkv][bs] */
  const float* v_scales;
  const float* codebook;  /* 4-bit: [16]; 3-bit keys: [8] key levels then [16] value levels */
  const float* sign;      /* codebook formats: [D] of +-1 */
  const int32_t* block_tables; /* [B][max_blocks] */
  const int32_t* context_lens; /* [B] */
  double scale, softcap;
  const float* alibi;     /* [Hq] ALiBi slopes, or NULL */
  int window, partition_size, split_threshold;
  const int32_t* out_row; /* [B*T*Hq]: output row of (b, j, h), or -1 when not requested */
  double* out;            /* [rows][D] */
  const double* H;        /* D x D Sylvester matrix (cb4) */
  int32_t* unit_b;        /* work units: (b, kv head g) with at least one requested head */
  int32_t* unit_g;
  int status;
} or_attn_job;

/* Dequantise token `t` of kv head g of sequence b (K if which == 0, else V) into x[D],
 * gathered through the block table: page t / bs, slot t % bs. Codebook sides are
 * decoded in their rotated basis and taken back to the original one with the dense H.
 * Codebooks: 4-bit formats use codebook[0..15]; the 3-bit-key format stores its 8 key
 * levels first and the 16 value levels after them. */
static int or_token(const or_attn_job* j, int b, int g, int t, int which, double* x) {
  int D = j->D, bs = j->bs, d, side = or_side(j->fmt, which);
  int32_t phys = j->block_tables[(int64_t)b * j->max_blocks + t / bs];
  int64_t row;
  const uint8_t* base = (const uint8_t*)(which ? j->v_cache : j->k_cache);
  if (phys < 0 || phys >= j->num_blocks) return OR_ERR_BLOCK;
  row = ((int64_t)phys * j->Hkv + g) * bs + t % bs; /* layout [num_blocks][Hkv][bs][...] */
  base += row * or_side_row_bytes(side, D);
  if (side == OR_SIDE_BF16) {
    const uint16_t* c = (const uint16_t*)base;
    for (d = 0; d < D; ++d) x[d] = or_bf16_decode(c[d]);
  } else if (side == OR_SIDE_FP8) {
    double s = (double)(which ? j->v_scales[0] : j->k_scales[0]);
    for (d = 0; d < D; ++d) x[d] = s * or_e4m3_decode(base[d]);
  } else {
    int bits = side == OR_SIDE_CB3 ? 3 : 4;
    const float* cb = j->codebook + ((j->fmt == OR_FMT_CB3K_CB4V && which) ? 8 : 0);
    float sc = (which ? j->v_scales : j->k_scales)[row];
    double r[1024];
    for (d = 0; d < D; ++d) r[d] = or_cb_rot_value(base, bits, d, sc, cb);
    or_unrotate(r, D, j->H, j->sign, x);
  }
  return OR_OK;
}

/* softmax(s) . V over n scores, with the maximum subtracted; out[D] = sum p V / sum p. */
static void or_softmax_pv(const double* s, const double* V, int n, int D, double* m_out, double* l_out, double* o) {
  double m = -INFINITY, l = 0.0;
  int t, d;
  for (t = 0; t < n; ++t)
    if (s[t] > m) m = s[t];
  for (d = 0; d < D; ++d) o[d] = 0.0;
  for (t = 0; t < n; ++t) {
    double p = exp(s[t] - m);
    l += p;
    for (d = 0; d < D; ++d) o[d] += p * V[(int64_t)t * D + d];
  }
  *m_out = m;
  *l_out = l;
}

/* One (sequence b, kv head g) unit: every requested query head of the group, for every
 * query token j (position L - T + j; T = 1 is ordinary decode). */
static void or_attn_task(void* ctx, int64_t u) {
  or_attn_job* j = (or_attn_job*)ctx;
  int b = j->unit_b[u], g = j->unit_g[u], D = j->D, G = j->Hq / j->Hkv, T = j->T;
  int L = j->context_lens[b];
  int s0 = or_window_start(L - T, j->window); /* first position any query token attends */
  int n = L - s0, t, d, i, hh, jq;
  double *K = NULL, *V = NULL, *s = NULL, *o = NULL, qh[1024];
  int32_t pst[4096], pen[4096];
  if (n < 0) n = 0;
  if (((int64_t)L + j->bs - 1) / j->bs > j->max_blocks) {
    j->status = OR_ERR_ARG; /* the sequence does not fit its block-table row */
    return;
  }
  if (n > 0) {
    K = (double*)malloc(sizeof(double) * (size_t)n * D);
    V = (double*)malloc(sizeof(double) * (size_t)n * D);
    s = (double*)malloc(sizeof(double) * (size_t)n);
    o = (double*)malloc(sizeof(double) * (size_t)D * 4097);
    if (!K || !V || !s || !o) {
      j->status = OR_ERR_NOMEM;
      goto done;
    }
    /* (1) gather and dequantise every attended key and value of kv head g */
    for (t = 0; t < n; ++t)
      if (or_token(j, b, g, s0 + t, 0, K + (int64_t)t * D) || or_token(j, b, g, s0 + t, 1, V + (int64_t)t * D)) {
        j->status = OR_ERR_BLOCK;
        goto done;
      }
  }
  for (jq = 0; jq < T; ++jq) {
    int pos = L - T + jq;                       /* position of query token jq */
    int a = or_window_start(pos, j->window), e = pos + 1; /* it attends [a, e) */
    for (hh = 0; hh < G; ++hh) {
      int h = g * G + hh; /* GQA: query head h reads kv head h / G (consecutive grouping) */
      int64_t qi = ((int64_t)b * T + jq) * j->Hq + h;
      int32_t row = j->out_row[qi];
      double* out;
      if (row < 0) continue;
      out = j->out + (int64_t)row * D;
      for (d = 0; d < D; ++d) out[d] = 0.0; /* nothing attended: zero output */
      if (pos < 0 || n == 0) continue;
      for (d = 0; d < D; ++d) qh[d] = or_bf16_decode(j->q[qi * D + d]);
      /* (2) scores s_t = scale * q . k_t, then the optional softcap cap * tanh(s / cap), then
       * the optional ALiBi bias slope_h * (t - pos): zero at the query's own position and
       * falling linearly with the distance (reading: the bias of the ALiBi method, added to
       * the finished score; the slopes are inputs) */
      for (t = a; t < e; ++t) {
        double acc = 0.0;
        for (d = 0; d < D; ++d) acc += qh[d] * K[(int64_t)(t - s0) * D + d];
        s[t - s0] = j->scale * acc;
        if (j->softcap > 0.0) s[t - s0] = j->softcap * tanh(s[t - s0] / j->softcap);
        if (j->alibi) s[t - s0] += (double)j->alibi[h] * (double)(t - pos);
      }
      /* (3) out = softmax(s) V over [a, e), in one piece or through per-partition partials */
      {
        int np = or_partition_bounds_span(s0, L, j->partition_size, j->split_threshold, pst, pen, 4096);
        if (np > 4096) {
          j->status = OR_ERR_ARG;
          goto done;
        }
        if (np == 1) {
          double m, l;
          or_softmax_pv(s + (a - s0), V + (int64_t)(a - s0) * D, e - a, D, &m, &l, out);
          for (d = 0; d < D; ++d) out[d] /= l;
        } else {
          /* per partition: running max m_p, sum l_p and the unnormalised o_p over the part of
           * it this query attends; then M = max m_p, Lsum = sum l_p e^(m_p - M),
           * out = sum o_p e^(m_p - M) / Lsum */
          double mp[4096], lp[4096], M = -INFINITY, Lsum = 0.0;
          for (i = 0; i < np; ++i) {
            int lo = pst[i] > a ? pst[i] : a, hi = pen[i] < e ? pen[i] : e;
            if (lo >= hi) {
              mp[i] = -INFINITY;
              lp[i] = 0.0;
              continue;
            }
            or_softmax_pv(s + (lo - s0), V + (int64_t)(lo - s0) * D, hi - lo, D, &mp[i], &lp[i], o + (int64_t)i * D);
            if (mp[i] > M) M = mp[i];
          }
          for (i = 0; i < np; ++i) {
            double w;
            if (lp[i] == 0.0) continue;
            w = exp(mp[i] - M);
            Lsum += lp[i] * w;
            for (d = 0; d < D; ++d) out[d] += o[(int64_t)i * D + d] * w;
          }
          for (d = 0; d < D; ++d) out[d] /= Lsum;
        }
      }
    }
  }
done:
  free(K);
  free(V);
  free(s);
  free(o);
}

/* out_row[(b * T + j) * Hq + h] selects the (b, j, h) outputs to compute (row index into
 * out, or -1); pass NULL to compute all of them into out[B][T][Hq][D]. T is the number of
 * query tokens per sequence (1 = ordinary decode). Returns OR_OK or an error;
 * *threads_used receives the thread count. */
int or_decode_attention(int B, int T, int Hq, int Hkv, int D, int block_size, int fmt, int num_blocks,
                        int max_blocks, const uint16_t* q, const void* k_cache, const void* v_cache,
                        const float* k_scales, const float* v_scales, const float* codebook, const float* sign,
                        const int32_t* block_tables, const int32_t* context_lens, double scale, double softcap,
                        const float* alibi_slopes, int window, int partition_size, int split_threshold,
                        const int32_t* out_row, double* out, int threads, int* threads_used) {
  or_attn_job j;
  int32_t* rows = NULL;
  double* H = NULL;
  int64_t nu = 0, b, g, hh, jq;
  int used;
  if (B < 0 || T < 1 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || D > 1024 || block_size <= 0) return OR_ERR_ARG;
  if (fmt < OR_FMT_BF16 || fmt > OR_FMT_CB3K_CB4V) return OR_ERR_ARG;
  if (fmt >= OR_FMT_CB4 && (D & (D - 1))) return OR_ERR_ARG;
  memset(&j, 0, sizeof j);
  if (!out_row) {
    rows = (int32_t*)malloc(sizeof(int32_t) * (size_t)((int64_t)B * T * Hq + 1));
    if (!rows) return OR_ERR_NOMEM;
    for (b = 0; b < (int64_t)B * T * Hq; ++b) rows[b] = (int32_t)b;
    out_row = rows;
  }
  j.unit_b = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B * Hkv + 1));
  j.unit_g = (int32_t*)malloc(sizeof(int32_t) * (size_t)(B * Hkv + 1));
  if (fmt >= OR_FMT_CB4) {
    H = (double*)malloc(sizeof(double) * D * D);
    if (H) or_hadamard(D, H);
  }
  if (!j.unit_b || !j.unit_g || (fmt >= OR_FMT_CB4 && !H)) {
    free(rows);
    free(j.unit_b);
    free(j.unit_g);
    free(H);
    return OR_ERR_NOMEM;
  }
  for (b = 0; b < B; ++b)
    for (g = 0; g < Hkv; ++g) {
      int want = 0;
      for (jq = 0; jq < T; ++jq)
        for (hh = 0; hh < Hq / Hkv; ++hh) want |= out_row[(b * T + jq) * Hq + g * (Hq / Hkv) + hh] >= 0;
      if (want) {
        j.unit_b[nu] = (int32_t)b;
        j.unit_g[nu] = (int32_t)g;
        ++nu;
      }
    }
  j.B = B;
  j.T = T;
  j.Hq = Hq;
  j.Hkv = Hkv;
  j.D = D;
  j.bs = block_size;
  j.fmt = fmt;
  j.num_blocks = num_blocks;
  j.max_blocks = max_blocks;
  j.q = q;
  j.k_cache = k_cache;
  j.v_cache = v_cache;
  j.k_scales = k_scales;
  j.v_scales = v_scales;
  j.codebook = codebook;
  j.sign = sign;
  j.block_tables = block_tables;
  j.context_lens = context_lens;
  j.scale = scale;
  j.softcap = softcap;
  j.alibi = alibi_slopes;
  j.window = window;
  j.partition_size = partition_size;
  j.split_threshold = split_threshold;
  j.out_row = out_row;
  j.out = out;
  j.H = H;
  j.status = OR_OK;
  used = or_parallel_for(or_attn_task, &j, nu, threads);
  if (threads_used) *threads_used = used;
  free(rows);
  free(j.unit_b);
  free(j.unit_g);
  free(H);
  return j.status;
}
