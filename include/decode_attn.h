/*
 * decode_attn.h -- C ABI of libdecode_attn, single-token (decode) grouped-query
 * attention over a paged KV cache on a GB300 (sm_103a) GPU.
 *
 * For every sequence b and query head h (kv head g = h / G, G = Hq / Hkv):
 *     out[b][h] = softmax_t( cap(scale * q[b][h] . K[b][g][t]) ) . V[b][g][t]
 * over the attended positions t of sequence b, where K/V rows are gathered through the
 * sequence's block table and dequantised from the cache format. Long contexts are split
 * into partitions, each producing a partial output with its running max and sum, and a
 * float reduce combines them.
 *   - Operation, formats, split-K + float reduce, features: attention.rs README,
 *     "KV Cache Formats" table and the paragraph under it (split-K decode kernels per
 *     format, used from 1024 tokens of context, with one fp32 reduce shared by all), and
 *     its feature list (softcap, sliding window, GQA/MQA, paged block tables).
 *   - Two-phase structure, partition size 512, ceil(kv_len / 512) partitions, partial
 *     output/max/sum buffers, f32 output [heads, head_dim], zero output for an empty
 *     context, codebook + sign_pattern inputs of the codebook format: turboquant-rs 0.4.1,
 *     src/cache/cuda/attention.rs, fused_attention() and its FFI call.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer unless its comment says "host". The caller
 *     owns every buffer; the library allocates no device memory and keeps no state
 *     between calls except what lives in the caller's workspace.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream) and runs asynchronously. No entry point synchronises, except
 *     decode_attn_get_device_error, which says so.
 *   - The partition kernel and the reduce are launched with programmatic stream
 *     serialisation: their CTAs may be scheduled while the previous kernel on `stream` is
 *     still running, and they wait inside the kernel, before their first read of any input
 *     or workspace, until that kernel has completed and its writes are visible. Stream order
 *     is therefore kept as for ordinary launches, also when the calls are captured into a
 *     CUDA graph; only the launch gap between kernels is hidden.
 *   - Return value: DA_OK (0) or a negative DA_ERR_* code. Argument checks happen on the
 *     host before anything is enqueued: a call that returns DA_ERR_INVALID_ARG,
 *     DA_ERR_UNSUPPORTED or DA_ERR_WORKSPACE has enqueued nothing.
 *   - Bad DATA found by a kernel (a block id outside [0, num_blocks), a context length
 *     outside [0, min(max_context_len, max_blocks_per_seq * block_size)]) does not fault:
 *     the kernel skips the bad page (or reads block 0 in its place) or clamps the length,
 *     sets a bit in the workspace's error word, and carries on. The affected outputs are
 *     then unspecified.
 *     decode_attn_get_device_error reports the bits.
 */
#ifndef DECODE_ATTN_H_
#define DECODE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* KV cache formats (attention.rs README, KV Cache Formats table). */
enum da_kv_format {
  /* Unquantized bfloat16. Cache layout [num_blocks][Hkv][block_size][D] bf16. */
  DA_KV_BF16 = 0,
  /* FP8 E4M3 (OCP "E4M3FN": bias 7, max 448, no infinity) with one fp32 dequant scale
   * per cache tensor: value = scale * e4m3(code). Layout [num_blocks][Hkv][block_size][D]
   * bytes; k_scales / v_scales point to ONE float each. */
  DA_KV_FP8_E4M3 = 1,
  /* 4-bit codebook on a random-sign Walsh-Hadamard basis ("Turbo4"). Each K or V vector x
   * is stored as r = H diag(sign) x / sqrt(D) (H: D x D Sylvester Hadamard matrix,
   * sign: sign_pattern), quantised per coordinate to the nearest of 16 codebook values
   * after division by ||x||_2. Layout: [num_blocks][Hkv][block_size][D/2] bytes, two
   * indices per byte, coordinate 2k in the low nibble of byte k; k_scales / v_scales are
   * [num_blocks][Hkv][block_size] fp32 norms; codebook is [16] fp32. The kernels rotate q
   * the same way, attend in the rotated basis and un-rotate the output once per head. */
  DA_KV_CB4 = 2,
  /* "Turbo8": keys as DA_KV_FP8_E4M3 (k_scales: one float), values as DA_KV_CB4 (v_scales:
   * per-token norms; codebook: the 16 value levels). */
  DA_KV_FP8K_CB4V = 3,
  /* "Turbo3": keys as a 3-bit codebook on the same rotated basis (8 levels; the codes of a
   * row form a little-endian bit stream, coordinate d at stream bits [3d, 3d+3), i.e. 3D/8
   * bytes per row; k_scales: per-token norms), values as DA_KV_CB4. codebook holds the 8 key
   * levels followed by the 16 value levels ([24] f32). */
  DA_KV_CB3K_CB4V = 4
};

enum da_status {
  DA_OK = 0,
  DA_ERR_INVALID_ARG = -1,  /* a required pointer is NULL, a size is negative or inconsistent */
  DA_ERR_UNSUPPORTED = -2,  /* valid arguments outside the built set (see da_params) */
  DA_ERR_WORKSPACE = -3,    /* workspace NULL, misaligned, or smaller than decode_attn_workspace_bytes */
  DA_ERR_LAUNCH = -4,       /* a kernel launch failed; see cudaGetLastError */
  DA_ERR_CUDA = -5,         /* another CUDA runtime call failed */
  DA_ERR_STATIC_WORKSPACE = -6 /* decode_attn_paged_static_workspace: the call needs more workspace
                                  than the library's fixed 64 MiB array holds */
};

/* Bits of the device error word (decode_attn_get_device_error). */
#define DA_DEVERR_BLOCK_ID 0x1u    /* a block-table entry used by the call was outside [0, num_blocks) */
#define DA_DEVERR_CONTEXT_LEN 0x2u /* a context length was < 0 or above the limits in the header comment */
#define DA_DEVERR_TIMEOUT 0x4u     /* a wait for a page copy gave up after 200 ms (never expected) */
#define DA_DEVERR_SMEM_LAYOUT 0x8u /* a partition kernel's shared-memory layout did not fit the CTA's
                                      window, so it computed nothing (never expected) */

typedef struct da_params {
  int32_t batch;              /* B >= 0 sequences (B == 0: nothing to do) */
  int32_t query_len;          /* T >= 1 query tokens per sequence (0 counts as 1). T = 1 is ordinary
                                 decode; T > 1 is multi-token decode with a causal mask: query token j
                                 sits at position L_b - T + j and attends positions up to its own (the
                                 last `window` of them when a window is set). T * G <= 32. */
  int32_t num_q_heads;        /* Hq >= 1 */
  int32_t num_kv_heads;       /* Hkv >= 1, Hq % Hkv == 0; group size G = Hq / Hkv in {1, 2, 4, 8} */
  int32_t head_dim;           /* D in {128, 256} */
  int32_t block_size;         /* tokens per page; 16 */
  int32_t num_blocks;         /* physical pages in the pool (>= 1) */
  int32_t max_blocks_per_seq; /* row length of block_tables */
  int32_t max_context_len;    /* upper bound on every context_lens[b]; sizes grid and workspace */
  int32_t kv_format;          /* enum da_kv_format */
  float softmax_scale;        /* scale applied to q . k (e.g. 1/sqrt(D)) */
  float softcap;              /* 0 = off; else s <- softcap * tanh(s / softcap) after scaling */
  int32_t window;             /* 0 = off; else attend only the last `window` tokens (t >= L - window) */
  int32_t partition_size;     /* tokens per split-K partition (512); 0 = never split. A span of
                                 max_context_len tokens may have at most 8192 partitions
                                 (decode_attn_max_partitions), else DA_ERR_UNSUPPORTED. */
  int32_t split_threshold;    /* split a sequence iff its attended length >= this (1024) */
  int32_t partition_schedule; /* how a partition kernel's warps share the work (results are the same
                                 up to rounding): 0 = chosen per call from the number of partitions,
                                 1 = the warps of a CTA share each partition, 2 = each warp owns whole
                                 partitions (no cross-warp merge; best when there are partitions
                                 for every warp the GPU holds at once). Other values are rejected. */
  int32_t partitions_per_cta; /* consecutive partitions of one (sequence, kv head) a CTA of a partition
                                 kernel takes, 0 = chosen per call, else 1 .. 64 (rounded up to a
                                 multiple of the CTA's warps when each warp owns partitions) */
  const float* alibi_slopes;  /* NULL = off; else DEVICE pointer to [Hq] f32 ALiBi slopes: the score of
                                 key position t for a query at position pos gets slope_h * (t - pos)
                                 added after scaling and softcap (attention.rs README, feature list:
                                 ALiBi slopes). 4-byte aligned. */
  void* workspace;            /* device memory, 256-byte aligned, decode_attn_workspace_bytes() long,
                                 zeroed once by decode_attn_workspace_init before first use */
  size_t workspace_bytes;     /* size of `workspace` in bytes */
} da_params;

/* Bytes of workspace a call with these parameters needs (0 if the parameters are invalid).
 * The workspace holds the error word, the rotated queries of the codebook formats
 * ([B][T][Hq][D] f32), the split-K partials -- output [B][T][Hq][P][D] f32 (unnormalised),
 * running max and running sum [B][T][Hq][P] f32, where P is the partition count of a
 * sequence of length max_context_len (the page's partial buffers, sized for a batch). */
size_t decode_attn_workspace_bytes(const da_params* p);

/* Zero the workspace (in particular its error word) on `stream`. Call once after
 * allocating it. Returns DA_OK, DA_ERR_WORKSPACE or DA_ERR_CUDA. */
int decode_attn_workspace_init(const da_params* p, void* stream);

/* Full decode attention: [codebook format: query rotation] -> partition kernel -> reduce.
 *   q            [B][T][Hq][D] bf16, the query tokens of each sequence (16-byte aligned).
 *   k_cache,
 *   v_cache      the paged caches, layout by format (enum da_kv_format), 16-byte aligned;
 *                num_blocks * Hkv * block_size must stay below 2^31.
 *   k_scales,
 *   v_scales     per side: FP8 one float; codebook [num_blocks][Hkv][block_size] f32 norms;
 *                BF16: ignored (may be NULL).
 *   codebook     formats with a codebook side: [16] f32 (DA_KV_CB3K_CB4V: [8 + 16]); else ignored.
 *   sign_pattern formats with a codebook side: [D] f32 of +1/-1; else ignored (may be NULL).
 *   block_tables [B][max_blocks_per_seq] int32: page i of sequence b lives in physical block
 *                block_tables[b][i]; token t of sequence b is slot t % block_size of page
 *                t / block_size. Only the pages holding attended tokens are read.
 *   context_lens [B] int32: L_b, tokens in sequence b. L_b == 0 gives an all-zero output row.
 *   out          [B][T][Hq][D] f32, fully written (rows of query tokens that attend nothing,
 *                i.e. L_b == 0 or position < 0, are zero).
 * Partitioning: the span attended by the sequence's query tokens runs from the first query
 * token's first attended position to L_b; with n_b its length (min(L_b, window + T - 1) with
 * a window), the sequence is split iff partition_size > 0 and n_b >= split_threshold, into
 * ceil(n_b / partition_size) partitions counted from the span start. */
int decode_attn_paged(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                      const float* v_scales, const float* codebook, const float* sign_pattern,
                      const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                      void* stream);

/* The phases of decode_attn_paged, for callers that schedule or time them one by one.
 * Same arguments and checks as decode_attn_paged; they must run in this order on one stream:
 *   decode_attn_rotate_q   formats whose keys are codebook codes (DA_KV_CB4, DA_KV_CB3K_CB4V;
 *                          returns DA_OK and does nothing for the others):
 *                          q_rot = H diag(sign) q / sqrt(D) into the workspace.
 *   decode_attn_partition  each CTA walks consecutive partitions of one (sequence, kv head)
 *                          (p->partition_schedule, p->partitions_per_cta): partial output, max
 *                          and sum of each partition into the workspace, or the normalised
 *                          output of an unsplit sequence whose values are not codebook codes.
 *   decode_attn_reduce     combines the partials of each (sequence, query token, head) into out
 *                          (and un-rotates it when the values are codebook codes). */
int decode_attn_rotate_q(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                         const float* v_scales, const float* codebook, const float* sign_pattern,
                         const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                         void* stream);
int decode_attn_partition(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                          const float* v_scales, const float* codebook, const float* sign_pattern,
                          const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                          void* stream);
int decode_attn_reduce(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                       const float* v_scales, const float* codebook, const float* sign_pattern,
                       const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                       void* stream);

/* decode_attn_paged for callers that cannot allocate device memory: code where device
 * allocation is forbidden or unavailable, such as a plugin inside a host framework that owns
 * every allocation and exposes none to its extensions, a real-time loop that must not call
 * the allocator (cudaMalloc can synchronise the device and take unbounded time), or a caller
 * with no CUDA allocator of its own. (This entry point has no counterpart in the pages; it is
 * an addition of this library.)
 * Same arguments, argument checks, status codes and results as decode_attn_paged, except
 * that p->workspace and p->workspace_bytes are ignored: the workspace is a fixed 64 MiB array
 * in device global memory defined by the library (every GPU that loads the library holds it
 * until the process exits). A call that passes decode_attn_paged's checks but whose
 * decode_attn_workspace_bytes(p) exceeds 64 MiB returns DA_ERR_STATIC_WORKSPACE. A rejected
 * call has enqueued nothing. Nothing is allocated and no allocating routine is called; each
 * accepted call clears the array's error word on `stream` first.
 * All calls share the one array: calls that overlap on the GPU (on different streams, or
 * from different host threads) race on it and must be serialised by the caller. The
 * device-side bad-input bits of these calls are not reported.
 * The first call on each device, and the first after the device's current context changed
 * (e.g. after cudaDeviceReset), looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that call before any stream capture. */
int decode_attn_paged_static_workspace(const void* q, const void* k_cache, const void* v_cache,
                                       const float* k_scales, const float* v_scales, const float* codebook,
                                       const float* sign_pattern, const int32_t* block_tables,
                                       const int32_t* context_lens, float* out, const da_params* p, void* stream);

/* Synchronises `stream`, then reads the workspace's error word into *err_out (host
 * pointer; DA_DEVERR_* bits, 0 = no bad input seen since the last read) and clears it. */
int decode_attn_get_device_error(const da_params* p, void* stream, uint32_t* err_out);

/* Static string describing a DA_* status code. */
const char* decode_attn_strerror(int status);

/* Partition count the grid is sized for: that of a sequence of length max_context_len. */
int decode_attn_max_partitions(const da_params* p);

/* ---- cache writers: the step that fills the quantised caches ------------------------- */

/* FP8 E4M3 encoding of one cache tensor (attention.rs README, KV Cache Formats table):
 * scale = max|x| / 448 (binary32; 1 for an all-zero tensor) is written to *scale_out
 * (device float), and codes[i] = round-to-nearest-even E4M3 of the binary32 quotient
 * x[i] / scale, saturating at +-448 (NaN stays NaN). x: n device floats, in the cache's
 * layout; codes: n device bytes. Three kernels on `stream`. */
int decode_attn_encode_fp8(const float* x, int64_t n, uint8_t* codes, float* scale_out, void* stream);

/* 4-bit codebook encoding of num_vectors vectors of head_dim floats (128 or 256), e.g. the
 * rows [num_blocks][Hkv][block_size] of a cache: r = H diag(sign) x / sqrt(D); scale =
 * ||x||_2 as binary32; idx_d = nearest codebook[16] value to r_d / scale (ties to the lower
 * index); packed[v][k] = idx_{2k} | idx_{2k+1} << 4; scales[v] = scale. The norm and the
 * rotation are evaluated in fp64 with index-ordered sums, so the codes do not depend on
 * the thread layout. All pointers are device pointers. */
int decode_attn_encode_cb4(const float* x, int64_t num_vectors, int32_t head_dim, const float* sign_pattern,
                           const float* codebook, uint8_t* packed, float* scales, void* stream);

/* The same for `bits`-bit codes (3 or 4) with a [2^bits] codebook; packed rows are
 * head_dim * bits / 8 bytes holding the codes as a little-endian bit stream (coordinate d
 * at stream bits [bits*d, bits*d + bits)). bits == 4 is decode_attn_encode_cb4. */
int decode_attn_encode_codebook(const float* x, int64_t num_vectors, int32_t head_dim, int32_t bits,
                                const float* sign_pattern, const float* codebook, uint8_t* packed, float* scales,
                                void* stream);

/* Host-side: the `levels`-level Lloyd-Max quantiser of N(0, sigma^2) (alternate midpoint
 * thresholds and conditional-mean levels until no level moves by 1e-14 sigma, then make it
 * exactly symmetric), written ascending as binary32 to codebook_host[levels]. The
 * codebook format uses levels = 16, sigma = 1/sqrt(D). Returns DA_OK or DA_ERR_INVALID_ARG. */
int decode_attn_codebook_lloyd_max(int32_t levels, double sigma, float* codebook_host);

/* ---- debug exports: the kernels' own device code, for bit-exact tests ---------------- */

/* bounds [B][P][2] int32 (P = decode_attn_max_partitions): [start, end) of partition p of
 * sequence b as the partition kernel computes it, or (-1, -1) where p is past the
 * sequence's last partition. */
int decode_attn_debug_partition_bounds(const int32_t* context_lens, int32_t* bounds, const da_params* p,
                                       void* stream);

/* out [n][Hkv][block_size][D] f32: the values the partition kernel computes from the cache
 * blocks block_ids[0..n) (device int32) of the K side (which == 0) or V side (which == 1) of
 * the format: BF16 exact; FP8 scale * e4m3(code) with scales[0]; codebook sides
 * scale_t * codebook[idx] in the rotated basis (codebook as in decode_attn_paged). */
int decode_attn_debug_dequant_blocks(const void* cache, const float* scales, const float* codebook,
                                     const int32_t* block_ids, int32_t n, int32_t which, float* out,
                                     const da_params* p, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DECODE_ATTN_H_ */
