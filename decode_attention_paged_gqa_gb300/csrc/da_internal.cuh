// da_internal.cuh -- definitions shared by the kernels and the C-ABI layer of libdecode_attn.
//
// Partition rules (turboquant-rs 0.4.1, src/cache/cuda/attention.rs, fused_attention():
// PARTITION_SIZE = 512 and num_partitions = ceil(kv_len / 512); attention.rs README, the
// sentence under the KV Cache Formats table: split-K decode only for contexts of 1024+
// tokens). With a sliding window the partitions are counted from the first attended token.
#pragma once

#include <cstddef>
#include <cstdint>
#include <type_traits>

#include <cuda_runtime.h>

#include "../../include/decode_attn.h"

namespace da {

constexpr int kBlockSize = 16;      // tokens per page (the only page size built)
constexpr int kMaxPartitions = 8192;
constexpr int kMaxColumns = 32;     // most (query token, head) pairs of one kv head: T * G

// Everything a kernel needs, passed by value (no pointers into host memory).
struct Args {
  const uint16_t* q;          // [B][T][Hq][D] bf16 bits
  const void* k_cache;        // layout by format, see decode_attn.h
  const void* v_cache;
  const float* k_scales;      // fp8: [1]; cb4: [num_blocks][Hkv][bs]
  const float* v_scales;
  const float* codebook;      // cb4: [16]
  const float* sign;          // cb4: [D]
  const float* alibi;         // [Hq] ALiBi slopes, or null
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* context_lens;  // [B]
  float* out;                 // [B][T][Hq][D]
  int B, T, Hq, Hkv, D, bs, num_blocks, max_blocks, max_ctx, fmt;  // T: query tokens per sequence
  float scale, softcap;
  int window, psize, thresh;
  int P;                      // partitions the grid and the workspace are sized for
  int ppc;                    // partitions a partition-kernel CTA walks (set by its launcher)
  int g_shift;                // log2 of the group size G = Hq / Hkv (a power of two)
  int ncg;                    // column groups: CTAs per partition chunk, each taking 8 of the T * G
                              // (query token, head) pairs when there are more than 8 (else 1)
  int ksub;                   // partials per partition: sub-items a partition's pages are dealt to
                              // by the codebook-value kernel when the batch has few partitions (a
                              // power of two <= 8; always 1 for the BF16 / FP8 kernel)
  uint32_t lut_stride;        // 128: entry stride of the codebook kernel's lookup tables (bytes)
  int schedule;               // da_params.partition_schedule (0 automatic, 1 shared, 2 owned)
  // Paired copies (set by a partition kernel's launcher): one 3-D tensor map spans both the K
  // and the V cache (or both per-token norm arrays), the third coordinate choosing the side,
  // so one copy fetches a page of both; *_zk is the side index of K (0 when K lies lower).
  int kv_pair, kv_zk, kn_pair, kn_zk;
  int ppc_req;                // da_params.partitions_per_cta (0 automatic)
  int owner;                  // 1: each warp of a partition kernel owns whole partitions, 0: the
                              // warps of a CTA share each partition (set by its launcher)
  // workspace pieces
  uint32_t* err;              // device error word (DA_DEVERR_* bits)
  uint32_t* claim;            // [2] next to it: the codebook-value kernel's item counter and count of
                              // warps done (zero between calls; zeroed with the workspace)
  float* q_rot;               // [B][T][Hq][D] (formats whose keys are on the rotated basis)
  float* part_o;              // [B][T][Hq][P * ksub][D], unnormalised partial outputs
  float* part_m;              // [B][T][Hq][P * ksub], running max in log2 units
  float* part_l;              // [B][T][Hq][P * ksub], running sum of 2^(s - m)
};

// First position attended by a query token at position `pos`: with a window of W tokens,
// the last W positions up to and including its own; else every position from 0.
__host__ __device__ __forceinline__ int window_start(int pos, int window) {
  const int s = window > 0 ? pos + 1 - window : 0;
  return s > 0 ? s : 0;
}

// First position attended by any of the T query tokens (positions L-T .. L-1) of a
// sequence of length L. With T = 1 this is max(0, L - window), or 0 without a window.
__host__ __device__ __forceinline__ int span_start(int L, int T, int window) { return window_start(L - T, window); }

// Partitions of an attended span of n tokens: 0 when empty, ceil(n / psize) when split, else 1.
__host__ __device__ __forceinline__ int num_partitions(int n, int psize, int thresh) {
  if (n <= 0) return 0;
  return (psize > 0 && n >= thresh) ? (n + psize - 1) / psize : 1;
}

__host__ __device__ __forceinline__ int seq_partitions(int L, int T, int window, int psize, int thresh) {
  return num_partitions(L - span_start(L, T, window), psize, thresh);
}

struct Range {
  int start, end;  // [start, end) token positions; start >= end means "no such partition"
};

// Token range of partition p of a sequence of (already clamped) length L with T query tokens
// and np partitions (seq_partitions); partitions are counted from the span start.
__host__ __device__ __forceinline__ Range partition_range_np(int L, int T, int p, int window, int psize, int np) {
  const int s = span_start(L, T, window);
  Range r{0, 0};
  if (p >= np) return r;
  if (np == 1) return Range{s, L};
  r.start = s + p * psize;
  r.end = r.start + psize < L ? r.start + psize : L;
  return r;
}

// The same with the partition count computed here.
__host__ __device__ __forceinline__ Range partition_range(int L, int T, int p, int window, int psize, int thresh) {
  return partition_range_np(L, T, p, window, psize, seq_partitions(L, T, window, psize, thresh));
}

// Largest length a context_lens entry may take.
__host__ __device__ __forceinline__ int max_valid_len(const Args& a) {
  const long long cap = (long long)a.max_blocks * a.bs;
  return cap < a.max_ctx ? (int)cap : a.max_ctx;
}

// Context length of sequence b, clamped into [0, max_valid_len]; flags bad input.
__device__ __forceinline__ int load_len(const Args& a, int b, bool report) {
  int L = __ldg(a.context_lens + b);
  const int lim = max_valid_len(a);
  if (L < 0 || L > lim) {
    if (report) atomicOr(a.err, DA_DEVERR_CONTEXT_LEN);
    L = L < 0 ? 0 : lim;
  }
  return L;
}

// Physical block of page `page` of sequence b, or -1 (flagged) when out of range.
__device__ __forceinline__ int load_block(const Args& a, int b, int page) {
  const int phys = __ldg(a.block_tables + (size_t)b * a.max_blocks + page);
  if (phys < 0 || phys >= a.num_blocks) {
    atomicOr(a.err, DA_DEVERR_BLOCK_ID);
    return -1;
  }
  return phys;
}

// Row of out and of the partials ([B][T][Hq] flattened) for virtual head vh = (query token) * G +
// (head within the group) of kv head g of sequence b (G = 2^g_shift).
__host__ __device__ __forceinline__ size_t query_row(const Args& a, int b, int g, int G, int vh) {
  return ((size_t)b * a.T + (vh >> a.g_shift)) * a.Hq + (size_t)g * G + (vh & (G - 1));
}

// Column groups of a partition kernel: one when the T * G pairs fit one 8-column MMA tile.
__host__ __device__ __forceinline__ int column_groups(int T, int G) { return T * G > 8 ? (T * G + 7) / 8 : 1; }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Workspace layout; every piece starts on a 256-byte boundary.
struct Layout {
  size_t err, q_rot, part_o, part_m, part_l, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline int query_len(const da_params& p) { return p.query_len > 1 ? p.query_len : 1; }

// Partition count of the longest possible span: that of a sequence of max_context_len tokens.
inline int host_max_partitions(const da_params& p) {
  long long n = p.max_context_len;
  if (p.window > 0 && n > (long long)p.window + query_len(p) - 1) n = (long long)p.window + query_len(p) - 1;
  const int np = num_partitions((int)n, p.partition_size, p.split_threshold);
  return np < 1 ? 1 : np;
}

// Partials per partition (Args::ksub): 1 for the BF16 / FP8 formats and when each warp is to
// own whole partitions (partition_schedule 2); else the smallest power of two (<= 8) that
// gives the batch at least kTargetItems items, at least 2 when the partitions are to be
// shared (partition_schedule 1), within kMaxPartitions partials per row. Depends on the
// parameters only, so the workspace size does too.
constexpr long long kTargetItems = 8192;
constexpr int kMaxKsub = 8;
inline int sub_items(const da_params& p) {
  if (p.kv_format == DA_KV_BF16 || p.kv_format == DA_KV_FP8_E4M3 || p.partition_schedule == 2) return 1;
  const int P = host_max_partitions(p);
  const long long units = (long long)p.batch * p.num_kv_heads * P *
                          column_groups(query_len(p), p.num_q_heads / p.num_kv_heads);
  int k = 1;
  while (k < kMaxKsub && units * k < kTargetItems) k *= 2;
  if (p.partition_schedule == 1 && k < 2) k = 2;
  while (k > 1 && (long long)P * k > kMaxPartitions) k /= 2;
  return k;
}

inline Layout workspace_layout(const da_params& p) {
  Layout l{};
  const size_t BH = (size_t)p.batch * query_len(p) * p.num_q_heads;
  const size_t P = (size_t)host_max_partitions(p) * sub_items(p);
  size_t off = 0;
  l.err = off;  // the error word, then the item counter and the count of warps done
  off = align256(off + 3 * sizeof(uint32_t));
  l.q_rot = off;
  const bool rotated_keys = p.kv_format == DA_KV_CB4 || p.kv_format == DA_KV_CB3K_CB4V;
  off = align256(off + (rotated_keys ? BH * p.head_dim * sizeof(float) : 0));
  l.part_o = off;
  off = align256(off + BH * P * p.head_dim * sizeof(float));
  l.part_m = off;
  off = align256(off + BH * P * sizeof(float));
  l.part_l = off;
  off = align256(off + BH * P * sizeof(float));
  l.total = off;
  return l;
}

// Per-device "done once" flags (up to 64 devices).
struct DeviceFlags {
  unsigned long long bits = 0;
};

// Raise a kernel's dynamic shared-memory limit once per device.
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel kern, size_t bytes, DeviceFlags& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(&done.bits, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) __atomic_fetch_or(&done.bits, bit, __ATOMIC_RELEASE);
  return e;
}

// The host-side checks of a call's parameters and tensors, without the workspace (the same
// checks and status codes as decode_attn_paged; decode_attn.cu).
int check_call(const void* q, const void* k, const void* v, const float* ks, const float* vs, const float* cb,
               const float* sign, const int32_t* bt, const int32_t* lens, const float* out, const da_params* p);

// The checked launch sequence behind decode_attn_paged and its phases (decode_attn.cu).
enum Phase { kRotate = 1, kPartition = 2, kReduce = 4, kAll = 7 };
int run_phases(int phases, const void* q, const void* k, const void* v, const float* ks, const float* vs,
               const float* cb, const float* sign, const int32_t* bt, const int32_t* lens, float* out,
               const da_params* p, void* stream);

// Partitions per CTA for a partition kernel with `per_sm` resident CTAs per SM: as requested,
// else enough that the CTAs walk consecutive partitions of one (sequence, kv head) with their
// pipelines full across partition boundaries, while the grid keeps about eight waves of CTAs.
// Also caches the device's SM count.
inline int partitions_per_cta(const Args& a, int per_sm, int* cached_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return a.ppc_req > 0 ? a.ppc_req : 1;
  if (cached_sms[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return a.ppc_req > 0 ? a.ppc_req : 1;
    cached_sms[dev] = sms;
  }
  if (a.ppc_req > 0) return a.ppc_req;
  const long long units = (long long)a.P * a.Hkv * a.B * a.ncg;
  const long long waves = units / (8ll * cached_sms[dev] * (per_sm > 0 ? per_sm : 1));
  return waves < 1 ? 1 : (waves > 8 ? 8 : (int)waves);
}

// CTAs of a kernel with `per_sm` resident CTAs per SM that the device holds at once (0 when
// the SM count is not known; partitions_per_cta caches it).
inline long long resident_slots(int per_sm, const int* cached_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cached_sms[dev] <= 0) return 0;
  return (long long)cached_sms[dev] * (per_sm > 0 ? per_sm : 1);
}

// Whether a partition kernel's warps own whole partitions: as requested, else when the
// batch has at least `min_fill_x2` / 2 partitions (counted at the longest possible span) for
// every warp the GPU holds at once. Below that, sharing each partition among a CTA's warps
// keeps more warps busy; above it, the owned schedule saves the per-partition merge. The
// break-even depends on the kernel: for the codebook kernel (eight warps sharing a partition
// at D = 128) it lies near half a warp per partition, for the tensor-core kernel between one
// and two (batches of varied lengths have fewer partitions than counted, so the latter errs
// high).
inline bool warps_own_partitions(const Args& a, int per_sm, int warps_per_cta, int min_fill_x2,
                                 const int* cached_sms) {
  if (a.schedule == 1) return false;
  if (a.schedule == 2) return true;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || cached_sms[dev] <= 0) return false;
  const long long units = (long long)a.P * a.Hkv * a.B * a.ncg;
  return 2ll * units >= (long long)min_fill_x2 * cached_sms[dev] * (per_sm > 0 ? per_sm : 1) * warps_per_cta;
}

// Launch with programmatic stream serialisation: the kernel's CTAs may be scheduled while the
// previous kernel on the stream finishes (the kernel waits in-kernel, grid_dependency_wait,
// before reading what that kernel writes), hiding the launch gap between the phases.
// The arguments are passed by address, so their types must be the kernel's parameter types.
template <typename... KArgs, typename... Params>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       const Params&... params) {
  static_assert(sizeof...(KArgs) == sizeof...(Params) && (std::is_same_v<std::remove_cv_t<KArgs>, Params> && ...),
                "launch_pdl: argument types must match the kernel's parameters");
  void* args[] = {const_cast<void*>(static_cast<const void*>(&params))...};
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kern), args);
}

// Launchers (one translation unit each). They return cudaGetLastError() of their launch.
cudaError_t launch_rotate_q(const Args& a, cudaStream_t s);
cudaError_t launch_partition(const Args& a, cudaStream_t s);     // dispatches on the format:
cudaError_t launch_partition_tc(const Args& a, cudaStream_t s);  //   BF16, FP8: TMA + tensor cores
cudaError_t launch_partition_cb(const Args& a, cudaStream_t s);  //   4-bit codebook values: lookup tables + tensor cores
cudaError_t launch_reduce(const Args& a, cudaStream_t s);
cudaError_t launch_encode_fp8(const float* x, long long n, uint8_t* codes, float* scale, cudaStream_t s);
cudaError_t launch_encode_codebook(const float* x, long long nvec, int D, int bits, const float* sign,
                                   const float* codebook, uint8_t* packed, float* scales, cudaStream_t s);
int lloyd_max_codebook(int levels, double sigma, float* out);
cudaError_t launch_debug_bounds(const Args& a, int32_t* bounds, cudaStream_t s);
cudaError_t launch_debug_dequant(const Args& a, const void* cache, const float* scales, const int32_t* ids, int n,
                                 int which, float* out, cudaStream_t s);

}  // namespace da
