// decode_attn.cu -- the C ABI of libdecode_attn (declared in include/decode_attn.h):
// host-side argument checks, workspace carving, and the launch sequence
//   [codebook format: query rotation] -> partition kernel -> reduce kernel
// on the caller's stream. Mirrors the host wrapper of turboquant-rs 0.4.1,
// src/cache/cuda/attention.rs, fused_attention(): device checks that refuse to launch
// (its bail! paths), an all-zero output for an empty context, the two-phase launch, and
// a launch-error check after it (check_cuda_kernel_launch) -- but the caller owns the
// partial buffers (workspace) instead of the wrapper allocating them per call.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "da_internal.cuh"
#include "kv_formats.cuh"

using namespace da;

namespace {

int check_params(const da_params* p) {
  if (!p) return DA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->query_len < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0 ||
      p->block_size <= 0 ||
      p->num_blocks <= 0 || p->max_blocks_per_seq <= 0 || p->max_context_len < 0 || p->window < 0 ||
      p->partition_size < 0 || p->split_threshold < 0 || p->partition_schedule < 0 || p->partition_schedule > 2 ||
      p->partitions_per_cta < 0 || p->partitions_per_cta > 64)
    return DA_ERR_INVALID_ARG;
  if (p->num_q_heads % p->num_kv_heads) return DA_ERR_INVALID_ARG;
  if (!std::isfinite(p->softmax_scale) || !std::isfinite(p->softcap) || p->softcap < 0.0f) return DA_ERR_INVALID_ARG;
  if (p->kv_format < DA_KV_BF16 || p->kv_format > DA_KV_CB3K_CB4V) return DA_ERR_INVALID_ARG;
  const int G = p->num_q_heads / p->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return DA_ERR_UNSUPPORTED;
  if ((long long)query_len(*p) * G > kMaxColumns) return DA_ERR_UNSUPPORTED;  // (query token, head) pairs
  if (p->head_dim != 128 && p->head_dim != 256) return DA_ERR_UNSUPPORTED;
  if (p->block_size != kBlockSize) return DA_ERR_UNSUPPORTED;
  if ((long long)p->batch * query_len(*p) > 65535 || p->num_kv_heads > 65535 || p->num_q_heads > 65535)
    return DA_ERR_UNSUPPORTED;
  if (host_max_partitions(*p) > kMaxPartitions) return DA_ERR_UNSUPPORTED;
  if ((long long)p->num_blocks * p->num_kv_heads * p->block_size >= (1ll << 31)) return DA_ERR_UNSUPPORTED;
  // the partition kernels index their work items with 32-bit integers
  if ((long long)p->batch * p->num_kv_heads * host_max_partitions(*p) * column_groups(query_len(*p), G) *
          kMaxKsub >= (1ll << 31))
    return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

int check_workspace(const da_params* p) {
  if (!p->workspace || (reinterpret_cast<uintptr_t>(p->workspace) & 255u)) return DA_ERR_WORKSPACE;
  if (p->workspace_bytes < workspace_layout(*p).total) return DA_ERR_WORKSPACE;
  return DA_OK;
}

bool aligned(const void* ptr, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0; }

int check_tensors(const void* q, const void* k, const void* v, const float* ks, const float* vs, const float* cb,
                  const float* sign, const int32_t* bt, const int32_t* lens, const float* out, const da_params* p) {
  if (!q || !k || !v || !bt || !lens || !out) return DA_ERR_INVALID_ARG;
  if (p->kv_format != DA_KV_BF16 && (!ks || !vs)) return DA_ERR_INVALID_ARG;
  if ((is_codebook(k_side(p->kv_format)) || is_codebook(v_side(p->kv_format))) && (!cb || !sign))
    return DA_ERR_INVALID_ARG;
  // vector loads: caches on 16-byte boundaries, q / out / scales on their element size
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(q, 16) || !aligned(out, 4) || !aligned(bt, 4) ||
      !aligned(lens, 4))
    return DA_ERR_INVALID_ARG;
  if (p->alibi_slopes && !aligned(p->alibi_slopes, 4)) return DA_ERR_INVALID_ARG;
  // per-token norms of a codebook side are copied 16 tokens (64 bytes) at a time
  if ((is_codebook(k_side(p->kv_format)) && !aligned(ks, 16)) || (is_codebook(v_side(p->kv_format)) && !aligned(vs, 16)))
    return DA_ERR_INVALID_ARG;
  return DA_OK;
}

Args make_args(const void* q, const void* k, const void* v, const float* ks, const float* vs, const float* cb,
               const float* sign, const int32_t* bt, const int32_t* lens, float* out, const da_params* p) {
  Args a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k_cache = k;
  a.v_cache = v;
  a.k_scales = ks;
  a.v_scales = vs;
  a.codebook = cb;
  a.sign = sign;
  a.block_tables = bt;
  a.context_lens = lens;
  a.out = out;
  a.B = p->batch;
  a.T = query_len(*p);
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.D = p->head_dim;
  a.bs = p->block_size;
  a.num_blocks = p->num_blocks;
  a.max_blocks = p->max_blocks_per_seq;
  a.max_ctx = p->max_context_len;
  a.fmt = p->kv_format;
  a.scale = p->softmax_scale;
  a.softcap = p->softcap;
  a.window = p->window;
  a.psize = p->partition_size;
  a.thresh = p->split_threshold;
  a.P = host_max_partitions(*p);
  a.ppc = 1;
  a.ncg = column_groups(a.T, a.Hq / a.Hkv);
  a.g_shift = 0;
  while ((1 << a.g_shift) < a.Hq / a.Hkv) ++a.g_shift;  // G is 1, 2, 4 or 8 (check_params)
  a.ksub = sub_items(*p);
  a.lut_stride = 128;
  a.alibi = p->alibi_slopes;
  a.schedule = p->partition_schedule;
  a.kv_pair = a.kv_zk = a.kn_pair = a.kn_zk = 0;
  a.ppc_req = p->partitions_per_cta;
  a.owner = 0;
  const Layout l = workspace_layout(*p);
  char* ws = static_cast<char*>(p->workspace);
  a.err = reinterpret_cast<uint32_t*>(ws + l.err);
  a.claim = a.err + 1;
  a.q_rot = reinterpret_cast<float*>(ws + l.q_rot);
  a.part_o = reinterpret_cast<float*>(ws + l.part_o);
  a.part_m = reinterpret_cast<float*>(ws + l.part_m);
  a.part_l = reinterpret_cast<float*>(ws + l.part_l);
  return a;
}

}  // namespace

namespace da {

int check_call(const void* q, const void* k, const void* v, const float* ks, const float* vs, const float* cb,
               const float* sign, const int32_t* bt, const int32_t* lens, const float* out, const da_params* p) {
  const int rc = check_params(p);
  return rc ? rc : check_tensors(q, k, v, ks, vs, cb, sign, bt, lens, out, p);
}

int run_phases(int phases, const void* q, const void* k, const void* v, const float* ks, const float* vs,
               const float* cb, const float* sign, const int32_t* bt, const int32_t* lens, float* out,
               const da_params* p, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_workspace(p))) return rc;
  if ((rc = check_tensors(q, k, v, ks, vs, cb, sign, bt, lens, out, p))) return rc;
  if (p->batch == 0) return DA_OK;
  const Args a = make_args(q, k, v, ks, vs, cb, sign, bt, lens, out, p);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((phases & kRotate) && is_codebook(k_side(a.fmt)) && launch_rotate_q(a, s) != cudaSuccess)
    return DA_ERR_LAUNCH;
  if ((phases & kPartition) && launch_partition(a, s) != cudaSuccess) return DA_ERR_LAUNCH;
  if ((phases & kReduce) && launch_reduce(a, s) != cudaSuccess) return DA_ERR_LAUNCH;
  return DA_OK;
}

}  // namespace da

extern "C" {

size_t decode_attn_workspace_bytes(const da_params* p) {
  if (check_params(p)) return 0;
  return workspace_layout(*p).total;
}

int decode_attn_workspace_init(const da_params* p, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_workspace(p))) return rc;
  return cudaMemsetAsync(p->workspace, 0, workspace_layout(*p).total, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? DA_OK
             : DA_ERR_CUDA;
}

int decode_attn_paged(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                      const float* v_scales, const float* codebook, const float* sign_pattern,
                      const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                      void* stream) {
  return run_phases(kAll, q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                    context_lens, out, p, stream);
}

int decode_attn_rotate_q(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                         const float* v_scales, const float* codebook, const float* sign_pattern,
                         const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                         void* stream) {
  return run_phases(kRotate, q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                    context_lens, out, p, stream);
}

int decode_attn_partition(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                          const float* v_scales, const float* codebook, const float* sign_pattern,
                          const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                          void* stream) {
  return run_phases(kPartition, q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                    context_lens, out, p, stream);
}

int decode_attn_reduce(const void* q, const void* k_cache, const void* v_cache, const float* k_scales,
                       const float* v_scales, const float* codebook, const float* sign_pattern,
                       const int32_t* block_tables, const int32_t* context_lens, float* out, const da_params* p,
                       void* stream) {
  return run_phases(kReduce, q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                    context_lens, out, p, stream);
}

int decode_attn_get_device_error(const da_params* p, void* stream, uint32_t* err_out) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_workspace(p))) return rc;
  if (!err_out) return DA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(static_cast<char*>(p->workspace) + workspace_layout(*p).err);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof v, s) != cudaSuccess) return DA_ERR_CUDA;
  *err_out = v;
  return DA_OK;
}

const char* decode_attn_strerror(int status) {
  switch (status) {
    case DA_OK: return "ok";
    case DA_ERR_INVALID_ARG: return "invalid argument";
    case DA_ERR_UNSUPPORTED: return "unsupported configuration (head_dim, group size, block size or partition count)";
    case DA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DA_ERR_LAUNCH: return "kernel launch failed";
    case DA_ERR_CUDA: return "CUDA runtime call failed";
    case DA_ERR_STATIC_WORKSPACE: return "the call needs more workspace than the library's static 64 MiB array holds";
  }
  return "unknown status";
}

int decode_attn_max_partitions(const da_params* p) {
  int rc = check_params(p);
  if (rc) return rc;
  return host_max_partitions(*p);
}

int decode_attn_encode_fp8(const float* x, int64_t n, uint8_t* codes, float* scale_out, void* stream) {
  if (n < 0 || !scale_out || (n > 0 && (!x || !codes)) || !aligned(scale_out, 4) || !aligned(x, 4))
    return DA_ERR_INVALID_ARG;
  return launch_encode_fp8(x, n, codes, scale_out, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DA_OK
             : DA_ERR_LAUNCH;
}

int decode_attn_encode_codebook(const float* x, int64_t num_vectors, int32_t head_dim, int32_t bits,
                                const float* sign_pattern, const float* codebook, uint8_t* packed, float* scales,
                                void* stream) {
  if (num_vectors < 0 || (num_vectors > 0 && (!x || !sign_pattern || !codebook || !packed || !scales)))
    return DA_ERR_INVALID_ARG;
  if ((head_dim != 128 && head_dim != 256) || (bits != 3 && bits != 4)) return DA_ERR_UNSUPPORTED;
  return launch_encode_codebook(x, num_vectors, head_dim, bits, sign_pattern, codebook, packed, scales,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DA_OK
             : DA_ERR_LAUNCH;
}

int decode_attn_encode_cb4(const float* x, int64_t num_vectors, int32_t head_dim, const float* sign_pattern,
                           const float* codebook, uint8_t* packed, float* scales, void* stream) {
  return decode_attn_encode_codebook(x, num_vectors, head_dim, 4, sign_pattern, codebook, packed, scales, stream);
}

int decode_attn_codebook_lloyd_max(int32_t levels, double sigma, float* codebook_host) {
  if (!codebook_host) return DA_ERR_INVALID_ARG;
  return lloyd_max_codebook(levels, sigma, codebook_host) == 0 ? DA_OK : DA_ERR_INVALID_ARG;
}

int decode_attn_debug_partition_bounds(const int32_t* context_lens, int32_t* bounds, const da_params* p,
                                       void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_workspace(p))) return rc;
  if (!context_lens || !bounds) return DA_ERR_INVALID_ARG;
  Args a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, context_lens, nullptr, p);
  return launch_debug_bounds(a, bounds, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DA_OK : DA_ERR_LAUNCH;
}

int decode_attn_debug_dequant_blocks(const void* cache, const float* scales, const float* codebook,
                                     const int32_t* block_ids, int32_t n, int32_t which, float* out,
                                     const da_params* p, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if ((rc = check_workspace(p))) return rc;
  if (!cache || !block_ids || !out || n < 0 || !aligned(cache, 16) || (which != 0 && which != 1))
    return DA_ERR_INVALID_ARG;
  const int side = which ? v_side(p->kv_format) : k_side(p->kv_format);
  if (side != kSideBF16 && !scales) return DA_ERR_INVALID_ARG;
  if (is_codebook(side) && !codebook) return DA_ERR_INVALID_ARG;
  Args a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, codebook, nullptr, nullptr, nullptr, nullptr, p);
  return launch_debug_dequant(a, cache, scales, block_ids, n, which, out, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? DA_OK
             : DA_ERR_LAUNCH;
}

}  // extern "C"
