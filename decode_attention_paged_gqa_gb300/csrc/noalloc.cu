// noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// decode_attn_paged needs a caller-provided workspace (the split-K partials, the rotated
// queries and the error word). Some callers have no way to provide one: code that runs where
// device allocation is forbidden or unavailable -- a plugin inside a host framework that owns
// every allocation and exposes none to its extensions, a real-time loop that must not call
// the allocator (cudaMalloc can synchronise the device and take unbounded time), or a caller
// with no CUDA allocator of its own at all. This entry point takes the workspace from a
// fixed-size array in device global memory that the library itself defines; it allocates
// nothing and calls no allocating routine.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "da_internal.cuh"

namespace {

// Largest workspace this entry point can serve: 64 MiB (the 32-sequence, 32-head,
// 32768-token codebook batch needs about 35 MB). Every GPU that loads the library holds
// this array until the process exits.
constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;

__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Device address of g_static_workspace, looked up once per device and context. In host code
// the array's name is only a host-side stand-in, never a device address. The address belongs
// to the context it was looked up in: when the device's current context changes (the primary
// context destroyed by cudaDeviceReset and created anew, or another context made current
// through the driver API), it is looked up again.
std::mutex g_mu;
void* g_addr[64] = {};
CUcontext g_ctx[64] = {};

PFN_cuCtxGetCurrent_v4000 ctx_get_current_fn() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

int static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DA_ERR_CUDA;
  auto get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;  // stays null while the runtime has made no context current yet
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!ctx || !g_addr[dev] || g_ctx[dev] != ctx) {
    // the lookup also makes the device's primary context current when none is
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return DA_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return DA_ERR_CUDA;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_paged_static_workspace(const void* q, const void* k_cache, const void* v_cache,
                                                  const float* k_scales, const float* v_scales,
                                                  const float* codebook, const float* sign_pattern,
                                                  const int32_t* block_tables, const int32_t* context_lens,
                                                  float* out, const da_params* p, void* stream) {
  // the checks of decode_attn_paged, with its status codes, before anything is enqueued
  int rc = da::check_call(q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                          context_lens, out, p);
  if (rc) return rc;
  if (p->batch == 0) return DA_OK;
  if (da::workspace_layout(*p).total > kStaticWorkspaceBytes) return DA_ERR_STATIC_WORKSPACE;
  void* ws = nullptr;
  if ((rc = static_workspace_address(&ws))) return rc;
  da_params local = *p;
  local.workspace = ws;
  local.workspace_bytes = kStaticWorkspaceBytes;
  // the array keeps the previous call's contents: the error word must start at zero
  // (the partials are always written before they are read)
  if (cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DA_ERR_CUDA;
  return da::run_phases(da::kAll, q, k_cache, v_cache, k_scales, v_scales, codebook, sign_pattern, block_tables,
                        context_lens, out, &local, stream);
}
