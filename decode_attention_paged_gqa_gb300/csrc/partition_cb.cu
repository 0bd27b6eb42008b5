// partition_cb.cu -- dispatch of the codebook-value partition kernel (partition_cb.cuh) by
// cache format, and of the partition phase by kernel.
#include "da_internal.cuh"

namespace da {

cudaError_t launch_partition_cb_cb4(const Args& a, cudaStream_t s);
cudaError_t launch_partition_cb_fp8k(const Args& a, cudaStream_t s);
cudaError_t launch_partition_cb_cb3k(const Args& a, cudaStream_t s);

cudaError_t launch_partition_cb(const Args& a, cudaStream_t s) {
  switch (a.fmt) {
    case DA_KV_CB4: return launch_partition_cb_cb4(a, s);
    case DA_KV_FP8K_CB4V: return launch_partition_cb_fp8k(a, s);
    case DA_KV_CB3K_CB4V: return launch_partition_cb_cb3k(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_partition(const Args& a, cudaStream_t s) {
  return a.fmt == DA_KV_BF16 || a.fmt == DA_KV_FP8_E4M3 ? launch_partition_tc(a, s) : launch_partition_cb(a, s);
}

}  // namespace da
