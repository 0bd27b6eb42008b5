// partition_cb_cb3k.cu -- the codebook-value partition kernel (partition_cb.cuh) for
// 3-bit keys and 4-bit values (DA_KV_CB3K_CB4V), in a translation unit of its own so the kernel variants compile in parallel.
#include "partition_cb.cuh"

namespace da {

cudaError_t launch_partition_cb_cb3k(const Args& a, cudaStream_t s) { return launch_d<kSideCB3>(a, s); }

}  // namespace da
