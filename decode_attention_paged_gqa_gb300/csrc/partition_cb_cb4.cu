// partition_cb_cb4.cu -- the codebook-value partition kernel (partition_cb.cuh) for
// 4-bit keys and values (DA_KV_CB4), in a translation unit of its own so the kernel variants compile in parallel.
#include "partition_cb.cuh"

namespace da {

cudaError_t launch_partition_cb_cb4(const Args& a, cudaStream_t s) { return launch_d<kSideCB4>(a, s); }

}  // namespace da
