// partition_cb_fp8k.cu -- the codebook-value partition kernel (partition_cb.cuh) for
// FP8 keys and 4-bit values (DA_KV_FP8K_CB4V), in a translation unit of its own so the kernel variants compile in parallel.
#include "partition_cb.cuh"

namespace da {

cudaError_t launch_partition_cb_fp8k(const Args& a, cudaStream_t s) { return launch_d<kSideFP8>(a, s); }

}  // namespace da
