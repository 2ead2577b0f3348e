// tcgen05 / TMA kernels of the chunkwise complex SSD forward (TF32 tensor cores).
#include <cuda_runtime.h>

#include "ssdc_kernels.h"

namespace ssdc {

bool tc_supported(int, int, int) { return false; }
int tc_launch_chunk_state(const Problem&, const Workspace&, cudaStream_t) { return SSDC_ERR_UNSUPPORTED; }
int tc_launch_chunk_scan(const Problem&, const Workspace&, cudaStream_t) { return SSDC_ERR_UNSUPPORTED; }

}  // namespace ssdc
