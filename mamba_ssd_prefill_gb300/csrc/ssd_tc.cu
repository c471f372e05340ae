// tcgen05 / TMA tensor-core kernel of the fused SSD prefill forward (bf16/fp16 I/O).
#include "ssd_common.cuh"
#include "ssd_internal.h"

namespace ssd {

bool tc_supports(int64_t, int64_t, int64_t, int) { return false; }
size_t tc_ring_bytes(int64_t, int64_t, int64_t, int) { return 0; }
uint32_t tc_total_units(int64_t, int64_t, int64_t, int64_t, int) { return 0; }
int tc_heads_per_unit(int64_t, int64_t, int64_t, int64_t, int) { return 1; }
cudaError_t launch_tc(Params, int, int, int, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ssd
