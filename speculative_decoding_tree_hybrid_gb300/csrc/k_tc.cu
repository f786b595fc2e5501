// tcgen05 tensor-core path (placeholder until the kernel lands).
#include "hta_launch.h"

namespace hta {
int tc_rows_per_group() { return 0; }
int tc_tile() { return 128; }
int tc_max_grid(int, int) { return 0; }
cudaError_t tc_launch(const AttnParams &, int, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace hta
