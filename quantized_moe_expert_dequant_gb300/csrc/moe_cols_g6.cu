// moe_cols_g6.cu -- the column split takes 4- and 8-bit gate/up codes only (its lanes hold 32
// columns of a row as whole bytes); 6-bit gate/up rows run on the row split, so these entry
// points refuse.
#include "moe_kernels.cuh"

namespace moe {
cudaError_t launch_cols_g6(const StackParams &, int, cudaStream_t) {
  return cudaErrorInvalidValue;
}
cudaError_t prepare_cols_g6(int, int, int, int *) { return cudaErrorInvalidValue; }
cudaError_t cols_occupancy_g6(int, int, size_t, int *per_sm) {
  *per_sm = 0;
  return cudaErrorInvalidValue;
}
}  // namespace moe
