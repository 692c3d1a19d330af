// moe_kernels_g6.cu -- the kernels of moe_fused.cuh whose gate/up codes (and, for kernel B
// alone, down codes) are 6-bit, in a translation unit of their own so that the families compile
// in parallel.
#include "moe_fused.cuh"

namespace moe {

MOE_KERNEL_FAMILY(6)

}  // namespace moe
