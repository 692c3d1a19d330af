// moe_kernels_g4.cu -- the kernels of moe_fused.cuh whose gate/up codes (and, for kernel B
// alone, down codes) are 4-bit, in a translation unit of their own so that the families compile
// in parallel.
#include "moe_fused.cuh"

namespace moe {

MOE_KERNEL_FAMILY(4)

}  // namespace moe
