// moe_grouped_g6.cu -- the fused grouped kernels of moe_fused.cuh whose gate/up codes are
// 6-bit, in a translation unit of their own so that the families compile in parallel.
#include "moe_fused.cuh"

namespace moe {

MOE_GROUPED_FAMILY(6)

}  // namespace moe
