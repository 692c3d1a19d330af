// moe_cols_g6.cu -- the column-split kernels with 6-bit gate/up codes (moe_cols.cuh).
#include "moe_cols.cuh"

namespace moe {
MOE_COLS_FAMILY(6)
}  // namespace moe
