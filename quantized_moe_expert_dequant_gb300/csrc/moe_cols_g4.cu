// moe_cols_g4.cu -- the column-split kernels with 4-bit gate/up codes (moe_cols.cuh).
#include "moe_cols.cuh"

namespace moe {
MOE_COLS_FAMILY(4)
}  // namespace moe
