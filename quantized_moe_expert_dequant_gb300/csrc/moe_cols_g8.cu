// moe_cols_g8.cu -- the column-split kernels with 8-bit gate/up codes (moe_cols.cuh).
#include "moe_cols.cuh"

namespace moe {
MOE_COLS_FAMILY(8)
}  // namespace moe
