// moe_mma.cuh -- parameters and launcher of the tensor-core batch variant (moe_mma.cu).
#pragma once

#include "moe_kernels.cuh"

namespace moe {

// The tensor-core batch variant (moe_mma.cu): m tokens of one layer, slots grouped by expert,
// gate/up and down on mma.sync bf16 tiles of 16 weight rows x 8 (token, slot) pairs.
struct MmaParams {
  LayerShape s;
  LayerPtrs w;
  int m;                    // tokens, m * top_k <= kMaxPairs, m <= kMaxGroupTokens
  const uint16_t *x;        // bf16 [m][din]
  const int32_t *ids;       // [m][top_k]
  const float *scores;      // [m][top_k]
  const void *resid;        // [m][din] bf16 or fp32
  void *out;                // [m][din] fp32 or bf16
  int resid_f32, out_f32;
  int32_t *route;           // [kMmaRouteInts]: U, uniq[U], offs[U + 1], pairs[offs[U]]
  float *sscal;             // [m] shared scalars
  float *act;               // [m][act_stride]
  int act_stride;           // top_k * dff + n_shared * dff_shared
  float *y;                 // [m][top_k + n_shared][din] per-slot down outputs
  int32_t *err;
  int32_t *ids_used;        // [m][top_k] or null
};
constexpr int kMmaRouteInts = 2 + 3 * kMaxPairs;
// Enqueues the route inversion, the gate/up and down tensor-core kernels and the tail.
cudaError_t launch_mma_layer(const MmaParams &p, int bits_gu, int bits_d, int bits_sh,
                             cudaStream_t stream);

}  // namespace moe
