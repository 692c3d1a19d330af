// moe_mma.cuh -- layout, parameters and launchers of the tensor-core batch variant (moe_mma.cu).
#pragma once

#include "moe_kernels.cuh"

namespace moe {

// ------------------------------------------------------------------ the tile-group copy
// The batch variant reads every projection from a copy made at create time, cut into blocks of
// one expert, one tile of 16 rows and one group of 64 columns, stored [expert][tile][group] (a
// work item's blocks are contiguous).  Inside a block, lane l = 4 g + q of the warp that consumes
// it finds, in "fragment order", the 32 codes it feeds the tensor core: codes 16 q .. 16 q + 15 of
// the group for rows g and g + 8 of the tile, arranged so that one shift and one mask yield the
// two codes of one fragment register (k-step j, register r: row g + 8 (r & 1), columns
// 16 q + 4 j + 2 (r >> 1) and that + 1).  Per projection and lane, 4 * bits bytes:
//   4 bits: one 16-byte word group: word j, nibble r = first code, nibble 4 + r = second code
//   8 bits: two 16-byte word groups: word 2 j + (r >> 1), byte (r & 1) = first, byte 2 + (r & 1)
//           = second
//   6 bits: the low nibbles as at 4 bits, then one 8-byte group of the high 2 bits: word j >> 1,
//           bits 2 p and 16 + 2 p with p = 4 (j & 1) + r
// each word group stored for all 32 lanes before the next ([group][lane][bytes]).
// A gate/up block holds gate codes, up codes, then per g one 16-byte record of fp16 (gate scale,
// gate bias of row g, the same of row g + 8, then up's four); a down block holds the codes, then
// per g one 8-byte record (scale, bias of row g, the same of row g + 8).  Sizes equal the
// canonical bytes of the same rows.
__host__ __device__ inline int mma_lane_bytes(int bits) { return 4 * bits; }
__host__ __device__ inline int mma_gu_block(int bits) { return 256 * bits + 128; }
__host__ __device__ inline int mma_dn_block(int bits) { return 128 * bits + 64; }

struct MmaLayerDev {
  const uint8_t *gu_r, *gu_s;   // [experts][dff / 16][din / 64] gate/up blocks (routed, shared)
  const uint8_t *dn_r, *dn_s;   // [experts][din / 16][dff / 64] down blocks
};

constexpr int kMmaMaxChunks = 8;   // work units split a row tile's groups in at most this many
constexpr int kMmaRouteInts = 2 + 3 * kMaxPairs;

// One layer, m tokens: the prep kernel (route, shared scalars, x's group sums and fp16 parts),
// gate/up, the activation pass (chunk sums, SwiGLU, coefficient, fp16 parts), down, tail.
struct MmaParams {
  LayerShape s;
  LayerPtrs w;              // canonical weights: only gate_vec is read
  MmaLayerDev t;            // the tile-group copy
  int bits_r, bits_s;       // gate/up code widths (routed, shared)
  int bits_dr, bits_ds;     // down code widths
  int m;                    // tokens, m * top_k <= kMaxPairs, m <= kMaxGroupTokens
  const uint16_t *x;        // bf16 [m][din]
  const int32_t *ids;       // [m][top_k]
  const float *scores;      // [m][top_k]
  const void *resid;        // [m][din] bf16 or fp32
  void *out;                // [m][din] fp32 or bf16
  int resid_f32, out_f32;
  int act_stride;           // top_k * dff + n_shared * dff_shared
  // workspace
  int32_t *route;           // [kMmaRouteInts]: U, uniq[U], offs[U + 1], pairs[offs[U]]
  int32_t *nc;              // [2] chunk counts the gate/up and down kernels chose
  float *sscal;             // [m] shared scalars
  float *xsum;              // [m][din / 64] group sums of x
  float *xinv;              // [m][din / 64] 2^-k of x's fp16 parts
  __half *x16;              // [m][din / 64][4][32] x scaled by 2^k: per q 16 high parts, 16 rests
  float2 *gu_part;          // [kMmaMaxChunks][m][act_stride] (gate, up) sums of each chunk
  __half *a16;              // [m][act_stride / 64][4][32] activation, like x16
  float *ainv, *asum;       // [m][act_stride / 64]
  float *y_part;            // [kMmaMaxChunks][m][top_k + n_shared][din]
  const float *zero;        // 256 zero bytes (the operand of an absent column)
  int32_t *err;
  int32_t *ids_used;        // [m][top_k] or null
};

// Enqueues the five kernels of one layer.
cudaError_t launch_mma_layer(const MmaParams &p, cudaStream_t stream);
// Writes the tile-group blocks of `experts` experts: gate/up (rows x din, both projections) or
// down (rows = din, cols = dff).
cudaError_t launch_repack_mma_gu(const uint8_t *g_codes, const __half *g_scales,
                                 const __half *g_biases, const uint8_t *u_codes,
                                 const __half *u_scales, const __half *u_biases, int experts,
                                 int rows, int din, int bits, uint8_t *out, cudaStream_t stream);
cudaError_t launch_repack_mma_down(const uint8_t *codes, const __half *scales,
                                   const __half *biases, int experts, int din, int dff, int bits,
                                   uint8_t *out, cudaStream_t stream);

}  // namespace moe
