// moe_kernels.cuh -- parameters, stage plans and launchers of the decode MoE kernels.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

struct ProjDev {
  const uint8_t *codes;   // [experts][rows][cols*bits/8], 16-byte aligned
  const __half *scales;   // [experts][rows][cols/64], 16-byte aligned
  const __half *biases;   // [experts][rows][cols/64], 16-byte aligned
};

struct LayerShape {
  int din, dff, top_k, n_experts, n_shared, dff_shared;
};

struct LayerPtrs {
  ProjDev gate, up, down, sh_gate, sh_up, sh_down;
  const uint16_t *gate_vec;  // bf16 [din] or nullptr (shared scalar 1)
};

constexpr int kMaxTopK = 64;
constexpr int kMaxPairs = 256;          // grouped tokens: m * top_k at most
constexpr int kMaxGroupTokens = 64;     // grouped tokens: m at most
constexpr int kMaxGroupExperts = 1024;  // grouped tokens: n_experts at most (one bitmap word a lane)
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarps = 1;           // issues the weight stream (bulk copies)
constexpr int kProducers = kProducerWarps * 32;
constexpr int kThreads = kConsumers + kProducers;
constexpr int kRingBytes = 208 * 1024;      // shared-memory ring of one CTA
constexpr int kMaxStages = 8;
constexpr int kMaxRowsB = 128;              // phase B: output rows one CTA owns, at most
constexpr int kMaxActRegs = 32;             // phase B: a thread owns at most this many codes' worth
                                            // of steps (one step at 4 and 6 bits, two at 8 bits)

// Phase A geometry of one class (routed or shared) of gate/up rows.
struct GateUpGeom {
  int bits;     // code width
  int rb;       // bytes per row
  int T;        // 16-B (6-bit: 48-B) steps per row
  int tpr;      // consumer threads per row group: T rounded up to 32, at most kConsumers
  int groups;   // row groups = kConsumers / tpr
  int R;        // rows per chunk = rows per thread * groups
  int sw;       // bytes reserved per scale/bias window in a stage
};

// Phase B geometry.
struct DownGeom {
  int bits_r, bits_s;  // code widths of routed / shared down rows
  int rb_r, rb_s;      // row bytes
  int G_r, G_s;        // groups per row
  int spr_r, spr_s;    // steps per row
  int T_r, T_s;        // steps over the concatenated contraction
  int tpr, groups;     // consumer threads per row group, row groups
  int spt;             // steps per consumer thread
  int R;               // rows per chunk (rows per thread * groups)
  int sw_r, sw_s;      // bytes reserved per scale/bias window
  int codes_bytes;     // code bytes of one stage
};

struct Plan {
  GateUpGeom geo_r, geo_s;
  DownGeom geo_b;
  int nst, stage_bytes;
  size_t smem;
};

// Stage plan of the grouped kernels (m > 1 tokens, each selected expert streamed once).
struct GroupPlan {
  GateUpGeom ga_r, ga_s;   // phase A rows (length din) of routed / shared experts
  GateUpGeom gb_r, gb_s;   // phase B rows (length dff / dff_shared) of routed / shared experts
  int t_sub;               // (token, slot) pairs whose operand rows one stage carries
  int op_off[4];           // operand rows' offset in a stage: A routed, A shared, B routed, B shared
  int nst, stage_bytes;
  size_t smem;
};

// Kernel A alone.
struct GateUpParams {
  LayerShape s;
  LayerPtrs w;
  Plan plan;
  const uint16_t *x;        // bf16 [din], read when v is null
  const float *v;           // fp32 [din] or null: x = RMSNorm(v) with weight gamma (bf16 [din])
  const uint16_t *gamma;
  float eps;
  const int32_t *ids;       // [top_k]
  const float *scores;      // [top_k]
  float *act;               // [top_k*dff + n_shared*dff_shared]
  int32_t *err;             // sticky error word
};

// Kernel B alone.
struct DownParams {
  LayerShape s;
  LayerPtrs w;
  Plan plan;
  const int32_t *ids;       // [top_k]
  const float *act;         // from kernel A
  const void *resid;        // [din] bf16 or fp32
  void *out;                // [din] fp32 or bf16
  int resid_f32, out_f32;
  int32_t *err;
};

// The fused persistent kernel over layers [0, L) and tokens [0, m): phase A, grid barrier,
// phase B, grid barrier, for each (layer, token).
struct StackParams {
  LayerShape s;
  Plan plan;
  const LayerPtrs *layers;  // device array [L]
  int L, m;
  const uint16_t *x;        // bf16 [L][m][din]; [m][din] (layer 0 only) when norm_w is set
  const uint16_t *norm_w;   // bf16 [L - 1][din] or null: layer l >= 1 reads x = RMSNorm(out of
  float norm_eps;           // layer l - 1) with weight row l - 1
  const int32_t *ids;       // [L][m][top_k]
  const float *scores;      // [L][m][top_k]
  const void *resid0;       // [m][din], bf16 or fp32: residual of layer 0
  int resid0_f32;
  float *ping0, *ping1;     // fp32 [m][din] outputs of the layers before the last
  void *out;                // [m][din] output of the last layer
  int out_f32;
  float *act;
  int32_t *err;
  uint32_t *bar;            // grid-barrier counter, zero at launch
  // grouped mode (m > 1): each selected expert streamed once per layer for all m tokens
  int grouped;
  GroupPlan gp;
  float *y;                 // [m][top_k + n_shared][din] partial outputs
  int act_stride;           // floats per token in act: top_k * dff + n_shared * dff_shared
};

// Host-side plan; false when the shape is outside what the kernels support.
bool make_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, Plan *plan);
// Grouped plan for up to m tokens; false when the shape or m is outside the grouped kernels.
bool make_group_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, int m,
                     GroupPlan *gp);

cudaError_t launch_gate_up(const GateUpParams &p, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_down(const DownParams &p, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_fused(const StackParams &p, int grid, cudaStream_t stream);
// Sets the kernels' dynamic shared-memory limits; *dyn_limit = the dynamic bytes all three allow.
cudaError_t prepare_kernels(int smem_optin, int bits_gu, int bits_d, int bits_sh, int *dyn_limit);
int fused_grid_limit(const Plan &plan, int bits_gu, int bits_d, int bits_sh);
cudaError_t launch_unpack(const uint8_t *packed, int64_t rows, int64_t cols, int bits,
                          uint8_t *codes, cudaStream_t stream);
// Router: per token the top_k of n_experts fp32 logits (ties to the lower id) and their softmax
// weights; n_experts <= 1024, top_k <= kMaxTopK.
cudaError_t launch_router(const float *logits, int m, int n_experts, int k, int32_t *ids,
                          float *scores, cudaStream_t stream);
// The kernels' bounded wait on a condition nothing satisfies (kind 0: grid-barrier count at cnt,
// which must be zero; kind 1: an mbarrier stage), giving up after `limit` cycles.
cudaError_t launch_wait_timeout(int kind, uint32_t *cnt, int32_t *err, long long limit,
                                cudaStream_t stream);
// Route inversion of ids [m][k] by the device code the grouped kernels use; writes
// out[0] = U, then uniq[U], offs[U + 1], pairs[offs[U]].
cudaError_t launch_route_invert(const int32_t *ids, int m, int k, int n_experts, int32_t *out,
                                cudaStream_t stream);

}  // namespace moe
