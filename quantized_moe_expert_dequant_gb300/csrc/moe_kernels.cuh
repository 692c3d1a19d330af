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
constexpr int kMaxStages = 12;             // ring slots a kernel's shared state holds
constexpr int kMaxRowStages = 8;           // ring slots the row-split plans use, at most
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

// ------------------------------------------------------------------ column-split mode
// The column-split kernel (moe_cols.cuh) gives each CTA a contiguous range of activation columns
// (the flattened routed-then-shared row space of the gate/up projections); it computes those
// activations locally and multiplies them into the matching columns of the down projections, so
// the down weights are read in a column-block-major copy made at create time:
//   codes  [experts][dff / cb][din] 32-bit words; word (jb, i) holds the cb = 32 / bits codes of
//          row i, columns jb * cb .. jb * cb + cb - 1, exactly as in the canonical row (LSB first);
//          6-bit codes are widened to one byte each (cb = 4, the 8-bit layout: exact, codes < 64)
//   sb     [experts][dff / 64][din] (scale, bias) pairs of row i, group g

// Code width of a projection as the column split stores and reads it: 6-bit codes are widened to
// one byte each (exact: codes < 64), so its kernels take 4- and 8-bit codes only.
__host__ __device__ inline int col_down_bits(int bits) { return bits == 6 ? 8 : bits; }
__host__ __device__ inline int col_gu_bits(int bits) { return bits == 6 ? 8 : bits; }
constexpr int kMaxColsCta = 256;     // activation columns one CTA owns, at most
constexpr int kMaxColPieces = 16;    // (segment, group) pieces of one CTA's columns, at most
constexpr int kMaxColBlocks = 64;    // down column blocks one CTA reads, at most
constexpr int kMaxOwnRows = 32;      // output rows one CTA sums from the partials, at most
constexpr int kColMaxGrid = 160;     // CTAs of a column-split launch, at most (the owner's sums
                                     // read five partial vectors per lane)

struct ColDownDev {
  const uint32_t *codes;   // [experts][dff / cb][din]
  const __half2 *sb;       // [experts][dff / 64][din]
};

// Gate/up rows of the column split as records, one per row pair j of each expert:
//   [gate codes: rb][up codes: rb][gate scales: G][gate biases: G][up scales: G][up biases: G],
// (6-bit codes stored as bytes, col_gu_bits)
// the four fp16 runs padded together to a multiple of 16 bytes (rec bytes per record), so that
// the R row pairs of a stage are one contiguous bulk copy.
struct ColPtrs {
  ColDownDev r, s;         // routed experts, shared experts
  const uint8_t *gu_r;     // [experts][dff][rec_r] gate/up records of the routed experts
  const uint8_t *gu_s;     // [n_shared][dff_shared][rec_s] those of the shared experts
};

struct ColPlan {
  int cb_r, cb_s;          // codes per 32-bit word of the routed / shared down projection
  int nbs;                 // column blocks per down stage, at most
  int ro;                  // output rows one CTA owns, at most (4 * its row quads)
  int rec_r, rec_s;        // bytes of one gate/up record, routed / shared
  int pack;                // down stages filled across pieces (stages of at most 2 blocks, no
                           // prefetch)
  int prefetch;            // ask L2 for the stages beyond the first ring-full (when they are at
                           // most one more ring-full)
  int32_t bounds[kColMaxGrid + 1];  // CTA c owns the activation columns [bounds[c], bounds[c+1])
};

// Bytes of one gate/up record of a row of `din` codes at `bits`.
__host__ __device__ inline int col_record_bytes(int din, int bits) {
  return 2 * (din * bits / 8) + ((8 * (din / 64) + 15) / 16) * 16;
}

// One piece of a CTA's columns: the columns [j0, j1) of one segment (routed slot or shared expert)
// that lie in one group of 64.
struct ColPiece {
  int seg;      // routed slot k (< top_k) or top_k + shared expert index
  int j0, j1;   // columns, expert coordinates
  int a0;       // index of column j0 in the CTA's activation range
  int blk0;     // first column block: j0 / cb
  int nb;       // column blocks
  int pb;       // index of the piece's first block in the CTA's block list
  int grp;      // group: j0 / 64
};

// The even split of U activation columns over n CTAs: CTA c's columns [u0, u1).  The plan starts
// from it and moves each boundary a few columns (ColPlan::bounds).
__host__ __device__ inline void col_range(int64_t U, int c, int n, int64_t *u0, int64_t *u1) {
  *u0 = U * c / n;
  *u1 = U * (c + 1) / n;
}

// Cuts the activation columns [u0, u1) into pieces; returns the piece count (-1 when more than
// kMaxColPieces or the blocks exceed kMaxColBlocks) and the block count in *nblocks.
__host__ __device__ inline int col_pieces(int top_k, int dff, int n_shared, int dff_shared,
                                          int cb_r, int cb_s, int64_t u0, int64_t u1,
                                          ColPiece *pc, int *nblocks) {
  const int64_t Ur = static_cast<int64_t>(top_k) * dff;
  int np = 0, nbk = 0;
  for (int64_t u = u0; u < u1;) {
    int seg, j, width, cb;
    if (u < Ur) {
      seg = static_cast<int>(u / dff);
      j = static_cast<int>(u - static_cast<int64_t>(seg) * dff);
      width = dff;
      cb = cb_r;
    } else {
      const int t = static_cast<int>((u - Ur) / dff_shared);
      seg = top_k + t;
      j = static_cast<int>(u - Ur - static_cast<int64_t>(t) * dff_shared);
      width = dff_shared;
      cb = cb_s;
    }
    int jend = (j / 64 + 1) * 64;
    if (jend > width) jend = width;
    if (static_cast<int64_t>(jend - j) > u1 - u) jend = j + static_cast<int>(u1 - u);
    if (np == kMaxColPieces) return -1;
    ColPiece &q = pc[np++];
    q.seg = seg;
    q.j0 = j;
    q.j1 = jend;
    q.a0 = static_cast<int>(u - u0);
    q.blk0 = j / cb;
    q.nb = (jend - 1) / cb - j / cb + 1;
    q.pb = nbk;
    q.grp = j / 64;
    nbk += q.nb;
    if (nbk > kMaxColBlocks) return -1;
    u += jend - j;
  }
  *nblocks = nbk;
  return np;
}

// The gate/up stages of a CTA of the column split: its activation columns [u0, u1) cut into
// chunks of at most R row pairs (R_s for the shared experts; kColFirstRows for the first) that
// never cross an expert, in column order.  Chunk i: segment seg[i] (routed slot, or top_k +
// shared expert), first row j[i] inside the expert, rows cnt[i], first column u[i] relative to
// u0.  Returns the chunk count and the routed chunks in *n_routed, or -1 beyond kMaxColChunks.
constexpr int kMaxColChunks = 96;
constexpr int kColFirstRows = 4;  // row pairs of a CTA's first gate/up stage of a layer
__host__ __device__ inline int col_chunks(int top_k, int dff, int n_shared, int dff_shared, int R,
                                          int R_s, int64_t u0, int64_t u1, short *seg, short *j,
                                          short *cnt, short *u, int *n_routed) {
  const int64_t Ur = static_cast<int64_t>(top_k) * dff;
  int nc = 0, nr = 0;
  for (int64_t x = u0; x < u1;) {
    const bool routed = x < Ur;
    const int width = routed ? dff : dff_shared;
    const int64_t rel = routed ? x : x - Ur;
    const int sg = static_cast<int>(rel / width);
    const int jj = static_cast<int>(rel - static_cast<int64_t>(sg) * width);
    int take = width - jj;
    // the CTA's first chunk is short, so that the first copy of a layer lands early
    const int lim = nc == 0 ? min(routed ? R : R_s, kColFirstRows) : (routed ? R : R_s);
    if (take > lim) take = lim;
    if (take > u1 - x) take = static_cast<int>(u1 - x);
    if (nc == kMaxColChunks) return -1;
    seg[nc] = static_cast<short>(routed ? sg : top_k + sg);
    j[nc] = static_cast<short>(jj);
    cnt[nc] = static_cast<short>(take);
    u[nc] = static_cast<short>(x - u0);
    nr += routed;
    ++nc;
    x += take;
  }
  *n_routed = nr;
  return nc;
}

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
  int32_t *ids_used;        // [top_k] or null: CTA 0 writes the ids it read
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
  // column-split mode (m = 1): repacked down projections per layer, plan, partial-sum slab
  const ColPtrs *cols;      // device array [L]
  ColPlan cp;
  float *slab;              // [2][grid][din]: each CTA's partial output vector, two passes
  int ahead;                // 1: every layer's ids are inputs known before the step: the weight
                            // stream runs on into the next layer (not the decode dependency)
  unsigned long long *tl;   // timeline builds: [grid][L][kTlPoints] time stamps; else null
  int32_t *ids_used;        // [L][m][top_k] or null: CTA 0 writes the ids its producer read
  int pool;                 // grouped path: gate/up without the score (or shared scalar); the
                            // tail forms resid + (sum_k score_k y_k + scalar * sum y_shared) from
                            // the per-slot outputs y, which it keeps
};

// Host-side plan; false when the shape is outside what the kernels support.
bool make_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, Plan *plan);
// Grouped plan for up to m tokens; false when the shape or m is outside the grouped kernels.
bool make_group_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, int m,
                     GroupPlan *gp);

// Column-split plan for a grid of `grid` CTAs (phase-A geometry and ring in *plan); false when
// the shape is outside the column-split kernels (down codes of 4 or 8 bits, din <= 4096, at most
// kColMaxGrid CTAs, and the per-CTA limits above).  A phase-A stage holds R (gate row, up row)
// pairs, R a power of two with R * ceil(din / 2048) <= 16 (one warp per 2048 columns of a pair).
bool make_col_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, int grid,
                   int ring_bytes, ColPlan *cp, Plan *plan);
cudaError_t launch_cols(const StackParams &p, int grid, cudaStream_t stream);
cudaError_t prepare_cols(int smem_optin, int bits_gu, int bits_d, int bits_sh, int *dyn_limit);
int cols_grid_limit(size_t smem, int bits_gu, int bits_d, int bits_sh);
// Writes the gate/up records (see ColPtrs) of `experts` experts of `rows` row pairs.
cudaError_t launch_repack_gate_up(const uint8_t *g_codes, const __half *g_scales,
                                  const __half *g_biases, const uint8_t *u_codes,
                                  const __half *u_scales, const __half *u_biases, int experts,
                                  int rows, int din, int bits, uint8_t *out, cudaStream_t stream);
// Writes the column-block-major copy of `experts` down projections (rows din, cols dff, bits).
cudaError_t launch_repack_down(const uint8_t *codes, const __half *scales, const __half *biases,
                               int experts, int din, int dff, int bits, uint32_t *out_codes,
                               __half2 *out_sb, cudaStream_t stream);

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
