// moe_cols.cuh -- the column-split decode kernel: one grid barrier per layer.
//
// The block computes, per token (the pages' two phases, "two-kernel decode-MoE that beats
// gather_qmm", What changed, step 2, and the tail of "Red Lite dev39 -- fused expert tail"):
//   act[u] = coef_u * silu(gate_u . x) * (up_u . x)          u over routed slots' and shared rows
//   out    = resid + sum_u W_down[:, u] * act[u]
// Kernel A and kernel B split that work by ROWS of each projection, so every CTA of kernel B needs
// every activation and the two phases meet at a device-wide exchange.  Here every CTA owns a
// contiguous, balanced range of the activation index u instead and carries its columns through
// both projections:
//   1. gate/up: the CTA's rows u, one warp per (gate row, up row) pair of a stage, each lane owning
//      one group of 64 codes of the row (so its integer sums run over a whole group and one scale
//      and bias apply to them); the activations stay in shared memory;
//   2. the matching COLUMNS u of the down projections, read from a column-block-major copy
//      (moe_kernels.cuh), multiplied by the local activations into a partial output for all din
//      rows, written to this CTA's vector of a slab in global memory;
//   3. an arrival on a device-wide counter (the consumers do not wait for it: they go on to the
//      next layer's x);
//   4. a helper warp waits for the counter, sums in a fixed order the grid's partials of the rows
//      this CTA owns and adds them to the running output it keeps in shared memory (and, after the
//      last layer, writes the output).
// The next layer's expert ids are read (by the producer warp) only after the counter shows that
// every CTA has finished the layer (its output exists as the partials), so no weight of a layer is
// requested before the previous layer is done.  With p.ahead (every layer's ids are inputs known
// before the step) the producer instead starts layer l + 1 as soon as its own CTA's consumers have
// finished layer l's gate/up phase (a CTA-local mbarrier); the arithmetic and its order are the
// same.
//
// Warps: 16 consumer warps, one producer warp (the bulk-copy stream of moe_phases.cuh), one helper
// warp (the owner's sums, the shared-expert scalar, the output).
//
// The down contraction over a CTA's columns uses integer dot products like the row kernels
// (moe_common.cuh): within one (segment, group of 64) piece the activations become 23-bit fixed
// point with one exponent, split into byte planes, and dp4a multiplies a 32-bit code word (4 codes
// at 8 bits, 8 at 4 bits, of ONE output row) by the plane word of the same columns.  The integer
// sums are exact over a whole piece; at the piece's end the group's scale and bias apply:
//   sum_j (s q_j + b) a_j = s * sum_j q_j a_j + b * sum_j a_j.
// Columns of a block outside the CTA's range get zero activations (a neighbour owns them).
#pragma once

#include "moe_fused.cuh"
#include "moe_timeline.cuh"

namespace moe {

constexpr int kColHelperWarp = kConsumerWarps + kProducerWarps;
constexpr int kColThreads = kThreads + 32;    // consumers, producer, helper
constexpr int kColMaxWpr = 4;                 // warps per gate/up row pair (32 columns a lane)
// Consumers test a stage's barrier from every lane (no broadcast from lane 0).
constexpr bool kColLaneWait = true;

// Consumer side: every lane tests the stage's full barrier until it completes (bounded; on the
// rare long wait the common path below takes over).
__device__ __forceinline__ bool cols_wait_full(Ring &r, int lane) {
  if (kColLaneWait) {
    for (int it = 0; it < 64; ++it) {
      if (mbar_test_wait(&r.full[r.st], r.ph)) return true;
      __nanosleep(32);
    }
  }
  return warp_wait_full(r, lane);
}

// ------------------------------------------------------------------ one lane's operand
// The lane's 32 values of x (half a group of 64 of a gate/up row) with ONE exponent, in the form
// its code width's dot product wants: dot() returns sum_c q_c * v_c / unit, the exact integer sum
// rounded once.  The two 16-byte chunks of an 8-bit lane are read in a rotated order (rot) so that
// the 8 lanes of a shared-memory wavefront hit distinct banks; the operand holds its chunks in the
// same order.
template <int BITS>
struct LaneOp;

template <>
struct LaneOp<8> {
  static constexpr int VEC = 2;  // uint4 chunks per lane and row
  uint32_t pl[8], pm[8], ph[8];
  float unit, sum;
  __device__ __forceinline__ static int rot(int lane) { return (lane >> 2) & 1; }
  __device__ __forceinline__ void set(const float (&v)[32]) {
    float mx = 0.f, sm = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      mx = fmaxf(mx, fabsf(v[c]));
      sm += v[c];
    }
    const int E = fixed_exponent(mx);
    const float sc = pow2f(22 - E);
    unit = pow2f(E - 22);
    sum = sm;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      byte_planes(__float2int_rn(v[4 * j] * sc), __float2int_rn(v[4 * j + 1] * sc),
                  __float2int_rn(v[4 * j + 2] * sc), __float2int_rn(v[4 * j + 3] * sc), pl[j],
                  pm[j], ph[j]);
  }
  __device__ __forceinline__ float dot(const uint4 (&c)[VEC]) const {
    uint32_t l = 0, m = 0;
    int h = 0;
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      const uint32_t w[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        l = dp4a_uu(w[i], pl[4 * k + i], l);
        m = dp4a_uu(w[i], pm[4 * k + i], m);
        h = dp4a_us(w[i], ph[4 * k + i], h);
      }
    }
    // l, m <= 32 * 255 * 255 < 2^21, so m * 256 + l < 2^30; |h| <= 32 * 255 * 64
    return fmaf(static_cast<float>(h), 65536.f, static_cast<float>(m * 256u + l));
  }
};

template <>
struct LaneOp<4> {
  static constexpr int VEC = 1;
  uint32_t el[4], em[4], eh[4];  // even columns of word j (low nibbles)
  uint32_t ol[4], om[4], oh[4];  // odd columns of word j (high nibbles, read as 16 q)
  float unit, sum;
  __device__ __forceinline__ static int rot(int) { return 0; }  // 16-B lanes: no conflict
  __device__ __forceinline__ void set(const float (&v)[32]) {
    float mx = 0.f, sm = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      mx = fmaxf(mx, fabsf(v[c]));
      sm += v[c];
    }
    const int E = fixed_exponent(mx);
    const float sc = pow2f(22 - E);
    unit = pow2f(E - 26);  // the dot below is 16 * sum q f
    sum = sm;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      byte_planes(__float2int_rn(v[8 * j] * sc), __float2int_rn(v[8 * j + 2] * sc),
                  __float2int_rn(v[8 * j + 4] * sc), __float2int_rn(v[8 * j + 6] * sc), el[j],
                  em[j], eh[j]);
      byte_planes(__float2int_rn(v[8 * j + 1] * sc), __float2int_rn(v[8 * j + 3] * sc),
                  __float2int_rn(v[8 * j + 5] * sc), __float2int_rn(v[8 * j + 7] * sc), ol[j],
                  om[j], oh[j]);
    }
  }
  __device__ __forceinline__ float dot(const uint4 (&c)[VEC]) const {
    const uint32_t w[4] = {c[0].x, c[0].y, c[0].z, c[0].w};
    uint32_t l0 = 0, m0 = 0, l1 = 0, m1 = 0;
    int h0 = 0, h1 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = w[j] & 0x0f0f0f0fu, hi = w[j] & 0xf0f0f0f0u;
      l0 = dp4a_uu(lo, el[j], l0);
      m0 = dp4a_uu(lo, em[j], m0);
      h0 = dp4a_us(lo, eh[j], h0);
      l1 = dp4a_uu(hi, ol[j], l1);
      m1 = dp4a_uu(hi, om[j], m1);
      h1 = dp4a_us(hi, oh[j], h1);
    }
    // 16 * sum q f: the even sums scaled by 16 join the odd ones (read as 16 q already);
    // l, m <= 16 * 15 * 255 * 16 + 16 * 240 * 255 < 2^21, so m * 256 + l < 2^30
    const uint32_t l = l0 * 16u + l1, m = m0 * 16u + m1;
    const int h = h0 * 16 + h1;
    return fmaf(static_cast<float>(h), 65536.f, static_cast<float>(m * 256u + l));
  }
};

// The lane's x operand: columns [32 k, 32 k + 32) of x (k = the lane's slot of the row), chunks
// in the lane's rotated order; zeros for a lane past the row.
template <int BITS>
__device__ __forceinline__ void load_lane_x(LaneOp<BITS> &op, const uint16_t *x, int k,
                                            bool active, int lane) {
  constexpr int VEC = LaneOp<BITS>::VEC;
  constexpr int CPC = 32 / VEC;  // columns per chunk
  const int rt = LaneOp<BITS>::rot(lane);
  float v[32];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int src = 32 * k + CPC * ((j + rt) % VEC);  // chunk j holds chunk j + rot
#pragma unroll
    for (int q = 0; q < CPC / 8; ++q) {
      const uint4 w = active ? *reinterpret_cast<const uint4 *>(x + src + 8 * q)
                             : make_uint4(0, 0, 0, 0);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v[CPC * j + 8 * q + 2 * h] = __uint_as_float(ww[h] << 16);
        v[CPC * j + 8 * q + 2 * h + 1] = __uint_as_float(ww[h] & 0xffff0000u);
      }
    }
  }
  op.set(v);
}

// ------------------------------------------------------------------ shared state
struct ColSmem {
  float2 red[kMaxColsCta][kColMaxWpr];    // (gate, up) sums of each column from each of the
                                          // warps that share its row pair
  uint32_t planes[kMaxColBlocks * 8];     // per block: byte planes (3 words at 8 bits, 6 at 4)
  float2 us[kMaxColPieces];               // per piece: (unit, sum of its activations)
  ColPiece pc[kMaxColPieces];
  float resid[kMaxOwnRows];               // the owned rows' running output (the next residual)
  float s_gate[2];                        // the shared-expert scalar of layers of each parity
  short ck_seg[kMaxColChunks], ck_j[kMaxColChunks], ck_n[kMaxColChunks], ck_u[kMaxColChunks];
  int nck, nck_r;                         // the CTA's gate/up chunks (col_chunks), routed first
  int np, nbk;
  int u0, ncols;
};

__device__ __forceinline__ bool col_valid(const LayerShape &s, const ColPiece &q, const int *ids,
                                          int *expert) {
  if (q.seg >= s.top_k) {
    *expert = q.seg - s.top_k;
    return true;
  }
  const int e = ids[q.seg];
  *expert = e;
  return e >= 0 && e < s.n_experts;
}

// The down stream of a layer in stages of C = cp.nbs + 1 slots of one column block (din 32-bit
// words): every valid piece's code blocks, then its (scale, bias) record, in piece order.  Packed
// (cp.pack): every slot filled, a piece may continue in the next stage and its record may open the
// next one.  Else a stage holds up to cp.nbs blocks of one piece, and the record rides in the
// piece's last stage.
struct DownWalk {
  int qi;     // the current piece (cs.np: none left)
  int done;   // its code blocks already placed
};

__device__ __forceinline__ int next_valid_piece(const LayerShape &s, const ColSmem &cs,
                                                const int *ids, int from) {
  for (int i = from; i < cs.np; ++i) {
    int e;
    if (col_valid(s, cs.pc[i], ids, &e)) return i;
  }
  return cs.np;
}

// One stage from w: seg(qi, piece, expert, b0, nk, slot) for each run of nk code blocks of a piece
// (b0: the run's first block inside the piece) and seg(qi, piece, expert, -1, 0, slot) for a
// piece's record; w moves past the stage.  The producer and the consumers walk the same stages.
template <class Seg>
__device__ __forceinline__ void col_down_stage(const LayerShape &s, const ColPlan &cp,
                                               const ColSmem &cs, const int *ids, DownWalk &w,
                                               Seg seg) {
  const int C = cp.nbs + 1;
  int k = 0;
  while (k < C && w.qi < cs.np) {
    const ColPiece q = cs.pc[w.qi];
    int e;
    col_valid(s, q, ids, &e);
    const int room = cp.pack ? C - k : cp.nbs;
    const int nk = min(q.nb - w.done, room);
    if (nk > 0) {
      seg(w.qi, q, e, w.done, nk, k);
      k += nk;
      w.done += nk;
    }
    if (w.done < q.nb) {
      if (!cp.pack) break;
      continue;           // packed: the stage is full
    }
    if (k == C) break;    // the record opens the next stage
    seg(w.qi, q, e, -1, 0, k);
    ++k;
    w.qi = next_valid_piece(s, cs, ids, w.qi + 1);
    w.done = 0;
    if (!cp.pack) break;
  }
}

// Named barrier 3: the consumer warps and the helper warp, once per layer (the helper's shared
// scalar is ready and its reads of the older slab pass are done).
__device__ __forceinline__ void consumers_helper_sync() {
  asm volatile("bar.sync 3, %0;" ::"n"(kConsumers + 32) : "memory");
}

// ------------------------------------------------------------------ gate/up
// The stages of one class (routed slots or shared experts) of the CTA's gate/up rows.  A stage
// holds up to R (gate row, up row) records (see ColPtrs); each pair is split among wpr lane sets of
// 32 lanes, each lane owning 32 columns of both rows (columns 32 (32 h + lane) ...), which makes
// T = R * wpr tasks (pair p, part h), task index p * wpr + h.  A warp takes two tasks of a stage,
// t and t + W (W = T / 2 warps per stage, slot t), so W warps work on a stage, by turns: with
// A = 16 / W warp sets, stage i of the phase goes to set i mod A and the sets overlap consecutive
// stages.  Every warp waits for and releases every stage.  The tasks' (gate, up) sums go to
// red[u - u0][h]; the caller forms the activations.
template <int BITS>
__device__ __forceinline__ void cols_a_task(const LaneOp<BITS> &xo, const uint8_t *rec, int koff,
                                            int rbc, int G, int k, bool on, int rt,
                                            float &gv, float &uv) {
  constexpr int VEC = LaneOp<BITS>::VEC;
  gv = uv = 0.f;
  if (!on) return;
  const uint8_t *rg = rec + koff;
  const uint8_t *ws = rec + 2 * rbc + (k >> 1) * 2;
  uint4 cg[VEC], cu[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    cg[j] = lds_u4(rg + 16 * ((j + rt) % VEC));
    cu[j] = lds_u4(rg + rbc + 16 * ((j + rt) % VEC));
  }
  const float sg = lds_half(ws), bg = lds_half(ws + 2 * G);
  const float su = lds_half(ws + 4 * G), bu = lds_half(ws + 6 * G);
  gv = fmaf(sg, xo.dot(cg) * xo.unit, bg * xo.sum);
  uv = fmaf(su, xo.dot(cu) * xo.unit, bu * xo.sum);
}

template <int BITS>
__device__ int cols_a_class(const LayerShape &s, const GateUpGeom &g, int count, int i0,
                            const LaneOp<BITS> &xo, ColSmem &cs, Ring &r, bool &waited,
                            bool &ok, int warp, int lane) {
  const int nk = s.din >> 5;                     // 32-column slots of a row
  const int wpr = (nk + 31) >> 5;
  const int T = g.R * wpr;                       // tasks of a full stage
  const int W = (T + 1) >> 1;                    // warps working on one stage
  const int A = kConsumerWarps / W;
  const int slot = warp % W, turn = warp / W;
  // the warp's two tasks: pair p and lane set h of each (the same h: W is a multiple of wpr)
  const int t1 = slot, t2 = slot + W;
  const int p1 = t1 / wpr, p2 = t2 / wpr, h = t1 - p1 * wpr;
  const int k = 32 * h + lane;                   // the lane's 32-column slot of the row
  const bool lane_on = k < nk;
  const int rt = LaneOp<BITS>::rot(lane);
  const int koff = k * (4 * BITS);               // the lane's bytes inside a row
  const int rbc = s.din * BITS / 8;              // code bytes of a row
  const int G = s.din / kGroup;
  int i = i0;
  for (int c = 0; c < count; ++c, ++i) {
    if (!waited) {
      if (warp == 0 && lane == 0) MOE_TL_STAGE_WAIT(r.used);
      ok = cols_wait_full(r, lane);
    }
    waited = false;
    if (warp == 0 && lane == 0) MOE_TL_STAGE_C(r.used);
    const StageDesc d = r.desc[r.st];
    const bool mine = ok && turn < A && (A == 1 || (i % A) == turn);
    const bool on1 = mine && t1 < T && p1 < d.n, on2 = mine && t2 < T && p2 < d.n;
    if (on1) {  // warp-uniform
      float v[4];
      const uint8_t *sb = r.stage();
      cols_a_task<BITS>(xo, sb + p1 * g.rb, koff, rbc, G, k, lane_on, rt, v[0], v[1]);
      cols_a_task<BITS>(xo, sb + p2 * g.rb, koff, rbc, G, k, lane_on && on2, rt, v[2], v[3]);
      warp_release(r, lane);
      // lanes 0-7 hold the gate sum of task 1, 8-15 its up sum, 16-23 and 24-31 task 2's
      const float val = warp_transpose_reduce<4>(v, lane);
      const int which = lane >> 3;
      if ((lane & 7) == 0 && (which < 2 || on2)) {
        float2 *dst = &cs.red[d.u + (which < 2 ? p1 : p2) - cs.u0][h];
        if (which & 1)
          dst->y = val;
        else
          dst->x = val;
      }
    } else {
      warp_release(r, lane);
    }
  }
  return i;
}

// Gate/up of one layer for the CTA's columns: x operands (built while the first stage is in
// flight), then the stages of both classes.  The first stage publishes the per-class stage
// counts (an empty stage when the CTA has no valid rows).
template <int BR, int BSH>
__device__ void cols_phase_a(const LayerShape &s, const GateUpGeom &gr, const GateUpGeom &gs,
                             const uint16_t *x, const int *cnt, ColSmem &cs, Ring &r, int warp,
                             int lane) {
  const int nk = s.din >> 5, wpr = (nk + 31) >> 5;
  const int kr = 32 * ((warp % ((gr.R * wpr + 1) >> 1)) % wpr) + lane;
  LaneOp<BR> xr;
  load_lane_x<BR>(xr, x, kr, kr < nk, lane);
  if (warp == 0 && lane == 0) {
    MOE_TL_HOOK(7);
    MOE_TL_STAGE_WAIT(r.used);
  }
  bool ok = cols_wait_full(r, lane), waited = true;
  if (warp == 0 && lane == 0) MOE_TL_HOOK(8);
  const int nr = cnt[0], ns = cnt[1];
  if (nr + ns == 0) {  // an empty stage
    warp_release(r, lane);
    return;
  }
  int i = cols_a_class<BR>(s, gr, nr, 0, xr, cs, r, waited, ok, warp, lane);
  if (ns > 0) {
    const int ks = 32 * ((warp % ((gs.R * wpr + 1) >> 1)) % wpr) + lane;
    LaneOp<BSH> xs;
    load_lane_x<BSH>(xs, x, ks, ks < nk, lane);
    cols_a_class<BSH>(s, gs, ns, i, xs, cs, r, waited, ok, warp, lane);
  }
}

// ------------------------------------------------------------------ down
// ------------------------------------------------------------------ the producer's layer
// The source of one segment of a down stage: nk code blocks of a piece from block b0, or
// (nk == 0) the piece's (scale, bias) record.
__device__ __forceinline__ const uint8_t *col_down_src(const LayerShape &s, const ColPlan &cp,
                                                       const ColPtrs &cw, const ColPiece &q, int e,
                                                       int b0, int nk) {
  const bool routed = q.seg < s.top_k;
  const ColDownDev &d = routed ? cw.r : cw.s;
  const int width = routed ? s.dff : s.dff_shared;
  if (nk > 0) {
    const int nblk = width / (routed ? cp.cb_r : cp.cb_s);
    return reinterpret_cast<const uint8_t *>(
        d.codes + (static_cast<int64_t>(e) * nblk + q.blk0 + b0) * s.din);
  }
  return reinterpret_cast<const uint8_t *>(
      d.sb + (static_cast<int64_t>(e) * (width / kGroup) + q.grp) * s.din);
}

// Lane 0 of the producer warp streams one layer, in the order the consumers take the stages: the
// CTA's gate/up chunks (routed, then shared; one empty stage when it has none), each ONE bulk copy
// of consecutive records (see ColPtrs), then the down column blocks of every valid piece (at most
// cp.nbs blocks a stage; the last stage of a piece also carries the piece's (scale, bias) group
// for all din rows).  false when a ring wait gave up.
__device__ __forceinline__ bool ring_claim_lane(Ring &r) {
  return r.used < r.nst || ring_wait(&r.empty[r.st], r.ph ^ 1u, r.abort, r.err);
}

// L2 prefetch of the layer's stages from index `from` on (the same walk as the copies).
__device__ inline void cols_prefetch_from(const LayerShape &s, const Plan &plan, const ColPlan &cp,
                                          const ColPtrs &cw, const ColSmem &cs, const int *ids,
                                          int from, uint64_t pol) {
  int i = 0;
  for (int c = 0; c < cs.nck; ++c) {
    const bool routed = c < cs.nck_r;
    const int sg = cs.ck_seg[c];
    const int e = routed ? ids[sg] : sg - s.top_k;
    if (routed && (e < 0 || e >= s.n_experts)) continue;
    if (i++ < from) continue;
    const GateUpGeom &g = routed ? plan.geo_r : plan.geo_s;
    const uint8_t *recs = routed ? cw.gu_r : cw.gu_s;
    const int rows_pe = routed ? s.dff : s.dff_shared;
    bulk_prefetch_l2(recs + (static_cast<int64_t>(e) * rows_pe + cs.ck_j[c]) * g.rb,
                     static_cast<uint32_t>(cs.ck_n[c]) * g.rb, pol);
  }
  if (cp.pack) {
    const uint32_t blk_bytes = static_cast<uint32_t>(s.din) * 4u;
    DownWalk w{next_valid_piece(s, cs, ids, 0), 0};
    while (w.qi < cs.np) {
      const bool want = i++ >= from;
      col_down_stage(s, cp, cs, ids, w, [&](int, const ColPiece &q, int e, int b0, int nk, int) {
        if (want)
          bulk_prefetch_l2(col_down_src(s, cp, cw, q, e, b0, nk),
                           static_cast<uint32_t>(nk > 0 ? nk : 1) * blk_bytes, pol);
      });
    }
    return;
  }
  const uint32_t blk_bytes = static_cast<uint32_t>(s.din) * 4u;
  for (int qi = 0; qi < cs.np; ++qi) {
    const ColPiece q = cs.pc[qi];
    int e;
    if (!col_valid(s, q, ids, &e)) continue;
    const bool routed = q.seg < s.top_k;
    const ColDownDev &d = routed ? cw.r : cw.s;
    const int width = routed ? s.dff : s.dff_shared;
    const int nblk = width / (routed ? cp.cb_r : cp.cb_s);
    const int G = width / kGroup;
    for (int bo = 0; bo < q.nb; bo += cp.nbs) {
      const int nk = (q.nb - bo) < cp.nbs ? (q.nb - bo) : cp.nbs;
      if (i++ < from) continue;
      bulk_prefetch_l2(d.codes + (static_cast<int64_t>(e) * nblk + q.blk0 + bo) * s.din,
                       static_cast<uint32_t>(nk) * blk_bytes, pol);
      if (bo + nk == q.nb)
        bulk_prefetch_l2(d.sb + (static_cast<int64_t>(e) * G + q.grp) * s.din, blk_bytes, pol);
    }
  }
}

template <int BR, int BSH>
__device__ bool cols_produce_layer(const LayerShape &s, const Plan &plan, const ColPlan &cp,
                                   const ColPtrs &cw, const ColSmem &cs, const int *ids,
                                   const float *scores, bool all_valid, int *cnt, Ring &r,
                                   uint64_t pol) {
  int nr = cs.nck_r;  // every slot names a valid expert: all routed chunks
  if (!all_valid) {
    nr = 0;
    for (int i = 0; i < cs.nck_r; ++i) {
      const int e = ids[cs.ck_seg[i]];
      nr += e >= 0 && e < s.n_experts;
    }
  }
  const int ns = cs.nck - cs.nck_r;
  cnt[0] = nr;
  cnt[1] = ns;
  MOE_TL_AT(::moe::tl_hook_row_p(), 53);
  int issued = 0;
  for (int i = 0; i < cs.nck; ++i) {
    const bool routed = i < cs.nck_r;
    const int sg = cs.ck_seg[i];
    const int e = routed ? ids[sg] : sg - s.top_k;
    if (routed && (e < 0 || e >= s.n_experts)) continue;
    if (cp.prefetch && issued++ == r.nst)
      cols_prefetch_from(s, plan, cp, cw, cs, ids, r.nst, pol);
    if (!ring_claim_lane(r)) return false;
    if (i == 0) MOE_TL_AT(::moe::tl_hook_row_p(), 54);
    const GateUpGeom &g = routed ? plan.geo_r : plan.geo_s;
    const uint8_t *recs = routed ? cw.gu_r : cw.gu_s;
    const int rows_pe = routed ? s.dff : s.dff_shared;
    const uint32_t bytes = static_cast<uint32_t>(cs.ck_n[i]) * g.rb;
    r.desc[r.st] = StageDesc{cs.u0 + cs.ck_u[i], cs.ck_n[i], routed ? scores[sg] : 0.f, 0};
    mbar_arrive_expect_tx(&r.full[r.st], bytes);
    bulk_g2s(r.stage(), recs + (static_cast<int64_t>(e) * rows_pe + cs.ck_j[i]) * g.rb, bytes,
             &r.full[r.st], pol);
    MOE_TL_STAGE_P(r.used);
    r.advance();
  }
  if (nr + ns == 0) {  // one empty stage, so the consumers always have a first stage to wait on
    if (!ring_claim_lane(r)) return false;
    r.desc[r.st] = StageDesc{0, 0, 0.f, 0};
    mbar_arrive_expect_tx(&r.full[r.st], 0);
    r.advance();
  }
  if (cp.pack) {
    const uint32_t blk_bytes = static_cast<uint32_t>(s.din) * 4u;
    DownWalk w{next_valid_piece(s, cs, ids, 0), 0};
    while (w.qi < cs.np) {
      if (cp.prefetch && issued++ == r.nst)
        cols_prefetch_from(s, plan, cp, cw, cs, ids, r.nst, pol);
      if (!ring_claim_lane(r)) return false;
      DownWalk probe = w;  // the stage's bytes first: the barrier expects them before the copies
      uint32_t total = 0;
      col_down_stage(s, cp, cs, ids, probe, [&](int, const ColPiece &, int, int, int nk, int) {
        total += static_cast<uint32_t>(nk > 0 ? nk : 1) * blk_bytes;
      });
      uint8_t *st = r.stage();
      mbar_arrive_expect_tx(&r.full[r.st], total);
      col_down_stage(s, cp, cs, ids, w, [&](int, const ColPiece &q, int e, int b0, int nk, int slot) {
        const uint8_t *src = col_down_src(s, cp, cw, q, e, b0, nk);
        bulk_g2s(st + static_cast<uint32_t>(slot) * blk_bytes, src,
                 static_cast<uint32_t>(nk > 0 ? nk : 1) * blk_bytes, &r.full[r.st], pol);
      });
      MOE_TL_STAGE_P(r.used);
      r.advance();
    }
    return true;
  }
  const uint32_t blk_bytes = static_cast<uint32_t>(s.din) * 4u;
  for (int qi = 0; qi < cs.np; ++qi) {
    const ColPiece q = cs.pc[qi];
    int e;
    if (!col_valid(s, q, ids, &e)) continue;
    const bool routed = q.seg < s.top_k;
    const ColDownDev &d = routed ? cw.r : cw.s;
    const int width = routed ? s.dff : s.dff_shared;
    const int nblk = width / (routed ? cp.cb_r : cp.cb_s);
    const int G = width / kGroup;
    for (int bo = 0; bo < q.nb; bo += cp.nbs) {
      const int nk = (q.nb - bo) < cp.nbs ? (q.nb - bo) : cp.nbs;
      const bool ends = bo + nk == q.nb;
      if (cp.prefetch && issued++ == r.nst)
        cols_prefetch_from(s, plan, cp, cw, cs, ids, r.nst, pol);
      if (!ring_claim_lane(r)) return false;
      const uint32_t code_bytes = static_cast<uint32_t>(nk) * blk_bytes;
      uint8_t *sb = r.stage();
      mbar_arrive_expect_tx(&r.full[r.st], code_bytes + (ends ? blk_bytes : 0u));
      bulk_g2s(sb, d.codes + (static_cast<int64_t>(e) * nblk + q.blk0 + bo) * s.din, code_bytes,
               &r.full[r.st], pol);
      if (ends)
        bulk_g2s(sb + code_bytes, d.sb + (static_cast<int64_t>(e) * G + q.grp) * s.din,
                 blk_bytes, &r.full[r.st], pol);
      MOE_TL_STAGE_P(r.used);
      r.advance();
    }
  }
  return true;
}

// Consumers: the activations of every valid piece and their byte planes, one warp per piece
// (pieces w, w + 16, ...): lane c holds columns c and c + 32 of the piece, forms
// act = coef * silu(gate) * up from the warps' (gate, up) sums (coef: the routed slot's score, or
// the shared scalar), and the piece's fixed-point exponent and activation sum come from warp
// reductions; lane b then gathers the fixed-point values of the piece's column block b with
// shuffles and writes its planes.
template <int BD, int BSD>
__device__ inline void col_planes(const LayerShape &s, const ColPlan &cp, ColSmem &cs,
                                  const int *ids, const float *scores, float shared_coef,
                                  int wprow, int warp, int lane) {
  for (int qi = warp; qi < cs.np; qi += kConsumerWarps) {
    const ColPiece q = cs.pc[qi];
    const bool routed = q.seg < s.top_k;
    // every load of the piece at once (the slot's id and score, the parked sums): the step is
    // a chain of latencies, so the loads share one round trip
    const int e = routed ? ids[q.seg] : 0;
    const float coef = routed ? scores[q.seg] : shared_coef;
    const int n = q.j1 - q.j0;  // at most 64
    float2 a[2][kColMaxWpr];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int h = 0; h < kColMaxWpr; ++h)
        a[t][h] = lane + 32 * t < n && h < wprow ? cs.red[q.a0 + lane + 32 * t][h]
                                                 : make_float2(0.f, 0.f);
    if (routed && (e < 0 || e >= s.n_experts)) continue;  // the slot names no valid expert
    const int bits = routed ? BD : BSD;
    const int cb = routed ? cp.cb_r : cp.cb_s;
    float v[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float2 g = a[t][0];
#pragma unroll
      for (int h = 1; h < kColMaxWpr; ++h) {
        if (h < wprow) {
          g.x += a[t][h].x;
          g.y += a[t][h].y;
        }
      }
      v[t] = lane + 32 * t < n ? coef * (silu_f(g.x) * g.y) : 0.f;
    }
    // the piece's largest magnitude and sum: two butterflies, interleaved (the same order as
    // warp_max and warp_sum)
    float mx = fmaxf(fabsf(v[0]), fabsf(v[1])), sm = v[0] + v[1];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
    }
    const int E = fixed_exponent(mx);
    const float sc = pow2f(22 - E);
    const int f0 = __float2int_rn(v[0] * sc), f1 = __float2int_rn(v[1] * sc);
    if (lane == 0) cs.us[qi] = make_float2(pow2f(bits == 8 ? E - 22 : E - 26), sm);
    // block b covers piece columns rel = (blk0 + b) * cb - j0 + k, k < cb
    const int rel0 = (q.blk0 + lane) * cb - q.j0;
    int f[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int rel = rel0 + k;
      const int src = rel & 31;
      const int g0 = __shfl_sync(0xffffffffu, f0, src);
      const int g1 = __shfl_sync(0xffffffffu, f1, src);
      f[k] = (k < cb && rel >= 0 && rel < n) ? (rel >= 32 ? g1 : g0) : 0;
    }
    if (lane < q.nb) {
      uint32_t *pl = cs.planes + (q.pb + lane) * 8;
      if (bits == 8) {
        byte_planes(f[0], f[1], f[2], f[3], pl[0], pl[1], pl[2]);
        pl[3] = pl[4] = pl[5] = pl[6] = pl[7] = 0u;
      } else {
        // low nibbles hold the even columns, high nibbles the odd ones
        byte_planes(f[0], f[2], f[4], f[6], pl[0], pl[1], pl[2]);
        byte_planes(f[1], f[3], f[5], f[7], pl[3], pl[4], pl[5]);
        pl[6] = pl[7] = 0u;
      }
    }
  }
}

// Consumers: the stages of one piece.  Thread t owns the row quads t and (QPT = 2) t + 512 (rows
// 4 quad .. 4 quad + 3).  Within a stage its sums over the stage's blocks are exact integers (one
// quad at a time); they join a per-row fp32 sum at the stage's end, and the piece's last stage
// applies the group's scale and bias to those sums into part[][].
template <int BITS, int QPT>
__device__ __forceinline__ void consume_piece(const ColPiece &q, float2 us, const ColPlan &cp,
                                              int din, const uint32_t *planes, Ring &r,
                                              int lane, int tid, float (&part)[2][4]) {
  constexpr int NPL = BITS == 8 ? 3 : 6;
  const int nquads = din >> 2;
  const uint32_t blk_bytes = static_cast<uint32_t>(din) * 4u;
  float dsum[QPT][4];
#pragma unroll
  for (int a = 0; a < QPT; ++a)
#pragma unroll
    for (int k = 0; k < 4; ++k) dsum[a][k] = 0.f;
  for (int bo = 0; bo < q.nb; bo += cp.nbs) {
    const int nk = (q.nb - bo) < cp.nbs ? (q.nb - bo) : cp.nbs;
    const bool ends = bo + nk == q.nb;
    if (tid == 0) MOE_TL_STAGE_WAIT(r.used);
    const bool ok = cols_wait_full(r, lane);
    if (tid == 0) MOE_TL_STAGE_C(r.used);
    const uint8_t *sb = r.stage();
    if (ok) {
#pragma unroll
      for (int a = 0; a < QPT; ++a) {
        const int quad = tid + a * kConsumers;
        if (quad < nquads) {
          uint32_t al[4][NPL];  // l and m planes (unsigned) and h planes (two's complement)
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int z = 0; z < NPL; ++z) al[k][z] = 0u;
#pragma unroll 4
          for (int b = 0; b < nk; ++b) {
            const uint4 pa = *reinterpret_cast<const uint4 *>(planes + (q.pb + bo + b) * 8);
            const uint4 pb = *reinterpret_cast<const uint4 *>(planes + (q.pb + bo + b) * 8 + 4);
            const uint4 w4 = lds_u4(sb + static_cast<uint32_t>(b) * blk_bytes + quad * 16);
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if constexpr (BITS == 8) {
                al[k][0] = dp4a_uu(w[k], pa.x, al[k][0]);
                al[k][1] = dp4a_uu(w[k], pa.y, al[k][1]);
                al[k][2] = static_cast<uint32_t>(dp4a_us(w[k], pa.z, static_cast<int>(al[k][2])));
              } else {
                const uint32_t lo = w[k] & 0x0f0f0f0fu, hi = w[k] & 0xf0f0f0f0u;
                al[k][0] = dp4a_uu(lo, pa.x, al[k][0]);
                al[k][1] = dp4a_uu(lo, pa.y, al[k][1]);
                al[k][2] = static_cast<uint32_t>(dp4a_us(lo, pa.z, static_cast<int>(al[k][2])));
                al[k][3] = dp4a_uu(hi, pa.w, al[k][3]);
                al[k][4] = dp4a_uu(hi, pb.x, al[k][4]);
                al[k][5] = static_cast<uint32_t>(dp4a_us(hi, pb.y, static_cast<int>(al[k][5])));
              }
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t l, m;
            int h;
            if constexpr (BITS == 8) {
              l = al[k][0];
              m = al[k][1];
              h = static_cast<int>(al[k][2]);
            } else {
              // the even sums scaled by 16 join the odd ones (read as 16 q)
              l = al[k][0] * 16u + al[k][3];
              m = al[k][1] * 16u + al[k][4];
              h = static_cast<int>(al[k][2]) * 16 + static_cast<int>(al[k][5]);
            }
            // l, m < 2^22 over at most a group of 64 columns, so m * 256 + l < 2^31
            dsum[a][k] += fmaf(static_cast<float>(h), 65536.f, static_cast<float>(m * 256u + l));
          }
        }
      }
      if (ends) {
        const uint8_t *sbp = sb + static_cast<uint32_t>(nk) * blk_bytes;
#pragma unroll
        for (int a = 0; a < QPT; ++a) {
          const int quad = tid + a * kConsumers;
          if (quad < nquads) {
            const uint4 h4 = lds_u4(sbp + quad * 16);
            const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __half2 sbh = *reinterpret_cast<const __half2 *>(&hw[k]);
              const float sc = __low2float(sbh), bi = __high2float(sbh);
              part[a][k] += fmaf(sc, dsum[a][k] * us.x, bi * us.y);
            }
          }
        }
      }
    }
    warp_release(r, lane);
  }
}

// Consumers: down blocks of one piece inside a stage.  Thread t owns the row quads t and (QPT = 2)
// t + 512 (rows 4 quad .. 4 quad + 3).  Its sums over the run of nk blocks are exact integers (one
// quad at a time); they join the piece's per-row fp32 sums dsum at the run's end (at most 64
// columns a piece keeps m * 256 + l below 2^31).  pl: the planes of the run's first block.
template <int BITS, int QPT>
__device__ __forceinline__ void down_blocks(const uint8_t *base, const uint32_t *pl, int nk,
                                            uint32_t blk_bytes, int nquads, int tid,
                                            float (&dsum)[QPT][4]) {
  constexpr int NPL = BITS == 8 ? 3 : 6;
#pragma unroll
  for (int a = 0; a < QPT; ++a) {
    const int quad = tid + a * kConsumers;
    if (quad < nquads) {
      uint32_t al[4][NPL];  // l and m planes (unsigned) and h planes (two's complement)
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int z = 0; z < NPL; ++z) al[k][z] = 0u;
#pragma unroll 4
      for (int b = 0; b < nk; ++b) {
        const uint4 pa = *reinterpret_cast<const uint4 *>(pl + b * 8);
        const uint4 pb = *reinterpret_cast<const uint4 *>(pl + b * 8 + 4);
        const uint4 w4 = lds_u4(base + static_cast<uint32_t>(b) * blk_bytes + quad * 16);
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if constexpr (BITS == 8) {
            al[k][0] = dp4a_uu(w[k], pa.x, al[k][0]);
            al[k][1] = dp4a_uu(w[k], pa.y, al[k][1]);
            al[k][2] = static_cast<uint32_t>(dp4a_us(w[k], pa.z, static_cast<int>(al[k][2])));
          } else {
            const uint32_t lo = w[k] & 0x0f0f0f0fu, hi = w[k] & 0xf0f0f0f0u;
            al[k][0] = dp4a_uu(lo, pa.x, al[k][0]);
            al[k][1] = dp4a_uu(lo, pa.y, al[k][1]);
            al[k][2] = static_cast<uint32_t>(dp4a_us(lo, pa.z, static_cast<int>(al[k][2])));
            al[k][3] = dp4a_uu(hi, pa.w, al[k][3]);
            al[k][4] = dp4a_uu(hi, pb.x, al[k][4]);
            al[k][5] = static_cast<uint32_t>(dp4a_us(hi, pb.y, static_cast<int>(al[k][5])));
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t l, m;
        int h;
        if constexpr (BITS == 8) {
          l = al[k][0];
          m = al[k][1];
          h = static_cast<int>(al[k][2]);
        } else {
          // the even sums scaled by 16 join the odd ones (read as 16 q)
          l = al[k][0] * 16u + al[k][3];
          m = al[k][1] * 16u + al[k][4];
          h = static_cast<int>(al[k][2]) * 16 + static_cast<int>(al[k][5]);
        }
        dsum[a][k] += fmaf(static_cast<float>(h), 65536.f, static_cast<float>(m * 256u + l));
      }
    }
  }
}

// A piece's (scale, bias) record (one half2 per row, at `base`): the group's scale and bias applied
// to the piece's sums into part[][]; the sums restart at zero for the next piece.
template <int QPT>
__device__ __forceinline__ void down_record(const uint8_t *base, float2 us, int nquads, int tid,
                                            float (&dsum)[QPT][4], float (&part)[2][4]) {
#pragma unroll
  for (int a = 0; a < QPT; ++a) {
    const int quad = tid + a * kConsumers;
    if (quad < nquads) {
      const uint4 h4 = lds_u4(base + quad * 16);
      const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 sbh = *reinterpret_cast<const __half2 *>(&hw[k]);
        const float sc = __low2float(sbh), bi = __high2float(sbh);
        part[a][k] += fmaf(sc, dsum[a][k] * us.x, bi * us.y);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) dsum[a][k] = 0.f;
  }
}

// Consumers: every down stage of the layer, walked like the producer packed them.
template <int BD, int BSD, int QPT>
__device__ void consume_down(const LayerShape &s, const ColPlan &cp, const ColSmem &cs,
                             const int *ids, const uint32_t *planes, Ring &r, int lane, int tid,
                             float (&part)[2][4]) {
  const int nquads = s.din >> 2;
  const uint32_t blk_bytes = static_cast<uint32_t>(s.din) * 4u;
  float dsum[QPT][4];
#pragma unroll
  for (int a = 0; a < QPT; ++a)
#pragma unroll
    for (int k = 0; k < 4; ++k) dsum[a][k] = 0.f;
  DownWalk w{next_valid_piece(s, cs, ids, 0), 0};
  while (w.qi < cs.np) {
    if (tid == 0) MOE_TL_STAGE_WAIT(r.used);
    const bool ok = cols_wait_full(r, lane);
    if (tid == 0) MOE_TL_STAGE_C(r.used);
    const uint8_t *st = r.stage();
    col_down_stage(s, cp, cs, ids, w,
                   [&](int qi, const ColPiece &q, int, int b0, int nk, int slot) {
                     if (!ok) return;
                     const uint8_t *base = st + static_cast<uint32_t>(slot) * blk_bytes;
                     if (nk > 0) {
                       const uint32_t *pl = planes + (q.pb + b0) * 8;
                       if (q.seg < s.top_k)
                         down_blocks<BD, QPT>(base, pl, nk, blk_bytes, nquads, tid, dsum);
                       else
                         down_blocks<BSD, QPT>(base, pl, nk, blk_bytes, nquads, tid, dsum);
                     } else {
                       down_record<QPT>(base, cs.us[qi], nquads, tid, dsum, part);
                     }
                   });
    warp_release(r, lane);
  }
}

// ------------------------------------------------------------------ the owner's sums
// CTA c owns the output rows of the row quads [nq c / n, nq (c + 1) / n), nq = din / 4.
__device__ __forceinline__ void col_owned_quads(int din, int c, int n, int *q0, int *q1) {
  const int nq = din >> 2;
  *q0 = static_cast<int>(static_cast<int64_t>(nq) * c / n);
  *q1 = static_cast<int>(static_cast<int64_t>(nq) * (c + 1) / n);
}

// Helper warp: the owned rows of one pass of the slab ([grid][din] partial vectors), summed over
// the grid's CTAs in a fixed order (lane l takes CTAs l, l + 32, ... in order, then a butterfly
// over the lanes), added to the running output; `out` (when set) receives the result.  Loads are
// issued for two quads at a time so that their L2 round trips overlap.
__device__ __forceinline__ void col_reduce(const float *slab, int din, ColSmem &cs, void *out,
                                           int out_f32, int lane) {
  const int n = gridDim.x;
  int q0, q1;
  col_owned_quads(din, blockIdx.x, n, &q0, &q1);
  for (int qa = q0; qa < q1; qa += 2) {
    float4 acc[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int quad = qa + j;
      float4 v[kColMaxGrid / 32];
#pragma unroll
      for (int k = 0; k < kColMaxGrid / 32; ++k) {
        const int cc = lane + 32 * k;
        v[k] = (quad < q1 && cc < n)
                   ? __ldcg(reinterpret_cast<const float4 *>(slab + static_cast<int64_t>(cc) * din) +
                            quad)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kColMaxGrid / 32; ++k) {
        acc[j].x += v[k].x;
        acc[j].y += v[k].y;
        acc[j].z += v[k].z;
        acc[j].w += v[k].w;
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int quad = qa + j;
      const float t[4] = {warp_sum(acc[j].x), warp_sum(acc[j].y), warp_sum(acc[j].z),
                          warp_sum(acc[j].w)};
      if (lane == 0 && quad < q1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int rr = 4 * (quad - q0) + k;
          const float o = cs.resid[rr] + t[k];
          cs.resid[rr] = o;
          if (out != nullptr) {
            const int i = 4 * quad + k;
            if (out_f32)
              static_cast<float *>(out)[i] = o;
            else
              static_cast<uint16_t *>(out)[i] = float_to_bf16_rn(o);
          }
        }
      }
    }
  }
}

// Helper warp for layers [0, L): the layer-0 residual, then per layer l the owner's sums of
// layer l - 1 (once every CTA has arrived), the shared scalar of layer l, and a meeting with the
// consumers; after the last layer, the output.
__device__ inline void cols_helper(const StackParams &p, ColSmem &cs, int *abort, int lane) {
  const LayerShape &s = p.s;
  const int n = gridDim.x;
  int q0, q1;
  col_owned_quads(s.din, blockIdx.x, n, &q0, &q1);
  for (int t = lane; t < 4 * (q1 - q0); t += 32) {
    const int i = 4 * q0 + t;
    cs.resid[t] = p.resid0_f32 ? static_cast<const float *>(p.resid0)[i]
                               : bf16_to_float(static_cast<const uint16_t *>(p.resid0)[i]);
  }
  const int64_t slab_pass = static_cast<int64_t>(n) * s.din;
  for (int l = 0; l < p.L; ++l) {
    [[maybe_unused]] unsigned long long *tlr = lane == 0 ? MOE_TL_ROW(p.tl, p.L, l) : nullptr;
    if (l > 0) {
      int ok = 1;
      if (lane == 0) ok = wait_count(p.bar, static_cast<uint32_t>(l) * n, abort, p.err);
      MOE_TL_AT(tlr, 52);
      MOE_TL_AT(tlr, 58);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) col_reduce(p.slab + ((l - 1) & 1) * slab_pass, s.din, cs, nullptr, 1, lane);
    }
    const LayerPtrs &w = p.layers[l];
    if (s.n_shared > 0) {
      float scalar = 1.f;
      if (w.gate_vec != nullptr) {
        const uint16_t *x = p.x + static_cast<int64_t>(l) * s.din;
        float dot = 0.f;
        for (int c = lane; c < s.din; c += 32)
          dot = fmaf(bf16_to_float(x[c]), bf16_to_float(w.gate_vec[c]), dot);
        dot = warp_sum(dot);
        scalar = 1.0f / (1.0f + expf(-dot));
      }
      if (lane == 0) cs.s_gate[l & 1] = scalar;
    }
    MOE_TL_AT(tlr, 15);
    consumers_helper_sync();
  }
  int ok = 1;
  if (lane == 0) ok = wait_count(p.bar, static_cast<uint32_t>(p.L) * n, abort, p.err);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) col_reduce(p.slab + ((p.L - 1) & 1) * slab_pass, s.din, cs, p.out, p.out_f32, lane);
}

// ------------------------------------------------------------------ the kernel
// One token per layer (m = 1), layers [0, L): see the top of this file.
template <int BR, int BD, int BSH>
__global__ void __launch_bounds__(kColThreads, 1) cols_kernel(const StackParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) RingSmem rs;
  __shared__ __align__(16) ColSmem cs;
  __shared__ LayerPtrs wpr;  // the producers' copy of the current layer's pointers
  __shared__ ColPtrs cpr;
  __shared__ int stop_pr;
  __shared__ int all_valid_pr;  // every slot of the producer's current layer names a valid expert
  // the expert ids and scores of layers l and l + 1 (the producer may be a layer ahead)
  __shared__ int ids2[2][kMaxTopK];
  __shared__ float sc2[2][kMaxTopK];
  __shared__ __align__(8) uint64_t a_done;  // phase l completes when layer l's gate/up phase has
                                            // been consumed (consumer thread 0 arrives)
  const LayerShape &s = p.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = gridDim.x;
  init_ring(rs.full, rs.empty, p.plan.nst, &rs.abort);
  if (tid == 0) {
    mbar_init(&a_done, 1);
    int nbk = 0;
    const int64_t u0 = p.cp.bounds[blockIdx.x], u1 = p.cp.bounds[blockIdx.x + 1];
    cs.np = col_pieces(s.top_k, s.dff, s.n_shared, s.dff_shared, p.cp.cb_r, p.cp.cb_s, u0, u1,
                       cs.pc, &nbk);
    cs.nbk = nbk;
    cs.u0 = static_cast<int>(u0);
    cs.ncols = static_cast<int>(u1 - u0);
    if (cs.np < 0) {  // outside the plan (the host checks every CTA): do nothing
      cs.np = 0;
      atomicOr(p.err, kDevErrPlan);
      rs.abort = 1;
    }
    cs.s_gate[0] = cs.s_gate[1] = 1.f;
    int nck_r = 0;
    cs.nck = col_chunks(s.top_k, s.dff, s.n_shared, s.dff_shared, p.plan.geo_r.R,
                        p.plan.geo_s.R, u0, u1, cs.ck_seg, cs.ck_j, cs.ck_n, cs.ck_u, &nck_r);
    cs.nck_r = nck_r;
    if (cs.nck < 0) {  // outside the plan (the host checks every CTA): do nothing
      cs.nck = cs.nck_r = 0;
      atomicOr(p.err, kDevErrPlan);
      rs.abort = 1;
    }
  }
  __syncthreads();
  Ring r = make_ring(rs.full, rs.empty, ring, rs.desc, p.plan, &rs.abort, p.err);

  if (warp == kColHelperWarp) {
    cols_helper(p, cs, &rs.abort, lane);
    return;
  }
  if (warp >= kConsumerWarps) {
    const uint64_t pol = policy_evict_first();
    const int pl = tid - kConsumers;
    for (int l = 0; l < p.L; ++l) {
      producer_sync();  // every producer is done with the previous layer's copies
      [[maybe_unused]] unsigned long long *tlr = pl == 0 ? MOE_TL_ROW(p.tl, p.L, l) : nullptr;
      MOE_TL_AT(tlr, 0);
      if (pl == 0) {
        wpr = p.layers[l];
        cpr = p.cols[l];
        if (l > 0) {
          if (p.ahead)  // this CTA's consumers are past layer l - 1's gate/up phase: they no
                        // longer read its stage counts, nor the ids of layer l - 2 (same slot)
            ring_wait(&a_done, static_cast<uint32_t>(l - 1) & 1u, &rs.abort, p.err);
          else          // every CTA has finished the previous layer before its ids are read
            wait_count(p.bar, static_cast<uint32_t>(l) * n, &rs.abort, p.err);
        }
        MOE_TL_AT(tlr, 1);
        MOE_TL_AT(tlr, 59);
        stop_pr = flag_abort(&rs.abort);
      }
      producer_sync();
      if (stop_pr) break;
      const int64_t ks = s.top_k;
      int *ids_l = ids2[l & 1];
      float *sc_l = sc2[l & 1];
      producer_load_token(s, p.ids + l * ks, p.scores + l * ks, ids_l, sc_l, p.err, pl,
                          p.ids_used ? p.ids_used + l * ks : nullptr, &all_valid_pr);
      MOE_TL_AT(tlr, 2);
      if (pl == 0) {
        MOE_TL_SET_HOOK_P(tlr);
        MOE_TL_STAGE_BASE_P(r.used);
        cols_produce_layer<BR, BSH>(s, p.plan, p.cp, cpr, cs, ids_l, sc_l, all_valid_pr != 0,
                                    rs.cnt, r, pol);
      }
      __syncwarp();
      MOE_TL_AT(tlr, 4);
    }
    ring_drain(r, pl);
    return;
  }

  // consumers
  const int64_t slab_pass = static_cast<int64_t>(n) * s.din;
  const int nquads = s.din >> 2;
  const bool two = s.din > 4 * kConsumers;  // a second row quad per thread
  for (int l = 0; l < p.L; ++l) {
    [[maybe_unused]] unsigned long long *tlr = tid == 0 ? MOE_TL_ROW(p.tl, p.L, l) : nullptr;
    MOE_TL_AT(tlr, 5);
    MOE_TL_AT(tlr, 56);
    if (tid == 0) {
      MOE_TL_SET_HOOK(tlr);
      MOE_TL_STAGE_BASE(r.used);
    }
    cols_phase_a<BR, BSH>(s, p.plan.geo_r, p.plan.geo_s, p.x + static_cast<int64_t>(l) * s.din,
                          rs.cnt, cs, r, warp, lane);
    MOE_TL_AT(tlr, 9);
    consumer_sync(kConsumers);  // every (gate, up) sum written; the ids were published by the
                                // phase's first stage
    MOE_TL_AT(tlr, 10);
    if (tid == 0) mbar_arrive(&a_done);
    const int *ids_l = ids2[l & 1];
    MOE_TL_AT(tlr, 3);
    consumers_helper_sync();  // the helper's shared scalar is ready
    MOE_TL_AT(tlr, 6);
    col_planes<BD, BSH>(s, p.cp, cs, ids_l, sc2[l & 1], cs.s_gate[l & 1],
                        ((s.din >> 5) + 31) >> 5, warp, lane);
    consumer_sync(kConsumers);
    MOE_TL_AT(tlr, 11);
    float part[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) part[a][k] = 0.f;
    if (p.cp.pack) {
      if (two)
        consume_down<BD, BSH, 2>(s, p.cp, cs, ids_l, cs.planes, r, lane, tid, part);
      else
        consume_down<BD, BSH, 1>(s, p.cp, cs, ids_l, cs.planes, r, lane, tid, part);
    } else {
      for (int qi = 0; qi < cs.np; ++qi) {
        const ColPiece q = cs.pc[qi];
        int e;
        if (!col_valid(s, q, ids_l, &e)) continue;
        if (q.seg < s.top_k) {
          if (two)
            consume_piece<BD, 2>(q, cs.us[qi], p.cp, s.din, cs.planes, r, lane, tid, part);
          else
            consume_piece<BD, 1>(q, cs.us[qi], p.cp, s.din, cs.planes, r, lane, tid, part);
        } else {
          if (two)
            consume_piece<BSH, 2>(q, cs.us[qi], p.cp, s.din, cs.planes, r, lane, tid, part);
          else
            consume_piece<BSH, 1>(q, cs.us[qi], p.cp, s.din, cs.planes, r, lane, tid, part);
        }
      }
    }
    MOE_TL_AT(tlr, 12);
    // this CTA's partial output of all din rows: one contiguous vector of the slab pass
    float *sl = p.slab + (l & 1) * slab_pass + static_cast<int64_t>(blockIdx.x) * s.din;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int quad = tid + a * kConsumers;
      if (quad < nquads)
        reinterpret_cast<float4 *>(sl)[quad] =
            make_float4(part[a][0], part[a][1], part[a][2], part[a][3]);
    }
    MOE_TL_AT(tlr, 13);
    consumer_sync(kConsumers);
    // bar.sync orders the CTA's partials before this thread's release, which is cumulative; the
    // consumers do not wait: the producer and the helper wait for the count
    if (tid == 0) red_release_add(p.bar, 1u);
    MOE_TL_AT(tlr, 14);
    MOE_TL_AT(tlr, 57);
  }
  if (tid == 0) MOE_TL_SET_HOOK(nullptr);
}

// Down code widths of the column-split kernels: 4 or 8 bits.
#define MOE_COLS_BITS(B, NAME, ...)                         \
  switch (B) {                                              \
    case 4: { constexpr int NAME = 4; __VA_ARGS__; break; } \
    case 8: { constexpr int NAME = 8; __VA_ARGS__; break; } \
    default: return cudaErrorInvalidValue;                  \
  }

template <int BR>
cudaError_t launch_cols_family(const StackParams &p, int grid, cudaStream_t stream) {
  MOE_COLS_BITS(p.cp.cb_r == 8 ? 4 : 8, BD, MOE_COLS_BITS(p.cp.cb_s == 8 ? 4 : 8, BSH,
      return launch(cols_kernel<BR, BD, BSH>, p, grid, p.plan.smem, stream, false, true,
                    kColThreads)));
  return cudaErrorInvalidValue;
}

template <int BR>
cudaError_t prepare_cols_family(int smem_optin, int bits_d, int bits_sh, int *lim) {
  cudaError_t e = cudaSuccess;
  MOE_COLS_BITS(bits_d, BD, MOE_COLS_BITS(bits_sh, BSH,
      e = set_smem_limit(reinterpret_cast<const void *>(cols_kernel<BR, BD, BSH>), smem_optin,
                         lim)));
  return e;
}

template <int BR>
cudaError_t cols_occupancy_family(int bits_d, int bits_sh, size_t smem, int *per_sm) {
  cudaError_t e = cudaSuccess;
  int nb = 0;
  MOE_COLS_BITS(bits_d, BD, MOE_COLS_BITS(bits_sh, BSH,
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, cols_kernel<BR, BD, BSH>,
                                                        kColThreads, smem)));
  *per_sm = nb;
  return e;
}
#undef MOE_COLS_BITS

#define MOE_COLS_FAMILY(B)                                                                       \
  cudaError_t launch_cols_g##B(const StackParams &p, int grid, cudaStream_t stream) {            \
    return launch_cols_family<B>(p, grid, stream);                                               \
  }                                                                                              \
  cudaError_t prepare_cols_g##B(int smem_optin, int bits_d, int bits_sh, int *lim) {             \
    return prepare_cols_family<B>(smem_optin, bits_d, bits_sh, lim);                             \
  }                                                                                              \
  cudaError_t cols_occupancy_g##B(int bits_d, int bits_sh, size_t smem, int *per_sm) {           \
    return cols_occupancy_family<B>(bits_d, bits_sh, smem, per_sm);                              \
  }

}  // namespace moe
