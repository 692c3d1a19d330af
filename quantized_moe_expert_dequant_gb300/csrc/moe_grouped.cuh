// moe_grouped.cuh -- a batch of m > 1 tokens per decode step, each selected expert streamed once.
//
// The tokens' slots are grouped by expert (route inversion, moe_phases.cuh).  Three phases per
// layer, each over all tokens at once:
//   A  every row j of every distinct routed expert (and of the shared experts): for each
//      (token, slot) that selected it, act[token][slot][j] = score * silu(gate_j . x) * (up_j . x)
//   B  every output row i of every distinct expert's down projection: for each (token, slot),
//      y[token][slot][i] = down_i . act[token][slot]
//   T  out[token][i] = resid[token][i] + (sum over valid slots, in slot order, of y + sum over
//      shared experts of y), the tail of "Red Lite dev39 -- fused expert tail" (Change)
// with a grid barrier after each.  A stage holds R rows of one expert plus the operand rows of up
// to t_sub of its (token, slot) pairs (x rows in phase A, activation rows in phase B), all copied
// by the bulk-copy engine, so consumers build each pair's operand from shared memory.  A shared
// expert, or a routed expert selected by more than t_sub pairs, is staged once per group of
// t_sub pairs (a segment); the repeats of its rows come from L2.
#pragma once

#include "moe_phases.cuh"

namespace moe {

// What the producer tells the consumers about a grouped stage.
struct GroupDesc {
  int u;       // flattened first row of the stage inside its class
  int n;       // rows (0: an empty stage that only publishes the phase's counts)
  int e;       // expert of the class: distinct-expert rank (routed) or shared expert index
  int pb, pe;  // the stage's pairs: [pb, pe) of the expert's pair list
  int delta;   // offset in bytes of the first row's first group inside each window
  int cls;     // class of the phase: 0 routed, 1 shared
  int j0;      // first row inside the expert
};

// Shared state of a grouped layer, written by the producer warp after it read the ids (except
// sscal, which the consumers compute).  It sits at the start of the dynamic shared memory, before
// the stage ring.
struct GroupSmem {
  Route rt;
  unsigned char pm[kMaxPairs];  // token of the q-th pair of the route's list
  unsigned char pk[kMaxPairs];  // its slot
  GroupDesc desc[kMaxStages];
  int cnt[4];                   // stages: A routed, A shared, B routed, B shared
  float sscal[kMaxGroupTokens]; // per-token shared scalar (consumers)
  int ids[kMaxPairs];           // the layer's ids [m][top_k] and scores
  float scores[kMaxPairs];
  // Work is split into segments: one distinct expert and one group of at most t_sub of its pairs
  // (shared experts: of the tokens).  Every segment spans the expert's rows once, so splitting
  // the flattened segment rows evenly across CTAs balances stages, not just weight rows.
  short seg_e[kMaxPairs];       // routed segment -> distinct-expert rank
  short seg_pb[kMaxPairs];      // -> its first pair in that expert's list
  int n_seg;                    // routed segments
};

constexpr int kGroupSmemBytes = (static_cast<int>(sizeof(GroupSmem)) + 127) / 128 * 128;

// The rows one CTA owns of a class pair (routed, shared) whose flattened row space is
// n_r * rows_r routed rows followed by n_s * rows_s shared rows.
struct RangeG {
  int64_t ra, rb, sa, sb, Ur;
};

__device__ __forceinline__ RangeG range_g(int64_t n_r, int rows_r, int64_t n_s, int rows_s) {
  const int64_t Ur = n_r * rows_r, U = Ur + n_s * rows_s;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  RangeG r;
  r.ra = u0;
  r.rb = u1 < Ur ? u1 : Ur;
  r.sa = u0 > Ur ? u0 : Ur;
  r.sb = u1;
  r.Ur = Ur;
  return r;
}

// How a class streams: its rows, projections and operand rows.
struct GClass {
  bool gated;        // phase A (gate and up rows, SwiGLU) or phase B (down rows)
  bool shared;       // shared experts (every token is a pair) or distinct routed experts
  int rows_pe;       // rows per expert
  int64_t base;      // first flattened row of the class
  ProjDev p0, p1;    // gate and up (A) or down (B; p1 unused)
  int cols;          // row length in codes
  int op_bytes;      // bytes of one operand row in a stage
};

__device__ __forceinline__ int pair_count(const GroupSmem &gs, const GClass &c, int e, int m) {
  return c.shared ? m : gs.rt.offs[e + 1] - gs.rt.offs[e];
}

// Segment k of a class: its expert (rank or shared index) and first pair; groups_sh = segments
// per shared expert.
__device__ __forceinline__ void segment(const GroupSmem &gs, const GClass &c, int k, int t_sub,
                                        int groups_sh, int &e, int &pb) {
  if (c.shared) {
    e = k / groups_sh;
    pb = (k - e * groups_sh) * t_sub;
  } else {
    e = gs.seg_e[k];
    pb = gs.seg_pb[k];
  }
}

// Routed segments after the route inversion: ceil(pairs / t_sub) per distinct expert, in rank
// order (one warp; U <= kMaxPairs, so eight experts per lane).
__device__ __forceinline__ void build_segments(GroupSmem &gs, int t_sub, int lane) {
  constexpr int PER = kMaxPairs / 32;
  const int U = gs.rt.n_uniq;
  int cnt[PER], sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int u = lane * PER + j;
    cnt[j] = u < U ? (gs.rt.offs[u + 1] - gs.rt.offs[u] + t_sub - 1) / t_sub : 0;
    sum += cnt[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int k = incl - sum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int u = lane * PER + j;
    for (int g = 0; g < cnt[j]; ++g, ++k) {
      gs.seg_e[k] = static_cast<short>(u);
      gs.seg_pb[k] = static_cast<short>(g * t_sub);
    }
  }
  if (lane == 31) gs.n_seg = incl;
  __syncwarp();
}

// Stages of a class in [a, b): one per chunk (a chunk never crosses a segment).
__device__ __forceinline__ int count_g(const GClass &c, const GateUpGeom &g, int64_t a, int64_t b) {
  ChunkIterA it(a, b, c.base, c.rows_pe, g.R);
  ChunkA ch;
  int n = 0;
  while (it.next(ch)) ++n;
  return n;
}

// Global address of the operand row of the q-th pair of expert e (class c) for a layer whose
// token data start at x_l (bf16 [m][din]) and whose activations are act ([m][act_stride]).
__device__ __forceinline__ const uint8_t *operand_src(const GroupSmem &gs, const GClass &c,
                                                      const LayerShape &s, int e, int q,
                                                      const uint16_t *x_l, const float *act,
                                                      int act_stride) {
  const int m = c.shared ? q : gs.pm[gs.rt.offs[e] + q];
  if (c.gated) return reinterpret_cast<const uint8_t *>(x_l + static_cast<int64_t>(m) * s.din);
  const int64_t col0 = c.shared ? static_cast<int64_t>(s.top_k) * s.dff +
                                      static_cast<int64_t>(e) * s.dff_shared
                                : static_cast<int64_t>(gs.pk[gs.rt.offs[e] + q]) * s.dff;
  return reinterpret_cast<const uint8_t *>(act + static_cast<int64_t>(m) * act_stride + col0);
}

// Operand copies of phase-B stages wait until the activations are complete (a grid barrier).
// Stages handed out before that carry only their weights: the producer raises the stage's
// expected bytes without arriving, and adds the operand rows and its arrival once the barrier has
// passed.  Before claiming a slot whose previous use is still waiting for its operands (which the
// consumers cannot release), the producer completes the waiting stages first.
struct Deferred {
  bool on;            // operand rows wait for the barrier
  bool ready;         // the barrier has passed
  int begin;          // first ring index (Ring::used) still waiting for its operand rows
  const uint32_t *bar;
  uint32_t target;
};

__device__ __forceinline__ void copy_operands(const LayerShape &s, const GroupSmem &gs,
                                              const GClass &c, const GroupDesc &d, uint8_t *sb,
                                              int op_off, const uint16_t *x_l, const float *act,
                                              int act_stride, uint64_t *full, int lane,
                                              uint64_t pol) {
  const int q = d.pb + lane - 8;  // lanes 8.. copy the operand rows
  if (lane >= 8 && q < d.pe)
    bulk_g2s(sb + op_off + (q - d.pb) * c.op_bytes,
             operand_src(gs, c, s, d.e, q, x_l, act, act_stride), c.op_bytes, full, pol);
}

// Completes the waiting stages [df.begin, r.used): waits for the barrier, then per stage adds the
// operand bytes with the producer's arrival and copies the rows.
__device__ inline void complete_deferred(const LayerShape &s, const GroupSmem &gs, const GClass *cls,
                                  const int *op_off, Deferred &df, Ring &r, int lane,
                                  const uint16_t *x_l, const float *act, int act_stride,
                                  uint64_t pol) {
  if (!df.ready) {
    if (lane == 0) wait_count(df.bar, df.target, r.abort, r.err);
    __syncwarp();
    // the operand rows were written through the generic proxy; the copies read them through
    // the async proxy
    asm volatile("fence.proxy.async.global;" ::: "memory");
    df.ready = true;
  }
  for (int i = df.begin; i < r.used; ++i) {
    const int st = i % r.nst;
    const GroupDesc d = gs.desc[st];
    const GClass &c = cls[d.cls];
    if (lane == 0)
      mbar_arrive_expect_tx(&r.full[st], static_cast<uint32_t>(d.pe - d.pb) * c.op_bytes);
    __syncwarp();
    copy_operands(s, gs, c, d, r.base + static_cast<size_t>(st) * r.stage_bytes, op_off[d.cls],
                  x_l, act, act_stride, &r.full[st], lane, pol);
  }
  df.begin = r.used;
}

// Producer of one class (index ci of cls): stages of R rows of one expert plus the operand rows
// of up to t_sub of its pairs.  Stage layout: codes (gated: gate then up, R rows each), 2 or 4
// scale/bias windows of g.sw bytes, then the operand rows at op_off[ci].
__device__ inline void produce_g_class(const LayerShape &s, const GroupSmem &gs, const GClass *cls,
                                int ci, const GateUpGeom &g, int64_t a, int64_t b, int m,
                                int t_sub, const int *op_off, const uint16_t *x_l,
                                const float *act, int act_stride, Ring &r, GroupDesc *desc,
                                Deferred &df, int lane, uint64_t pol) {
  const GClass &c = cls[ci];
  const int G = c.cols / kGroup;
  const int groups_sh = (m + t_sub - 1) / t_sub;
  ChunkIterA it(a, b, c.base, c.rows_pe, g.R);
  ChunkA ch;
  const int nproj = c.gated ? 2 : 1;
  const uint64_t pol_first = policy_evict_first(), pol_again = policy_evict_normal();
  while (it.next(ch)) {
    int e, pb;
    segment(gs, c, ch.k, t_sub, groups_sh, e, pb);
    const int expert = c.shared ? e : gs.rt.uniq[e];
    const int np = pair_count(gs, c, e, m);
    const int pe = pb + t_sub < np ? pb + t_sub : np;
    // rows staged again for the expert's other pair groups stay in L2 for them
    const uint64_t pol = np > t_sub ? pol_again : pol_first;
    const int64_t row = static_cast<int64_t>(expert) * c.rows_pe + ch.j;
    const uint32_t code_bytes = static_cast<uint32_t>(ch.n) * g.rb;
    const int64_t ng = static_cast<int64_t>(ch.n) * G;
    {
      // the slot's previous use must be releasable: complete waiting stages first
      if (df.on && !df.ready && df.begin < r.used && r.used - r.nst >= df.begin)
        complete_deferred(s, gs, cls, op_off, df, r, lane, x_l, act, act_stride, pol_first);
      if (!ring_claim(r, lane)) return;
      uint8_t *sb = r.stage();
      const Window w0 = window_of(c.p0.scales + row * G, ng);
      const Window w1 = window_of(c.p0.biases + row * G, ng);
      uint32_t wbytes = nproj * code_bytes + w0.bytes + w1.bytes;
      Window w2{}, w3{};
      if (c.gated) {
        w2 = window_of(c.p1.scales + row * G, ng);
        w3 = window_of(c.p1.biases + row * G, ng);
        wbytes += w2.bytes + w3.bytes;
      }
      const uint32_t obytes = static_cast<uint32_t>(pe - pb) * c.op_bytes;
      const bool later = df.on && !df.ready;
      const GroupDesc d{ch.u - static_cast<int>(c.base), ch.n, e, pb, pe,
                        static_cast<int>(w0.delta), ci, ch.j};
      uint8_t *wb = sb + nproj * g.R * g.rb;
      if (lane == 0) {
        desc[r.st] = d;
        if (later)
          mbar_expect_tx(&r.full[r.st], wbytes);
        else
          mbar_arrive_expect_tx(&r.full[r.st], wbytes + obytes);
      }
      __syncwarp();
      if (lane == 0) bulk_g2s(sb, c.p0.codes + row * g.rb, code_bytes, &r.full[r.st], pol);
      if (lane == 1) bulk_g2s(wb, w0.src, w0.bytes, &r.full[r.st], pol);
      if (lane == 2) bulk_g2s(wb + g.sw, w1.src, w1.bytes, &r.full[r.st], pol);
      if (c.gated) {
        if (lane == 3) bulk_g2s(sb + g.R * g.rb, c.p1.codes + row * g.rb, code_bytes, &r.full[r.st],
                                pol);
        if (lane == 4) bulk_g2s(wb + 2 * g.sw, w2.src, w2.bytes, &r.full[r.st], pol);
        if (lane == 5) bulk_g2s(wb + 3 * g.sw, w3.src, w3.bytes, &r.full[r.st], pol);
      }
      if (!later)
        copy_operands(s, gs, c, d, sb, op_off[ci], x_l, act, act_stride, &r.full[r.st], lane,
                      pol_first);
      r.advance();
    }
  }
}

// Producer of one grouped phase (two classes of n_r and n_s segments): counts its stages into
// cnt[0..1], streams them, and hands out one empty stage when the CTA has none.  With deferred
// operands, the waiting stages are completed at the end.
__device__ inline void produce_g_phase(const LayerShape &s, const GroupSmem &gs, GroupDesc *desc,
                                int *cnt, const GClass *cls, const GateUpGeom &gr,
                                const GateUpGeom &gsh, int64_t n_r, int64_t n_s, int m,
                                int t_sub, const int *op_off, const uint16_t *x_l,
                                const float *act, int act_stride, Deferred &df, Ring &r,
                                int lane, uint64_t pol) {
  const RangeG rg = range_g(n_r, cls[0].rows_pe, n_s, cls[1].rows_pe);
  const int nr = count_g(cls[0], gr, rg.ra, rg.rb);
  const int ns = count_g(cls[1], gsh, rg.sa, rg.sb);
  if (lane == 0) {
    cnt[0] = nr;
    cnt[1] = ns;
  }
  __syncwarp();
  df.begin = r.used;
  produce_g_class(s, gs, cls, 0, gr, rg.ra, rg.rb, m, t_sub, op_off, x_l, act, act_stride, r,
                  desc, df, lane, pol);
  if (flag_abort(r.abort)) return;
  produce_g_class(s, gs, cls, 1, gsh, rg.sa, rg.sb, m, t_sub, op_off, x_l, act, act_stride, r,
                  desc, df, lane, pol);
  if (flag_abort(r.abort)) return;
  if (nr + ns == 0) {
    if (!ring_claim(r, lane)) return;
    if (lane == 0) {
      desc[r.st] = GroupDesc{0, 0, 0, 0, 0, 0, 0, 0};
      mbar_arrive_expect_tx(&r.full[r.st], 0);
    }
    r.advance();
    df.begin = r.used;
  }
  // Only stages handed out before the barrier wait; those after it were issued complete (a
  // second arrival on them would complete their next use early).
  if (df.on && !df.ready && df.begin < r.used)
    complete_deferred(s, gs, cls, op_off, df, r, lane, x_l, act, act_stride, pol);
}

// The Operand of a thread's C columns of an operand row in shared memory: bf16 (x) or fp32
// (activations).
template <int BITS>
__device__ __forceinline__ void operand_from_smem(Operand<BITS> &op, const uint8_t *row, bool bf16,
                                                  int c0, bool active) {
  constexpr int C = Operand<BITS>::C;
  float v[C];
  if (bf16) {
#pragma unroll
    for (int q = 0; q < C / 8; ++q) {
      const uint4 w = active ? lds_u4(row + (c0 + 8 * q) * 2) : make_uint4(0, 0, 0, 0);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v[8 * q + 2 * h] = __uint_as_float(ww[h] << 16);
        v[8 * q + 2 * h + 1] = __uint_as_float(ww[h] & 0xffff0000u);
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < C / 4; ++q) {
      const uint4 w = active ? lds_u4(row + (c0 + 4 * q) * 4) : make_uint4(0, 0, 0, 0);
      v[4 * q] = __uint_as_float(w.x);
      v[4 * q + 1] = __uint_as_float(w.y);
      v[4 * q + 2] = __uint_as_float(w.z);
      v[4 * q + 3] = __uint_as_float(w.w);
    }
  }
  op.set(v);
}

// Sums the parked partials of the held items across warps and writes them: gated items get
// coef * silu(gate) * up, plain items the sum.
__device__ __forceinline__ void flush_g(SmemA &sm, int held, int wpg, bool gated, float *outp,
                                        int tid, bool trailing) {
  consumer_sync(kConsumers);
  for (int t = tid; t < held; t += kConsumers) {
    float gs = 0.f, us = 0.f;
    for (int w = 0; w < wpg; ++w) {
      gs += sm.red[0][t * wpg + w];
      if (gated) us += sm.red[1][t * wpg + w];
    }
    outp[sm.row_u[t]] = gated ? sm.coef[t] * (silu_f(gs) * us) : gs;
  }
  if (trailing) consumer_sync(kConsumers);
}

// Where a class's items go: the activation or partial-output index of the stage's first row for
// the q-th pair of expert e, and the item's coefficient.
struct GOut {
  int stride;      // per token: act_stride (A) or (K + n_shared) * din (B)
  int col_shared;  // first column of shared expert 0 in a token's vector
  int col_pe;      // columns per routed slot: dff (A) or din (B)
  int col_sh;      // columns per shared expert: dff_sh (A) or din (B)
};

// Consumers of one class of a grouped phase: `count` stages (the first may already be waited).
template <int BITS, bool GATED>
__device__ int consume_g_class(const LayerShape &s, const GroupSmem &gs, const GClass &c,
                               const GateUpGeom &g, const GOut &go, int count, int op_off,
                               const float *scores_s, float *outp, Ring &r, SmemA &sm,
                               bool &waited, bool &ok, int tid, bool fold = true) {
  constexpr int VEC = Fmt<BITS>::kVecs, C = Operand<BITS>::C;
  constexpr int RPT = GATED ? rows_per_thread_a<BITS>() : rows_per_thread_gb<BITS>();
  constexpr int V = GATED ? 2 * RPT : RPT;
  int held = 0;
  if (count == 0) return held;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = c.cols / kGroup;
  const int my_group = tid / g.tpr, my_step = tid % g.tpr;
  const bool grp_ok = my_group < g.groups;
  const bool active = grp_ok && my_step < g.T;
  const int wpg = g.tpr / 32;
  const int wslot = warp - my_group * wpg;
  const int code_off = my_step * 16 * VEC;
  const int win_off = ((my_step * C) / kGroup) * 2;
  const int idx = (lane >> (5 - Log2<V>::v)) & (V - 1);
  const bool writer = grp_ok && (lane & ((32 / V) - 1)) == 0;
  const int w_kind = GATED ? idx / RPT : 0, w_row = (idx % RPT) * g.groups + my_group;
  const int cap = kRedA / wpg < kBatchA ? kRedA / wpg : kBatchA;
  const int nproj = GATED ? 2 : 1;
  const int wbase = nproj * g.R * g.rb + win_off;

  for (int i = 0; i < count; ++i) {
    if (!waited) ok = warp_wait_full(r, lane);
    waited = false;
    const GroupDesc d = gs.desc[r.st];
    const uint8_t *sb = r.stage();
    const uint8_t *ws = sb + wbase + d.delta;
    const int j0 = d.j0;
    for (int q = d.pb; q < d.pe; ++q) {
      int m, col;
      float coef;
      if (c.shared) {
        m = q;
        col = go.col_shared + d.e * go.col_sh;
        coef = GATED && fold ? gs.sscal[m] : 1.f;
      } else {
        const int o = gs.rt.offs[d.e] + q;
        m = gs.pm[o];
        const int k = gs.pk[o];
        col = k * go.col_pe;
        coef = GATED && fold ? scores_s[m * s.top_k + k] : 1.f;
      }
      if (held + d.n > cap) {
        flush_g(sm, held, wpg, GATED, outp, tid, true);
        held = 0;
      }
      if (tid < d.n) {
        sm.row_u[held + tid] = m * go.stride + col + j0 + tid;
        sm.coef[held + tid] = coef;
      }
      Operand<BITS> op;
      operand_from_smem<BITS>(op, sb + op_off + (q - d.pb) * c.op_bytes, GATED, my_step * C,
                              active && ok);
      float v[V];
#pragma unroll
      for (int t = 0; t < V; ++t) v[t] = 0.f;
      if (active && ok) {
#pragma unroll
        for (int t = 0; t < RPT; ++t) {
          const int rr = t * g.groups + my_group;
          if (rr < d.n) {
            uint4 cg[VEC];
            const uint8_t *pg = sb + rr * g.rb + code_off;
#pragma unroll
            for (int w = 0; w < VEC; ++w) cg[w] = lds_u4(pg + 16 * w);
            const uint8_t *wr = ws + rr * G * 2;
            v[t] = fmaf(lds_half(wr), op.dot(cg) * op.unit, lds_half(wr + g.sw) * op.sum);
            if (GATED) {
              uint4 cu[VEC];
#pragma unroll
              for (int w = 0; w < VEC; ++w) cu[w] = lds_u4(pg + g.R * g.rb + 16 * w);
              v[(RPT + t) % V] = fmaf(lds_half(wr + 2 * g.sw), op.dot(cu) * op.unit,
                                      lds_half(wr + 3 * g.sw) * op.sum);
            }
          }
        }
      }
      const float val = warp_transpose_reduce<V>(v, lane);
      if (writer && w_row < d.n) sm.red[w_kind][(held + w_row) * wpg + wslot] = val;
      held += d.n;
    }
    warp_release(r, lane);
  }
  return held;
}

// Consumers of one grouped phase: the first stage publishes the counts.
template <int BR, int BS, bool GATED>
__device__ void consume_g_phase(const LayerShape &s, const GroupSmem &gs, const GClass *cls,
                                const GateUpGeom &gr, const GateUpGeom &gsh, const GOut &go,
                                const int *op_off, const float *scores_s, float *outp, Ring &r,
                                SmemA &sm, int tid, bool fold = true) {
  const int lane = tid & 31;
  bool ok = warp_wait_full(r, lane), waited = true;
  const int nr = gs.cnt[GATED ? 0 : 2], ns = gs.cnt[GATED ? 1 : 3];
  if (nr + ns == 0) {
    warp_release(r, lane);
    return;
  }
  int held = consume_g_class<BR, GATED>(s, gs, cls[0], gr, go, nr, op_off[0], scores_s, outp, r,
                                        sm, waited, ok, tid, fold);
  if (held > 0) flush_g(sm, held, gr.tpr / 32, GATED, outp, tid, ns > 0);
  held = consume_g_class<BS, GATED>(s, gs, cls[1], gsh, go, ns, op_off[1], scores_s, outp, r, sm,
                                    waited, ok, tid, fold);
  if (held > 0) flush_g(sm, held, gsh.tpr / 32, GATED, outp, tid, false);
}

// Tail of a grouped layer for the CTA's output rows: out = resid + (routed + shared), routed
// summed over the valid slots in slot order.  y and the residual are complete (grid barrier).
// pool: y holds the slots' and shared experts' outputs without their coefficients, and the tail
// is the one of "Red Lite dev39 -- fused expert tail" (Change) as written:
//   out = resid + (sum_k score_k * y_k + scalar * sum_s y_s).
__device__ inline void tail_g(const LayerShape &s, const int *ids_s, int m, const float *y, int y_stride,
                       const void *resid, int resid_f32, void *out, int out_f32, int tid,
                       bool pool = false, const float *scores_s = nullptr,
                       const float *sscal = nullptr) {
  int i0, i1;
  range_b(s, i0, i1);
  const int rows = i1 - i0;
  for (int t = tid; t < m * rows; t += kConsumers) {
    const int tok = t / rows, i = i0 + (t - tok * rows);
    const float *yt = y + static_cast<int64_t>(tok) * y_stride + i;
    float routed = 0.f, shared = 0.f;
    for (int k = 0; k < s.top_k; ++k) {
      const int e = ids_s[tok * s.top_k + k];
      if (e >= 0 && e < s.n_experts) {
        const float yk = yt[static_cast<int64_t>(k) * s.din];
        routed = pool ? fmaf(scores_s[tok * s.top_k + k], yk, routed) : routed + yk;
      }
    }
    for (int sh = 0; sh < s.n_shared; ++sh)
      shared += yt[static_cast<int64_t>(s.top_k + sh) * s.din];
    const int64_t o = static_cast<int64_t>(tok) * s.din + i;
    const float rs = resid_f32 ? static_cast<const float *>(resid)[o]
                               : bf16_to_float(static_cast<const uint16_t *>(resid)[o]);
    const float v = pool ? rs + (s.n_shared > 0 ? fmaf(sscal[tok], shared, routed) : routed)
                         : rs + (routed + shared);
    if (out_f32)
      static_cast<float *>(out)[o] = v;
    else
      static_cast<uint16_t *>(out)[o] = float_to_bf16_rn(v);
  }
}

// Per-token shared scalars sigmoid(x_t . g) into gs.sscal (one warp per token, no block-wide
// synchronisation; the caller publishes them).
__device__ __forceinline__ void shared_scalars_g(const LayerShape &s, const uint16_t *x_l,
                                                 const uint16_t *gate_vec, int m, float *sscal,
                                                 int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  for (int t = warp; t < m; t += kConsumerWarps) {
    float v = 1.f;
    if (gate_vec != nullptr) {
      float dot = 0.f;
      const uint16_t *xt = x_l + static_cast<int64_t>(t) * s.din;
      for (int c = lane; c < s.din; c += 32)
        dot = fmaf(bf16_to_float(xt[c]), bf16_to_float(gate_vec[c]), dot);
      dot = warp_sum(dot);
      v = 1.0f / (1.0f + expf(-dot));
    }
    if (lane == 0) sscal[t] = v;
  }
}

// The classes of a grouped layer: phase A (gate/up) and phase B (down), routed then shared; the
// shared class's rows follow n_seg routed segments.
__device__ __forceinline__ void group_classes(const LayerShape &s, const LayerPtrs &w, int n_seg,
                                              GClass *ca, GClass *cb) {
  const int dsh = s.n_shared > 0 ? s.dff_shared : s.dff;
  ca[0] = GClass{true, false, s.dff, 0, w.gate, w.up, s.din, s.din * 2};
  ca[1] = GClass{true, true, dsh, static_cast<int64_t>(n_seg) * s.dff, w.sh_gate, w.sh_up, s.din,
                 s.din * 2};
  cb[0] = GClass{false, false, s.din, 0, w.down, w.down, s.dff, s.dff * 4};
  cb[1] = GClass{false, true, s.din, static_cast<int64_t>(n_seg) * s.din, w.sh_down, w.sh_down,
                 dsh, dsh * 4};
}

// One launch over L layers of m tokens, each selected expert streamed once per layer.  Barriers
// per layer: activations complete (3l + 1), partial outputs complete (3l + 2), layer output
// complete (3l + 3, before the next layer's ids are read).
template <int BR, int BD, int BSH>
__device__ void fused_grouped(const StackParams &p, uint8_t *dyn, uint64_t *full, uint64_t *empty,
                              StageDesc *sdesc, int *abort, SmemA &sm, LayerPtrs &wl,
                              LayerPtrs &wpr, int &stop, int tid) {
  GroupSmem &gs = *reinterpret_cast<GroupSmem *>(dyn);
  Plan rp;
  rp.nst = p.gp.nst;
  rp.stage_bytes = p.gp.stage_bytes;
  Ring r = make_ring(full, empty, dyn + kGroupSmemBytes, sdesc, rp, abort, p.err);
  const LayerShape &s = p.s;
  const int m = p.m, K = s.top_k, P = m * K;
  const uint32_t n = gridDim.x;
  const int y_stride = (K + s.n_shared) * s.din;
  if ((tid >> 5) >= kConsumerWarps) {
    const uint64_t pol = policy_evict_first();
    const int pl = tid - kConsumers;
    for (int l = 0; l < p.L; ++l) {
      producer_sync();  // every producer is done with the previous layer's copies
      if (pl == 0) {
        wpr = p.layers[l];
        if (l > 0) wait_count(p.bar, 3u * l * n, abort, p.err);  // the previous output
        stop = flag_abort(abort);
      }
      producer_sync();
      if (stop) break;
      const int32_t *ids = p.ids + static_cast<int64_t>(l) * P;
      const float *scores = p.scores + static_cast<int64_t>(l) * P;
      for (int q = pl; q < P; q += kProducers) {
        const int e = ids[q];
        gs.ids[q] = e;
        gs.scores[q] = scores[q];
        if (e < 0 || e >= s.n_experts) atomicOr(p.err, kDevErrBadId);
        if (p.ids_used != nullptr && blockIdx.x == 0) p.ids_used[static_cast<int64_t>(l) * P + q] = e;
      }
      producer_sync();
      route_invert_warp(gs.ids, P, s.n_experts, gs.rt, pl);
      for (int q = pl; q < gs.rt.n_pairs; q += kProducers) {
        const int pp = gs.rt.pairs[q];
        gs.pm[q] = static_cast<unsigned char>(pp / K);
        gs.pk[q] = static_cast<unsigned char>(pp % K);
      }
      build_segments(gs, p.gp.t_sub, pl);
      const int n_seg_s = s.n_shared * ((m + p.gp.t_sub - 1) / p.gp.t_sub);
      const uint16_t *x_l = p.x + static_cast<int64_t>(l) * m * s.din;
      GClass ca[2], cb[2];
      group_classes(s, wpr, gs.n_seg, ca, cb);
      Deferred none{false, true, 0, p.bar, 0};
      produce_g_phase(s, gs, gs.desc, gs.cnt, ca, p.gp.ga_r, p.gp.ga_s, gs.n_seg, n_seg_s, m,
                      p.gp.t_sub, p.gp.op_off, x_l, p.act, p.act_stride, none, r, pl, pol);
      if (flag_abort(abort)) break;
      Deferred df{true, false, 0, p.bar, (3u * l + 1u) * n};
      produce_g_phase(s, gs, gs.desc, gs.cnt + 2, cb, p.gp.gb_r, p.gp.gb_s, gs.n_seg, n_seg_s, m,
                      p.gp.t_sub, p.gp.op_off + 2, x_l, p.act, p.act_stride, df, r, pl, pol);
      if (flag_abort(abort)) break;
    }
    ring_drain(r, pl);  // never leave with copies in flight
    return;
  }

  for (int l = 0; l < p.L; ++l) {
    if (tid == 0) wl = p.layers[l];
    consumer_sync(kConsumers);
    const uint16_t *x_l = p.x + static_cast<int64_t>(l) * m * s.din;
    if (s.n_shared > 0) {
      shared_scalars_g(s, x_l, wl.gate_vec, m, gs.sscal, tid);
      consumer_sync(kConsumers);  // publishes sscal
    }
    GClass ca[2], cb[2];
    group_classes(s, wl, 0, ca, cb);  // the consumers use no row bases
    const GOut goa{p.act_stride, K * s.dff, s.dff, s.n_shared > 0 ? s.dff_shared : s.dff};
    consume_g_phase<BR, BSH, true>(s, gs, ca, p.gp.ga_r, p.gp.ga_s, goa, p.gp.op_off, gs.scores,
                                   p.act, r, sm, tid, !p.pool);
    consumers_grid_barrier(p.bar, (3u * l + 1u) * n, tid, abort, p.err);
    const GOut gob{y_stride, K * s.din, s.din, s.din};
    consume_g_phase<BD, BSH, false>(s, gs, cb, p.gp.gb_r, p.gp.gb_s, gob, p.gp.op_off + 2,
                                    gs.scores, p.y, r, sm, tid);
    consumers_grid_barrier(p.bar, (3u * l + 2u) * n, tid, abort, p.err);
    const void *resid;
    int resid_f32;
    if (l == 0) {
      resid = p.resid0;
      resid_f32 = p.resid0_f32;
    } else {
      resid = (l - 1) & 1 ? p.ping1 : p.ping0;
      resid_f32 = 1;
    }
    void *out;
    int out_f32;
    if (l == p.L - 1) {
      out = p.out;
      out_f32 = p.out_f32;
    } else {
      out = l & 1 ? p.ping1 : p.ping0;
      out_f32 = 1;
    }
    tail_g(s, gs.ids, m, p.y, y_stride, resid, resid_f32, out, out_f32, tid, p.pool != 0,
           gs.scores, gs.sscal);
    if (l < p.L - 1) consumers_grid_barrier(p.bar, (3u * l + 3u) * n, tid, abort, p.err);
  }
}

}  // namespace moe

