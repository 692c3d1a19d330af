// moe_kernels.cu -- the decode MoE kernels built from the phases of moe_phases.cuh:
//
//   gate_up_kernel   kernel A alone (phase A), launched with programmatic dependent launch
//   down_kernel      kernel B alone (phase B); its producer streams down weights before the
//                    activations are ready, its consumers wait for kernel A
//   fused_kernel     both phases for every layer and token of a stack in one cooperative launch:
//                    phase A, grid barrier (activations complete), phase B, grid barrier (layer
//                    output complete).  The producer warp streams phase B's down weights right
//                    after phase A's gate/up weights, so the down weights are in shared memory
//                    when the barrier opens; it starts the next layer's gate/up weights only
//                    after the barrier that completes the previous layer's output, because in a
//                    decoder a layer's expert ids depend on that output.
//
// The split into two GEMV phases with the activation in global memory between them follows
// "two-kernel decode-MoE that beats gather_qmm" (What changed, step 2); the fused launch keeps
// that split (every row is computed once by threads spread over all SMs) and replaces the kernel
// boundary with a device-wide barrier, which on GB300 also lets the second phase's weight stream
// run under the first phase's arithmetic.
#include "moe_grouped.cuh"

namespace moe {

__device__ __forceinline__ void init_ring(uint64_t *full, uint64_t *empty, int nst, int *abort) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);  // the producer's arrive.expect_tx; the bulk copies complete it
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort = 0;
    mbar_fence_init();
  }
}

// Shared state of the stage ring besides the stages themselves.
struct RingSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  StageDesc desc[kMaxStages];
  int cnt[2];              // phase A chunks of the current token: routed, shared
  int ids[kMaxTopK];       // the producer's copy of the current token's expert ids
  float scores[kMaxTopK];  // and scores
  int abort;
};

template <int BR, int BS>
__global__ void __launch_bounds__(kThreads, 1) gate_up_kernel(const GateUpParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) RingSmem rs;
  __shared__ SmemA sm;
  init_ring(rs.full, rs.empty, p.plan.nst, &rs.abort);
  // Token data (x, ids, scores) may come from the previous kernel on the stream.
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  Ring r = make_ring(rs.full, rs.empty, ring, rs.desc, p.plan, &rs.abort, p.err);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp >= kConsumerWarps) {
    const int pl = tid - kConsumers;
    producer_load_token(p.s, p.ids, p.scores, rs.ids, rs.scores, p.err, pl);
    produce_a<BR, BS>(p.s, p.w, p.plan.geo_r, p.plan.geo_s, rs.ids, rs.scores, rs.cnt, r, pl,
                      policy_evict_first());
    ring_drain(r, pl);
    return;
  }
  consume_a<BR, BS>(p.s, p.w, p.plan.geo_r, p.plan.geo_s, p.x, rs.cnt, p.act, r, sm, tid);
}

template <int BD, int BSD>
__global__ void __launch_bounds__(kThreads, 1) down_kernel(const DownParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) RingSmem rs;
  __shared__ SmemB sm;
  __shared__ float resid_s[kMaxRowsB];
  init_ring(rs.full, rs.empty, p.plan.nst, &rs.abort);
  pdl_launch_dependents();
  __syncthreads();
  Ring r = make_ring(rs.full, rs.empty, ring, rs.desc, p.plan, &rs.abort, p.err);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp >= kConsumerWarps) {
    // The ids were complete before kernel A started (A waits on its predecessor before it lets
    // this kernel launch), so the weight stream may start before the activations are ready.
    const int pl = tid - kConsumers;
    producer_load_token(p.s, p.ids, nullptr, rs.ids, rs.scores, p.err, pl);
    produce_b(p.s, p.w, p.plan.geo_b, rs.ids, r, pl, policy_evict_first());
    ring_drain(r, pl);
    return;
  }
  pdl_wait();  // the activations come from kernel A (and, in a stack, resid from the kernel
               // before it)
  load_resid_rows(p.s, p.resid, p.resid_f32, resid_s, tid);
  consumer_sync(kConsumers);  // publishes resid_s
  consume_b<BD, BSD>(p.s, p.plan.geo_b, rs.ids, p.act, resid_s, p.out, p.out_f32, r, sm, tid);
}

template <int BR, int BD, int BSH>
__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const StackParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) RingSmem rs;
  __shared__ SmemAB sm;
  __shared__ float resid_s[kMaxRowsB];
  __shared__ LayerPtrs wl;   // the consumers' copy of the current layer's pointers
  __shared__ LayerPtrs wpr;  // the producers' copy
  __shared__ int stop_pr;
  init_ring(rs.full, rs.empty, p.grouped ? p.gp.nst : p.plan.nst, &rs.abort);
  __syncthreads();
  const int tid = threadIdx.x, warp = tid >> 5;
  if (p.grouped) {
    fused_grouped<BR, BD, BSH>(p, ring, rs.full, rs.empty, rs.desc, &rs.abort, sm.a, wl, wpr,
                               stop_pr, tid);
    return;
  }
  Ring r = make_ring(rs.full, rs.empty, ring, rs.desc, p.plan, &rs.abort, p.err);
  const LayerShape &s = p.s;
  const uint32_t n = gridDim.x;
  const int64_t xs = static_cast<int64_t>(s.din), ks = s.top_k;

  if (warp >= kConsumerWarps) {
    // Producers work from their own shared copies of the layer's pointers and expert ids.
    const uint64_t pol = policy_evict_first();
    const int pl = tid - kConsumers;
    int pass = 0;
    for (int l = 0; l < p.L; ++l) {
      for (int t = 0; t < p.m; ++t, ++pass) {
        producer_sync();  // every producer is done with the previous pass's copies
        if (pl == 0) {
          wpr = p.layers[l];  // weight addresses do not depend on the ids: fetch them early
          // the previous (layer, token) output is complete before these ids are read
          if (pass > 0) wait_count(p.bar, 2u * pass * n, &rs.abort, p.err);
          stop_pr = flag_abort(&rs.abort);
        }
        producer_sync();      // orders every lane's id loads after lane 0's acquire
        if (stop_pr) break;
        const int64_t tok = static_cast<int64_t>(l) * p.m + t;
        producer_load_token(s, p.ids + tok * ks, p.scores + tok * ks, rs.ids, rs.scores, p.err,
                            pl);
        produce_a<BR, BSH>(s, wpr, p.plan.geo_r, p.plan.geo_s, rs.ids, rs.scores, rs.cnt, r, pl,
                           pol);
        produce_b(s, wpr, p.plan.geo_b, rs.ids, r, pl, pol);
      }
      if (stop_pr) break;
    }
    ring_drain(r, pl);  // never leave with copies in flight
    return;
  }

  int pass = 0;
  for (int l = 0; l < p.L; ++l) {
    if (tid == 0) wl = p.layers[l];
    consumer_sync(kConsumers);
    const LayerPtrs &w = wl;
    for (int t = 0; t < p.m; ++t, ++pass) {
      const int64_t tok = static_cast<int64_t>(l) * p.m + t;
      // The residual is an input (layer 0) or the previous layer's output, complete since the
      // last grid barrier: fetch it now, off the path between the two phases.
      if (l == 0)
        load_resid_rows(s, static_cast<const char *>(p.resid0) + t * xs * (p.resid0_f32 ? 4 : 2),
                        p.resid0_f32, resid_s, tid);
      else
        load_resid_rows(s, ((l - 1) & 1 ? p.ping1 : p.ping0) + t * xs, 1, resid_s, tid);
      consume_a<BR, BSH>(s, w, p.plan.geo_r, p.plan.geo_s, p.x + tok * xs, rs.cnt, p.act, r, sm.a,
                         tid);
      consumers_grid_barrier(p.bar, (2u * pass + 1u) * n, tid, &rs.abort, p.err);
      void *out;
      int out_f32;
      if (l == p.L - 1) {
        out = static_cast<char *>(p.out) + t * xs * (p.out_f32 ? 4 : 2);
        out_f32 = p.out_f32;
      } else {
        out = (l & 1 ? p.ping1 : p.ping0) + t * xs;
        out_f32 = 1;
      }
      consume_b<BD, BSH>(s, p.plan.geo_b, rs.ids, p.act, resid_s, out, out_f32, r, sm.b, tid);
      if (!(l == p.L - 1 && t == p.m - 1))
        consumers_grid_barrier(p.bar, (2u * pass + 2u) * n, tid, &rs.abort, p.err);
    }
  }
}

// ================================================================== debug unpack
template <int BITS>
__global__ void unpack_kernel(const uint8_t *packed, int64_t rows, int64_t cols, uint8_t *codes) {
  constexpr int V = Fmt<BITS>::kVecs, C = Fmt<BITS>::kCodes;
  const int64_t steps_per_row = cols / C;
  const int64_t n = rows * steps_per_row;
  for (int64_t s = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; s < n;
       s += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = s / steps_per_row, t = s - r * steps_per_row;
    const uint4 *vp = reinterpret_cast<const uint4 *>(packed + r * (cols * BITS / 8)) + t * V;
    uint4 v[V];
#pragma unroll
    for (int w = 0; w < V; ++w) v[w] = vp[w];
    uint32_t m[C];
    step_masks<BITS>(v, m);
#pragma unroll
    for (int j = 0; j < C; ++j)
      codes[r * cols + t * C + j] = static_cast<uint8_t>(m[j] >> code_offset<BITS>(j));
  }
}

// ================================================================== router
// One warp per token: lane l holds logits l, l + 32, ... (n_experts <= 1024).  k rounds of a warp
// arg-max on (logit, then lower id) pick the pool in order; the weights are the softmax of the
// picked logits, exponentials by lanes t < k and a fixed-order warp sum.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

__global__ void router_kernel(const float *logits, int m, int n_experts, int k, int32_t *ids,
                              float *scores) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= m) return;
  const float *lg = logits + static_cast<int64_t>(warp) * n_experts;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < n_experts ? lg[e] : 0.f;
  }
  uint32_t taken = 0u;       // bit j: expert lane + 32 j is in the pool
  float first = 0.f;         // the largest logit (first pick)
  float pick0 = 0.f, pick1 = 0.f;  // this lane's picks: pool positions lane and lane + 32
  int id0 = 0, id1 = 0;
  for (int t = 0; t < k; ++t) {
    float bv = 0.f;
    int bi = -1;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int e = lane + 32 * j;
      if (e < n_experts && !((taken >> j) & 1u) && (bi < 0 || better(v[j], e, bv, bi))) {
        bv = v[j];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi >= 0 && (bi < 0 || better(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (t == 0) first = bv;
    if (t == lane) {
      pick0 = bv;
      id0 = bi;
    } else if (t == lane + 32) {
      pick1 = bv;
      id1 = bi;
    }
  }
  const float w0 = lane < k ? expf(pick0 - first) : 0.f;
  const float w1 = lane + 32 < k ? expf(pick1 - first) : 0.f;
  const float sum = warp_sum(w0 + w1);
  int32_t *ids_t = ids + static_cast<int64_t>(warp) * k;
  float *sc_t = scores + static_cast<int64_t>(warp) * k;
  if (lane < k) {
    ids_t[lane] = id0;
    sc_t[lane] = w0 / sum;
  }
  if (lane + 32 < k) {
    ids_t[lane + 32] = id1;
    sc_t[lane + 32] = w1 / sum;
  }
}

// ================================================================== bounded waits
// Waits, with the kernels' own wait functions and a short limit, on a condition nothing will
// satisfy: kind 0 a grid-barrier count (a zeroed counter that nobody increments), kind 1 an
// mbarrier stage that no producer fills.  The wait gives up, records the time-out in the error
// word and the kernel returns normally.
__global__ void wait_timeout_kernel(int kind, uint32_t *cnt, int32_t *err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_s = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (kind == 0)
    wait_count(cnt, 1u, &abort_s, err, limit);
  else
    ring_wait(&bar, 0u, &abort_s, err, limit);
}

// ================================================================== debug route inversion
__global__ void route_invert_kernel(const int32_t *ids, int n, int n_experts, int32_t *out) {
  __shared__ Route rt;
  __shared__ int ids_s[kMaxPairs];
  for (int p = threadIdx.x; p < n; p += 32) ids_s[p] = ids[p];
  __syncwarp();
  route_invert_warp(ids_s, n, n_experts, rt, threadIdx.x);
  __syncwarp();
  const int U = rt.n_uniq;
  if (threadIdx.x == 0) out[0] = U;
  for (int u = threadIdx.x; u < U; u += 32) out[1 + u] = rt.uniq[u];
  for (int u = threadIdx.x; u <= U; u += 32) out[1 + U + u] = rt.offs[u];
  for (int q = threadIdx.x; q < rt.n_pairs; q += 32) out[2 + 2 * U + q] = rt.pairs[q];
}

// ================================================================== host side
static int fmt_codes(int bits) { return bits == 4 ? 32 : bits == 8 ? 16 : 64; }
static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Rows of `cols` codes, `rpt` rows per thread in a stage; the rows' partial sums are parked per
// warp, so R * warps-per-row must fit the parking area (kRedA entries, kBatchA rows).
static bool geom_rows(int cols, int bits, int rpt, GateUpGeom *g) {
  const int C = fmt_codes(bits);
  g->bits = bits;
  g->T = cols / C;
  if (g->T < 1 || g->T > kConsumers) return false;
  g->tpr = align_up(g->T, 32);
  g->groups = kConsumers / g->tpr;
  g->R = rpt * g->groups;
  g->rb = cols * bits / 8;
  g->sw = align_up(g->R * (cols / 64) * 2 + 14, 16);
  return g->R * (g->tpr / 32) <= kRedA && g->R <= kBatchA;
}

static bool geom_a(int din, int bits, GateUpGeom *g) {
  return geom_rows(din, bits, rows_per_thread_a_host(bits), g);
}

static int stage_a(const GateUpGeom &g) { return align_up(2 * g.R * g.rb + 4 * g.sw, 128); }

static bool geom_b(const LayerShape &s, int bits_d, int bits_sd, DownGeom *g) {
  const int CR = fmt_codes(bits_d), CS = fmt_codes(bits_sd);
  const int cmax = CR > CS ? CR : CS;
  g->bits_r = bits_d;
  g->bits_s = bits_sd;
  g->rb_r = s.dff * bits_d / 8;
  g->rb_s = s.dff_shared * bits_sd / 8;
  g->G_r = s.dff / 64;
  g->G_s = s.dff_shared / 64;
  g->spr_r = s.dff / CR;
  g->spr_s = s.n_shared > 0 ? s.dff_shared / CS : 0;
  g->T_r = s.top_k * g->spr_r;
  g->T_s = s.n_shared * g->spr_s;
  const int T = g->T_r + g->T_s;
  g->tpr = align_up(T, 32) < kConsumers ? align_up(T, 32) : kConsumers;
  g->groups = kConsumers / g->tpr;
  g->spt = (T + g->tpr - 1) / g->tpr;
  const int sptmax = kMaxActRegs / cmax > 0 ? kMaxActRegs / cmax : 1;
  if (g->spt < 1 || g->spt > sptmax) return false;
  const int row_bytes =
      s.top_k * (g->rb_r + 4 * g->G_r) + s.n_shared * (g->rb_s + 4 * g->G_s);
  const int rmax = rows_per_thread_b_max(bits_d, bits_sd);
  int rpt = (64 * 1024) / (g->groups * row_bytes);
  rpt = rpt < 1 ? 1 : (rpt > rmax ? rmax : rpt);
  g->R = rpt * g->groups;
  g->sw_r = align_up(g->R * g->G_r * 2 + 14, 16);
  g->sw_s = s.n_shared > 0 ? align_up(g->R * g->G_s * 2 + 14, 16) : 0;
  g->codes_bytes = g->R * (s.top_k * g->rb_r + s.n_shared * g->rb_s);
  return g->R <= kMaxRowsB;  // partial sums are parked per CTA row, not per stage
}

static int stage_b(const LayerShape &s, const DownGeom &g) {
  return align_up(g.codes_bytes + 2 * (s.top_k * g.sw_r + s.n_shared * g.sw_s), 128);
}

// bits_sh is the shared experts' code width; a layer without shared experts passes bits_d, so
// that phase B's register sizing (which depends on both widths) matches the plan.
bool make_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, Plan *plan) {
  if (!geom_a(s.din, bits_gu, &plan->geo_r) || !geom_a(s.din, bits_sh, &plan->geo_s)) return false;
  if (!geom_b(s, bits_d, bits_sh, &plan->geo_b)) return false;
  int st = stage_b(s, plan->geo_b);
  if (s.top_k > 0 && stage_a(plan->geo_r) > st) st = stage_a(plan->geo_r);
  if (s.n_shared > 0 && stage_a(plan->geo_s) > st) st = stage_a(plan->geo_s);
  int n = kRingBytes / st;
  if (n > kMaxStages) n = kMaxStages;
  if (n < 2) return false;
  plan->nst = n;
  plan->stage_bytes = st;
  plan->smem = static_cast<size_t>(n) * st;
  return true;
}

bool make_group_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, int m,
                     GroupPlan *gp) {
  if (m < 2 || m > kMaxGroupTokens || m * s.top_k > kMaxPairs || s.n_experts > kMaxGroupExperts)
    return false;
  const int dsh = s.n_shared > 0 ? s.dff_shared : s.dff;
  if (!geom_a(s.din, bits_gu, &gp->ga_r) || !geom_a(s.din, bits_sh, &gp->ga_s) ||
      !geom_rows(s.dff, bits_d, rows_per_thread_gb_host(bits_d), &gp->gb_r) ||
      !geom_rows(dsh, bits_sh, rows_per_thread_gb_host(bits_sh), &gp->gb_s))
    return false;
  const GateUpGeom *g[4] = {&gp->ga_r, &gp->ga_s, &gp->gb_r, &gp->gb_s};
  const int op_bytes[4] = {s.din * 2, s.din * 2, s.dff * 4, dsh * 4};
  for (int c = 0; c < 4; ++c) {
    const int nproj = c < 2 ? 2 : 1;
    gp->op_off[c] = align_up(nproj * g[c]->R * g[c]->rb + 2 * nproj * g[c]->sw, 16);
  }
  // as many pairs per stage as keep at least four stages in the ring (at least one pair)
  const int ring_bytes = kRingBytes - kGroupSmemBytes;  // the route state precedes the ring
  int t = m < 8 ? m : 8, st = 0;
  for (; t >= 1; --t) {
    st = 0;
    for (int c = 0; c < 4; ++c) {
      const int b = align_up(gp->op_off[c] + t * op_bytes[c], 128);
      st = b > st ? b : st;
    }
    if (st * 4 <= ring_bytes) break;
  }
  if (t < 1) {
    t = 1;
    st = 0;
    for (int c = 0; c < 4; ++c) {
      const int b = align_up(gp->op_off[c] + op_bytes[c], 128);
      st = b > st ? b : st;
    }
  }
  int n = ring_bytes / st;
  if (n > kMaxStages) n = kMaxStages;
  if (n < 2) return false;
  gp->t_sub = t;
  gp->nst = n;
  gp->stage_bytes = st;
  gp->smem = static_cast<size_t>(kGroupSmemBytes) + static_cast<size_t>(n) * st;
  return true;
}

template <typename Kern, typename P>
static cudaError_t launch(Kern kern, const P &p, int grid, size_t smem, cudaStream_t stream,
                          bool pdl, bool cooperative) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

#define MOE_BITS_SWITCH(B, NAME, ...)                       \
  switch (B) {                                              \
    case 4: { constexpr int NAME = 4; __VA_ARGS__; break; } \
    case 6: { constexpr int NAME = 6; __VA_ARGS__; break; } \
    case 8: { constexpr int NAME = 8; __VA_ARGS__; break; } \
    default: return cudaErrorInvalidValue;                  \
  }

cudaError_t launch_gate_up(const GateUpParams &p, int grid, cudaStream_t stream, bool pdl) {
  MOE_BITS_SWITCH(p.plan.geo_r.bits, BR, MOE_BITS_SWITCH(p.plan.geo_s.bits, BS,
      return launch(gate_up_kernel<BR, BS>, p, grid, p.plan.smem, stream, pdl, false)));
  return cudaErrorInvalidValue;
}

cudaError_t launch_down(const DownParams &p, int grid, cudaStream_t stream, bool pdl) {
  MOE_BITS_SWITCH(p.plan.geo_b.bits_r, BD, MOE_BITS_SWITCH(p.plan.geo_b.bits_s, BSD,
      return launch(down_kernel<BD, BSD>, p, grid, p.plan.smem, stream, pdl, false)));
  return cudaErrorInvalidValue;
}

// shared-expert bits as the kernels see them: the routed ones when there is no shared expert
static int sh_bits(const Plan &plan) { return plan.geo_s.bits; }

cudaError_t launch_fused(const StackParams &p, int grid, cudaStream_t stream) {
  const size_t smem = p.grouped ? p.gp.smem : p.plan.smem;
  MOE_BITS_SWITCH(p.plan.geo_r.bits, BR, MOE_BITS_SWITCH(p.plan.geo_b.bits_r, BD,
      MOE_BITS_SWITCH(sh_bits(p.plan), BSH,
          return launch(fused_kernel<BR, BD, BSH>, p, grid, smem, stream, false, true))));
  return cudaErrorInvalidValue;
}

cudaError_t prepare_kernels(int smem_optin, int bits_gu, int bits_d, int bits_sh,
                            int *dyn_limit) {
  // The attribute is global to a kernel instance: set it to the most the device allows next to
  // the kernel's static shared memory, so one handle can never lower it below what another
  // handle launches with.  *dyn_limit is the smallest of the three kernels' limits.
  cudaError_t e = cudaSuccess;
  int lim = smem_optin;
  auto set = [&](const void *fn) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return;
    const int dyn = smem_optin - static_cast<int>(fa.sharedSizeBytes);
    if (dyn < lim) lim = dyn;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  };
  MOE_BITS_SWITCH(bits_gu, BR, MOE_BITS_SWITCH(bits_sh, BS,
      set(reinterpret_cast<const void *>(gate_up_kernel<BR, BS>))));
  if (e != cudaSuccess) return e;
  MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sh, BSD,
      set(reinterpret_cast<const void *>(down_kernel<BD, BSD>))));
  if (e != cudaSuccess) return e;
  MOE_BITS_SWITCH(bits_gu, BR, MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sh, BSH,
      set(reinterpret_cast<const void *>(fused_kernel<BR, BD, BSH>)))));
  *dyn_limit = lim;
  return e;
}

// Largest grid the fused kernel can run with every CTA resident (0 on error).
int fused_grid_limit(const Plan &plan, int bits_gu, int bits_d, int bits_sh) {
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  cudaError_t e = cudaErrorInvalidValue;
  switch (bits_gu * 100 + bits_d * 10 + bits_sh) {
#define MOE_OCC(a, b, c)                                                                        \
  case a * 100 + b * 10 + c:                                                                   \
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_kernel<a, b, c>, kThreads, \
                                                      plan.smem);                              \
    break;
    MOE_OCC(4, 4, 4) MOE_OCC(4, 4, 6) MOE_OCC(4, 4, 8) MOE_OCC(4, 6, 4) MOE_OCC(4, 6, 6)
    MOE_OCC(4, 6, 8) MOE_OCC(4, 8, 4) MOE_OCC(4, 8, 6) MOE_OCC(4, 8, 8)
    MOE_OCC(6, 4, 4) MOE_OCC(6, 4, 6) MOE_OCC(6, 4, 8) MOE_OCC(6, 6, 4) MOE_OCC(6, 6, 6)
    MOE_OCC(6, 6, 8) MOE_OCC(6, 8, 4) MOE_OCC(6, 8, 6) MOE_OCC(6, 8, 8)
    MOE_OCC(8, 4, 4) MOE_OCC(8, 4, 6) MOE_OCC(8, 4, 8) MOE_OCC(8, 6, 4) MOE_OCC(8, 6, 6)
    MOE_OCC(8, 6, 8) MOE_OCC(8, 8, 4) MOE_OCC(8, 8, 6) MOE_OCC(8, 8, 8)
#undef MOE_OCC
    default:
      break;
  }
  if (e != cudaSuccess) return 0;
  return per_sm * sms;
}

cudaError_t launch_unpack(const uint8_t *packed, int64_t rows, int64_t cols, int bits,
                          uint8_t *codes, cudaStream_t stream) {
  const int64_t steps = rows * (cols / fmt_codes(bits));
  int grid = (int)((steps + 255) / 256);
  grid = grid < 1 ? 1 : (grid > 65535 ? 65535 : grid);
  MOE_BITS_SWITCH(bits, B, unpack_kernel<B><<<grid, 256, 0, stream>>>(packed, rows, cols, codes));
  return cudaGetLastError();
}

cudaError_t launch_router(const float *logits, int m, int n_experts, int k, int32_t *ids,
                          float *scores, cudaStream_t stream) {
  const int warps_per_block = 8;
  const int grid = (m + warps_per_block - 1) / warps_per_block;
  router_kernel<<<grid, warps_per_block * 32, 0, stream>>>(logits, m, n_experts, k, ids, scores);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(int kind, uint32_t *cnt, int32_t *err, long long limit,
                                cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(kind, cnt, err, limit);
  return cudaGetLastError();
}

cudaError_t launch_route_invert(const int32_t *ids, int m, int k, int n_experts, int32_t *out,
                                cudaStream_t stream) {
  route_invert_kernel<<<1, 32, 0, stream>>>(ids, m * k, n_experts, out);
  return cudaGetLastError();
}

}  // namespace moe
