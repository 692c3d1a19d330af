// moe_kernels.cu -- host side of the decode MoE kernels: geometry and plans, and the dispatch
// to the kernels of moe_fused.cuh (instantiated per gate/up code width in moe_kernels_g4.cu,
// moe_kernels_g6.cu and moe_kernels_g8.cu); plus the small kernels (debug unpack, router, bounded
// waits, debug route inversion).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "moe_grouped.cuh"

namespace moe {

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

// ================================================================== column-block-major down copy
// out_codes[e][jb][i] = word jb of canonical row (e, i); out_sb[e][g][i] = (scale, bias)[e][i][g].
// Consecutive threads write consecutive rows i.
__global__ void repack_down_kernel(const uint32_t *codes, const __half *scales,
                                   const __half *biases, int experts, int din, int words,
                                   int groups, uint32_t *out_codes, __half2 *out_sb) {
  const int64_t nc = static_cast<int64_t>(experts) * words * din;
  const int64_t ns = static_cast<int64_t>(experts) * groups * din;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < nc;
       x += stride) {
    const int64_t i = x % din, t = x / din;
    const int64_t jb = t % words, e = t / words;
    out_codes[x] = codes[(e * din + i) * words + jb];
  }
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < ns;
       x += stride) {
    const int64_t i = x % din, t = x / din;
    const int64_t g = t % groups, e = t / groups;
    const int64_t src = (e * din + i) * groups + g;
    out_sb[x] = __halves2half2(scales[src], biases[src]);
  }
}

// Gate/up records: one thread per 16-byte word of a record's codes, then one per fp16 of its
// scale/bias runs (and the padding, zeroed).
__global__ void repack_gate_up_kernel(const uint4 *g_codes, const __half *g_scales,
                                      const __half *g_biases, const uint4 *u_codes,
                                      const __half *u_scales, const __half *u_biases,
                                      int64_t records, int rb16, int G, int rec, uint8_t *out) {
  const int codes_bytes = rec - ((8 * G + 15) / 16) * 16;  // the two code rows
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t nc = records * 2 * rb16;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < nc;
       x += stride) {
    const int64_t r = x / (2 * rb16);
    const int w = static_cast<int>(x - r * 2 * rb16);
    const uint4 v = w < rb16 ? g_codes[r * rb16 + w] : u_codes[r * rb16 + (w - rb16)];
    reinterpret_cast<uint4 *>(out + r * rec)[w] = v;
  }
  const int tail = (rec - codes_bytes) / 2;  // fp16 slots after the codes
  const int64_t ns = records * tail;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < ns;
       x += stride) {
    const int64_t r = x / tail;
    const int k = static_cast<int>(x - r * tail);
    const int run = k / G, g = k - run * G;
    __half v = __float2half(0.f);
    if (run < 4) {
      const __half *src = run == 0 ? g_scales : run == 1 ? g_biases : run == 2 ? u_scales : u_biases;
      v = src[r * G + g];
    }
    reinterpret_cast<__half *>(out + r * rec + codes_bytes)[k] = v;
  }
}

// Column-block-major copy of 6-bit down projections, widened to bytes: word (jb, i) holds codes
// 4 jb .. 4 jb + 3 of row i, one per byte (the canonical row packs 16 codes in 3 words, LSB first).
__global__ void repack_down6_kernel(const uint32_t *codes, int experts, int din, int dff,
                                    uint32_t *out_codes) {
  const int words = dff * 6 / 32;  // canonical words per row
  const int nblk = dff / 4;
  const int64_t nc = static_cast<int64_t>(experts) * nblk * din;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < nc;
       x += stride) {
    const int64_t i = x % din, t = x / din;
    const int64_t jb = t % nblk, e = t / nblk;
    const uint32_t *row = codes + (e * din + i) * words;
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t bit = (jb * 4 + k) * 6;
      const int wi = static_cast<int>(bit >> 5), sh = static_cast<int>(bit & 31);
      uint64_t v = row[wi];
      if (sh + 6 > 32) v |= static_cast<uint64_t>(row[wi + 1]) << 32;
      w |= static_cast<uint32_t>((v >> sh) & 63u) << (8 * k);
    }
    out_codes[x] = w;
  }
}

// Gate/up records of 6-bit rows, codes widened to bytes (the scale/bias runs are written by
// repack_gate_up_kernel with no code words): one thread per byte-quad of a record's codes.
__global__ void repack_gate_up6_kernel(const uint32_t *g_codes, const uint32_t *u_codes,
                                       int64_t records, int din, int rec, uint8_t *out) {
  const int words = din * 6 / 32;  // canonical words per row
  const int quads = din / 4;       // 32-bit words of a widened row
  const int64_t n = records * 2 * quads;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
       x += stride) {
    const int64_t r = x / (2 * quads);
    const int q = static_cast<int>(x - r * 2 * quads);
    const bool up = q >= quads;
    const int qq = up ? q - quads : q;
    const uint32_t *row = (up ? u_codes : g_codes) + r * words;
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int bit = (qq * 4 + k) * 6;
      const int wi = bit >> 5, sh = bit & 31;
      uint64_t v = row[wi];
      if (sh + 6 > 32) v |= static_cast<uint64_t>(row[wi + 1]) << 32;
      w |= static_cast<uint32_t>((v >> sh) & 63u) << (8 * k);
    }
    reinterpret_cast<uint32_t *>(out + r * rec)[q] = w;
  }
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
  if (n > kMaxRowStages) n = kMaxRowStages;
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
  if (n > kMaxRowStages) n = kMaxRowStages;
  if (n < 2) return false;
  gp->t_sub = t;
  gp->nst = n;
  gp->stage_bytes = st;
  gp->smem = static_cast<size_t>(kGroupSmemBytes) + static_cast<size_t>(n) * st;
  return true;
}

// Phase-A geometry of the column split: R (gate, up) row pairs per stage, about 32 KB of codes,
// each pair taken by one warp per 1024 columns (a lane owns 32 columns of both rows).
static bool geom_cols_a(int din, int bits, GateUpGeom *g) {
  if (bits != 4 && bits != 8) return false;
  const int nk = din / 32, wpr = (nk + 31) / 32;
  if (din < 64 || wpr > 4) return false;
  g->bits = bits;
  g->rb = col_record_bytes(din, bits);   // a stage holds R records
  int R = 1;
  while ((R * 2) * 2 * (din * bits / 8) <= 32 * 1024 && R * 2 * wpr <= kConsumerWarps) R *= 2;
  if (R < 2) return false;  // a warp takes two tasks of the same lane set: R even
  g->R = R;
  g->T = nk;
  g->tpr = 32 * wpr;
  g->groups = kConsumerWarps / (R * wpr);
  g->sw = 0;
  return true;
}

// What the columns [u0, u1) cost the CTA that owns them in one layer when every slot names a valid
// expert: its stages (gate/up chunks, then down stages: unpacked, or packed when `pack`) in the
// high bits, its bytes in the low 40.  -1 when the range breaks a per-CTA limit.
static int64_t col_cost(const LayerShape &s, const ColPlan &cp, const Plan &plan, int64_t u0,
                        int64_t u1, bool pack) {
  if (u1 < u0 || u1 - u0 > kMaxColsCta) return -1;
  ColPiece pc[kMaxColPieces];
  int nbk = 0;
  const int np = col_pieces(s.top_k, s.dff, s.n_shared, s.dff_shared, cp.cb_r, cp.cb_s, u0, u1,
                            pc, &nbk);
  if (np < 0) return -1;
  short sg[kMaxColChunks], jj[kMaxColChunks], nn[kMaxColChunks], uu[kMaxColChunks];
  int nrt = 0;
  const int nck = col_chunks(s.top_k, s.dff, s.n_shared, s.dff_shared, plan.geo_r.R,
                             plan.geo_s.R, u0, u1, sg, jj, nn, uu, &nrt);
  if (nck < 0) return -1;
  int down = 0;
  if (pack) {
    down = (nbk + np + cp.nbs) / (cp.nbs + 1);  // every slot of a stage filled
  } else {
    for (int i = 0; i < np; ++i) down += (pc[i].nb + cp.nbs - 1) / cp.nbs;
  }
  int64_t bytes = static_cast<int64_t>(nbk + np) * s.din * 4;  // code blocks and records
  for (int i = 0; i < nck; ++i) bytes += static_cast<int64_t>(nn[i]) * (i < nrt ? cp.rec_r : cp.rec_s);
  return (static_cast<int64_t>(nck + down) << 40) | bytes;
}

// The CTAs' column ranges of an unpacked plan (cp->bounds): starting from the even split, each
// inner boundary moves at most kColSlack columns so that the costliest CTA (stages first, then
// bytes) costs as little as possible, and among those splits the total bytes (blocks read by two
// CTAs, records of cut groups) are least.  A layer waits for its slowest CTA, and a CTA whose
// columns end a few columns into a new group carries one more down stage than its neighbours: the
// even split of the qwen3 8-bit shape (768 columns a slot over 19 CTAs) gives 4 CTAs of every 19
// five down stages, this one none.  false when no split within the slack keeps every CTA inside
// the limits.
constexpr int kColSlack = 16;
static bool col_balance(const LayerShape &s, ColPlan *cp, const Plan &plan, int grid) {
  const int64_t U = static_cast<int64_t>(s.top_k) * s.dff +
                    static_cast<int64_t>(s.n_shared) * s.dff_shared;
  const int D = static_cast<int>(std::min<int64_t>(kColSlack, U / grid / 2));
  const int W = 2 * D + 1;
  const int64_t kInf = INT64_MAX;
  // boundary c sits at U c / grid + (i - D), window slot i; boundaries 0 and grid are fixed
  auto pos = [&](int c, int i) -> int64_t {
    const int64_t v = U * c / grid + (i - D);
    return (c == 0 || c == grid || v < 0 || v > U) ? -1 : v;
  };
  auto slot_ok = [&](int c, int i) {
    return (c == 0 || c == grid) ? i == D : pos(c, i) >= 0;
  };
  auto at = [&](int c, int i) -> int64_t { return (c == 0) ? 0 : (c == grid ? U : pos(c, i)); };
  std::vector<int64_t> cost(static_cast<size_t>(grid) * W * W, -1);
  for (int c = 0; c < grid; ++c)
    for (int i = 0; i < W; ++i) {
      if (!slot_ok(c, i)) continue;
      for (int j = 0; j < W; ++j)
        if (slot_ok(c + 1, j) && at(c + 1, j) >= at(c, i))
          cost[(static_cast<size_t>(c) * W + i) * W + j] =
              col_cost(s, *cp, plan, at(c, i), at(c + 1, j), false);
    }
  // pass 1: the least possible cost of the costliest CTA
  std::vector<int64_t> best(static_cast<size_t>(grid + 1) * W, kInf);
  best[static_cast<size_t>(grid) * W + D] = 0;
  for (int c = grid - 1; c >= 0; --c)
    for (int i = 0; i < W; ++i)
      for (int j = 0; j < W; ++j) {
        const int64_t k = cost[(static_cast<size_t>(c) * W + i) * W + j];
        const int64_t rest = best[static_cast<size_t>(c + 1) * W + j];
        if (k < 0 || rest == kInf) continue;
        int64_t &b = best[static_cast<size_t>(c) * W + i];
        b = std::min(b, std::max(k, rest));
      }
  const int64_t M = best[D];
  if (M == kInf) return false;
  // pass 2: within that bound, the least total bytes
  const int64_t mask = (int64_t{1} << 40) - 1;
  std::vector<int64_t> sum(static_cast<size_t>(grid + 1) * W, kInf);
  std::vector<int> next(static_cast<size_t>(grid) * W, -1);
  sum[static_cast<size_t>(grid) * W + D] = 0;
  for (int c = grid - 1; c >= 0; --c)
    for (int i = 0; i < W; ++i)
      for (int j = 0; j < W; ++j) {
        const int64_t k = cost[(static_cast<size_t>(c) * W + i) * W + j];
        const int64_t rest = sum[static_cast<size_t>(c + 1) * W + j];
        if (k < 0 || k > M || rest == kInf) continue;
        const int64_t v = rest + (k & mask);
        if (v < sum[static_cast<size_t>(c) * W + i]) {
          sum[static_cast<size_t>(c) * W + i] = v;
          next[static_cast<size_t>(c) * W + i] = j;
        }
      }
  if (sum[D] == kInf) return false;
  int i = D;
  for (int c = 0; c < grid; ++c) {
    cp->bounds[c] = static_cast<int32_t>(at(c, i));
    i = next[static_cast<size_t>(c) * W + i];
  }
  cp->bounds[grid] = static_cast<int32_t>(U);
  return true;
}

bool make_col_plan(const LayerShape &s, int bits_gu, int bits_d, int bits_sh, int grid,
                   int ring_bytes, ColPlan *cp, Plan *plan) {
  const bool sh = s.n_shared > 0;
  bits_gu = col_gu_bits(bits_gu);   // 6-bit codes are stored widened to bytes
  const int bits_sh_gu = col_gu_bits(bits_sh);
  bits_d = col_down_bits(bits_d);
  bits_sh = col_down_bits(bits_sh);
  if (grid < 1 || grid > kColMaxGrid || (bits_d != 4 && bits_d != 8) ||
      (sh && bits_sh != 4 && bits_sh != 8))
    return false;
  if (s.din > 4 * 2 * kConsumers || s.din % 64) return false;  // two row quads per thread
  if (s.dff > 32767 || s.dff_shared > 32767) return false;    // chunk rows are 16-bit
  if (!geom_cols_a(s.din, bits_gu, &plan->geo_r) || !geom_cols_a(s.din, bits_sh_gu, &plan->geo_s))
    return false;
  cp->cb_r = 32 / bits_d;
  cp->cb_s = sh ? 32 / bits_sh : cp->cb_r;
  const int blk = s.din * 4;  // one column block of all din rows
  int sa = 0;
  if (s.top_k > 0) sa = align_up(plan->geo_r.R * plan->geo_r.rb, 128);
  if (sh && align_up(plan->geo_s.R * plan->geo_s.rb, 128) > sa)
    sa = align_up(plan->geo_s.R * plan->geo_s.rb, 128);
  cp->rec_r = plan->geo_r.rb;
  cp->rec_s = plan->geo_s.rb;
  int nbs = sa / blk - 1;
  nbs = nbs < 1 ? 1 : (nbs > 16 ? 16 : nbs);
  int st = align_up((nbs + 1) * blk, 128);
  st = st > sa ? st : sa;
  int n = ring_bytes / st;
  if (n > kMaxStages) n = kMaxStages;
  if (n < 2) return false;
  cp->nbs = nbs;
  cp->ro = 4 * ((s.din / 4 + grid - 1) / grid);   // the owner's row quads
  if (cp->ro > kMaxOwnRows) return false;
  const int64_t U = (int64_t)s.top_k * s.dff + (int64_t)s.n_shared * s.dff_shared;
  if ((U + grid - 1) / grid > kMaxColsCta || U > (int64_t{1} << 30)) return false;
  // the column ranges, balanced for the unpacked stages; the stages of the costliest CTA decide
  // the prefetch and the packing
  if (!col_balance(s, cp, *plan, grid)) return false;
  int max_stages = 0;
  for (int c = 0; c < grid; ++c)
    max_stages = std::max(max_stages, static_cast<int>(
                              col_cost(s, *cp, *plan, cp->bounds[c], cp->bounds[c + 1], false) >> 40));
  // The prefetches queue on the bulk-copy engine ahead of the ring's next copies: worth it only
  // for a short overflow (measured: qwen3 8-bit, 10-11 stages on a 6-slot ring, +1%; dots-like,
  // 20-30 stages, -17%).
  cp->prefetch = max_stages <= 2 * n;
  // Packing pays where a piece's record would otherwise take a stage of its own next to one or
  // two blocks and nothing is prefetched (measured, prefetch off: dots-like stack, 2-slot stages,
  // +11%; qwen3 8-bit, 4-slot stages, -3%; with the prefetch on, packing measured slower).
  cp->pack = nbs <= 2 && !cp->prefetch;
  // A packed plan keeps the even split (measured, dots-like stack: 619.7 tok/s even, 615.4 with
  // the unpacked balance, 606.0 with a split weighted for the packed stages, which lowered its
  // costliest CTA from 30 stages to 29; the unpacked plans gained 0.6-4.6% from the balance).
  if (cp->pack) {
    for (int c = 0; c <= grid; ++c) cp->bounds[c] = static_cast<int32_t>(U * c / grid);
    for (int c = 0; c < grid; ++c)
      if (col_cost(s, *cp, *plan, cp->bounds[c], cp->bounds[c + 1], true) < 0) return false;
  }
  std::memset(&plan->geo_b, 0, sizeof plan->geo_b);
  plan->nst = n;
  plan->stage_bytes = st;
  plan->smem = static_cast<size_t>(n) * st;
  return true;
}

#define MOE_BITS_SWITCH(B, NAME, ...)                       \
  switch (B) {                                              \
    case 4: { constexpr int NAME = 4; __VA_ARGS__; break; } \
    case 6: { constexpr int NAME = 6; __VA_ARGS__; break; } \
    case 8: { constexpr int NAME = 8; __VA_ARGS__; break; } \
    default: return cudaErrorInvalidValue;                  \
  }

// Two translation units per gate/up code width hold the launchable kernels (moe_fused.cuh):
// moe_kernels_g<B>.cu (kernel A, kernel B, fused token kernels), moe_grouped_g<B>.cu (fused
// grouped kernels).
#define MOE_FAMILY_DECL(B)                                                                    \
  cudaError_t launch_fused_g##B(const StackParams &, int, size_t, cudaStream_t);              \
  cudaError_t launch_gate_up_g##B(const GateUpParams &, int, cudaStream_t, bool);             \
  cudaError_t launch_down_g##B(const DownParams &, int, cudaStream_t, bool);                  \
  cudaError_t prepare_g##B(int, int, int, bool, int *);                                       \
  cudaError_t fused_occupancy_g##B(int, int, size_t, int *);                                 \
  cudaError_t launch_grouped_g##B(const StackParams &, int, size_t, cudaStream_t);            \
  cudaError_t prepare_grouped_g##B(int, int, int, int *);                                     \
  cudaError_t grouped_occupancy_g##B(int, int, size_t, int *);                               \
  cudaError_t launch_cols_g##B(const StackParams &, int, cudaStream_t);                       \
  cudaError_t prepare_cols_g##B(int, int, int, int *);                                        \
  cudaError_t cols_occupancy_g##B(int, int, size_t, int *);
MOE_FAMILY_DECL(4)
MOE_FAMILY_DECL(6)
MOE_FAMILY_DECL(8)
#undef MOE_FAMILY_DECL

#define MOE_FAMILY_CALL(B, FN, ...)                   \
  switch (B) {                                        \
    case 4: return FN##_g4(__VA_ARGS__);              \
    case 6: return FN##_g6(__VA_ARGS__);              \
    case 8: return FN##_g8(__VA_ARGS__);              \
    default: return cudaErrorInvalidValue;            \
  }

cudaError_t launch_gate_up(const GateUpParams &p, int grid, cudaStream_t stream, bool pdl) {
  MOE_FAMILY_CALL(p.plan.geo_r.bits, launch_gate_up, p, grid, stream, pdl);
}

cudaError_t launch_down(const DownParams &p, int grid, cudaStream_t stream, bool pdl) {
  MOE_FAMILY_CALL(p.plan.geo_b.bits_r, launch_down, p, grid, stream, pdl);
}

cudaError_t launch_fused(const StackParams &p, int grid, cudaStream_t stream) {
  if (p.grouped) {
    MOE_FAMILY_CALL(p.plan.geo_r.bits, launch_grouped, p, grid, p.gp.smem, stream);
  }
  MOE_FAMILY_CALL(p.plan.geo_r.bits, launch_fused, p, grid, p.plan.smem, stream);
}

// Sets every kernel's shared-memory limit; *dyn_limit is the smallest of them.
cudaError_t prepare_kernels(int smem_optin, int bits_gu, int bits_d, int bits_sh,
                            int *dyn_limit) {
  int lim = smem_optin;
  cudaError_t e;
  auto fam = [&](int b, int bd, int bs, bool down) -> cudaError_t {
    MOE_FAMILY_CALL(b, prepare, smem_optin, bd, bs, down, &lim);
  };
  auto grp = [&]() -> cudaError_t {
    MOE_FAMILY_CALL(bits_gu, prepare_grouped, smem_optin, bits_d, bits_sh, &lim);
  };
  e = fam(bits_gu, bits_d, bits_sh, false);
  if (e == cudaSuccess) e = fam(bits_d, bits_d, bits_sh, true);
  if (e == cudaSuccess) e = grp();
  *dyn_limit = lim;
  return e;
}

// Largest grid the fused kernel can run with every CTA resident (0 on error).
int fused_grid_limit(const Plan &plan, int bits_gu, int bits_d, int bits_sh) {
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  per_sm = 1 << 30;
  auto occ = [&]() -> cudaError_t {
    MOE_FAMILY_CALL(bits_gu, fused_occupancy, bits_d, bits_sh, plan.smem, &per_sm);
  };
  auto occ_g = [&]() -> cudaError_t {
    MOE_FAMILY_CALL(bits_gu, grouped_occupancy, bits_d, bits_sh, plan.smem, &per_sm);
  };
  if (occ() != cudaSuccess || occ_g() != cudaSuccess) return 0;
  return per_sm * sms;
}
cudaError_t launch_cols(const StackParams &p, int grid, cudaStream_t stream) {
  MOE_FAMILY_CALL(p.plan.geo_r.bits, launch_cols, p, grid, stream);
}

cudaError_t prepare_cols(int smem_optin, int bits_gu, int bits_d, int bits_sh, int *dyn_limit) {
  int lim = smem_optin;
  auto fam = [&]() -> cudaError_t {
    MOE_FAMILY_CALL(bits_gu, prepare_cols, smem_optin, bits_d, bits_sh, &lim);
  };
  const cudaError_t e = fam();
  *dyn_limit = lim;
  return e;
}

int cols_grid_limit(size_t smem, int bits_gu, int bits_d, int bits_sh) {
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  auto occ = [&]() -> cudaError_t {
    MOE_FAMILY_CALL(bits_gu, cols_occupancy, bits_d, bits_sh, smem, &per_sm);
  };
  if (occ() != cudaSuccess) return 0;
  return per_sm * sms;
}
#undef MOE_FAMILY_CALL

cudaError_t launch_repack_gate_up(const uint8_t *g_codes, const __half *g_scales,
                                  const __half *g_biases, const uint8_t *u_codes,
                                  const __half *u_scales, const __half *u_biases, int experts,
                                  int rows, int din, int bits, uint8_t *out, cudaStream_t stream) {
  if (experts < 1 || rows < 1) return cudaSuccess;
  const int wb = col_gu_bits(bits);               // stored width
  const int rb = din * wb / 8, G = din / 64;
  const int rec = col_record_bytes(din, wb);
  const int64_t records = static_cast<int64_t>(experts) * rows;
  const int64_t n = records * (2 * rb / 16 > 4 * G ? 2 * rb / 16 : 4 * G);
  int64_t grid = (n + 255) / 256;
  grid = grid < 1 ? 1 : (grid > 8192 ? 8192 : grid);
  // codes as they are (4, 8 bits), the scale/bias runs and the padding
  repack_gate_up_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(
      reinterpret_cast<const uint4 *>(g_codes), g_scales, g_biases,
      reinterpret_cast<const uint4 *>(u_codes), u_scales, u_biases, records,
      wb == bits ? rb / 16 : 0, G, rec, out);
  if (wb != bits)  // 6-bit rows: the codes widened to bytes
    repack_gate_up6_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(
        reinterpret_cast<const uint32_t *>(g_codes), reinterpret_cast<const uint32_t *>(u_codes),
        records, din, rec, out);
  return cudaGetLastError();
}

cudaError_t launch_repack_down(const uint8_t *codes, const __half *scales, const __half *biases,
                               int experts, int din, int dff, int bits, uint32_t *out_codes,
                               __half2 *out_sb, cudaStream_t stream) {
  if (experts < 1) return cudaSuccess;
  const int words = dff * bits / 32, groups = dff / 64;
  const int64_t n = static_cast<int64_t>(experts) * din * (words > groups ? words : groups);
  int64_t grid = (n + 255) / 256;
  grid = grid < 1 ? 1 : (grid > 4096 ? 4096 : grid);
  // the scale/bias pairs (and, below 6 bits, the codes as they are)
  repack_down_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(
      reinterpret_cast<const uint32_t *>(codes), scales, biases, experts, din,
      bits == 6 ? 0 : words, groups, out_codes, out_sb);
  if (bits == 6)
    repack_down6_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(
        reinterpret_cast<const uint32_t *>(codes), experts, din, dff, out_codes);
  return cudaGetLastError();
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
