// moe_kernels.cu -- kernel A (dequant gate/up GEMV + SwiGLU) and kernel B (dequant down GEMV,
// summed over slots and shared experts, fused with the residual tail) for one decode token.
//
// The split follows "two-kernel decode-MoE that beats gather_qmm" (What changed, step 2): every
// GEMV output row is an independent warp spread over all SMs and every weight is read once;
// the activation crosses between the two kernels through global memory.  The tail of "Red Lite
// dev39 -- fused expert tail" (Change) is B's epilogue, grid-parallel (one warp per output row
// pair; that page found a one-core tail slower than the dispatches it saved).
//
// Both kernels are persistent (one CTA per SM, grid-stride over their rows) and launch with
// programmatic dependent launch: A waits for the previous kernel on the stream before it reads
// any token data, then lets B launch; B stages its first weight loads before it waits for A.
#include "moe_common.cuh"
#include "moe_kernels.cuh"

namespace moe {

// ------------------------------------------------------------------ streaming loads
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ __half ld_half(const __half *p) {
  unsigned short r;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return __ushort_as_half(r);
}

// ------------------------------------------------------------------ block reductions
// Deterministic: warp butterflies, then warp 0 folds the warps in index order.
__device__ __forceinline__ float block_sum(float v, float *red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    float s = 0.f;
    for (int i = 0; i < nw; ++i) s += red[i];
    if (lane == 0) red[32] = s;
  }
  __syncthreads();
  return red[32];
}

__device__ __forceinline__ float block_max(float v, float *red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    float s = 0.f;
    for (int i = 0; i < nw; ++i) s = fmaxf(s, red[i]);
    if (lane == 0) red[32] = s;
  }
  __syncthreads();
  return red[32];
}

// Two dots of one step against the same activations (gate and up rows share x).
template <int BITS>
__device__ __forceinline__ void step_dot2(const uint4 *vg, const uint4 *vu, const float *xs,
                                          float &dg, float &du) {
  constexpr int N = Fmt<BITS>::kCodes;
  uint32_t mg[N], mu[N];
  step_masks<BITS>(vg, mg);
  step_masks<BITS>(vu, mu);
  float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
  for (int j = 0; j < N; j += 4) {
    const float4 x4 = *reinterpret_cast<const float4 *>(xs + j);
    g0 = fmaf(__uint_as_float(mg[j + 0]), x4.x, g0);
    u0 = fmaf(__uint_as_float(mu[j + 0]), x4.x, u0);
    g1 = fmaf(__uint_as_float(mg[j + 1]), x4.y, g1);
    u1 = fmaf(__uint_as_float(mu[j + 1]), x4.y, u1);
    g0 = fmaf(__uint_as_float(mg[j + 2]), x4.z, g0);
    u0 = fmaf(__uint_as_float(mu[j + 2]), x4.z, u0);
    g1 = fmaf(__uint_as_float(mg[j + 3]), x4.w, g1);
    u1 = fmaf(__uint_as_float(mu[j + 3]), x4.w, u1);
  }
  dg = g0 + g1;
  du = u0 + u1;
}

// ================================================================== kernel A
template <int BITS, int NB>
struct PairBatch {
  uint4 g[NB][Fmt<BITS>::kVecs];
  uint4 u[NB][Fmt<BITS>::kVecs];
  __half gs[NB], gb[NB], us[NB], ub[NB];
};

// Row pair u of one class: its gate and up rows, or nullptr rows when the slot's id is invalid.
struct PairRows {
  const uint8_t *g, *u;
  const __half *gs, *gb, *us, *ub;
};

template <int BITS, int NB>
__device__ __forceinline__ void load_pair(PairBatch<BITS, NB> &B, const PairRows &r, int b,
                                          int nsteps, int lane) {
  constexpr int V = Fmt<BITS>::kVecs, C = Fmt<BITS>::kCodes;
#pragma unroll
  for (int v = 0; v < NB; ++v) {
    const int t = (b * NB + v) * 32 + lane;
    if (r.g != nullptr && t < nsteps) {
      const uint4 *gp = reinterpret_cast<const uint4 *>(r.g) + t * V;
      const uint4 *up = reinterpret_cast<const uint4 *>(r.u) + t * V;
#pragma unroll
      for (int w = 0; w < V; ++w) {
        B.g[v][w] = ld_stream(gp + w);
        B.u[v][w] = ld_stream(up + w);
      }
      const int grp = (t * C) / kGroup;
      B.gs[v] = ld_half(r.gs + grp);
      B.gb[v] = ld_half(r.gb + grp);
      B.us[v] = ld_half(r.us + grp);
      B.ub[v] = ld_half(r.ub + grp);
    } else {
#pragma unroll
      for (int w = 0; w < V; ++w) {
        B.g[v][w] = make_uint4(0, 0, 0, 0);
        B.u[v][w] = make_uint4(0, 0, 0, 0);
      }
      B.gs[v] = B.gb[v] = B.us[v] = B.ub[v] = __float2half(0.f);
    }
  }
}

template <int BITS, int NB>
__device__ __forceinline__ void compute_pair(const PairBatch<BITS, NB> &B, const float *xs,
                                             const float *xsum, float twoS, int b, int nsteps,
                                             int lane, float &gacc, float &uacc) {
  constexpr int C = Fmt<BITS>::kCodes;
#pragma unroll
  for (int v = 0; v < NB; ++v) {
    const int t = (b * NB + v) * 32 + lane;
    if (t < nsteps) {
      float dg, du;
      step_dot2<BITS>(B.g[v], B.u[v], xs + t * C, dg, du);
      const float xsm = xsum[t];
      gacc = fmaf(__half2float(B.gs[v]), dg * twoS, gacc);
      gacc = fmaf(__half2float(B.gb[v]), xsm, gacc);
      uacc = fmaf(__half2float(B.us[v]), du * twoS, uacc);
      uacc = fmaf(__half2float(B.ub[v]), xsm, uacc);
    }
  }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Rows of unit u (global unit index) of one class.  Routed units are k*dff + j, shared units are
// K*dff + s*dff_shared + j.
__device__ __forceinline__ PairRows pair_rows(const GateUpParams &p, const ProjDev &gate,
                                              const ProjDev &up, int64_t expert, int j, int rows,
                                              int rowbytes) {
  PairRows r;
  const int64_t row = expert * rows + j;
  const int64_t groups = p.din / kGroup;
  r.g = gate.codes + row * rowbytes;
  r.u = up.codes + row * rowbytes;
  r.gs = gate.scales + row * groups;
  r.gb = gate.biases + row * groups;
  r.us = up.scales + row * groups;
  r.ub = up.biases + row * groups;
  return r;
}

template <int BITS, int NB>
__device__ void gate_up_rows(const GateUpParams &p, bool shared_class, int u_first, int u_end,
                             const float *xs, const float *xsum, float twoS, const int *ids_s,
                             const float *coef_s, float shared_scalar) {
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  constexpr int C = Fmt<BITS>::kCodes;
  const int nsteps = p.din / C;
  const int nb = (nsteps + 32 * NB - 1) / (32 * NB);
  const int rowbytes = p.din * BITS / 8;
  const int units_r = p.top_k * p.dff;

  auto rows_of = [&](int u) -> PairRows {
    if (!shared_class) {
      const int k = u / p.dff, j = u - k * p.dff;
      const int e = ids_s[k];
      if (e < 0 || e >= p.n_experts) {
        PairRows z{};
        return z;
      }
      return pair_rows(p, p.gate, p.up, e, j, p.dff, rowbytes);
    }
    const int us = u - units_r;
    const int s = us / p.dff_shared, j = us - s * p.dff_shared;
    return pair_rows(p, p.sh_gate, p.sh_up, s, j, p.dff_shared, rowbytes);
  };

  if (u_first >= u_end) return;
  int u = u_first, b = 0;
  PairRows rows = rows_of(u);
  PairBatch<BITS, NB> cur;
  load_pair<BITS, NB>(cur, rows, b, nsteps, lane);
  float gacc = 0.f, uacc = 0.f;
  while (true) {
    int nu = u, nbb = b + 1;
    if (nbb == nb) {
      nbb = 0;
      nu = u + nwarps;
    }
    const bool has_next = nu < u_end;
    PairRows nrows = rows;
    PairBatch<BITS, NB> nxt;
    if (has_next) {
      if (nu != u) nrows = rows_of(nu);
      load_pair<BITS, NB>(nxt, nrows, nbb, nsteps, lane);
    }
    compute_pair<BITS, NB>(cur, xs, xsum, twoS, b, nsteps, lane, gacc, uacc);
    if (b == nb - 1) {
      gacc = warp_sum(gacc);
      uacc = warp_sum(uacc);
      if (lane == 0) {
        float coef;
        if (shared_class) {
          coef = shared_scalar;
        } else {
          const int k = u / p.dff;
          coef = coef_s[k];
          if (rows.g == nullptr) atomicOr(p.err, 1);
        }
        p.act[u] = coef * (silu_f(gacc) * uacc);
      }
      gacc = uacc = 0.f;
    }
    if (!has_next) break;
    cur = nxt;
    rows = nrows;
    u = nu;
    b = nbb;
  }
}

template <int BR, int BS>
__global__ void __launch_bounds__(kAThreads, 1) gate_up_kernel(const GateUpParams p) {
  extern __shared__ __align__(16) float smem[];
  __shared__ float red[33];
  __shared__ int ids_s[kMaxTopK];
  __shared__ float coef_s[kMaxTopK];

  const int din = p.din;
  const bool separate = (BS != BR) && p.n_shared > 0;
  float *xs_r = smem;
  float *xs_s = separate ? smem + din : smem;
  float *xsum_r = smem + (separate ? 2 : 1) * din;
  float *xsum_s = separate ? xsum_r + din / Fmt<BR>::kCodes : xsum_r;

  // Token data (x, ids, scores) may be produced by the previous kernel on the stream.
  pdl_wait();
  pdl_launch_dependents();

  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int k = tid; k < p.top_k; k += nthr) {
    ids_s[k] = p.ids[k];
    coef_s[k] = p.scores[k];
  }
  float mx = 0.f, dot = 0.f;
  for (int c = tid; c < din; c += nthr) {
    const float v = bf16_to_float(p.x[c]);
    mx = fmaxf(mx, fabsf(v));
    if (p.gate_vec != nullptr) dot = fmaf(v, bf16_to_float(p.gate_vec[c]), dot);
  }
  mx = block_max(mx, red);
  dot = block_sum(dot, red);
  const int S = choose_shift(mx);
  const float twoS = pow2f(S);
  const float shared_scalar = p.gate_vec != nullptr ? 1.0f / (1.0f + expf(-dot)) : 1.0f;
  for (int c = tid; c < din; c += nthr) {
    const float v = bf16_to_float(p.x[c]);
    xs_r[c] = v * pow2f(149 - S - code_offset<BR>(c));
    if (separate) xs_s[c] = v * pow2f(149 - S - code_offset<BS>(c));
  }
  for (int t = tid; t < din / Fmt<BR>::kCodes; t += nthr) {
    float s = 0.f;
    for (int j = 0; j < Fmt<BR>::kCodes; ++j) s += bf16_to_float(p.x[t * Fmt<BR>::kCodes + j]);
    xsum_r[t] = s;
  }
  if (separate) {
    for (int t = tid; t < din / Fmt<BS>::kCodes; t += nthr) {
      float s = 0.f;
      for (int j = 0; j < Fmt<BS>::kCodes; ++j) s += bf16_to_float(p.x[t * Fmt<BS>::kCodes + j]);
      xsum_s[t] = s;
    }
  }
  __syncthreads();

  const int warp = blockIdx.x * (nthr >> 5) + (tid >> 5);
  const int nwarps = gridDim.x * (nthr >> 5);
  const int units_r = p.top_k * p.dff;
  const int units = units_r + p.n_shared * p.dff_shared;
  constexpr int NBR = Fmt<BR>::kVecs == 1 ? 2 : 1;
  constexpr int NBS = Fmt<BS>::kVecs == 1 ? 2 : 1;
  gate_up_rows<BR, NBR>(p, false, warp, units_r, xs_r, xsum_r, twoS, ids_s, coef_s, 1.f);
  int first_s = warp;
  if (first_s < units_r) first_s += ((units_r - warp + nwarps - 1) / nwarps) * nwarps;
  gate_up_rows<BS, NBS>(p, true, first_s, units, xs_s, xsum_s, twoS, ids_s, coef_s,
                        shared_scalar);
}

// ================================================================== kernel B
template <int BD, int BSD>
struct DownFmt {
  static constexpr int kVecs = Fmt<BD>::kVecs > Fmt<BSD>::kVecs ? Fmt<BD>::kVecs : Fmt<BSD>::kVecs;
};

template <int BD, int BSD, int NB>
struct DownBatch {
  uint4 c[NB][kBRows][DownFmt<BD, BSD>::kVecs];
  __half s[NB][kBRows], b[NB][kBRows];
};

struct DownGeom {
  int T_r, T_s;          // routed / shared steps over the concatenated contraction
  int spr_r, spr_s;      // steps per row of one routed / shared expert
  int rb_r, rb_s;        // row bytes
  int V_r, V_s;          // per-lane step slots
  int nb_r, nb_s;        // batches per tile
};

template <int BITS, int BD, int BSD, int NB>
__device__ __forceinline__ void load_down_class(DownBatch<BD, BSD, NB> &B, const ProjDev &pr,
                                                const int *ids_s, bool shared_class, int v0,
                                                int T, int spr, int rowbytes, int i0,
                                                const DownParams &p, int lane) {
  constexpr int V = Fmt<BITS>::kVecs, C = Fmt<BITS>::kCodes;
  const int G = (shared_class ? p.dff_shared : p.dff) / kGroup;
#pragma unroll
  for (int v = 0; v < NB; ++v) {
    const int t = (v0 + v) * 32 + lane;
    int64_t expert = -1;
    int j = 0;
    if (t < T) {
      const int k = t / spr;
      j = t - k * spr;
      if (shared_class) {
        expert = k;
      } else {
        const int e = ids_s[k];
        expert = (e >= 0 && e < p.n_experts) ? e : -1;
      }
    }
#pragma unroll
    for (int r = 0; r < kBRows; ++r) {
      if (expert >= 0) {
        const int64_t row = expert * p.din + i0 + r;
        const uint4 *cp = reinterpret_cast<const uint4 *>(pr.codes + row * rowbytes) + j * V;
#pragma unroll
        for (int w = 0; w < V; ++w) B.c[v][r][w] = ld_stream(cp + w);
        const int64_t gi = row * G + (j * C) / kGroup;
        B.s[v][r] = ld_half(pr.scales + gi);
        B.b[v][r] = ld_half(pr.biases + gi);
      } else {
#pragma unroll
        for (int w = 0; w < V; ++w) B.c[v][r][w] = make_uint4(0, 0, 0, 0);
        B.s[v][r] = B.b[v][r] = __float2half(0.f);
      }
    }
  }
}

template <int BITS, int BD, int BSD, int NB>
__device__ __forceinline__ void compute_down_class(const DownBatch<BD, BSD, NB> &B,
                                                   const float *as, const float *asum, int v0,
                                                   int T, float twoS, int lane,
                                                   float (&acc)[kBRows]) {
  constexpr int C = Fmt<BITS>::kCodes;
#pragma unroll
  for (int v = 0; v < NB; ++v) {
    const int t = (v0 + v) * 32 + lane;
    if (t < T) {
      const float *xp = as + t * C;
      const float sm = asum[t];
#pragma unroll
      for (int r = 0; r < kBRows; ++r) {
        const float d = step_dot<BITS>(B.c[v][r], xp);
        acc[r] = fmaf(__half2float(B.s[v][r]), d * twoS, acc[r]);
        acc[r] = fmaf(__half2float(B.b[v][r]), sm, acc[r]);
      }
    }
  }
}

template <int BD, int BSD, int NB>
__device__ __forceinline__ void load_down(DownBatch<BD, BSD, NB> &B, const DownParams &p,
                                          const DownGeom &g, const int *ids_s, int tile, int b,
                                          int lane) {
  const int i0 = tile * kBRows;
  if (b < g.nb_r)
    load_down_class<BD, BD, BSD, NB>(B, p.down, ids_s, false, b * NB, g.T_r, g.spr_r, g.rb_r, i0,
                                     p, lane);
  else
    load_down_class<BSD, BD, BSD, NB>(B, p.sh_down, ids_s, true, (b - g.nb_r) * NB, g.T_s,
                                      g.spr_s, g.rb_s, i0, p, lane);
}

template <int BD, int BSD>
__global__ void __launch_bounds__(kBThreads, 1) down_kernel(const DownParams p) {
  extern __shared__ __align__(16) float smem[];
  __shared__ float red[33];
  __shared__ int ids_s[kMaxTopK];
  constexpr int NB = 2;

  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
  const int Lr = p.top_k * p.dff, Ls = p.n_shared * p.dff_shared;
  DownGeom g;
  g.spr_r = p.dff / Fmt<BD>::kCodes;
  g.spr_s = p.dff_shared / Fmt<BSD>::kCodes;
  g.T_r = p.top_k * g.spr_r;
  g.T_s = p.n_shared * g.spr_s;
  g.rb_r = p.dff * BD / 8;
  g.rb_s = p.dff_shared * BSD / 8;
  g.V_r = (g.T_r + 31) / 32;
  g.V_s = (g.T_s + 31) / 32;
  g.nb_r = (g.V_r + NB - 1) / NB;
  g.nb_s = (g.V_s + NB - 1) / NB;
  const int nbt = g.nb_r + g.nb_s;

  float *as_r = smem;
  float *as_s = smem + Lr;
  float *asum_r = as_s + Ls;
  float *asum_s = asum_r + g.T_r;

  // ids were complete before kernel A started; reading them here is allowed before the wait.
  for (int k = tid; k < p.top_k; k += nthr) ids_s[k] = p.ids[k];
  __syncthreads();

  const int warp = blockIdx.x * (nthr >> 5) + (tid >> 5);
  const int nwarps = gridDim.x * (nthr >> 5);
  const int tiles = p.din / kBRows;
  int tile = warp, b = 0;
  DownBatch<BD, BSD, NB> cur;
  if (tile < tiles && nbt > 0) load_down<BD, BSD, NB>(cur, p, g, ids_s, tile, b, lane);

  // The activations come from kernel A.
  pdl_wait();
  pdl_launch_dependents();

  float mx = 0.f;
  for (int i = tid; i < Lr + Ls; i += nthr) mx = fmaxf(mx, fabsf(p.act[i]));
  mx = block_max(mx, red);
  const int S = choose_shift(mx);
  const float twoS = pow2f(S);
  for (int i = tid; i < Lr; i += nthr) as_r[i] = p.act[i] * pow2f(149 - S - code_offset<BD>(i));
  for (int i = tid; i < Ls; i += nthr)
    as_s[i] = p.act[Lr + i] * pow2f(149 - S - code_offset<BSD>(i));
  for (int t = tid; t < g.T_r; t += nthr) {
    float s = 0.f;
    for (int j = 0; j < Fmt<BD>::kCodes; ++j) s += p.act[t * Fmt<BD>::kCodes + j];
    asum_r[t] = s;
  }
  for (int t = tid; t < g.T_s; t += nthr) {
    float s = 0.f;
    for (int j = 0; j < Fmt<BSD>::kCodes; ++j) s += p.act[Lr + t * Fmt<BSD>::kCodes + j];
    asum_s[t] = s;
  }
  __syncthreads();

  if (tile >= tiles) return;
  int bad = 0;
  for (int k = 0; k < p.top_k; ++k) bad |= (ids_s[k] < 0 || ids_s[k] >= p.n_experts);
  if (bad && blockIdx.x == 0 && tid == 0) atomicOr(p.err, 1);

  float acc[kBRows];
#pragma unroll
  for (int r = 0; r < kBRows; ++r) acc[r] = 0.f;
  while (true) {
    int nt = tile, nbb = b + 1;
    if (nbb == nbt) {
      nbb = 0;
      nt = tile + nwarps;
    }
    const bool has_next = nt < tiles;
    DownBatch<BD, BSD, NB> nxt;
    if (has_next) load_down<BD, BSD, NB>(nxt, p, g, ids_s, nt, nbb, lane);
    if (b < g.nb_r)
      compute_down_class<BD, BD, BSD, NB>(cur, as_r, asum_r, b * NB, g.T_r, twoS, lane, acc);
    else
      compute_down_class<BSD, BD, BSD, NB>(cur, as_s, asum_s, (b - g.nb_r) * NB, g.T_s, twoS,
                                           lane, acc);
    if (b == nbt - 1) {
#pragma unroll
      for (int r = 0; r < kBRows; ++r) acc[r] = warp_sum(acc[r]);
      if (lane < kBRows) {
        float a = acc[0];
#pragma unroll
        for (int r = 1; r < kBRows; ++r)
          if (lane == r) a = acc[r];
        const int i = tile * kBRows + lane;
        const float res = p.resid_f32 ? static_cast<const float *>(p.resid)[i]
                                      : bf16_to_float(static_cast<const uint16_t *>(p.resid)[i]);
        const float o = res + a;
        if (p.out_f32)
          static_cast<float *>(p.out)[i] = o;
        else
          static_cast<uint16_t *>(p.out)[i] = float_to_bf16_rn(o);
      }
#pragma unroll
      for (int r = 0; r < kBRows; ++r) acc[r] = 0.f;
    }
    if (!has_next) break;
    cur = nxt;
    tile = nt;
    b = nbb;
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

// ================================================================== host side
static int fmt_codes(int bits) { return bits == 4 ? 32 : bits == 8 ? 16 : 64; }

size_t gate_up_smem_bytes(int din, int bits_r, int bits_s, int n_shared) {
  const bool separate = bits_s != bits_r && n_shared > 0;
  size_t n = (separate ? 2 : 1) * (size_t)din + din / fmt_codes(bits_r);
  if (separate) n += din / fmt_codes(bits_s);
  return n * sizeof(float);
}

size_t down_smem_bytes(int dff, int top_k, int n_shared, int dff_shared, int bits_d,
                       int bits_sd) {
  const size_t Lr = (size_t)top_k * dff, Ls = (size_t)n_shared * dff_shared;
  return (Lr + Ls + Lr / fmt_codes(bits_d) + Ls / fmt_codes(bits_sd)) * sizeof(float);
}

template <typename Kern, typename P>
static cudaError_t launch(Kern kern, const P &p, int grid, int threads, size_t smem,
                          cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

#define MOE_BITS_SWITCH(B, NAME, ...)                      \
  switch (B) {                                             \
    case 4: { constexpr int NAME = 4; __VA_ARGS__; break; } \
    case 6: { constexpr int NAME = 6; __VA_ARGS__; break; } \
    case 8: { constexpr int NAME = 8; __VA_ARGS__; break; } \
    default: return cudaErrorInvalidValue;                 \
  }

cudaError_t launch_gate_up(const GateUpParams &p, int bits_r, int bits_s, int grid, size_t smem,
                           cudaStream_t stream, bool pdl) {
  MOE_BITS_SWITCH(bits_r, BR, MOE_BITS_SWITCH(bits_s, BS,
      return launch(gate_up_kernel<BR, BS>, p, grid, kAThreads, smem, stream, pdl)));
  return cudaErrorInvalidValue;
}

cudaError_t launch_down(const DownParams &p, int bits_d, int bits_sd, int grid, size_t smem,
                        cudaStream_t stream, bool pdl) {
  MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sd, BSD,
      return launch(down_kernel<BD, BSD>, p, grid, kBThreads, smem, stream, pdl)));
  return cudaErrorInvalidValue;
}

cudaError_t prepare_kernels(int smem_optin, int bits_r, int bits_s, int bits_d, int bits_sd) {
  // The attribute is global to a kernel instance: set it to the device's opt-in maximum so one
  // handle can never lower it below what another handle launches with.
  cudaError_t e = cudaSuccess;
  MOE_BITS_SWITCH(bits_r, BR, MOE_BITS_SWITCH(bits_s, BS,
      e = cudaFuncSetAttribute(gate_up_kernel<BR, BS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin)));
  if (e != cudaSuccess) return e;
  MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sd, BSD,
      e = cudaFuncSetAttribute(down_kernel<BD, BSD>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin)));
  return e;
}

cudaError_t launch_unpack(const uint8_t *packed, int64_t rows, int64_t cols, int bits,
                          uint8_t *codes, cudaStream_t stream) {
  const int64_t steps = rows * (cols / fmt_codes(bits));
  int grid = (int)((steps + 255) / 256);
  grid = grid < 1 ? 1 : (grid > 65535 ? 65535 : grid);
  MOE_BITS_SWITCH(bits, B, unpack_kernel<B><<<grid, 256, 0, stream>>>(packed, rows, cols, codes));
  return cudaGetLastError();
}

}  // namespace moe
