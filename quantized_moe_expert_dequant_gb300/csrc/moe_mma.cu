// moe_mma.cu -- the tensor-core batch variant of the block (MOE_KERNELS_MMA): m tokens, their
// slots grouped by expert, every projection on bf16 tensor-core tiles.
//
// The block is the same as in every mode (the two phases of "two-kernel decode-MoE that beats
// gather_qmm", What changed, step 2, and the tail of "Red Lite dev39 -- fused expert tail"):
//   act[t][k][j] = coef * silu(gate_j . x_t) * (up_j . x_t)      coef: the slot's score (routed)
//                                                                or the shared scalar (shared)
//   y[t][k][i]   = down_i . act[t][k]
//   out[t][i]    = resid[t][i] + (sum over the token's valid slots, in slot order, and its shared
//                  experts of y[t][.][i])
// With several tokens per expert a row of weights meets several vectors: a small dense
// contraction.  A warp takes a tile of 16 weight rows of one expert and up to 8 (token, slot)
// pairs that name it and runs mma.sync.m16n8k16 (bf16 operands, fp32 accumulation) over one
// group of 64 codes at a time.  The codes enter the tensor core exactly: bf16 holds every integer
// below 256, and a code q < 128 is formed as the bf16 (128 + q) by one OR (0x4300 | q) minus 128
// (an exact bf16x2 subtraction); an 8-bit code is split into its nibbles, 16 * hi formed by one
// bf16x2 FMA, and both nibble tiles accumulate into the same sum; x is bf16 already, so the gate/up
// products are exact.  The down projection meets the fp32 activation instead, on fp16 tiles: a
// code (any width, < 1024) is the fp16 (1024 + q) - 1024, and the activation's 64 values of one
// group and one column are scaled by one power of two 2^k that puts their largest magnitude in
// [2^14, 2^15), then split into an fp16 high part and an fp16 remainder (two tiles, 22
// significant bits); the column's sum is multiplied by 2^-k.  Per group the accumulator
// D = sum_c q_c v_c becomes the group's dequantised dot
//   sum_c (s q_c + b) v_c = s * D + b * sum_c v_c,
// added to the row's fp32 sum.  Fragments come straight from global memory: inside a group lane
// (g, q) owns codes 16 q .. 16 q + 15 of rows g and g + 8 (and the same 16 entries of its column's
// vector); the four k-steps take them as k slots in one permutation that A and B share (a sum does
// not depend on its order).  Nothing is staged in shared memory: each weight byte is read once by
// the one warp whose tile holds it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_mma.cuh"
#include "moe_phases.cuh"

namespace moe {
namespace mma {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCtasPerSm = 4;      // gate/up: 64 registers a thread
constexpr int kCtasPerSmDown = 3;  // down: the activation's two bf16 parts need more

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_u32(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_h2(uint32_t u) { return *reinterpret_cast<const __half2 *>(&u); }

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 h) {
  return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) {
  return *reinterpret_cast<const __nv_bfloat162 *>(&u);
}

// The bf16 pair (c0, c1) of two values below 128 (4/6-bit codes, nibbles).
__device__ __forceinline__ uint32_t code_pair(uint32_t c0, uint32_t c1) {
  const uint32_t biased = 0x43004300u | c0 | (c1 << 16);  // (128 + c0, 128 + c1), exact
  return as_u32(__hsub2(as_bf2(biased), as_bf2(0x43004300u)));
}
// The bf16 pair (16 h0, 16 h1) of two high nibbles: (128 + h) * 16 - 2048, exact in one FMA.
__device__ __forceinline__ uint32_t hi_pair(uint32_t h0, uint32_t h1) {
  const uint32_t biased = 0x43004300u | h0 | (h1 << 16);
  return as_u32(__hfma2(as_bf2(biased), as_bf2(0x41804180u), as_bf2(0xC500C500u)));
}

// The fp16 pair (c0, c1) of two codes below 1024: (1024 + c) - 1024, exact.
__device__ __forceinline__ uint32_t code_pair_h(uint32_t c0, uint32_t c1) {
  const uint32_t biased = 0x64006400u | c0 | (c1 << 16);
  return h2_u32(__hsub2(u32_h2(biased), u32_h2(0x64006400u)));
}

// The raw words of one lane's slice of one group of one row (codes 16 q .. 16 q + 15 of the group,
// LSB first): 2 words at 4 bits, 4 at 8 bits, 3 at 6 bits; zeros for a row past the projection.
template <int BITS>
__device__ __forceinline__ void lane_words(const uint8_t *grp, int q, bool ok, uint32_t (&w)[4]) {
  w[0] = w[1] = w[2] = w[3] = 0u;
  if (!ok) return;
  if constexpr (BITS == 4) {
    const uint2 v = *reinterpret_cast<const uint2 *>(grp + 8 * q);
    w[0] = v.x;
    w[1] = v.y;
  } else if constexpr (BITS == 8) {
    const uint4 v = *reinterpret_cast<const uint4 *>(grp + 16 * q);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
    const uint32_t *p = reinterpret_cast<const uint32_t *>(grp + 12 * q);
    w[0] = p[0];
    w[1] = p[1];
    w[2] = p[2];
  }
}

// Code i (0..15) of a lane's slice.
template <int BITS>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&w)[4], int i) {
  const int b = BITS * i, wi = b >> 5, o = b & 31;
  if (o + BITS <= 32) return (w[wi] >> o) & ((1u << BITS) - 1u);
  return __funnelshift_r(w[wi], w[wi + 1], o) & ((1u << BITS) - 1u);
}

// A fragments of k-step j from the words of rows g (wa) and g + 8 (wb): codes 4 j, 4 j + 1 in k
// slots 2q, 2q + 1 and 4 j + 2, 4 j + 3 in slots 2q + 8, 2q + 9.  PART 0: the whole code; 1: 16
// times the high nibble; 2: the low nibble (8-bit codes).
template <int BITS, int PART>
__device__ __forceinline__ void a_frag(const uint32_t (&wa)[4], const uint32_t (&wb)[4], int j,
                                       uint32_t (&a)[4]) {
  uint32_t x[4], y[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t u = code_at<BITS>(wa, 4 * j + t), v = code_at<BITS>(wb, 4 * j + t);
    x[t] = PART == 1 ? u >> 4 : (PART == 2 ? u & 15u : u);
    y[t] = PART == 1 ? v >> 4 : (PART == 2 ? v & 15u : v);
  }
  if constexpr (PART == 1) {
    a[0] = hi_pair(x[0], x[1]);
    a[1] = hi_pair(y[0], y[1]);
    a[2] = hi_pair(x[2], x[3]);
    a[3] = hi_pair(y[2], y[3]);
  } else {
    a[0] = code_pair(x[0], x[1]);  // row g, k slots 2q, 2q + 1
    a[1] = code_pair(y[0], y[1]);  // row g + 8
    a[2] = code_pair(x[2], x[3]);  // row g, k slots 2q + 8, 2q + 9
    a[3] = code_pair(y[2], y[3]);
  }
}

// D += codes(rows g, g + 8) x B over one group, bf16 tiles; B as 8 registers (pairs of the lane's
// 16 values).
template <int BITS>
__device__ __forceinline__ void group_mma(const uint32_t (&ca)[4], const uint32_t (&cb)[4],
                                          const uint32_t (&b)[8], float (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    if constexpr (BITS == 8) {
      a_frag<BITS, 1>(ca, cb, j, a);
      mma_bf16(d, a, b[2 * j], b[2 * j + 1]);
      a_frag<BITS, 2>(ca, cb, j, a);
      mma_bf16(d, a, b[2 * j], b[2 * j + 1]);
    } else {
      a_frag<BITS, 0>(ca, cb, j, a);
      mma_bf16(d, a, b[2 * j], b[2 * j + 1]);
    }
  }
}

// fp16 A fragments of k-step j (the slot layout of a_frag, whole codes of any width).
template <int BITS>
__device__ __forceinline__ void a_frag_h(const uint32_t (&wa)[4], const uint32_t (&wb)[4], int j,
                                         uint32_t (&a)[4]) {
  const int i = 4 * j;
  a[0] = code_pair_h(code_at<BITS>(wa, i), code_at<BITS>(wa, i + 1));
  a[1] = code_pair_h(code_at<BITS>(wb, i), code_at<BITS>(wb, i + 1));
  a[2] = code_pair_h(code_at<BITS>(wa, i + 2), code_at<BITS>(wa, i + 3));
  a[3] = code_pair_h(code_at<BITS>(wb, i + 2), code_at<BITS>(wb, i + 3));
}

// D += codes(rows g, g + 8) x (high + remainder) over one group, fp16 tiles.
template <int BITS>
__device__ __forceinline__ void group_mma_down(const uint32_t (&ca)[4], const uint32_t (&cb)[4],
                                               const uint32_t (&b)[2][8], float (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
    a_frag_h<BITS>(ca, cb, j, a);
    mma_f16(d, a, b[0][2 * j], b[0][2 * j + 1]);
    mma_f16(d, a, b[1][2 * j], b[1][2 * j + 1]);
  }
}

// One lane's 16 bf16 values of a group as B registers, and their sum.
__device__ __forceinline__ float b_from_bf16(const uint16_t *v, bool ok, uint32_t (&b)[8]) {
  uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
  if (ok) {
    w0 = *reinterpret_cast<const uint4 *>(v);
    w1 = *reinterpret_cast<const uint4 *>(v + 8);
  }
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    b[i] = w[i];
    s += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xffff0000u);
  }
  return s;
}

// One lane's 16 fp32 values of a group of column g as fp16 B registers: scaled by 2^k, where
// 2^k puts the largest magnitude of the column's 64 values of the group (the four lanes of g) in
// [2^14, 2^15) (k at most 126, for an all-zero or tiny group), high parts in b[0] and remainders
// in b[1].  Returns the plain fp32 sum of the 16 values; *inv = 2^-k.
__device__ __forceinline__ float b_from_f32(const float *v, bool ok, uint32_t (&b)[2][8],
                                            float *inv) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const float4 t = ok ? *reinterpret_cast<const float4 *>(v + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    a[i] = t.x;
    a[i + 1] = t.y;
    a[i + 2] = t.z;
    a[i + 3] = t.w;
  }
  float mx = 0.f, s = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    mx = fmaxf(mx, fabsf(a[i]));
    s += a[i];
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const int E = static_cast<int>((__float_as_uint(mx) >> 23) & 255u);  // biased exponent
  const int k = min(141 - E, 126);                                       // 14 - (E - 127)
  const float sc = pow2f(k);
  *inv = pow2f(-k);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float v0 = a[2 * i] * sc, v1 = a[2 * i + 1] * sc;
    const __half2 h = __floats2half2_rn(v0, v1);
    b[0][i] = h2_u32(h);
    b[1][i] = h2_u32(__floats2half2_rn(v0 - __low2float(h), v1 - __high2float(h)));
  }
  return s;
}

// The group sums of this lane's two D columns (2q, 2q + 1) from each lane's partial sum of its 16
// values of column g.
__device__ __forceinline__ void column_sums(float part, int q, float *s0, float *s1) {
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  *s0 = __shfl_sync(0xffffffffu, part, 8 * q);
  *s1 = __shfl_sync(0xffffffffu, part, 8 * q + 4);
}

// The batch's route in shared memory and the phase's work items: for every distinct expert u,
// ceil(pairs_u / 8) pair tiles x `tiles` row tiles (ibase[u] = first item of u), then the shared
// experts, ceil(m / 8) pair tiles x `tiles_s` row tiles each.
struct MmaSmem {
  int U, n_items_r;
  int uniq[kMaxPairs];
  int offs[kMaxPairs + 1];
  int pairs[kMaxPairs];
  int ibase[kMaxPairs + 1];
};

__device__ void load_route(const int32_t *route, int tiles, MmaSmem &sm) {
  const int U = route[0];
  if (threadIdx.x == 0) sm.U = U;
  for (int u = threadIdx.x; u < U; u += blockDim.x) sm.uniq[u] = route[1 + u];
  for (int u = threadIdx.x; u <= U; u += blockDim.x) sm.offs[u] = route[1 + U + u];
  __syncthreads();
  const int np = sm.offs[U];
  for (int i = threadIdx.x; i < np; i += blockDim.x) sm.pairs[i] = route[2 + 2 * U + i];
  if (threadIdx.x < 32) {  // exclusive scan of the items per expert, 8 experts a lane
    const int lane = threadIdx.x;
    constexpr int PER = kMaxPairs / 32;
    int loc[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int u = lane * PER + j;
      loc[j] = u < U ? ((sm.offs[u + 1] - sm.offs[u] + 7) / 8) * tiles : 0;
      sum += loc[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int u = lane * PER + j;
      if (u <= U) sm.ibase[u] = run;
      run += loc[j];
    }
    if (lane == 31) sm.n_items_r = incl;
  }
  __syncthreads();
}

struct Item {
  bool shared;
  int e;        // expert id (routed) or shared expert index
  int tile;     // 16-row tile
  int pb, pe;   // pair range: routed pairs [pb, pe) of the route's list; shared: tokens
};

__device__ __forceinline__ bool item_of(int idx, const MmaSmem &sm, int m, int n_shared,
                                        int tiles, int tiles_s, Item &it) {
  if (idx < sm.n_items_r) {
    int lo = 0, hi = sm.U;  // ibase[lo] <= idx < ibase[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sm.ibase[mid] <= idx) lo = mid;
      else hi = mid;
    }
    const int rel = idx - sm.ibase[lo];
    const int pt = rel / tiles;
    it.shared = false;
    it.e = sm.uniq[lo];
    it.tile = rel - pt * tiles;
    it.pb = sm.offs[lo] + 8 * pt;
    it.pe = min(it.pb + 8, sm.offs[lo + 1]);
    return true;
  }
  idx -= sm.n_items_r;
  const int pts = (m + 7) / 8, per = pts * tiles_s;
  if (idx >= per * n_shared) return false;
  const int sh = idx / per, rel = idx - sh * per, pt = rel / tiles_s;
  it.shared = true;
  it.e = sh;
  it.tile = rel - pt * tiles_s;
  it.pb = 8 * pt;
  it.pe = min(it.pb + 8, m);
  return true;
}

// (token, slot) of entry p of an item's pair range; slot -1 for a shared expert's token.
__device__ __forceinline__ void pair_of(const Item &it, const MmaSmem &sm, int p, int K, int *t,
                                        int *k) {
  if (it.shared) {
    *t = p;
    *k = -1;
  } else {
    const int v = sm.pairs[p];
    *t = v / K;
    *k = v - *t * K;
  }
}

// Activation segment of a (token, slot) column inside the token's act row.
__device__ __forceinline__ int64_t act_segment(const Item &it, const LayerShape &s, int k) {
  return it.shared ? static_cast<int64_t>(s.top_k) * s.dff + static_cast<int64_t>(it.e) * s.dff_shared
                   : static_cast<int64_t>(k) * s.dff;
}

// ------------------------------------------------------------------ gate/up
template <int BITS>
__device__ void gate_up_item(const MmaParams &p, const ProjDev &gate, const ProjDev &up,
                             int rows_pe, const Item &it, const MmaSmem &sm, int lane) {
  const LayerShape &s = p.s;
  const int g = lane >> 2, q = lane & 3;
  const int K = s.top_k, G = s.din / kGroup;
  constexpr int GB = kGroup * BITS / 8;  // bytes of one group of one row
  const int64_t rb = static_cast<int64_t>(s.din) * BITS / 8;
  const int r0 = 16 * it.tile;
  const int64_t rowA = static_cast<int64_t>(it.e) * rows_pe + r0 + g, rowB = rowA + 8;
  const bool okA = r0 + g < rows_pe, okB = r0 + g + 8 < rows_pe;
  int tb = 0, kb = 0;
  const bool okT = it.pb + g < it.pe;  // this lane's B column: pair pb + g
  if (okT) pair_of(it, sm, it.pb + g, K, &tb, &kb);
  const uint16_t *xv = p.x + static_cast<int64_t>(tb) * s.din + 16 * q;
  const uint8_t *gA = gate.codes + rowA * rb, *gB = gate.codes + rowB * rb;
  const uint8_t *uA = up.codes + rowA * rb, *uB = up.codes + rowB * rb;
  float Gs[4] = {0.f, 0.f, 0.f, 0.f}, Us[4] = {0.f, 0.f, 0.f, 0.f};
  for (int gi = 0; gi < G; ++gi) {
    uint32_t b[8];
    const float part = b_from_bf16(xv + gi * kGroup, okT, b);
    uint32_t ca[4], cb[4];
    float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
    lane_words<BITS>(gA + gi * GB, q, okA, ca);
    lane_words<BITS>(gB + gi * GB, q, okB, cb);
    group_mma<BITS>(ca, cb, b, dg);
    lane_words<BITS>(uA + gi * GB, q, okA, ca);
    lane_words<BITS>(uB + gi * GB, q, okB, cb);
    group_mma<BITS>(ca, cb, b, du);
    float sx0, sx1;
    column_sums(part, q, &sx0, &sx1);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const bool second = h >= 2;
      if (second ? okB : okA) {
        const int64_t gidx = (second ? rowB : rowA) * G + gi;
        const float sx = (h & 1) ? sx1 : sx0;
        Gs[h] += fmaf(__half2float(gate.scales[gidx]), dg[h], __half2float(gate.biases[gidx]) * sx);
        Us[h] += fmaf(__half2float(up.scales[gidx]), du[h], __half2float(up.biases[gidx]) * sx);
      }
    }
  }
  // the lane's four entries: rows g, g + 8 of the tile, columns 2q, 2q + 1
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int pp = it.pb + 2 * q + (h & 1);
    const int row = r0 + g + (h >= 2 ? 8 : 0);
    if (pp < it.pe && row < rows_pe) {
      int t, k;
      pair_of(it, sm, pp, K, &t, &k);
      const float coef = it.shared ? p.sscal[t] : p.scores[t * K + k];
      p.act[static_cast<int64_t>(t) * p.act_stride + act_segment(it, s, k) + row] =
          coef * (silu_f(Gs[h]) * Us[h]);
    }
  }
}

// ------------------------------------------------------------------ down
template <int BITS>
__device__ void down_item(const MmaParams &p, const ProjDev &down, int cols, const Item &it,
                          const MmaSmem &sm, int lane) {
  const LayerShape &s = p.s;
  const int g = lane >> 2, q = lane & 3;
  const int K = s.top_k, G = cols / kGroup, ny = K + s.n_shared;
  constexpr int GB = kGroup * BITS / 8;
  const int64_t rb = static_cast<int64_t>(cols) * BITS / 8;
  const int r0 = 16 * it.tile;
  const int64_t rowA = static_cast<int64_t>(it.e) * s.din + r0 + g, rowB = rowA + 8;
  const bool okA = r0 + g < s.din, okB = r0 + g + 8 < s.din;
  int tb = 0, kb = 0;
  const bool okT = it.pb + g < it.pe;
  if (okT) pair_of(it, sm, it.pb + g, K, &tb, &kb);
  const float *av = p.act + static_cast<int64_t>(tb) * p.act_stride + act_segment(it, s, kb) + 16 * q;
  const uint8_t *cA = down.codes + rowA * rb, *cB = down.codes + rowB * rb;
  float Y[4] = {0.f, 0.f, 0.f, 0.f};
  for (int gi = 0; gi < G; ++gi) {
    uint32_t b[2][8];
    float inv;
    const float part = b_from_f32(av + gi * kGroup, okT, b, &inv);
    uint32_t ca[4], cb[4];
    lane_words<BITS>(cA + gi * GB, q, okA, ca);
    lane_words<BITS>(cB + gi * GB, q, okB, cb);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    group_mma_down<BITS>(ca, cb, b, d);
    float sv0, sv1;
    column_sums(part, q, &sv0, &sv1);
    const float inv0 = __shfl_sync(0xffffffffu, inv, 8 * q), inv1 = __shfl_sync(0xffffffffu, inv, 8 * q + 4);
    d[0] *= inv0;
    d[1] *= inv1;
    d[2] *= inv0;
    d[3] *= inv1;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const bool second = h >= 2;
      if (second ? okB : okA) {
        const int64_t gidx = (second ? rowB : rowA) * G + gi;
        const float sv = (h & 1) ? sv1 : sv0;
        Y[h] += fmaf(__half2float(down.scales[gidx]), d[h], __half2float(down.biases[gidx]) * sv);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int pp = it.pb + 2 * q + (h & 1);
    const int row = r0 + g + (h >= 2 ? 8 : 0);
    if (pp < it.pe && row < s.din) {
      int t, k;
      pair_of(it, sm, pp, K, &t, &k);
      const int slot = it.shared ? K + it.e : k;
      p.y[(static_cast<int64_t>(t) * ny + slot) * s.din + row] = Y[h];
    }
  }
}

// ------------------------------------------------------------------ kernels
// Block 0: route inversion, the ids export and the bad-id flag; block t < m: token t's shared
// scalar sigmoid(x_t . gate_vec) (1 without a gate vector).
__global__ void __launch_bounds__(kThreads) mma_prep_kernel(const MmaParams p) {
  const LayerShape &s = p.s;
  const int t = blockIdx.x;
  if (s.n_shared > 0) {
    float v = 1.f;
    if (p.w.gate_vec != nullptr) {
      __shared__ float part[kWarps];
      float dot = 0.f;
      for (int c = threadIdx.x; c < s.din; c += kThreads)
        dot = fmaf(bf16_to_float(p.x[static_cast<int64_t>(t) * s.din + c]),
                   bf16_to_float(p.w.gate_vec[c]), dot);
      dot = warp_sum(dot);
      if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = dot;
      __syncthreads();
      dot = 0.f;
      for (int w = 0; w < kWarps; ++w) dot += part[w];
      v = 1.0f / (1.0f + expf(-dot));
    }
    if (threadIdx.x == 0) p.sscal[t] = v;
  }
  if (blockIdx.x != 0) return;
  const int n = p.m * s.top_k;
  __shared__ Route rt;
  __shared__ int ids_s[kMaxPairs];
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const int e = p.ids[i];
    ids_s[i] = e;
    if (p.ids_used != nullptr) p.ids_used[i] = e;
    if (e < 0 || e >= s.n_experts) atomicOr(p.err, kDevErrBadId);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    route_invert_warp(ids_s, n, s.n_experts, rt, lane);
    __syncwarp();
    const int U = rt.n_uniq;
    if (lane == 0) p.route[0] = U;
    for (int u = lane; u < U; u += 32) p.route[1 + u] = rt.uniq[u];
    for (int u = lane; u <= U; u += 32) p.route[1 + U + u] = rt.offs[u];
    for (int i = lane; i < rt.n_pairs; i += 32) p.route[2 + 2 * U + i] = rt.pairs[i];
  }
}

template <int BR, int BS>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) gate_up_mma_kernel(const MmaParams p) {
  __shared__ MmaSmem sm;
  const LayerShape &s = p.s;
  const int tiles = (s.dff + 15) / 16, tiles_s = (s.dff_shared + 15) / 16;
  load_route(p.route, tiles, sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * kWarps;
  for (int idx = blockIdx.x * kWarps + warp;; idx += nw) {
    Item it;
    if (!item_of(idx, sm, p.m, s.n_shared, tiles, tiles_s, it)) break;
    if (it.shared)
      gate_up_item<BS>(p, p.w.sh_gate, p.w.sh_up, s.dff_shared, it, sm, lane);
    else
      gate_up_item<BR>(p, p.w.gate, p.w.up, s.dff, it, sm, lane);
  }
}

template <int BD, int BS>
__global__ void __launch_bounds__(kThreads, kCtasPerSmDown) down_mma_kernel(const MmaParams p) {
  __shared__ MmaSmem sm;
  const LayerShape &s = p.s;
  const int tiles = (s.din + 15) / 16;
  load_route(p.route, tiles, sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * kWarps;
  for (int idx = blockIdx.x * kWarps + warp;; idx += nw) {
    Item it;
    if (!item_of(idx, sm, p.m, s.n_shared, tiles, tiles, it)) break;
    if (it.shared)
      down_item<BS>(p, p.w.sh_down, s.dff_shared, it, sm, lane);
    else
      down_item<BD>(p, p.w.down, s.dff, it, sm, lane);
  }
}

// out[t][i] = resid[t][i] + (the token's valid slots in slot order, then its shared experts).
__global__ void tail_mma_kernel(const MmaParams p) {
  const LayerShape &s = p.s;
  const int ny = s.top_k + s.n_shared;
  const int64_t n = static_cast<int64_t>(p.m) * s.din;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(x / s.din);
    const int i = static_cast<int>(x - static_cast<int64_t>(t) * s.din);
    const float *yt = p.y + static_cast<int64_t>(t) * ny * s.din + i;
    float sum = 0.f;
    for (int k = 0; k < s.top_k; ++k) {
      const int e = p.ids[t * s.top_k + k];
      if (e >= 0 && e < s.n_experts) sum += yt[static_cast<int64_t>(k) * s.din];
    }
    for (int sh = 0; sh < s.n_shared; ++sh) sum += yt[static_cast<int64_t>(s.top_k + sh) * s.din];
    const float r = p.resid_f32 ? static_cast<const float *>(p.resid)[x]
                                : bf16_to_float(static_cast<const uint16_t *>(p.resid)[x]);
    const float v = r + sum;
    if (p.out_f32)
      static_cast<float *>(p.out)[x] = v;
    else
      static_cast<uint16_t *>(p.out)[x] = float_to_bf16_rn(v);
  }
}

}  // namespace mma

#define MOE_MMA_BITS(B, NAME, ...)                            \
  switch (B) {                                                \
    case 4: { constexpr int NAME = 4; __VA_ARGS__; } break;   \
    case 6: { constexpr int NAME = 6; __VA_ARGS__; } break;   \
    case 8: { constexpr int NAME = 8; __VA_ARGS__; } break;   \
    default: return cudaErrorInvalidValue;                    \
  }

cudaError_t launch_mma_layer(const MmaParams &p, int bits_gu, int bits_d, int bits_sh,
                             cudaStream_t stream) {
  if (p.m < 1 || p.m > kMaxGroupTokens || p.m * p.s.top_k > kMaxPairs ||
      p.s.n_experts > kMaxGroupExperts)
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int grid = mma::kCtasPerSm * sms, grid_d = mma::kCtasPerSmDown * sms;
  mma::mma_prep_kernel<<<p.m, mma::kThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int bs = p.s.n_shared > 0 ? bits_sh : 4;
  MOE_MMA_BITS(bits_gu, BR, MOE_MMA_BITS(bs, BS,
      (mma::gate_up_mma_kernel<BR, BS><<<grid, mma::kThreads, 0, stream>>>(p))));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  MOE_MMA_BITS(bits_d, BD, MOE_MMA_BITS(bs, BS,
      (mma::down_mma_kernel<BD, BS><<<grid_d, mma::kThreads, 0, stream>>>(p))));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n = static_cast<int64_t>(p.m) * p.s.din;
  const int tg = static_cast<int>((n + 255) / 256);
  mma::tail_mma_kernel<<<tg, 256, 0, stream>>>(p);
  return cudaGetLastError();
}
#undef MOE_MMA_BITS

}  // namespace moe
