// moe_mma.cu -- the tensor-core batch variant of the block (MOE_KERNELS_MMA): m tokens, their
// slots grouped by expert, every projection on tensor-core tiles.
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
// pairs that name it and runs mma.sync.m16n8k16 (fp32 accumulation) over one group of 64 codes
// at a time, then adds s * D + b * sum(v) for the group's scale s and bias b:
//   sum_c (s q_c + b) v_c = s * (sum_c q_c v_c) + b * sum_c v_c.
// Codes enter the tensor core exactly, as the 16-bit floats M + q: a shift and one mask-and-OR
// place a code pair in the mantissas of a float pair whose exponent fields hold M (M = 16, 64 or
// 256 for 4-, 6- or 8-bit codes: the binade [M, 2M) spaces its floats by 1 or finer), and the
// epilogue removes the bias in fp32, sum_c (M + q_c) v_c - M sum_c v_c.  4- and 6-bit gate/up
// codes meet x on bf16 tiles (x is bf16: the products are exact); 8-bit gate/up codes (256 + q
// does not fit bf16's 8 significant bits) and every down projection use fp16 tiles, the vector
// scaled per group by a power of two 2^k that puts its largest magnitude in [2^14, 2^15) and split
// into an fp16 high part and an fp16 remainder (two tiles, 22 significant bits); the column's
// group sum is multiplied by 2^-k.
//
// Data path: each warp streams its blocks of the tile-group copy (moe_mma.cuh) through a private
// ring of kStages shared-memory slots, each holding up to kGroupsPerStage consecutive blocks and
// filled by one bulk copy (the TMA engine) on an mbarrier; the vector operands (x, or the
// activation's fp16 parts) and the per-(column, group) sums are read from global memory (L2)
// when a stage is consumed.  Work units are (item, chunk): a chunk is a
// balanced range of the item's groups, the chunk count chosen from the route so that every warp
// gets several units; chunk sums are added in chunk order by the next kernel (deterministic).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "moe_mma.cuh"
#include "moe_phases.cuh"

namespace moe {
namespace mma {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;          // ring slots per warp
constexpr int kGroupsPerStage = 2;  // blocks one bulk copy carries, at most
constexpr int kMinCtas = 2;         // CTAs per SM the register budget is sized for
constexpr int kUnitsPerWarp = 6;    // the chunk count aims at this many units per warp

// ------------------------------------------------------------------ tensor-core instructions
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

__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
  return *reinterpret_cast<const uint32_t *>(&h);
}

// ------------------------------------------------------------------ code words
// One lane's code words of one projection in a block region (layout in moe_mma.cuh).
template <int BITS>
__device__ __forceinline__ void lds_codes(const uint8_t *region, int lane, uint32_t (&w)[8]) {
  const uint4 a = *reinterpret_cast<const uint4 *>(region + 16 * lane);
  w[0] = a.x;
  w[1] = a.y;
  w[2] = a.z;
  w[3] = a.w;
  if constexpr (BITS == 8) {
    const uint4 b = *reinterpret_cast<const uint4 *>(region + 512 + 16 * lane);
    w[4] = b.x;
    w[5] = b.y;
    w[6] = b.z;
    w[7] = b.w;
  } else if constexpr (BITS == 6) {
    const uint2 h = *reinterpret_cast<const uint2 *>(region + 512 + 8 * lane);
    w[4] = h.x;
    w[5] = h.y;
  }
}

// x shifted left by s bits (right by -s): s is a compile-time constant after unrolling.
__device__ __forceinline__ uint32_t shl(uint32_t x, int s) { return s >= 0 ? x << s : x >> -s; }

// The bias M of a code width: 16, 64 or 256.
template <int BITS>
struct Bias {
  static constexpr float M = BITS == 4 ? 16.f : (BITS == 6 ? 64.f : 256.f);
};

// Fragment register r of k-step j: the code pair as the 16-bit floats (M + q0, M + q1), bf16
// (F16 false: 4- and 6-bit codes) or fp16.  The code's bits go to the mantissa's top bits
// below the exponent field that holds M.
template <int BITS, bool F16>
__device__ __forceinline__ uint32_t biased_pair(const uint32_t (&w)[8], int j, int r) {
  if constexpr (BITS == 4) {
    // bf16 16 + q: q at bits 3..6 under 0x4180; fp16 16 + q: q at bits 6..9 under 0x4c00
    constexpr int pos = F16 ? 6 : 3;
    constexpr uint32_t mask = 0x000f000fu << pos, magic = F16 ? 0x4c004c00u : 0x41804180u;
    return (shl(w[j], pos - 4 * r) & mask) | magic;
  } else if constexpr (BITS == 8) {
    // fp16 256 + q: q at bits 2..9 under 0x5c00
    return (shl(w[2 * j + (r >> 1)], 2 - 8 * (r & 1)) & 0x03fc03fcu) | 0x5c005c00u;
  } else {
    // bf16 64 + q: q at bits 1..6 under 0x4280; fp16 64 + q: q at bits 4..9 under 0x5400
    constexpr int pos = F16 ? 4 : 1;
    constexpr uint32_t lo_mask = 0x000f000fu << pos, hi_mask = 0x00030003u << (pos + 4);
    constexpr uint32_t magic = F16 ? 0x54005400u : 0x42804280u;
    const int p = 4 * (j & 1) + r;
    const uint32_t hi = (shl(w[4 + (j >> 1)], pos + 4 - 2 * p) & hi_mask) | magic;
    return (shl(w[j], pos - 4 * r) & lo_mask) | hi;
  }
}

// D += (M + codes) x B over one group: bf16 tiles (B = bf16 pairs) or fp16 tiles (B = high parts
// and remainders).
template <int BITS, bool F16>
__device__ __forceinline__ void group_mma(const uint32_t (&w)[8], const uint32_t (&bh)[8],
                                          const uint32_t (&bl)[8], float (&d)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t a[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = biased_pair<BITS, F16>(w, j, r);
    if constexpr (F16) {
      mma_f16(d, a, bh[2 * j], bh[2 * j + 1]);
      mma_f16(d, a, bl[2 * j], bl[2 * j + 1]);
    } else {
      mma_bf16(d, a, bh[2 * j], bh[2 * j + 1]);
    }
  }
}

// ------------------------------------------------------------------ route and work units
struct MmaSmem {
  int U, n_items_r, n_items, nc;
  int uniq[kMaxPairs];
  int offs[kMaxPairs + 1];
  int pairs[kMaxPairs];
  int ibase[kMaxPairs + 1];
  uint64_t bar[kWarps][kStages];
};

struct Item {
  bool shared;
  int e;        // expert id (routed) or shared expert index
  int tile;     // 16-row tile
  int pb, pe;   // pairs [pb, pe): entries of the route's pair list (routed) or tokens (shared)
};

// The route into shared memory, the item counts (ibase[u] = first item of distinct expert u:
// ceil(pairs_u / 8) pair tiles x tiles_r row tiles; then each shared expert: ceil(m / 8) x
// tiles_s) and the chunk count: about kUnitsPerWarp units per warp, at most kMmaMaxChunks and
// g_min (every chunk of every class holds a group).  CTA 0 publishes the chunk count.
__device__ void load_route(const MmaParams &p, int tiles_r, int tiles_s, int g_min,
                           int32_t *nc_out, MmaSmem &sm) {
  const int32_t *route = p.route;
  const int U = route[0];
  if (threadIdx.x == 0) sm.U = U;
  for (int u = threadIdx.x; u < U; u += blockDim.x) sm.uniq[u] = route[1 + u];
  for (int u = threadIdx.x; u <= U; u += blockDim.x) sm.offs[u] = route[1 + U + u];
  __syncthreads();
  const int np = sm.offs[U];
  for (int i = threadIdx.x; i < np; i += blockDim.x) sm.pairs[i] = route[2 + 2 * U + i];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    constexpr int PER = kMaxPairs / 32;
    int loc[PER], sum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int u = lane * PER + j;
      loc[j] = u < U ? ((sm.offs[u + 1] - sm.offs[u] + 7) / 8) * tiles_r : 0;
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
    if (lane == 31) {
      const int items = incl + ((p.m + 7) / 8) * tiles_s * p.s.n_shared;
      const int64_t want = static_cast<int64_t>(kUnitsPerWarp) * gridDim.x * kWarps;
      int nc = items > 0 ? static_cast<int>((want + items - 1) / items) : 1;
      nc = min(nc, min(kMmaMaxChunks, g_min));
      nc = max(nc, 1);
      sm.n_items_r = incl;
      sm.n_items = items;
      sm.nc = nc;
      if (blockIdx.x == 0) *nc_out = nc;
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void item_of(int idx, const MmaSmem &sm, int m, int tiles_r,
                                        int tiles_s, Item &it) {
  if (idx < sm.n_items_r) {
    int lo = 0, hi = sm.U;  // ibase[lo] <= idx < ibase[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sm.ibase[mid] <= idx) lo = mid;
      else hi = mid;
    }
    const int rel = idx - sm.ibase[lo];
    const int pt = rel / tiles_r;
    it.shared = false;
    it.e = sm.uniq[lo];
    it.tile = rel - pt * tiles_r;
    it.pb = sm.offs[lo] + 8 * pt;
    it.pe = min(it.pb + 8, sm.offs[lo + 1]);
    return;
  }
  idx -= sm.n_items_r;
  const int per = ((m + 7) / 8) * tiles_s;
  const int sh = idx / per, rel = idx - sh * per, pt = rel / tiles_s;
  it.shared = true;
  it.e = sh;
  it.tile = rel - pt * tiles_s;
  it.pb = 8 * pt;
  it.pe = min(it.pb + 8, m);
}

// (token, slot) of pair entry i of an item; slot -1 for a shared expert's token.
__device__ __forceinline__ void pair_of(const Item &it, const MmaSmem &sm, int i, int K, int *t,
                                        int *k) {
  if (it.shared) {
    *t = i;
    *k = -1;
  } else {
    const int v = sm.pairs[i];
    *t = v / K;
    *k = v - *t * K;
  }
}

// Geometry of one kernel's two classes.
struct Geo {
  int tiles_r, tiles_s;   // row tiles per expert
  int G_r, G_s;           // groups per row tile
  int B_r, B_s;           // block bytes
  const uint8_t *base_r, *base_s;
};

// A warp's position in its stream of stages.
struct Cursor {
  int unit;              // -1 past the end
  Item it;
  int c;                 // chunk of the item
  int g, g1;             // next group, chunk end
  int bb;                // block bytes of the item's class
  const uint8_t *src;    // block of group g
};

__device__ __forceinline__ void cursor_at(Cursor &cu, int unit, const MmaSmem &sm, int m,
                                          const Geo &geo) {
  if (unit >= sm.n_items * sm.nc) {
    cu.unit = -1;
    return;
  }
  cu.unit = unit;
  const int item = unit / sm.nc;
  item_of(item, sm, m, geo.tiles_r, geo.tiles_s, cu.it);
  cu.c = unit - item * sm.nc;
  const bool s = cu.it.shared;
  const int G = s ? geo.G_s : geo.G_r, tiles = s ? geo.tiles_s : geo.tiles_r;
  cu.g = cu.c * G / sm.nc;
  cu.g1 = (cu.c + 1) * G / sm.nc;
  cu.bb = s ? geo.B_s : geo.B_r;
  cu.src = (s ? geo.base_s : geo.base_r) +
           (static_cast<int64_t>(cu.it.e * tiles + cu.it.tile) * G + cu.g) * cu.bb;
}

// Groups of the cursor's next stage.
__device__ __forceinline__ int stage_groups(const Cursor &cu) {
  return min(kGroupsPerStage, cu.g1 - cu.g);
}

// Issues the bulk copy of the cursor's next stage (consecutive blocks) and moves past it.
__device__ __forceinline__ void issue_stage(Cursor &pc, const MmaSmem &sm, int m, const Geo &geo,
                                            int nw, uint8_t *dst, uint64_t *bar,
                                            uint64_t policy) {
  const int n = stage_groups(pc);
  const uint32_t bytes = static_cast<uint32_t>(n * pc.bb);
  mbar_arrive_expect_tx(bar, bytes);
  bulk_g2s(dst, pc.src, bytes, bar, policy);
  pc.g += n;
  pc.src += bytes;
  if (pc.g == pc.g1) cursor_at(pc, pc.unit + nw, sm, m, geo);
}

// Per lane, for the current unit: where the vector operand of its B column (pair pb + g) and the
// sums and 2^-k of its two D columns (pairs pb + 2q, pb + 2q + 1) are, as pointers to the unit's
// first group and steps per group (step 0 on a zero page for an absent column), and the D
// columns' (token, slot) for the unit's end.
struct Feed {
  const uint4 *b;
  int bstep;
  const float *sum[2], *inv[2];
  int sstep[2];
  int t[2], k[2];
};

// act_vectors false: x (bf16, or its fp16 parts when f16), groups of din; true: the activation's
// fp16 parts, groups of the activation row.
__device__ __forceinline__ void feed_of(const Cursor &cu, const MmaSmem &sm, const MmaParams &p,
                                        bool act_vectors, bool f16, int lane, Feed &f) {
  const LayerShape &s = p.s;
  const int g = lane >> 2, q = lane & 3, K = s.top_k;
  const int groups = act_vectors ? p.act_stride / kGroup : s.din / kGroup;
  auto seg = [&](int k) {
    if (!act_vectors) return 0;
    return cu.it.shared ? (K * s.dff + cu.it.e * s.dff_shared) / kGroup : k * s.dff / kGroup;
  };
  const uint4 *zero = reinterpret_cast<const uint4 *>(p.zero);
  f.b = zero;
  f.bstep = 0;
  if (cu.it.pb + g < cu.it.pe) {
    int t, k;
    pair_of(cu.it, sm, cu.it.pb + g, K, &t, &k);
    const int64_t grp = static_cast<int64_t>(t) * groups + seg(k) + cu.g;
    if (f16) {
      const __half *v16 = act_vectors ? p.a16 : p.x16;
      f.b = reinterpret_cast<const uint4 *>(v16 + (grp * 4 + q) * 32);
      f.bstep = 16;   // 128 halves per group
    } else {
      f.b = reinterpret_cast<const uint4 *>(p.x + grp * kGroup + 16 * q);
      f.bstep = 8;    // 64 bf16 per group
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = cu.it.pb + 2 * q + h;
    f.sum[h] = f.inv[h] = p.zero;
    f.sstep[h] = 0;
    f.t[h] = -1;
    f.k[h] = -1;
    if (i < cu.it.pe) {
      int t, k;
      pair_of(cu.it, sm, i, K, &t, &k);
      const int64_t grp = static_cast<int64_t>(t) * groups + seg(k) + cu.g;
      f.sum[h] = (act_vectors ? p.asum : p.xsum) + grp;
      f.inv[h] = (act_vectors ? p.ainv : p.xinv) + grp;
      f.sstep[h] = 1;
      f.t[h] = t;
      f.k[h] = k;
    }
  }
}

__device__ __forceinline__ void feed_skip(Feed &f, int n) {
  f.b += n * f.bstep;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    f.sum[h] += n * f.sstep[h];
    f.inv[h] += n * f.sstep[h];
  }
}

// The vector operand of one group for this lane, and its D columns' (sum, 2^-k).
struct Operand {
  uint32_t h[8], l[8];
  float sum[2], inv[2];
};

__device__ __forceinline__ void unpack4(uint4 v, uint32_t *o) {
  o[0] = v.x;
  o[1] = v.y;
  o[2] = v.z;
  o[3] = v.w;
}

// Group i of the feed's current stage.
template <bool F16>
__device__ __forceinline__ void load_operand(const Feed &f, int i, Operand &o) {
  const uint4 *b = f.b + i * f.bstep;
  unpack4(__ldg(b), o.h);
  unpack4(__ldg(b + 1), o.h + 4);
  if constexpr (F16) {
    unpack4(__ldg(b + 2), o.l);
    unpack4(__ldg(b + 3), o.l + 4);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    o.sum[h] = __ldg(f.sum[h] + i * f.sstep[h]);
    o.inv[h] = F16 ? __ldg(f.inv[h] + i * f.sstep[h]) : 1.f;
  }
}

// ------------------------------------------------------------------ the streaming loop
// Streams a warp's units through its ring, one stage (up to kGroupsPerStage blocks) at a time:
// consume(cursor, feed, stage, groups) adds the stage's groups, finish(cursor, feed) ends a unit.
template <class Consume, class Finish>
__device__ void stream_units(const MmaParams &p, MmaSmem &sm, const Geo &geo, uint8_t *ring,
                             int slot_bytes, bool act_vectors, bool f16_r, bool f16_s,
                             Consume consume, Finish finish) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = gridDim.x * kWarps;
  uint64_t *bar = sm.bar[warp];
  uint8_t *myring = ring + static_cast<size_t>(warp) * kStages * slot_bytes;
  const uint64_t policy = policy_evict_first();
  Cursor cu;
  cursor_at(cu, blockIdx.x * kWarps + warp, sm, p.m, geo);
  Cursor pc = cu;
  int issued = 0, pslot = 0;
  if (lane == 0) {
    for (; issued < kStages && pc.unit >= 0; ++issued, ++pslot)
      issue_stage(pc, sm, p.m, geo, nw, myring + pslot * slot_bytes, &bar[pslot], policy);
    if (pslot == kStages) pslot = 0;
  }
  Feed feed;
  if (cu.unit >= 0) feed_of(cu, sm, p, act_vectors, cu.it.shared ? f16_s : f16_r, lane, feed);
  int used = 0, slot = 0;
  uint32_t phase = 0;
  while (cu.unit >= 0) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar[slot], phase));
    if (!ok) {
      // a copy that never landed: flag it, wait (bounded) for the others in flight, give up
      if (lane == 0) atomicOr(p.err, kDevErrTimeout);
      const int inflight = __shfl_sync(0xffffffffu, issued, 0) - used;
      for (int i = 1; i < inflight; ++i)
        mbar_wait(&bar[(slot + i) % kStages], phase ^ static_cast<uint32_t>((slot + i) >= kStages));
      return;
    }
    const int ng = stage_groups(cu);
    consume(cu, feed, myring + slot * slot_bytes, ng);
    __syncwarp();
    if (lane == 0 && pc.unit >= 0) {
      issue_stage(pc, sm, p.m, geo, nw, myring + pslot * slot_bytes, &bar[pslot], policy);
      ++issued;
      if (++pslot == kStages) pslot = 0;
    }
    ++used;
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
    cu.g += ng;
    feed_skip(feed, ng);
    if (cu.g == cu.g1) {
      finish(cu, feed);
      cursor_at(cu, cu.unit + nw, sm, p.m, geo);
      if (cu.unit >= 0) feed_of(cu, sm, p, act_vectors, cu.it.shared ? f16_s : f16_r, lane, feed);
    }
  }
}

__device__ __forceinline__ void init_bars(MmaSmem &sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&sm.bar[warp][i], 1);
    mbar_fence_init();
  }
  __syncwarp();
}

// acc[h] += s * (D'[h] * inv - M * sum) + b * sum for this lane's rows g (h < 2) and g + 8, with
// (s, b) of the two rows in sbA, sbB.
template <int BITS>
__device__ __forceinline__ void group_epilogue(const float (&d)[4], __half2 sbA, __half2 sbB,
                                               const Operand &o, float (&acc)[4]) {
  constexpr float M = Bias<BITS>::M;
  const float2 A = __half22float2(sbA), B = __half22float2(sbB);
  const float ms0 = -M * o.sum[0], ms1 = -M * o.sum[1];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float2 sb = h < 2 ? A : B;
    const float sum = o.sum[h & 1];
    const float dot = fmaf(d[h], o.inv[h & 1], (h & 1) ? ms1 : ms0);   // sum_c q_c v_c
    acc[h] = fmaf(sb.x, dot, fmaf(sb.y, sum, acc[h]));
  }
}

// ------------------------------------------------------------------ gate/up
// One gate/up block: both projections against the same operand.
template <int BITS>
__device__ __forceinline__ void gu_block(const uint8_t *blk, int lane, const Operand &o,
                                         float (&acc_g)[4], float (&acc_u)[4]) {
  constexpr bool F16 = BITS == 8;
  constexpr int region = 32 * 4 * BITS;
  const int g = lane >> 2;
  float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t w[8];
  lds_codes<BITS>(blk, lane, w);
  group_mma<BITS, F16>(w, o.h, o.l, dg);
  lds_codes<BITS>(blk + region, lane, w);
  group_mma<BITS, F16>(w, o.h, o.l, du);
  const uint4 sbw = *reinterpret_cast<const uint4 *>(blk + 2 * region + 16 * g);
  group_epilogue<BITS>(dg, *reinterpret_cast<const __half2 *>(&sbw.x),
                       *reinterpret_cast<const __half2 *>(&sbw.y), o, acc_g);
  group_epilogue<BITS>(du, *reinterpret_cast<const __half2 *>(&sbw.z),
                       *reinterpret_cast<const __half2 *>(&sbw.w), o, acc_u);
}

template <int BITS>
__device__ __forceinline__ void gu_stage(const Feed &f, const uint8_t *stage, int ng, int lane,
                                         float (&acc_g)[4], float (&acc_u)[4]) {
  constexpr bool F16 = BITS == 8;
  constexpr int bb = 256 * BITS + 128;
  if (ng == 2 && !F16) {
    Operand o0, o1;
    load_operand<F16>(f, 0, o0);
    load_operand<F16>(f, 1, o1);
    gu_block<BITS>(stage, lane, o0, acc_g, acc_u);
    gu_block<BITS>(stage + bb, lane, o1, acc_g, acc_u);
  } else {
    for (int i = 0; i < ng; ++i) {
      Operand o;
      load_operand<F16>(f, i, o);
      gu_block<BITS>(stage + i * bb, lane, o, acc_g, acc_u);
    }
  }
}

template <int BR, int BS>
__global__ void __launch_bounds__(kThreads, kMinCtas) gate_up_mma_kernel(const MmaParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ MmaSmem sm;
  const LayerShape &s = p.s;
  Geo geo;
  geo.tiles_r = s.dff / 16;
  geo.tiles_s = s.dff_shared / 16;
  geo.G_r = geo.G_s = s.din / kGroup;
  geo.B_r = mma_gu_block(BR);
  geo.B_s = mma_gu_block(BS);
  geo.base_r = p.t.gu_r;
  geo.base_s = p.t.gu_s;
  const int slot_bytes =
      kGroupsPerStage * max(s.top_k > 0 ? geo.B_r : 0, s.n_shared > 0 ? geo.B_s : 0);
  init_bars(sm);
  load_route(p, geo.tiles_r, geo.tiles_s, geo.G_r, &p.nc[0], sm);
  const int lane = threadIdx.x & 31, g = lane >> 2;
  float acc_g[4] = {0.f, 0.f, 0.f, 0.f}, acc_u[4] = {0.f, 0.f, 0.f, 0.f};

  auto consume = [&](const Cursor &cu, const Feed &f, const uint8_t *stage, int ng) {
    if (!cu.it.shared) gu_stage<BR>(f, stage, ng, lane, acc_g, acc_u);
    else gu_stage<BS>(f, stage, ng, lane, acc_g, acc_u);
  };
  auto finish = [&](const Cursor &cu, const Feed &f) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int col = h & 1;
      if (f.t[col] >= 0) {
        const int row = 16 * cu.it.tile + g + (h >= 2 ? 8 : 0);
        const int64_t seg = cu.it.shared
                                ? static_cast<int64_t>(s.top_k) * s.dff +
                                      static_cast<int64_t>(cu.it.e) * s.dff_shared
                                : static_cast<int64_t>(f.k[col]) * s.dff;
        p.gu_part[(static_cast<int64_t>(cu.c) * p.m + f.t[col]) * p.act_stride + seg + row] =
            make_float2(acc_g[h], acc_u[h]);
      }
      acc_g[h] = acc_u[h] = 0.f;
    }
  };
  stream_units(p, sm, geo, ring, slot_bytes, false, BR == 8, BS == 8, consume, finish);
}

// ------------------------------------------------------------------ down
template <int BITS>
__device__ __forceinline__ void down_block(const uint8_t *blk, int lane, const Operand &o,
                                           float (&acc)[4]) {
  constexpr int region = 32 * 4 * BITS;
  const int g = lane >> 2;
  float d[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t w[8];
  lds_codes<BITS>(blk, lane, w);
  group_mma<BITS, true>(w, o.h, o.l, d);
  const uint2 sbw = *reinterpret_cast<const uint2 *>(blk + region + 8 * g);
  group_epilogue<BITS>(d, *reinterpret_cast<const __half2 *>(&sbw.x),
                       *reinterpret_cast<const __half2 *>(&sbw.y), o, acc);
}

template <int BITS>
__device__ __forceinline__ void down_stage(const Feed &f, const uint8_t *stage, int ng, int lane,
                                           float (&acc)[4]) {
  constexpr int bb = 128 * BITS + 64;
  if (ng == 2) {
    Operand o0, o1;
    load_operand<true>(f, 0, o0);
    load_operand<true>(f, 1, o1);
    down_block<BITS>(stage, lane, o0, acc);
    down_block<BITS>(stage + bb, lane, o1, acc);
  } else {
    Operand o;
    load_operand<true>(f, 0, o);
    down_block<BITS>(stage, lane, o, acc);
  }
}

template <int BR, int BS>
__global__ void __launch_bounds__(kThreads, kMinCtas) down_mma_kernel(const MmaParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ MmaSmem sm;
  const LayerShape &s = p.s;
  Geo geo;
  geo.tiles_r = geo.tiles_s = s.din / 16;
  geo.G_r = s.dff / kGroup;
  geo.G_s = s.n_shared > 0 ? s.dff_shared / kGroup : geo.G_r;
  geo.B_r = mma_dn_block(BR);
  geo.B_s = mma_dn_block(BS);
  geo.base_r = p.t.dn_r;
  geo.base_s = p.t.dn_s;
  const int slot_bytes =
      kGroupsPerStage * max(s.top_k > 0 ? geo.B_r : 0, s.n_shared > 0 ? geo.B_s : 0);
  init_bars(sm);
  const int g_min = s.top_k > 0 ? min(geo.G_r, geo.G_s) : geo.G_s;
  load_route(p, geo.tiles_r, geo.tiles_s, g_min, &p.nc[1], sm);
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const int ny = s.top_k + s.n_shared;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  auto consume = [&](const Cursor &cu, const Feed &f, const uint8_t *stage, int ng) {
    if (!cu.it.shared) down_stage<BR>(f, stage, ng, lane, acc);
    else down_stage<BS>(f, stage, ng, lane, acc);
  };
  auto finish = [&](const Cursor &cu, const Feed &f) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int col = h & 1;
      if (f.t[col] >= 0) {
        const int row = 16 * cu.it.tile + g + (h >= 2 ? 8 : 0);
        const int slot = cu.it.shared ? s.top_k + cu.it.e : f.k[col];
        p.y_part[((static_cast<int64_t>(cu.c) * p.m + f.t[col]) * ny + slot) * s.din + row] =
            acc[h];
      }
      acc[h] = 0.f;
    }
  };
  stream_units(p, sm, geo, ring, slot_bytes, true, true, true, consume, finish);
}

// ------------------------------------------------------------------ small kernels
// Writes a group of 64 values held two per lane (v0, v1 = values 2 lane, 2 lane + 1) as fp16
// parts scaled by 2^k (the x16 / a16 layout), its 2^-k and its sum.
__device__ __forceinline__ void pack_group(float v0, float v1, __half *dst, float *inv_out,
                                           float *sum_out, int lane) {
  const float mx = warp_max(fmaxf(fabsf(v0), fabsf(v1)));
  const float sum = warp_sum(v0 + v1);
  const int E = static_cast<int>((__float_as_uint(mx) >> 23) & 255u);
  const int k = min(141 - E, 126);  // puts mx in [2^14, 2^15); an all-zero group takes 2^126
  const float sc = pow2f(k);
  const float a = v0 * sc, b = v1 * sc;
  const __half2 hi = __floats2half2_rn(a, b);
  const __half2 lo = __floats2half2_rn(a - __low2float(hi), b - __high2float(hi));
  const int q = lane >> 3, i = 2 * (lane & 7);
  *reinterpret_cast<__half2 *>(dst + q * 32 + i) = hi;
  *reinterpret_cast<__half2 *>(dst + q * 32 + 16 + i) = lo;
  if (lane == 0) {
    *inv_out = pow2f(-k);
    *sum_out = sum;
  }
}

// Block t < m: x's group sums (and fp16 parts when an 8-bit gate/up class reads them) and the
// shared scalar sigmoid(x_t . gate_vec) (1 without a gate vector); block 0 also inverts the
// route, exports the ids and flags invalid ones.
__global__ void __launch_bounds__(kThreads) mma_prep_kernel(const MmaParams p) {
  const LayerShape &s = p.s;
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ Route rt;
  __shared__ int ids_s[kMaxPairs];
  __shared__ float part[kWarps];
  const int n = p.m * s.top_k;
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const int e = p.ids[i];
      ids_s[i] = e;
      if (p.ids_used != nullptr) p.ids_used[i] = e;
      if (e < 0 || e >= s.n_experts) atomicOr(p.err, kDevErrBadId);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0 && warp == 0) {
    route_invert_warp(ids_s, n, s.n_experts, rt, lane);
    __syncwarp();
    const int U = rt.n_uniq;
    if (lane == 0) p.route[0] = U;
    for (int u = lane; u < U; u += 32) p.route[1 + u] = rt.uniq[u];
    for (int u = lane; u <= U; u += 32) p.route[1 + U + u] = rt.offs[u];
    for (int i = lane; i < rt.n_pairs; i += 32) p.route[2 + 2 * U + i] = rt.pairs[i];
  }
  const int Gx = s.din / kGroup;
  const bool need16 = (s.top_k > 0 && p.bits_r == 8) || (s.n_shared > 0 && p.bits_s == 8);
  const uint16_t *xt = p.x + static_cast<int64_t>(t) * s.din;
  // a warp's groups kPrepBatch at a time: every load issued before the first reduction
  constexpr int kPrepBatch = 8;
  for (int g0 = warp; g0 < Gx; g0 += kWarps * kPrepBatch) {
    uint32_t two[kPrepBatch];
#pragma unroll
    for (int b = 0; b < kPrepBatch; ++b) {
      const int gi = g0 + b * kWarps;
      two[b] = gi < Gx ? *reinterpret_cast<const uint32_t *>(xt + gi * kGroup + 2 * lane) : 0u;
    }
#pragma unroll
    for (int b = 0; b < kPrepBatch; ++b) {
      const int gi = g0 + b * kWarps;
      if (gi >= Gx) break;
      const float v0 = __uint_as_float(two[b] << 16), v1 = __uint_as_float(two[b] & 0xffff0000u);
      const int64_t ix = static_cast<int64_t>(t) * Gx + gi;
      if (need16) {
        pack_group(v0, v1, p.x16 + ix * 128, p.xinv + ix, p.xsum + ix, lane);
      } else {
        const float sum = warp_sum(v0 + v1);
        if (lane == 0) p.xsum[ix] = sum;
      }
    }
  }
  if (s.n_shared > 0) {
    float v = 1.f;
    if (p.w.gate_vec != nullptr) {
      float dot = 0.f;
      for (int c = threadIdx.x; c < s.din; c += kThreads)
        dot = fmaf(bf16_to_float(xt[c]), bf16_to_float(p.w.gate_vec[c]), dot);
      dot = warp_sum(dot);
      if (lane == 0) part[warp] = dot;
      __syncthreads();
      dot = 0.f;
      for (int w = 0; w < kWarps; ++w) dot += part[w];
      v = 1.0f / (1.0f + expf(-dot));
    }
    if (threadIdx.x == 0) p.sscal[t] = v;
  }
}

// One warp per (token, group of 64 activation rows): the chunk sums in chunk order, SwiGLU times
// the slot's score (or the shared scalar), then the fp16 parts, 2^-k and sum of the group.
__global__ void __launch_bounds__(kThreads) mma_act_kernel(const MmaParams p) {
  const LayerShape &s = p.s;
  const int lane = threadIdx.x & 31;
  const int Ga = p.act_stride / kGroup;
  const int w = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (w >= p.m * Ga) return;
  const int t = w / Ga, ga = w - t * Ga;
  const int r0 = ga * kGroup, K = s.top_k;
  float coef;
  if (r0 < K * s.dff) {
    const int k = r0 / s.dff, e = p.ids[t * K + k];
    if (e < 0 || e >= s.n_experts) return;   // a dropped slot: nothing reads its groups
    coef = p.scores[t * K + k];
  } else {
    coef = p.sscal[t];
  }
  const int nc = p.nc[0];
  float v[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float gs = 0.f, us = 0.f;
    for (int c = 0; c < nc; ++c) {
      const float2 gu =
          p.gu_part[(static_cast<int64_t>(c) * p.m + t) * p.act_stride + r0 + 2 * lane + i];
      gs += gu.x;
      us += gu.y;
    }
    v[i] = coef * (silu_f(gs) * us);
  }
  const int64_t ix = static_cast<int64_t>(t) * Ga + ga;
  pack_group(v[0], v[1], p.a16 + ix * 128, p.ainv + ix, p.asum + ix, lane);
}

// out[t][i] = resid[t][i] + (the token's valid slots in slot order, then its shared experts),
// each slot's output the sum of its down chunks in chunk order.
__global__ void mma_tail_kernel(const MmaParams p) {
  const LayerShape &s = p.s;
  const int ny = s.top_k + s.n_shared;
  const int nc = p.nc[1];
  const int64_t n = static_cast<int64_t>(p.m) * s.din;
  const int64_t cstride = n * ny;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(x / s.din);
    const int i = static_cast<int>(x - static_cast<int64_t>(t) * s.din);
    const float *yt = p.y_part + static_cast<int64_t>(t) * ny * s.din + i;
    // eight slots at a time: every load issued first (a dropped slot's value is read, not used)
    float sum = 0.f;
    for (int k0 = 0; k0 < ny; k0 += 8) {
      float yv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float yk = 0.f;
        if (k0 + j < ny)
          for (int c = 0; c < nc; ++c)
            yk += yt[c * cstride + static_cast<int64_t>(k0 + j) * s.din];
        yv[j] = yk;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int k = k0 + j;
        if (k >= ny) break;
        bool valid = true;
        if (k < s.top_k) {
          const int e = p.ids[t * s.top_k + k];
          valid = e >= 0 && e < s.n_experts;
        }
        if (valid) sum += yv[j];
      }
    }
    const float r = p.resid_f32 ? static_cast<const float *>(p.resid)[x]
                                : bf16_to_float(static_cast<const uint16_t *>(p.resid)[x]);
    const float v = r + sum;
    if (p.out_f32)
      static_cast<float *>(p.out)[x] = v;
    else
      static_cast<uint16_t *>(p.out)[x] = float_to_bf16_rn(v);
  }
}

// ------------------------------------------------------------------ create-time repack
// Code c of row `row` of a canonical packed matrix with `rb` bytes per row.
__device__ __forceinline__ uint32_t canon_code(const uint8_t *codes, int64_t row, int64_t rb,
                                               int c, int bits) {
  const int64_t bit = static_cast<int64_t>(c) * bits;
  const uint8_t *b = codes + row * rb + (bit >> 3);
  const int o = static_cast<int>(bit & 7);
  uint32_t v = b[0];
  if (o + bits > 8) v |= static_cast<uint32_t>(b[1]) << 8;
  return (v >> o) & ((1u << bits) - 1u);
}

// Word wi of the lane payloads of one projection in a block (tile rows from row0, the group's
// columns from col0); layout in moe_mma.cuh.
__device__ uint32_t payload_word(const uint8_t *codes, int64_t row0, int64_t rb, int col0,
                                 int bits, int wi) {
  int lane, word;  // the lane, and the index of the word in its logical words w[0..7]
  if (bits == 4) {
    lane = wi >> 2;
    word = wi & 3;
  } else if (bits == 8) {
    lane = (wi & 127) >> 2;
    word = (wi >> 7) * 4 + (wi & 3);
  } else if (wi < 128) {
    lane = wi >> 2;
    word = wi & 3;
  } else {
    lane = (wi - 128) >> 1;
    word = 4 + ((wi - 128) & 1);
  }
  const int g = lane >> 2, q = lane & 3;
  auto code = [&](int r, int j, int second) {
    const int64_t row = row0 + g + 8 * (r & 1);
    const int c = col0 + 16 * q + 4 * j + 2 * (r >> 1) + second;
    return canon_code(codes, row, rb, c, bits);
  };
  uint32_t out = 0;
  if (bits == 4) {
    for (int r = 0; r < 4; ++r)
      out |= (code(r, word, 0) << (4 * r)) | (code(r, word, 1) << (16 + 4 * r));
  } else if (bits == 8) {
    const int j = word >> 1;
    for (int b = 0; b < 2; ++b) {
      const int r = 2 * (word & 1) + b;
      out |= (code(r, j, 0) << (8 * b)) | (code(r, j, 1) << (16 + 8 * b));
    }
  } else if (word < 4) {
    for (int r = 0; r < 4; ++r)
      out |= ((code(r, word, 0) & 15u) << (4 * r)) | ((code(r, word, 1) & 15u) << (16 + 4 * r));
  } else {
    const int jh = word - 4;
    for (int pp = 0; pp < 8; ++pp) {
      const int j = 2 * jh + (pp >> 2), r = pp & 3;
      out |= ((code(r, j, 0) >> 4) << (2 * pp)) | ((code(r, j, 1) >> 4) << (16 + 2 * pp));
    }
  }
  return out;
}

__global__ void repack_mma_gu_kernel(const uint8_t *gc, const __half *gs, const __half *gb,
                                     const uint8_t *uc, const __half *us, const __half *ub,
                                     int experts, int rows, int din, int bits, uint32_t *out) {
  const int G = din / kGroup, T = rows / 16;
  const int pw = 8 * mma_lane_bytes(bits);            // payload words per projection
  const int bw = mma_gu_block(bits) / 4;              // words per block
  const int64_t rb = static_cast<int64_t>(din) * bits / 8;
  const int64_t n = static_cast<int64_t>(experts) * T * G * bw;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int wi = static_cast<int>(x % bw);
    const int64_t blk = x / bw;
    const int gi = static_cast<int>(blk % G);
    const int64_t et = blk / G;                 // e * T + tile
    const int64_t row0 = (et / T) * rows + (et % T) * 16;
    uint32_t v;
    if (wi < 2 * pw) {
      const bool up = wi >= pw;
      v = payload_word(up ? uc : gc, row0, rb, gi * kGroup, bits, wi - (up ? pw : 0));
    } else {
      const int k = wi - 2 * pw;                // record g = k / 4, word k % 4
      const int g = k >> 2, part = k & 3;
      const int64_t row = row0 + g + ((part & 1) ? 8 : 0);
      const __half *S = part < 2 ? gs : us, *B = part < 2 ? gb : ub;
      const int64_t ix = row * G + gi;
      v = h2_bits(__halves2half2(S[ix], B[ix]));
    }
    out[x] = v;
  }
}

__global__ void repack_mma_down_kernel(const uint8_t *c, const __half *sc, const __half *bi,
                                       int experts, int din, int dff, int bits, uint32_t *out) {
  const int G = dff / kGroup, T = din / 16;
  const int pw = 8 * mma_lane_bytes(bits);
  const int bw = mma_dn_block(bits) / 4;
  const int64_t rb = static_cast<int64_t>(dff) * bits / 8;
  const int64_t n = static_cast<int64_t>(experts) * T * G * bw;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < n;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int wi = static_cast<int>(x % bw);
    const int64_t blk = x / bw;
    const int gi = static_cast<int>(blk % G);
    const int64_t et = blk / G;
    const int64_t row0 = (et / T) * din + (et % T) * 16;
    uint32_t v;
    if (wi < pw) {
      v = payload_word(c, row0, rb, gi * kGroup, bits, wi);
    } else {
      const int k = wi - pw;                    // record g = k / 2, word k % 2
      const int64_t row = row0 + (k >> 1) + ((k & 1) ? 8 : 0);
      const int64_t ix = row * G + gi;
      v = h2_bits(__halves2half2(sc[ix], bi[ix]));
    }
    out[x] = v;
  }
}

}  // namespace mma

cudaError_t launch_repack_mma_gu(const uint8_t *g_codes, const __half *g_scales,
                                 const __half *g_biases, const uint8_t *u_codes,
                                 const __half *u_scales, const __half *u_biases, int experts,
                                 int rows, int din, int bits, uint8_t *out, cudaStream_t stream) {
  if (rows % 16 || din % kGroup || (bits != 4 && bits != 6 && bits != 8))
    return cudaErrorInvalidValue;
  mma::repack_mma_gu_kernel<<<2048, 256, 0, stream>>>(g_codes, g_scales, g_biases, u_codes,
                                                      u_scales, u_biases, experts, rows, din,
                                                      bits, reinterpret_cast<uint32_t *>(out));
  return cudaGetLastError();
}

cudaError_t launch_repack_mma_down(const uint8_t *codes, const __half *scales,
                                   const __half *biases, int experts, int din, int dff, int bits,
                                   uint8_t *out, cudaStream_t stream) {
  if (din % 16 || dff % kGroup || (bits != 4 && bits != 6 && bits != 8))
    return cudaErrorInvalidValue;
  mma::repack_mma_down_kernel<<<2048, 256, 0, stream>>>(codes, scales, biases, experts, din, dff,
                                                        bits, reinterpret_cast<uint32_t *>(out));
  return cudaGetLastError();
}

namespace {

// A streaming kernel with every warp's ring in dynamic shared memory, one CTA per resident slot
// (the units are strided over the whole grid).
template <class K>
cudaError_t launch_streaming(K kernel, int slot_bytes, const MmaParams &p, cudaStream_t stream) {
  const int dyn = mma::kWarps * mma::kStages * mma::kGroupsPerStage * slot_bytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, mma::kThreads, dyn)) !=
      cudaSuccess)
    return e;
  if (per < 1) return cudaErrorInvalidConfiguration;
  kernel<<<per * sms, mma::kThreads, dyn, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

#define MOE_MMA_BITS(B, NAME, ...)                            \
  switch (B) {                                                \
    case 4: { constexpr int NAME = 4; __VA_ARGS__; } break;   \
    case 6: { constexpr int NAME = 6; __VA_ARGS__; } break;   \
    case 8: { constexpr int NAME = 8; __VA_ARGS__; } break;   \
    default: return cudaErrorInvalidValue;                    \
  }

cudaError_t launch_mma_layer(const MmaParams &p, cudaStream_t stream) {
  const LayerShape &s = p.s;
  if (p.m < 1 || p.m > kMaxGroupTokens || p.m * s.top_k > kMaxPairs ||
      s.n_experts > kMaxGroupExperts || s.din % kGroup || s.dff % kGroup ||
      (s.n_shared > 0 && s.dff_shared % kGroup))
    return cudaErrorInvalidValue;
  cudaError_t e;
  mma::mma_prep_kernel<<<p.m, mma::kThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int br = s.top_k > 0 ? p.bits_r : p.bits_s, bs = s.n_shared > 0 ? p.bits_s : p.bits_r;
  const int dr = s.top_k > 0 ? p.bits_dr : p.bits_ds, ds = s.n_shared > 0 ? p.bits_ds : p.bits_dr;
  const int gu_slot = std::max(s.top_k > 0 ? mma_gu_block(br) : 0,
                               s.n_shared > 0 ? mma_gu_block(bs) : 0);
  const int dn_slot = std::max(s.top_k > 0 ? mma_dn_block(dr) : 0,
                               s.n_shared > 0 ? mma_dn_block(ds) : 0);
  e = cudaErrorInvalidValue;
  MOE_MMA_BITS(br, BR, MOE_MMA_BITS(bs, BS,
      e = launch_streaming(mma::gate_up_mma_kernel<BR, BS>, gu_slot, p, stream)));
  if (e != cudaSuccess) return e;
  const int na = p.m * (p.act_stride / kGroup);
  mma::mma_act_kernel<<<(na + mma::kWarps - 1) / mma::kWarps, mma::kThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = cudaErrorInvalidValue;
  MOE_MMA_BITS(dr, BD, MOE_MMA_BITS(ds, BS,
      e = launch_streaming(mma::down_mma_kernel<BD, BS>, dn_slot, p, stream)));
  if (e != cudaSuccess) return e;
  const int64_t n = static_cast<int64_t>(p.m) * s.din;
  mma::mma_tail_kernel<<<static_cast<int>((n + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}
#undef MOE_MMA_BITS

}  // namespace moe
