// moe_phases.cuh -- the two phases of the decode MoE block as device functions, shared by the
// separate kernels (kernel A, kernel B) and the fused persistent kernel.
//
// Phase A ("two-kernel decode-MoE that beats gather_qmm", What changed, step 2, kernel A):
//   act[u] = coef_u * silu(gate_u . x) * (up_u . x) for every gate/up row pair u of the routed slots
//   (coef = the slot's score) and of the shared experts (coef = the shared scalar).
// Phase B (same step, kernel B, fused with the tail of "Red Lite dev39 -- fused expert tail"):
//   out[i] = resid[i] + sum over slots and shared experts of W_down[i, :] . act_segment.
//
// Both phases run on one CTA per SM: 16 consumer warps and one producer warp.
//  * Each CTA owns a contiguous, balanced range of rows.  The producer streams those rows' packed
//    codes, scales and biases into a ring of shared-memory stages with bulk asynchronous copies
//    (TMA, 1-D form) completing on mbarriers; consumers release a stage on its "empty" barrier.
//  * Each consumer thread owns fixed 16-byte code steps (48 bytes at 6 bits) of a row and keeps
//    the matching activations, pre-scaled for the decoding of moe_common.cuh, in registers, so
//    shared memory carries codes only and each code costs one bitwise op and half a packed FMA.
//  * Per-row partial sums leave a warp through a transpose-reduction and are summed across warps
//    in a fixed order, so results are bitwise reproducible.
#pragma once

#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "moe_tma.cuh"
#include "moe_timeline.cuh"

namespace moe {

// ------------------------------------------------------------------ helpers
template <int BITS>
__host__ __device__ constexpr int rows_per_thread_a() {
  return BITS == 6 ? 1 : 2;
}

// Grouped phase B builds an operand per (stage, pair) and uses it for this many rows per thread.
template <int BITS>
__host__ __device__ constexpr int rows_per_thread_gb() {
  return BITS == 6 ? 2 : 4;
}

inline int rows_per_thread_a_host(int bits) { return bits == 6 ? 1 : 2; }
inline int rows_per_thread_gb_host(int bits) { return bits == 6 ? 2 : 4; }

// Phase B (token path): rows per thread in a stage, at most.  A 6-bit operand holds 64 registers,
// which leaves room for fewer accumulators.
__host__ __device__ constexpr int rows_per_thread_b_max(int bits_d, int bits_sd) {
  return bits_d == 6 || bits_sd == 6 ? 4 : 8;
}

template <int V>
struct Log2 {
  static constexpr int v = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : -1;
};

// Sums V values over the 32 lanes of a warp: log2(V) exchange steps that halve the values a lane
// holds, then a butterfly over the rest.  Lane l returns the warp sum of value
// (l >> (5 - log2 V)) & (V - 1).
template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[V], int lane) {
#pragma unroll
  for (int k = V / 2, off = 16; k >= 1; k >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < k; ++j) {
      const float send = upper ? v[j] : v[j + k];
      const float keep = upper ? v[j + k] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int off = 16 / V; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
  return v[0];
}

// Deterministic reductions over the consumer threads (red holds kConsumerWarps floats).
__device__ __forceinline__ float consumers_max(float v, float *red, int warp, int lane) {
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  consumer_sync(kConsumers);
  float m = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) m = fmaxf(m, red[w]);
  consumer_sync(kConsumers);
  return m;
}

__device__ __forceinline__ float consumers_sum(float v, float *red, int warp, int lane) {
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  consumer_sync(kConsumers);
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) s += red[w];
  consumer_sync(kConsumers);
  return s;
}

// 16-B aligned window around a contiguous fp16 run [p, p + n): start, length, offset of p.
struct Window {
  const uint8_t *src;
  uint32_t bytes;
  uint32_t delta;
};

__device__ __forceinline__ Window window_of(const __half *p, int64_t n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uintptr_t lo = a & ~uintptr_t(15);
  const uintptr_t hi = (a + uintptr_t(n) * 2 + 15) & ~uintptr_t(15);
  return Window{reinterpret_cast<const uint8_t *>(lo), static_cast<uint32_t>(hi - lo),
                static_cast<uint32_t>(a - lo)};
}

__device__ __forceinline__ float lds_half(const uint8_t *p) {
  return __half2float(*reinterpret_cast<const __half *>(p));
}

__device__ __forceinline__ uint4 lds_u4(const uint8_t *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

// The Operand of C bf16 values of x from column c0 (x + c0 16-byte aligned); zeros when the
// thread has no step.
template <int BITS>
__device__ __forceinline__ void load_x_operand(Operand<BITS> &op, const uint16_t *x, int c0,
                                               bool active) {
  constexpr int C = Operand<BITS>::C;
  float v[C];
#pragma unroll
  for (int q = 0; q < C / 8; ++q) {
    const uint4 w =
        active ? *reinterpret_cast<const uint4 *>(x + c0 + 8 * q) : make_uint4(0, 0, 0, 0);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * q + 2 * h] = __uint_as_float(ww[h] << 16);
      v[8 * q + 2 * h + 1] = __uint_as_float(ww[h] & 0xffff0000u);
    }
  }
  op.set(v);
}

// Phase A's input vector x: bf16 values in memory, or, in a stack with the next layer's RMSNorm
// folded in ("Red Lite dev39 -- fused expert tail", Measurements: the tail variant that also
// folded in the next layer's RMSNorm), the previous layer's fp32 output v normalised on the fly:
//   x_c = bf16( gamma_c * (v_c * r) ),  r = 1 / sqrt(mean(v^2) + eps)
// with both products in fp32 and the result rounded to the nearest bf16 (ties to even).
struct XSource {
  const uint16_t *x;      // bf16 [din] (v == nullptr)
  const float *v;         // fp32 [din]: the previous layer's output
  const uint16_t *gamma;  // bf16 [din]: the norm's weight
  float eps;
  float r;                // set by load_x_class_norm before any value is read
};

__device__ __forceinline__ XSource xsource_plain(const uint16_t *x) {
  return XSource{x, nullptr, nullptr, 0.f, 1.f};
}

__device__ __forceinline__ float norm_value(float v, float gamma, float r) {
  return bf16_to_float(float_to_bf16_rn(gamma * (v * r)));
}

__device__ __forceinline__ float x_value(const XSource &xs, int c) {
  return xs.v == nullptr ? bf16_to_float(xs.x[c])
                         : norm_value(xs.v[c], bf16_to_float(xs.gamma[c]), xs.r);
}

// The Operand of C values of x from column c0 (16-byte aligned) once x.r is known; zeros when the
// thread has no step.
template <int BITS>
__device__ __forceinline__ void load_x_operand(Operand<BITS> &op, const XSource &xs, int c0,
                                               bool active) {
  if (xs.v == nullptr) {
    load_x_operand<BITS>(op, xs.x, c0, active);
    return;
  }
  constexpr int C = Operand<BITS>::C;
  float v[C];
#pragma unroll
  for (int q = 0; q < C / 8; ++q) {
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 a = active ? *reinterpret_cast<const float4 *>(xs.v + c0 + 8 * q) : zero;
    const float4 b = active ? *reinterpret_cast<const float4 *>(xs.v + c0 + 8 * q + 4) : zero;
    const uint4 g =
        active ? *reinterpret_cast<const uint4 *>(xs.gamma + c0 + 8 * q) : make_uint4(0, 0, 0, 0);
    const float vv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * q + 2 * h] = norm_value(vv[2 * h], __uint_as_float(gw[h] << 16), xs.r);
      v[8 * q + 2 * h + 1] = norm_value(vv[2 * h + 1], __uint_as_float(gw[h] & 0xffff0000u), xs.r);
    }
  }
  op.set(v);
}

// The thread's operand of a class of rows when x is normalised on the fly (XSource with v set):
// computes r, sets x.r and builds the operand.  The threads of the first row group hold every
// column once, so r comes from their steps: squares summed in fp32 per thread, then in fp64
// across those warps in a fixed order (the same in every CTA and in both kernel modes), and
// 1 / sqrt(mean + eps) in fp64 by one thread, rounded to fp32.  The operand then re-reads the
// thread's values (from L1 for the first group).
template <int BITS>
__device__ __forceinline__ void load_x_class_norm(Operand<BITS> &op, const GateUpGeom &g,
                                                  XSource &x, int din, double *red, float *rsh,
                                                  int warp, int lane, int tid) {
  constexpr int C = Operand<BITS>::C;
  const int my_group = tid / g.tpr, my_step = tid % g.tpr;
  const bool active = my_group < g.groups && my_step < g.T;
  if (tid < g.tpr) {  // the first group's warps (tpr is a multiple of 32)
    float ss = 0.f;
    if (my_step < g.T) {
#pragma unroll
      for (int q = 0; q < C / 4; ++q) {
        const float4 a = *reinterpret_cast<const float4 *>(x.v + my_step * C + 4 * q);
        ss = fmaf(a.x, a.x, ss);
        ss = fmaf(a.y, a.y, ss);
        ss = fmaf(a.z, a.z, ss);
        ss = fmaf(a.w, a.w, ss);
      }
    }
    double d = ss;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) red[warp] = d;
  }
  consumer_sync(kConsumers);
  if (tid == 0) {
    double t = 0.0;
    for (int w = 0; w < g.tpr / 32; ++w) t += red[w];
    *rsh = static_cast<float>(1.0 / sqrt(t / din + static_cast<double>(x.eps)));
  }
  consumer_sync(kConsumers);
  x.r = *rsh;
  load_x_operand<BITS>(op, x, my_step * C, active);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// ------------------------------------------------------------------ ring and grid barrier
// What the producer tells the consumers about a phase-A stage (written before the stage's
// arrive.expect_tx, whose release makes it visible to every consumer that waited on the stage).
struct StageDesc {
  int u;        // act index of the stage's first row
  int n;        // rows in the stage (0: an empty stage that only carries the phase's counts)
  float coef;   // the routed slot's score (unused for shared experts)
  int delta;    // byte offset of the first row's first group inside each scale/bias window
};

struct Ring {
  uint64_t *full;
  uint64_t *empty;
  uint8_t *base;
  StageDesc *desc;  // [kMaxStages]
  int nst, stage_bytes;
  int st;           // the next stage this role hands out (producer) or takes (consumers)
  uint32_t ph;      // the parity of that stage's current use
  int used;         // stages handed out or taken so far
  int *abort;       // shared flag: a wait timed out, stop waiting
  int32_t *err;
  __device__ __forceinline__ void advance() {
    if (++st == nst) {
      st = 0;
      ph ^= 1u;
    }
    ++used;
  }
  __device__ __forceinline__ uint8_t *stage() const {
    return base + static_cast<size_t>(st) * stage_bytes;
  }
};

__device__ __forceinline__ Ring make_ring(uint64_t *full, uint64_t *empty, uint8_t *base,
                                          StageDesc *desc, const Plan &plan, int *abort,
                                          int32_t *err) {
  Ring r;
  r.full = full;
  r.empty = empty;
  r.base = base;
  r.desc = desc;
  r.nst = plan.nst;
  r.stage_bytes = plan.stage_bytes;
  r.st = 0;
  r.ph = 0;
  r.used = 0;
  r.abort = abort;
  r.err = err;
  return r;
}

__device__ __forceinline__ bool flag_abort(int *abort) {
  return *reinterpret_cast<volatile int *>(abort) != 0;
}

__device__ __forceinline__ void set_timeout(int *abort, int32_t *err) {
  atomicOr(err, kDevErrTimeout);
  *reinterpret_cast<volatile int *>(abort) = 1;
}

__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, int *abort,
                                          int32_t *err, long long limit = kWaitCycles) {
  // a completed phase is the common case: test it without the suspending wait's fixed cost
  if (mbar_test_wait(bar, parity)) return true;
  if (flag_abort(abort)) return false;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (flag_abort(abort)) return false;
    if (clock64() - t0 > limit) {
      set_timeout(abort, err);
      return false;
    }
    __nanosleep(64);  // leave the issue slots to the warps that have work
  }
  return true;
}

// Consumer side: lane 0 of each warp waits for the current stage and the warp follows it.  One
// waiter per warp instead of 32 keeps the barrier word free for the arrivals that complete it.
__device__ __forceinline__ bool warp_wait_full(Ring &r, int lane) {
  int ok = 1;
  if (lane == 0) ok = ring_wait(&r.full[r.st], r.ph, r.abort, r.err);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Consumer side: the warp is done reading the current stage.
__device__ __forceinline__ void warp_release(Ring &r, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&r.empty[r.st]);
  r.advance();
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Producer side: claims the current stage (waits until its previous use was released).
__device__ __forceinline__ bool ring_claim(Ring &r, int lane) {
  int good = 1;
  if (r.used >= r.nst && lane == 0) good = ring_wait(&r.empty[r.st], r.ph ^ 1u, r.abort, r.err);
  return __shfl_sync(0xffffffffu, good, 0) != 0;
}

// Producer side, at exit: the copies into the last use of every stage have landed.
__device__ __forceinline__ void ring_drain(Ring &r, int lane) {
  if (lane != 0) return;
  for (int s = r.used - r.nst < 0 ? 0 : r.used - r.nst; s < r.used; ++s)
    mbar_wait(&r.full[s % r.nst], (s / r.nst) & 1);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *cnt >= target (bounded).  Only meaningful when every CTA of the grid is resident.
__device__ __forceinline__ bool wait_count(const uint32_t *cnt, uint32_t target, int *abort,
                                           int32_t *err, long long limit = kWaitCycles) {
  if (ld_acquire(cnt) >= target) return true;
  const long long t0 = clock64();
  while (ld_acquire(cnt) < target) {
    if (flag_abort(abort)) return false;
    if (clock64() - t0 > limit) {
      set_timeout(abort, err);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Grid barrier among the consumer threads of all CTAs: every CTA's consumers finished their writes.
__device__ __forceinline__ void consumers_grid_barrier(uint32_t *cnt, uint32_t target, int tid,
                                                       int *abort, int32_t *err) {
  consumer_sync(kConsumers);
  if (tid == 0) {
    // bar.sync orders the CTA's writes before this thread's release, which is cumulative
    red_release_add(cnt, 1u);
    wait_count(cnt, target, abort, err);
  }
  consumer_sync(kConsumers);
}

// Producer side, at the start of a (layer, token): the expert ids and scores into shared memory
// (lanes in parallel) and the error bit for ids outside [0, n_experts); with ids_used set, CTA 0
// also writes the ids it read there (the route the kernel took, for the caller to check).  The caller has already
// waited for whatever makes them complete; the producer_sync after the loads orders them before
// the producer's first arrive on a stage, which publishes them to the consumers.
__device__ __forceinline__ void producer_load_token(const LayerShape &s, const int32_t *ids,
                                                    const float *scores, int *ids_s,
                                                    float *scores_s, int32_t *err, int lane,
                                                    int32_t *ids_used = nullptr,
                                                    int *all_valid = nullptr) {
  int bad = 0;
  for (int k = lane; k < s.top_k; k += kProducers) {
    // both loads before either store: one round trip
    const int e = ids[k];
    const float sc = scores != nullptr ? scores[k] : 0.f;
    ids_s[k] = e;
    scores_s[k] = sc;
    const bool b = e < 0 || e >= s.n_experts;
    bad |= b;
    if (b) atomicOr(err, kDevErrBadId);
    if (ids_used != nullptr && blockIdx.x == 0) ids_used[k] = e;  // what this kernel read
  }
  if (all_valid != nullptr) {  // the whole warp calls this
    const unsigned any = __ballot_sync(0xffffffffu, bad);
    if (lane == 0) *all_valid = any == 0u;
  }
  producer_sync();
}

// ================================================================== route inversion
// A batch of tokens is grouped by expert so that each selected expert is streamed once per
// layer: the distinct valid ids in ascending order, and for each the (token, slot) pairs that
// name it, p = token * K + slot, ascending.  The grouping of the routers' top-k pools by expert
// ("Red Lite dev39 -- fused expert tail", Change) is the step before that stream.
struct Route {
  int n_uniq;                                // U
  int n_pairs;                               // valid pairs (offs[U])
  int uniq[kMaxPairs];                       // expert ids, ascending
  int offs[kMaxPairs + 1];                   // pairs of uniq[u]: pairs[offs[u] .. offs[u + 1])
  short pairs[kMaxPairs];                    // token * K + slot
  int cnt[kMaxPairs];                        // scratch: pairs per expert, then placement cursor
  uint32_t bitmap[kMaxGroupExperts / 32];    // scratch: which experts occur
  int wbase[kMaxGroupExperts / 32];          // scratch: experts below each bitmap word
};

__device__ __forceinline__ int route_rank(const Route &rt, int e) {
  const int w = e >> 5;
  return rt.wbase[w] + __popc(rt.bitmap[w] & ((1u << (e & 31)) - 1u));
}

// One warp inverts ids[0 .. n) (n = m * K <= kMaxPairs; n_experts <= kMaxGroupExperts) into rt.
// Deterministic: experts by bitmap rank, pairs placed in index order within each expert.
__device__ __forceinline__ void route_invert_warp(const int *ids, int n, int n_experts, Route &rt,
                                                  int lane) {
  const int words = (n_experts + 31) >> 5;
  for (int w = lane; w < kMaxGroupExperts / 32; w += 32) rt.bitmap[w] = 0u;
  __syncwarp();
  for (int p = lane; p < n; p += 32) {
    const int e = ids[p];
    if (e >= 0 && e < n_experts) atomicOr(&rt.bitmap[e >> 5], 1u << (e & 31));
  }
  __syncwarp();
  // experts below each word (exclusive scan of popcounts; one word per lane)
  const int c = lane < words ? __popc(rt.bitmap[lane]) : 0;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  rt.wbase[lane] = incl - c;
  const int U = __shfl_sync(0xffffffffu, incl, 31);
  if (lane < words) {
    uint32_t bits = rt.bitmap[lane];
    int r = incl - c;
    while (bits) {
      const int b = __ffs(bits) - 1;
      rt.uniq[r++] = (lane << 5) + b;
      bits &= bits - 1u;
    }
  }
  for (int u = lane; u < U; u += 32) rt.cnt[u] = 0;
  __syncwarp();
  for (int p = lane; p < n; p += 32) {
    const int e = ids[p];
    if (e >= 0 && e < n_experts) atomicAdd(&rt.cnt[route_rank(rt, e)], 1);
  }
  __syncwarp();
  // offsets: exclusive scan of the counts, U <= kMaxPairs = 8 per lane
  constexpr int PER = kMaxPairs / 32;
  int local[PER];
  int lsum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int u = lane * PER + j;
    local[j] = u < U ? rt.cnt[u] : 0;
    lsum += local[j];
  }
  int lin = lsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, lin, o);
    if (lane >= o) lin += t;
  }
  int run = lin - lsum;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int u = lane * PER + j;
    if (u < U) rt.offs[u] = run;
    run += local[j];
  }
  const int total = __shfl_sync(0xffffffffu, lin, 31);
  if (lane == 0) {
    rt.offs[U] = total;
    rt.n_uniq = U;
    rt.n_pairs = total;
  }
  __syncwarp();
  for (int u = lane; u < U; u += 32) rt.cnt[u] = 0;
  __syncwarp();
  // stable placement, 32 pairs at a time: equal experts in one batch are ordered by lane
  for (int b = 0; b < n; b += 32) {
    const int p = b + lane;
    const int e = p < n ? ids[p] : -1;
    const bool valid = e >= 0 && e < n_experts;
    const int key = valid ? e : -1 - lane;  // invalid lanes match nobody
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    int r = 0, pos = 0;
    if (valid) {
      r = route_rank(rt, e);
      pos = rt.offs[r] + rt.cnt[r] + __popc(peers & ((1u << lane) - 1u));
      rt.pairs[pos] = static_cast<short>(p);
    }
    __syncwarp();
    if (valid && (__ffs(peers) - 1) == lane) rt.cnt[r] += __popc(peers);
    __syncwarp();
  }
}

// ================================================================== phase A
struct ChunkA {
  int k;   // slot (routed) or shared expert index
  int j;   // first row inside the expert
  int n;   // rows in the chunk
  int u;   // flattened index of the first row (= its act index)
};

// Walks the chunks of a CTA's row range [a, b) of one class: at most R rows each, never crossing
// an expert's block of rows_pe rows.  One division per range, 32-bit arithmetic (the flattened
// row space is below 2^24 rows).
struct ChunkIterA {
  int u, b, k, j, rows_pe, R;
  __device__ __forceinline__ ChunkIterA(int64_t a, int64_t b_, int64_t base_u, int rows_pe_, int R_)
      : u(static_cast<int>(a)), b(static_cast<int>(b_)), rows_pe(rows_pe_), R(R_) {
    const int v = static_cast<int>(a - base_u);
    k = rows_pe_ > 0 ? v / rows_pe_ : 0;
    j = v - k * rows_pe_;
  }
  __device__ __forceinline__ bool next(ChunkA &c) {
    if (u >= b) return false;
    int n = b - u;
    if (n > R) n = R;
    if (n > rows_pe - j) n = rows_pe - j;
    c.k = k;
    c.j = j;
    c.n = n;
    c.u = u;
    u += n;
    j += n;
    if (j == rows_pe) {
      j = 0;
      ++k;
    }
    return true;
  }
};

// The rows a CTA owns in phase A: [u0, u1) of the flattened routed-then-shared row space.
struct RangeA {
  int64_t ra, rb;   // routed rows
  int64_t sa, sb;   // shared rows
  int64_t Ur;       // routed row count
};

__device__ __forceinline__ RangeA range_a(const LayerShape &s) {
  const int64_t Ur = static_cast<int64_t>(s.top_k) * s.dff;
  const int64_t U = Ur + static_cast<int64_t>(s.n_shared) * s.dff_shared;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  RangeA r;
  r.ra = u0;
  r.rb = u1 < Ur ? u1 : Ur;
  r.sa = u0 > Ur ? u0 : Ur;
  r.sb = u1;
  r.Ur = Ur;
  return r;
}

// Chunks of one class that carry data (routed chunks of a slot with an invalid id are skipped).
__device__ __forceinline__ int count_a_class(const LayerShape &s, int R, bool shared_class,
                                             int64_t a, int64_t b, int64_t base_u, int rows_pe,
                                             const int *ids) {
  ChunkIterA it(a, b, base_u, rows_pe, R);
  ChunkA c;
  int n = 0;
  while (it.next(c)) {
    const int e = shared_class ? c.k : ids[c.k];
    n += shared_class || (e >= 0 && e < s.n_experts);
  }
  return n;
}

template <int BITS>
__device__ void produce_a_class(const LayerShape &s, const GateUpGeom &g, const ProjDev &gate,
                                const ProjDev &up, bool shared_class, int64_t a, int64_t b,
                                int64_t base_u, int rows_pe, const int *ids, const float *scores,
                                Ring &r, int lane, uint64_t pol) {
  const int G = s.din / kGroup;
  ChunkIterA it(a, b, base_u, rows_pe, g.R);
  ChunkA c;
  while (it.next(c)) {
    const int e = shared_class ? c.k : ids[c.k];
    if (!shared_class && (e < 0 || e >= s.n_experts)) continue;
    if (!ring_claim(r, lane)) return;
    uint8_t *sb = r.stage();
    const int64_t row = static_cast<int64_t>(e) * rows_pe + c.j;
    const uint32_t code_bytes = static_cast<uint32_t>(c.n) * g.rb;
    const int64_t ng = static_cast<int64_t>(c.n) * G;
    const Window w0 = window_of(gate.scales + row * G, ng);
    const Window w1 = window_of(gate.biases + row * G, ng);
    const Window w2 = window_of(up.scales + row * G, ng);
    const Window w3 = window_of(up.biases + row * G, ng);
    uint8_t *wb = sb + 2 * g.R * g.rb;
    if (lane == 0) {
      r.desc[r.st] = StageDesc{c.u, c.n, shared_class ? 0.f : scores[c.k],
                               static_cast<int>(w0.delta)};
      mbar_arrive_expect_tx(&r.full[r.st],
                            2 * code_bytes + w0.bytes + w1.bytes + w2.bytes + w3.bytes);
    }
    __syncwarp();
    if (lane == 0) bulk_g2s(sb, gate.codes + row * g.rb, code_bytes, &r.full[r.st], pol);
    if (lane == 1) bulk_g2s(sb + g.R * g.rb, up.codes + row * g.rb, code_bytes, &r.full[r.st], pol);
    if (lane == 2) bulk_g2s(wb + 0 * g.sw, w0.src, w0.bytes, &r.full[r.st], pol);
    if (lane == 3) bulk_g2s(wb + 1 * g.sw, w1.src, w1.bytes, &r.full[r.st], pol);
    if (lane == 4) bulk_g2s(wb + 2 * g.sw, w2.src, w2.bytes, &r.full[r.st], pol);
    if (lane == 5) bulk_g2s(wb + 3 * g.sw, w3.src, w3.bytes, &r.full[r.st], pol);
    r.advance();
  }
}

// Producer of phase A for one token: counts the CTA's chunks per class (the consumers learn them
// from the phase's first stage), then streams them.  A CTA without any phase-A chunk still hands
// out one empty stage, so the consumers always have a first stage to wait on.
template <int BR, int BS>
__device__ void produce_a(const LayerShape &s, const LayerPtrs &w, const GateUpGeom &gr,
                          const GateUpGeom &gs, const int *ids, const float *scores, int *cnt,
                          Ring &r, int lane, uint64_t pol) {
  const RangeA ra = range_a(s);
  const int nr = count_a_class(s, gr.R, false, ra.ra, ra.rb, 0, s.dff, ids);
  const int ns = count_a_class(s, gs.R, true, ra.sa, ra.sb, ra.Ur, s.dff_shared, ids);
  if (lane == 0) {
    cnt[0] = nr;
    cnt[1] = ns;
  }
  __syncwarp();
  produce_a_class<BR>(s, gr, w.gate, w.up, false, ra.ra, ra.rb, 0, s.dff, ids, scores, r, lane,
                      pol);
  if (flag_abort(r.abort)) return;
  produce_a_class<BS>(s, gs, w.sh_gate, w.sh_up, true, ra.sa, ra.sb, ra.Ur, s.dff_shared, ids,
                      scores, r, lane, pol);
  if (nr + ns == 0 && !flag_abort(r.abort)) {
    if (!ring_claim(r, lane)) return;
    if (lane == 0) {
      r.desc[r.st] = StageDesc{0, 0, 0.f, 0};
      mbar_arrive_expect_tx(&r.full[r.st], 0);
    }
    r.advance();
  }
}

// Scratch of the consumer side of both phases.  Per-row partial sums are reduced within a warp as
// soon as a stage is consumed, parked in shared memory (one slot per row and warp), and summed
// across warps once per batch of rows, so warps run through the stages independently and the
// only block-wide synchronisation in a phase is the final one.
constexpr int kRedA = 1024;   // phase A: parked partial sums per kind (gate, up)
constexpr int kBatchA = 256;  // phase A: rows parked before a flush, at most

struct SmemA {
  float red[2][kRedA];        // [gate/up][held row * warps-per-group + warp slot]
  int row_u[kBatchA];         // act index of each held row
  float coef[kBatchA];        // its coefficient: the slot's score or the shared scalar
  float stat[kConsumerWarps];
  double dstat[kConsumerWarps];
  float rnorm;                // r of the folded RMSNorm, broadcast
};

struct SmemB {
  float red[kMaxRowsB * kConsumerWarps];  // [row - first row][warp slot]
};

// Phase A and phase B never hold scratch at the same time (a grid barrier or a kernel boundary
// separates them), so they share it.
union SmemAB {
  SmemA a;
  SmemB b;
};

// Sums the parked partials of the held rows across warps (fixed order) and writes the
// activations.  `trailing` adds the barrier that frees the buffer for reuse.
__device__ __forceinline__ void flush_a(SmemA &sm, int held, int wpg, float *act, int tid,
                                        bool trailing, int u_base = 0) {
  consumer_sync(kConsumers);
  for (int t = tid; t < held; t += kConsumers) {
    float gs = 0.f, us = 0.f;
    for (int w = 0; w < wpg; ++w) {
      gs += sm.red[0][t * wpg + w];
      us += sm.red[1][t * wpg + w];
    }
    act[sm.row_u[t] - u_base] = sm.coef[t] * (silu_f(gs) * us);
  }
  if (trailing) consumer_sync(kConsumers);
}

// Consumes the `count` stages of one class (routed slots or shared experts) of a CTA's phase A
// rows.  `waited`: the current stage has already been waited on (the phase's first stage is
// waited before the counts are read).  Returns the rows still parked, which the caller flushes
// (the two classes may have different warps per row, so a batch never mixes them).
// The thread's x operand for one class's geometry.
template <int BITS, typename XS>
__device__ __forceinline__ void load_x_class(Operand<BITS> &op, const GateUpGeom &g,
                                             const XS &x, int tid) {
  const int my_group = tid / g.tpr, my_step = tid % g.tpr;
  load_x_operand<BITS>(op, x, my_step * Operand<BITS>::C, my_group < g.groups && my_step < g.T);
}

template <int BITS>
__device__ int consume_a_class(const LayerShape &s, const GateUpGeom &g, bool shared_class,
                               int count, const Operand<BITS> &xo, float *act, float shared_scalar,
                               Ring &r, SmemA &sm, bool &waited, bool &ok, int tid,
                               int u_base = 0) {
  constexpr int C = Fmt<BITS>::kCodes, VEC = Fmt<BITS>::kVecs;
  constexpr int RPT = rows_per_thread_a<BITS>();
  constexpr int V = 2 * RPT;        // values per stage: gate and up of RPT rows
  int held = 0;
  if (count == 0) return held;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = s.din / kGroup;
  const int my_group = tid / g.tpr, my_step = tid % g.tpr;
  const bool grp_ok = my_group < g.groups;
  const bool active = grp_ok && my_step < g.T;
  const int wpg = g.tpr / 32;
  const int wslot = warp - my_group * wpg;
  const float xunit = xo.unit, xsum = xo.sum;
  const int code_off = my_step * 16 * VEC;          // the thread's step inside a row
  const int win_off = ((my_step * C) / kGroup) * 2;  // its group's scale inside a row's run
  // after the transpose-reduction, lane l holds value idx of the stage
  const int idx = (lane >> (5 - Log2<V>::v)) & (V - 1);
  const bool writer = grp_ok && (lane & ((32 / V) - 1)) == 0;
  const int w_kind = idx / RPT, w_row = (idx % RPT) * g.groups + my_group;
  const int cap = kRedA / wpg < kBatchA ? kRedA / wpg : kBatchA;
  const int wbase = 2 * g.R * g.rb + win_off;

  for (int i = 0; i < count; ++i) {
    if (!waited) ok = warp_wait_full(r, lane);
    waited = false;
    const StageDesc d = r.desc[r.st];
    if (held + d.n > cap) {
      flush_a(sm, held, wpg, act, tid, true, u_base);
      held = 0;
    }
    if (tid < d.n) {
      sm.row_u[held + tid] = d.u + tid;
      sm.coef[held + tid] = shared_class ? shared_scalar : d.coef;
    }
    const uint8_t *sb = r.stage();
    const uint8_t *ws = sb + wbase + d.delta;
    float v[V];
#pragma unroll
    for (int q = 0; q < V; ++q) v[q] = 0.f;
    // rows q < nq of this stage are the thread's (row q sits at q * groups + my_group)
    int nq = (d.n - my_group + g.groups - 1) / g.groups;
    nq = nq > RPT ? RPT : nq;
    if (active && ok && nq > 0) {
      // every row's codes, scales and biases first, then the dot products; a row past nq reads
      // row 0's bytes (in the stage) and is dropped
      uint4 cg[RPT][VEC], cu[RPT][VEC];
      float h[RPT][4];
#pragma unroll
      for (int q = 0; q < RPT; ++q) {
        const int rr = (q < nq ? q : 0) * g.groups + my_group;
        const uint8_t *pg = sb + rr * g.rb + code_off;
        const uint8_t *pu = pg + g.R * g.rb;
#pragma unroll
        for (int w = 0; w < VEC; ++w) {
          cg[q][w] = lds_u4(pg + 16 * w);
          cu[q][w] = lds_u4(pu + 16 * w);
        }
        const uint8_t *wr = ws + rr * G * 2;
#pragma unroll
        for (int k = 0; k < 4; ++k) h[q][k] = lds_half(wr + k * g.sw);
      }
#pragma unroll
      for (int q = 0; q < RPT; ++q) {
        if (q < nq) {
          v[q] = fmaf(h[q][0], xo.dot(cg[q]) * xunit, h[q][1] * xsum);
          v[RPT + q] = fmaf(h[q][2], xo.dot(cu[q]) * xunit, h[q][3] * xsum);
        }
      }
    }
    warp_release(r, lane);
    const float val = warp_transpose_reduce<V>(v, lane);
    if (writer && w_row < d.n) sm.red[w_kind][(held + w_row) * wpg + wslot] = val;
    held += d.n;
  }
  return held;
}

// Consumers of phase A for one token of one layer: x is read here; the stages' descriptors carry
// the rest.  Ends with the activations written and a consumer_sync-free tail: callers
// synchronise as needed.
// CHAIN: x may be normalised on the fly (XSource with v set); otherwise x.x is read.
template <int BR, int BS, bool CHAIN>
__device__ void consume_a(const LayerShape &s, const LayerPtrs &w, const GateUpGeom &gr,
                          const GateUpGeom &gs, XSource x, const int *cnt, float *act,
                          Ring &r, SmemA &sm, int tid, int u_base = 0) {
  const int warp = tid >> 5, lane = tid & 31;
  Operand<BR> xr;   // x for the routed rows, loaded while the first stage is in flight
  if constexpr (CHAIN) {
    if (x.v != nullptr)
      load_x_class_norm<BR>(xr, gr, x, s.din, sm.dstat, &sm.rnorm, warp, lane, tid);
    else
      load_x_class<BR>(xr, gr, x.x, tid);
  } else {
    load_x_class<BR>(xr, gr, x.x, tid);
  }
  float shared_scalar = 1.0f;
  if (w.gate_vec != nullptr && s.n_shared > 0) {
    float dot = 0.f;
    for (int c = tid; c < s.din; c += kConsumers) {
      const float xc = CHAIN ? x_value(x, c) : bf16_to_float(x.x[c]);
      dot = fmaf(xc, bf16_to_float(w.gate_vec[c]), dot);
    }
    dot = consumers_sum(dot, sm.stat, warp, lane);
    shared_scalar = 1.0f / (1.0f + expf(-dot));
  }
  // the phase's first stage publishes the counts
  bool ok = warp_wait_full(r, lane), waited = true;
  const int nr = cnt[0], ns = cnt[1];
  if (nr + ns == 0) {   // an empty stage
    warp_release(r, lane);
    return;
  }
  int held =
      consume_a_class<BR>(s, gr, false, nr, xr, act, 1.f, r, sm, waited, ok, tid, u_base);
  if (held > 0) flush_a(sm, held, gr.tpr / 32, act, tid, ns > 0, u_base);
  if (ns > 0) {
    Operand<BS> xsh;
    if constexpr (CHAIN)
      load_x_class<BS>(xsh, gs, x, tid);
    else
      load_x_class<BS>(xsh, gs, x.x, tid);
    held = consume_a_class<BS>(s, gs, true, ns, xsh, act, shared_scalar, r, sm, waited, ok, tid,
                               u_base);
    if (held > 0) flush_a(sm, held, gs.tpr / 32, act, tid, false, u_base);
  }
}

// ================================================================== phase B
struct SegB {
  const ProjDev *pr;
  int64_t expert;   // -1 when the slot's id is invalid
  int rb, G, sw;
  int code_off, win_off;
};

__device__ __forceinline__ SegB seg_b(const LayerShape &s, const LayerPtrs &w, const DownGeom &g,
                                      int expert_id, int q) {
  SegB sg;
  if (q < s.top_k) {
    sg.pr = &w.down;
    sg.expert = (expert_id >= 0 && expert_id < s.n_experts) ? expert_id : -1;
    sg.rb = g.rb_r;
    sg.G = g.G_r;
    sg.sw = g.sw_r;
    sg.code_off = q * g.R * g.rb_r;
    sg.win_off = q * g.sw_r;
  } else {
    const int t = q - s.top_k;
    sg.pr = &w.sh_down;
    sg.expert = t;
    sg.rb = g.rb_s;
    sg.G = g.G_s;
    sg.sw = g.sw_s;
    sg.code_off = s.top_k * g.R * g.rb_r + t * g.R * g.rb_s;
    sg.win_off = s.top_k * g.sw_r + t * g.sw_s;
  }
  return sg;
}

__device__ __forceinline__ void range_b(const LayerShape &s, int &i0, int &i1) {
  i0 = static_cast<int>(static_cast<int64_t>(s.din) * blockIdx.x / gridDim.x);
  i1 = static_cast<int>(static_cast<int64_t>(s.din) * (blockIdx.x + 1) / gridDim.x);
}

// Producer of phase B: per stage, lane q handles segment q (and q + 32, ...): the codes of R
// output rows of that slot's (or shared expert's) down projection plus their scale and bias
// windows.  `ids` is the producer's shared copy.
__device__ inline void produce_b(const LayerShape &s, const LayerPtrs &w, const DownGeom &g,
                          const int *ids, Ring &r, int lane, uint64_t pol) {
  int i0, i1;
  range_b(s, i0, i1);
  const int nseg = s.top_k + s.n_shared;
  const int wins = s.top_k * g.sw_r + s.n_shared * g.sw_s;
  for (int r0 = i0; r0 < i1; r0 += g.R) {
    const int n = (i1 - r0) < g.R ? (i1 - r0) : g.R;
    if (!ring_claim(r, lane)) return;
    uint8_t *sb = r.stage();
    uint8_t *wb = sb + g.codes_bytes;
    uint32_t tx = 0;
    for (int q = lane; q < nseg; q += 32) {
      const SegB sg = seg_b(s, w, g, q < s.top_k ? ids[q] : 0, q);
      if (sg.expert < 0) continue;
      const int64_t row = sg.expert * s.din + r0;
      const int64_t ng = static_cast<int64_t>(n) * sg.G;
      tx += static_cast<uint32_t>(n) * sg.rb + window_of(sg.pr->scales + row * sg.G, ng).bytes +
            window_of(sg.pr->biases + row * sg.G, ng).bytes;
    }
    tx = warp_sum_u32(tx);
    if (lane == 0) mbar_arrive_expect_tx(&r.full[r.st], tx);
    __syncwarp();
    for (int q = lane; q < nseg; q += 32) {
      const SegB sg = seg_b(s, w, g, q < s.top_k ? ids[q] : 0, q);
      if (sg.expert < 0) continue;
      const int64_t row = sg.expert * s.din + r0;
      const int64_t ng = static_cast<int64_t>(n) * sg.G;
      const Window ws = window_of(sg.pr->scales + row * sg.G, ng);
      const Window wbi = window_of(sg.pr->biases + row * sg.G, ng);
      bulk_g2s(sb + sg.code_off, sg.pr->codes + row * sg.rb, static_cast<uint32_t>(n) * sg.rb,
               &r.full[r.st], pol);
      bulk_g2s(wb + sg.win_off, ws.src, ws.bytes, &r.full[r.st], pol);
      bulk_g2s(wb + wins + sg.win_off, wbi.src, wbi.bytes, &r.full[r.st], pol);
    }
    r.advance();
  }
}

// A thread's step of the down contraction: routed (BD-bit codes) or shared (BSD-bit codes).
template <int BD, int BSD>
struct DownOperand {
  union {
    Operand<BD> r;
    Operand<BSD> s;
  };
};

// One thread's step of a stage's rows q < nq (row q sits at q * groups + my_group): the codes,
// scales and biases of QB rows are loaded before any of their dot products, so the loads and the
// rows' integer chains overlap.  A row past nq reads row q0's bytes (in the stage) and adds
// nothing; each acc[q] sums its terms in the order of the callers' step loop.
template <int BITS, int VS>
__device__ __forceinline__ void down_rows(const uint8_t *cp, const uint8_t *sp, int rb, int G,
                                          int wins, int groups, int my_group, int nq,
                                          const Operand<BITS> &op, float (&acc)[VS]) {
  constexpr int VEC = Fmt<BITS>::kVecs;
  // rows in flight (a 6-bit operand already holds 64 registers)
  constexpr int QB = VEC == 1 ? 4 : 1;
#pragma unroll
  for (int q0 = 0; q0 < VS; q0 += QB) {
    if (q0 >= nq) break;
    uint4 cv[QB][VEC];
    float hs[QB], hb[QB];
#pragma unroll
    for (int j = 0; j < QB; ++j) {
      const int rr = (q0 + j < nq ? q0 + j : q0) * groups + my_group;
#pragma unroll
      for (int w = 0; w < VEC; ++w) cv[j][w] = lds_u4(cp + rr * rb + 16 * w);
      const uint8_t *wr = sp + rr * G * 2;
      hs[j] = lds_half(wr);
      hb[j] = lds_half(wr + wins);
    }
#pragma unroll
    for (int j = 0; j < QB; ++j) {
      const float t = fmaf(hs[j], op.dot(cv[j]) * op.unit, hb[j] * op.sum);
      if (q0 + j < nq) acc[q0 + j] += t;
    }
  }
}

// The Operand of C activations from act + base (16-byte aligned); zeros when not owned.
template <int BITS>
__device__ __forceinline__ void load_act_operand(Operand<BITS> &op, const float *act, int base,
                                                 bool own) {
  constexpr int C = Operand<BITS>::C;
  float v[C];
  const float4 *ap = reinterpret_cast<const float4 *>(act + base);
#pragma unroll
  for (int c = 0; c < C; c += 4) {
    const float4 a4 = own ? ap[c / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
    v[c] = a4.x;
    v[c + 1] = a4.y;
    v[c + 2] = a4.z;
    v[c + 3] = a4.w;
  }
  op.set(v);
}

// The CTA's residual rows of phase B into shared memory (the tail adds them).  The residual may
// be read at any time during the layer: it is an input or the previous layer's complete output.
__device__ __forceinline__ void load_resid_rows(const LayerShape &s, const void *resid,
                                                int resid_f32, float *dst, int tid) {
  int i0, i1;
  range_b(s, i0, i1);
  for (int t = tid; t < i1 - i0; t += kConsumers)
    dst[t] = resid_f32 ? static_cast<const float *>(resid)[i0 + t]
                       : bf16_to_float(static_cast<const uint16_t *>(resid)[i0 + t]);
}

// Consumers of phase B for one token, each thread owning at most SPTMAX steps of the
// concatenated contraction.  act must be complete (the caller waited for phase A);
// resid_s holds the CTA's residual rows (load_resid_rows, before a consumer_sync); ids_s is the
// producer's shared copy of the expert ids, published by the first stage the consumers wait on.
template <int BD, int BSD, int SPTMAX>
__device__ void consume_b_spt(const LayerShape &s, const DownGeom &g, const int *ids_s,
                              const float *act, const float *resid_s, void *out, int out_f32,
                              Ring &r, SmemB &sm, int tid) {
  constexpr int CR = Fmt<BD>::kCodes, CS = Fmt<BSD>::kCodes;
  constexpr int VS = rows_per_thread_b_max(BD, BSD);  // rows per thread per stage, at most
  const int warp = tid >> 5, lane = tid & 31;
  int i0, i1;
  range_b(s, i0, i1);
  if (i1 <= i0) return;
  const int my_group = tid / g.tpr, my_step = tid % g.tpr;
  const bool grp_ok = my_group < g.groups;
  const int wpg = g.tpr / 32;
  const int wslot = warp - my_group * wpg;
  const int Lr = s.top_k * s.dff;

  // this thread's steps of the concatenated contraction and their activations (each thread
  // scales its own operands)
  DownOperand<BD, BSD> op[SPTMAX];
  int seg[SPTMAX], jst[SPTMAX];
  bool own[SPTMAX], shr[SPTMAX];
#pragma unroll
  for (int i = 0; i < SPTMAX; ++i) {
    const int t = my_step + g.tpr * i;
    own[i] = grp_ok && i < g.spt && t < g.T_r + g.T_s;
    shr[i] = t >= g.T_r;
    if (!shr[i]) {
      seg[i] = t / g.spr_r;
      jst[i] = t - seg[i] * g.spr_r;
      load_act_operand<BD>(op[i].r, act, t * CR, own[i]);
    } else {
      const int ts = t - g.T_r;
      const int si = ts / (g.spr_s > 0 ? g.spr_s : 1);
      seg[i] = s.top_k + si;
      jst[i] = ts - si * g.spr_s;
      load_act_operand<BSD>(op[i].s, act, Lr + ts * CS, own[i]);
    }
  }

  // the first stage publishes the ids
  bool ok = warp_wait_full(r, lane);
  // Per-thread constants of each owned step: where its codes and its group's scale/bias sit in
  // a stage, and its expert's first row (for the window offset).
  const int wins = s.top_k * g.sw_r + s.n_shared * g.sw_s;
  bool seg_ok[SPTMAX];
  int cbase[SPTMAX], sbase[SPTMAX], rbs[SPTMAX], Gs[SPTMAX];
  uint32_t rowbase[SPTMAX];
#pragma unroll
  for (int i = 0; i < SPTMAX; ++i) {
    const bool routed = seg[i] < s.top_k;
    const int e = routed ? ids_s[seg[i]] : seg[i] - s.top_k;
    seg_ok[i] = own[i] && (!routed || (e >= 0 && e < s.n_experts));
    const int t = seg[i] - s.top_k;
    const int code_off = routed ? seg[i] * g.R * g.rb_r : s.top_k * g.R * g.rb_r + t * g.R * g.rb_s;
    const int win_off = routed ? seg[i] * g.sw_r : s.top_k * g.sw_r + t * g.sw_s;
    const int C = shr[i] ? CS : CR;
    cbase[i] = code_off + jst[i] * 16 * (shr[i] ? Fmt<BSD>::kVecs : Fmt<BD>::kVecs);
    sbase[i] = win_off + ((jst[i] * C) / kGroup) * 2;
    rbs[i] = routed ? g.rb_r : g.rb_s;
    Gs[i] = routed ? g.G_r : g.G_s;
    rowbase[i] = static_cast<uint32_t>(e) * static_cast<uint32_t>(s.din);
  }
  const int rpt = g.R / g.groups;
  // after the transpose-reduction, lane l holds the sum of row slot q_w
  const int q_w = (lane >> (5 - Log2<VS>::v)) & (VS - 1);
  const bool writer = grp_ok && (lane & ((32 / VS) - 1)) == 0;
  const int w_row = q_w * g.groups + my_group;

  for (int r0 = i0; r0 < i1; r0 += g.R) {
    if (r0 != i0) ok = warp_wait_full(r, lane);
    const int n = (i1 - r0) < g.R ? (i1 - r0) : g.R;
    const uint8_t *sb = r.stage();
    const uint8_t *wb = sb + g.codes_bytes;
    float acc[VS];
#pragma unroll
    for (int q = 0; q < VS; ++q) acc[q] = 0.f;
    // rows q < nq of this stage are the thread's: q < rpt and q * groups + my_group < n
    int nq = (n - my_group + g.groups - 1) / g.groups;
    nq = nq < 0 ? 0 : (nq > rpt ? rpt : nq);
    if (ok) {
#pragma unroll
      for (int i = 0; i < SPTMAX; ++i) {
        if (!seg_ok[i]) continue;
        // windows start at the 16-B boundary below the first group of row r0 (arrays 16-B
        // aligned), so the group sits (row * G mod 8) halves in
        const uint32_t delta = (((rowbase[i] + r0) * static_cast<uint32_t>(Gs[i])) & 7u) * 2u;
        const uint8_t *cp = sb + cbase[i];
        const uint8_t *sp = wb + sbase[i] + delta;
        if (shr[i])
          down_rows<BSD, VS>(cp, sp, rbs[i], Gs[i], wins, g.groups, my_group, nq, op[i].s, acc);
        else
          down_rows<BD, VS>(cp, sp, rbs[i], Gs[i], wins, g.groups, my_group, nq, op[i].r, acc);
      }
    }
    warp_release(r, lane);
    const float val = warp_transpose_reduce<VS>(acc, lane);
    if (writer && q_w < rpt && w_row < n) sm.red[(r0 - i0 + w_row) * wpg + wslot] = val;
  }
  consumer_sync(kConsumers);
  for (int t = tid; t < i1 - i0; t += kConsumers) {
    float sum = 0.f;
    for (int ww = 0; ww < wpg; ++ww) sum += sm.red[t * wpg + ww];
    const float o = resid_s[t] + sum;
    if (out_f32)
      static_cast<float *>(out)[i0 + t] = o;
    else
      static_cast<uint16_t *>(out)[i0 + t] = float_to_bf16_rn(o);
  }
}

// Phase B with the activation registers sized for the plan's steps per thread.
template <int BD, int BSD>
__device__ void consume_b(const LayerShape &s, const DownGeom &g, const int *ids_s,
                          const float *act, const float *resid_s, void *out, int out_f32,
                          Ring &r, SmemB &sm, int tid) {
  constexpr int CMAX = Fmt<BD>::kCodes > Fmt<BSD>::kCodes ? Fmt<BD>::kCodes : Fmt<BSD>::kCodes;
  constexpr int SPT_LIMIT = kMaxActRegs / CMAX > 0 ? kMaxActRegs / CMAX : 1;
  if (SPT_LIMIT >= 2 && g.spt >= 2)
    consume_b_spt<BD, BSD, (SPT_LIMIT >= 2 ? 2 : 1)>(s, g, ids_s, act, resid_s, out, out_f32, r,
                                                      sm, tid);
  else
    consume_b_spt<BD, BSD, 1>(s, g, ids_s, act, resid_s, out, out_f32, r, sm, tid);
}

}  // namespace moe
