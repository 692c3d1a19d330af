// moe_cols.cuh -- the column-split decode kernel: one grid barrier per layer.
//
// The block computes, per token (the pages' two phases, "two-kernel decode-MoE that beats
// gather_qmm", What changed, step 2, and the tail of "Red Lite dev39 -- fused expert tail"):
//   act[u] = coef_u * silu(gate_u . x) * (up_u . x)          u over routed slots' and shared rows
//   out    = resid + sum_u W_down[:, u] * act[u]
// Kernel A and kernel B split that work by ROWS of each projection, so every CTA of kernel B needs
// every activation and the two phases meet at a device-wide exchange.  Here every CTA owns a
// contiguous, balanced range of the activation index u instead (the same balanced split phase A
// uses) and carries its columns through both projections:
//   1. phase A on the CTA's gate/up rows (the rows u of its range), activations kept in shared
//      memory;
//   2. the matching COLUMNS u of the down projections, read from a column-block-major copy
//      (moe_kernels.cuh), multiplied by the local activations into a partial output for all din
//      rows, written to a slab in global memory;
//   3. one grid barrier;
//   4. at the start of the next layer (or after the last one) each CTA sums, in a fixed order, the
//      partials of the din / grid rows it owns and adds the residual, which it keeps in shared
//      memory from layer to layer.
// The next layer's expert ids are read only after that barrier, when every CTA has finished the
// layer (its output exists as the partials), so no weight of a layer is requested before the
// previous layer is done.  With p.ahead (every layer's ids are inputs known before the step) the
// producer instead starts layer l + 1 as soon as its own CTA's consumers have finished layer l's
// gate/up phase (a CTA-local mbarrier), so the weight stream runs on across the layer boundary;
// the arithmetic and its order are the same.
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

namespace moe {

struct ColSmem {
  float act[kMaxColsCta];                 // the CTA's activations, index u - u0
  uint32_t planes[kMaxColBlocks * 8];     // per block: byte planes (3 words at 8 bits, 6 at 4)
  float2 us[kMaxColPieces];               // per piece: (unit, sum of its activations)
  ColPiece pc[kMaxColPieces];
  float resid[kMaxOwnRows];               // the owned rows' running output (the next residual)
  int np, nbk;
  int u0;
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

// Producer: the down column blocks of every valid piece, at most cp.nbs blocks per stage; the
// last stage of a piece also carries the piece's group of (scale, bias) pairs for all din rows.
__device__ inline void produce_down_cols(const LayerShape &s, const ColPlan &cp, const ColPtrs &cw,
                                  const ColSmem &cs, const int *ids, Ring &r, int lane,
                                  uint64_t pol) {
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
      if (!ring_claim(r, lane)) return;
      uint8_t *sb = r.stage();
      const uint32_t code_bytes = static_cast<uint32_t>(nk) * blk_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&r.full[r.st], code_bytes + (ends ? blk_bytes : 0u));
      __syncwarp();
      if (lane == 0)
        bulk_g2s(sb,
                 d.codes + (static_cast<int64_t>(e) * nblk + q.blk0 + bo) * s.din,
                 code_bytes, &r.full[r.st], pol);
      if (lane == 1 && ends)
        bulk_g2s(sb + code_bytes, d.sb + (static_cast<int64_t>(e) * G + q.grp) * s.din, blk_bytes,
                 &r.full[r.st], pol);
      r.advance();
    }
  }
}

// Consumers: byte planes of every block of every valid piece, from the local activations.
// Warp w handles pieces w, w + 16, ...; lane b the piece's block b.
template <int BD, int BSD>
__device__ inline void col_planes(const LayerShape &s, const ColPlan &cp, ColSmem &cs, const int *ids,
                           int warp, int lane) {
  for (int qi = warp; qi < cs.np; qi += kConsumerWarps) {
    const ColPiece q = cs.pc[qi];
    int e;
    if (!col_valid(s, q, ids, &e)) continue;
    const bool routed = q.seg < s.top_k;
    const int bits = routed ? BD : BSD;
    const int cb = routed ? cp.cb_r : cp.cb_s;
    const int n = q.j1 - q.j0;  // at most 64
    const float v0 = lane < n ? cs.act[q.a0 + lane] : 0.f;
    const float v1 = lane + 32 < n ? cs.act[q.a0 + lane + 32] : 0.f;
    const float mx = warp_max(fmaxf(fabsf(v0), fabsf(v1)));
    const float sm = warp_sum(v0 + v1);
    const int E = fixed_exponent(mx);
    const float sc = pow2f(22 - E);
    if (lane == 0) cs.us[qi] = make_float2(pow2f(bits == 8 ? E - 22 : E - 26), sm);
    for (int b = lane; b < q.nb; b += 32) {
      const int c0 = (q.blk0 + b) * cb;  // first column of the block, expert coordinates
      int f[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + k;
        f[k] = (k < cb && c >= q.j0 && c < q.j1) ? __float2int_rn(cs.act[q.a0 + c - q.j0] * sc)
                                                 : 0;
      }
      uint32_t *pl = cs.planes + (q.pb + b) * 8;
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
// 4 quad .. 4 quad + 3); its exact integer sums run over all of the piece's blocks, and the
// piece's last stage applies the group's scale and bias to them into part[][].
template <int BITS, int QPT>
__device__ __forceinline__ void consume_piece(const ColPiece &q, float2 us, const ColPlan &cp,
                                              int din, const uint32_t *planes, Ring &r,
                                              int lane, int tid, float (&part)[2][4]) {
  constexpr int NPL = BITS == 8 ? 3 : 6;
  const int nquads = din >> 2;
  const uint32_t blk_bytes = static_cast<uint32_t>(din) * 4u;
  uint32_t al[QPT][4][NPL];  // l and m planes (unsigned) and h planes (two's complement) per row
#pragma unroll
  for (int a = 0; a < QPT; ++a)
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int z = 0; z < NPL; ++z) al[a][k][z] = 0u;
  for (int bo = 0; bo < q.nb; bo += cp.nbs) {
    const int nk = (q.nb - bo) < cp.nbs ? (q.nb - bo) : cp.nbs;
    const bool ends = bo + nk == q.nb;
    const bool ok = warp_wait_full(r, lane);
    const uint8_t *sb = r.stage();
    if (ok) {
      for (int b = 0; b < nk; ++b) {
        const uint4 pa = *reinterpret_cast<const uint4 *>(planes + (q.pb + bo + b) * 8);
        const uint4 pb = *reinterpret_cast<const uint4 *>(planes + (q.pb + bo + b) * 8 + 4);
        const uint8_t *cp_b = sb + static_cast<uint32_t>(b) * blk_bytes;
#pragma unroll
        for (int a = 0; a < QPT; ++a) {
          const int quad = tid + a * kConsumers;
          if (quad < nquads) {
            const uint4 w4 = lds_u4(cp_b + quad * 16);
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              if constexpr (BITS == 8) {
                al[a][k][0] = dp4a_uu(w[k], pa.x, al[a][k][0]);
                al[a][k][1] = dp4a_uu(w[k], pa.y, al[a][k][1]);
                al[a][k][2] = static_cast<uint32_t>(
                    dp4a_us(w[k], pa.z, static_cast<int>(al[a][k][2])));
              } else {
                const uint32_t lo = w[k] & 0x0f0f0f0fu, hi = w[k] & 0xf0f0f0f0u;
                al[a][k][0] = dp4a_uu(lo, pa.x, al[a][k][0]);
                al[a][k][1] = dp4a_uu(lo, pa.y, al[a][k][1]);
                al[a][k][2] = static_cast<uint32_t>(
                    dp4a_us(lo, pa.z, static_cast<int>(al[a][k][2])));
                al[a][k][3] = dp4a_uu(hi, pa.w, al[a][k][3]);
                al[a][k][4] = dp4a_uu(hi, pb.x, al[a][k][4]);
                al[a][k][5] = static_cast<uint32_t>(
                    dp4a_us(hi, pb.y, static_cast<int>(al[a][k][5])));
              }
            }
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
              uint32_t l, m;
              int h;
              if constexpr (BITS == 8) {
                l = al[a][k][0];
                m = al[a][k][1];
                h = static_cast<int>(al[a][k][2]);
              } else {
                // the even sums scaled by 16 join the odd ones (read as 16 q)
                l = al[a][k][0] * 16u + al[a][k][3];
                m = al[a][k][1] * 16u + al[a][k][4];
                h = static_cast<int>(al[a][k][2]) * 16 + static_cast<int>(al[a][k][5]);
              }
              // l, m < 2^22 over a group of 64 columns, so m * 256 + l < 2^31
              const float dot = fmaf(static_cast<float>(h), 65536.f, static_cast<float>(m * 256u + l));
              const __half2 sbh = *reinterpret_cast<const __half2 *>(&hw[k]);
              const float sc = __low2float(sbh), bi = __high2float(sbh);
              part[a][k] += fmaf(sc, dot * us.x, bi * us.y);
            }
          }
        }
      }
    }
    warp_release(r, lane);
  }
}

// The owner's rows [i0, i1) of the partials of one pass: fixed-order sums over the grid's CTAs,
// added to the running output in shared memory; `out` (when set) receives the result.
__device__ __forceinline__ void col_reduce(const float *slab, int din, int ro, ColSmem &cs,
                                           void *out, int out_f32, int warp, int lane) {
  const int n = gridDim.x, c = blockIdx.x;
  const int i0 = static_cast<int>(static_cast<int64_t>(din) * c / n);
  const int i1 = static_cast<int>(static_cast<int64_t>(din) * (c + 1) / n);
  const float *blk = slab + static_cast<int64_t>(c) * n * ro;
  for (int rr = warp; rr < i1 - i0; rr += kConsumerWarps) {
    float t = 0.f;
    for (int cc = lane; cc < n; cc += 32) t += __ldcg(blk + static_cast<int64_t>(cc) * ro + rr);
    t = warp_sum(t);
    if (lane == 0) {
      const float o = cs.resid[rr] + t;
      cs.resid[rr] = o;
      if (out != nullptr) {
        if (out_f32)
          static_cast<float *>(out)[i0 + rr] = o;
        else
          static_cast<uint16_t *>(out)[i0 + rr] = float_to_bf16_rn(o);
      }
    }
  }
}

// One token per layer (m = 1), layers [0, L): see the top of this file.
template <int BR, int BD, int BSH>
__global__ void __launch_bounds__(kThreads, 1) cols_kernel(const StackParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) RingSmem rs;
  __shared__ SmemA sma;
  __shared__ __align__(16) ColSmem cs;
  __shared__ LayerPtrs wl;   // the consumers' copy of the current layer's pointers
  __shared__ LayerPtrs wpr;  // the producers' copy
  __shared__ ColPtrs cpr;
  __shared__ int stop_pr;
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
    int64_t u0 = 0;
    cs.np = col_pieces(s.top_k, s.dff, s.n_shared, s.dff_shared, p.cp.cb_r, p.cp.cb_s,
                       blockIdx.x, n, cs.pc, &nbk, &u0);
    cs.nbk = nbk;
    cs.u0 = static_cast<int>(u0);
    if (cs.np < 0) {  // outside the plan (the host checks every CTA): do nothing
      cs.np = 0;
      atomicOr(p.err, kDevErrTimeout);
      rs.abort = 1;
    }
  }
  __syncthreads();
  Ring r = make_ring(rs.full, rs.empty, ring, rs.desc, p.plan, &rs.abort, p.err);

  if (warp >= kConsumerWarps) {
    const uint64_t pol = policy_evict_first();
    const int pl = tid - kConsumers;
    for (int l = 0; l < p.L; ++l) {
      producer_sync();  // every producer is done with the previous layer's copies
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
        stop_pr = flag_abort(&rs.abort);
      }
      producer_sync();
      if (stop_pr) break;
      const int64_t ks = s.top_k;
      int *ids_l = ids2[l & 1];
      float *sc_l = sc2[l & 1];
      producer_load_token(s, p.ids + l * ks, p.scores + l * ks, ids_l, sc_l, p.err, pl);
      produce_a<BR, BSH>(s, wpr, p.plan.geo_r, p.plan.geo_s, ids_l, sc_l, rs.cnt, r, pl, pol);
      produce_down_cols(s, p.cp, cpr, cs, ids_l, r, pl, pol);
    }
    ring_drain(r, pl);
    return;
  }

  // the owned rows' residual (layer 0's input)
  {
    const int i0 = static_cast<int>(static_cast<int64_t>(s.din) * blockIdx.x / n);
    const int i1 = static_cast<int>(static_cast<int64_t>(s.din) * (blockIdx.x + 1) / n);
    for (int t = tid; t < i1 - i0; t += kConsumers)
      cs.resid[t] = p.resid0_f32 ? static_cast<const float *>(p.resid0)[i0 + t]
                                 : bf16_to_float(static_cast<const uint16_t *>(p.resid0)[i0 + t]);
  }
  const int64_t slab_pass = static_cast<int64_t>(n) * n * p.cp.ro;
  const int nquads = s.din >> 2;
  for (int l = 0; l < p.L; ++l) {
    if (tid == 0) wl = p.layers[l];
    consumer_sync(kConsumers);
    // the previous layer's output rows this CTA owns (the barrier has passed)
    if (l > 0) col_reduce(p.slab + ((l - 1) & 1) * slab_pass, s.din, p.cp.ro, cs, nullptr, 1,
                          warp, lane);
    consume_a<BR, BSH, false>(s, wl, p.plan.geo_r, p.plan.geo_s,
                              xsource_plain(p.x + static_cast<int64_t>(l) * s.din), rs.cnt,
                              cs.act, r, sma, tid, cs.u0);
    consumer_sync(kConsumers);  // activations complete; the ids were published by phase A
    if (tid == 0) mbar_arrive(&a_done);
    const int *ids_l = ids2[l & 1];
    col_planes<BD, BSH>(s, p.cp, cs, ids_l, warp, lane);
    consumer_sync(kConsumers);
    float part[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) part[a][k] = 0.f;
    for (int qi = 0; qi < cs.np; ++qi) {
      const ColPiece q = cs.pc[qi];
      int e;
      if (!col_valid(s, q, ids_l, &e)) continue;
      const bool two = s.din > 4 * kConsumers;  // a second row quad per thread
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
    // partials of all din rows into the slab, grouped by the row's owner CTA
    float *sl = p.slab + (l & 1) * slab_pass;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int quad = tid + a * kConsumers;
      if (quad < nquads) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 4 * quad + k;
          const int o = static_cast<int>((static_cast<int64_t>(i + 1) * n - 1) / s.din);
          const int rr = i - static_cast<int>(static_cast<int64_t>(s.din) * o / n);
          sl[(static_cast<int64_t>(o) * n + blockIdx.x) * p.cp.ro + rr] = part[a][k];
        }
      }
    }
    consumers_grid_barrier(p.bar, static_cast<uint32_t>(l + 1) * n, tid, &rs.abort, p.err);
  }
  col_reduce(p.slab + ((p.L - 1) & 1) * slab_pass, s.din, p.cp.ro, cs, p.out, p.out_f32, warp,
             lane);
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
      return launch(cols_kernel<BR, BD, BSH>, p, grid, p.plan.smem, stream, false, true)));
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
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, cols_kernel<BR, BD, BSH>, kThreads,
                                                        smem)));
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
