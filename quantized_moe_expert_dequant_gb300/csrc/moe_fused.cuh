// moe_fused.cuh -- the decode MoE kernels built from the phases of moe_phases.cuh:
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
#pragma once

#include "moe_grouped.cuh"

namespace moe {

__device__ __forceinline__ void init_ring(uint64_t *full, uint64_t *empty, int nst, int *abort) {
  if (threadIdx.x == 0) {
    MOE_TL_SET_HOOK(nullptr);  // timeline builds: no phase stamps unless a kernel asks for them
    MOE_TL_SET_HOOK_P(nullptr);
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

template <int BR, int BS, bool CHAIN>
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
    producer_load_token(p.s, p.ids, p.scores, rs.ids, rs.scores, p.err, pl, p.ids_used);
    produce_a<BR, BS>(p.s, p.w, p.plan.geo_r, p.plan.geo_s, rs.ids, rs.scores, rs.cnt, r, pl,
                      policy_evict_first());
    ring_drain(r, pl);
    return;
  }
  const XSource xs = CHAIN ? XSource{nullptr, p.v, p.gamma, p.eps, 1.f} : xsource_plain(p.x);
  consume_a<BR, BS, CHAIN>(p.s, p.w, p.plan.geo_r, p.plan.geo_s, xs, rs.cnt, p.act, r, sm, tid);
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

// What a fused kernel instance runs: tokens one at a time, the same with the next layer's RMSNorm
// folded in (p.norm_w set), or batches grouped by expert (p.grouped).  Each is its own instance so
// that none carries the others' registers.
enum FusedMode { kTokens = 0, kTokensNorm = 1, kGrouped = 2 };

template <int BR, int BD, int BSH, int MODE>
__global__ void __launch_bounds__(kThreads, 1) fused_kernel(const StackParams p) {
  constexpr bool CHAIN = MODE == kTokensNorm;
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
  if constexpr (MODE == kGrouped) {
    fused_grouped<BR, BD, BSH>(p, ring, rs.full, rs.empty, rs.desc, &rs.abort, sm.a, wl, wpr,
                               stop_pr, tid);
    return;
  } else {
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
                              pl, p.ids_used ? p.ids_used + tok * ks : nullptr);
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
        // x: the layer's input, or (norm folded in) the previous layer's output, normalised
        XSource xsrc = xsource_plain(p.x + tok * xs);
        if (CHAIN && l > 0)
          xsrc = XSource{nullptr, ((l - 1) & 1 ? p.ping1 : p.ping0) + t * xs,
                         p.norm_w + static_cast<int64_t>(l - 1) * xs, p.norm_eps, 1.f};
        consume_a<BR, BSH, CHAIN>(s, w, p.plan.geo_r, p.plan.geo_s, xsrc, rs.cnt, p.act, r, sm.a,
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
  }  // token modes
}

template <typename Kern, typename P>
inline cudaError_t launch(Kern kern, const P &p, int grid, size_t smem, cudaStream_t stream,
                          bool pdl, bool cooperative, int threads = kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
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


// ------------------------------------------------------------------ families of kernels
// The kernels are instantiated per gate/up code width BR in translation units of their own, so
// that they compile in parallel: moe_kernels_g<BR>.cu holds kernel A, the down kernels of width BR
// and the fused token kernels (both modes); moe_grouped_g<BR>.cu holds the fused grouped kernels.

template <int BR>
cudaError_t launch_fused_family(const StackParams &p, int grid, size_t smem,
                                cudaStream_t stream) {
  const bool chain = p.norm_w != nullptr;
  MOE_BITS_SWITCH(p.plan.geo_b.bits_r, BD, MOE_BITS_SWITCH(p.plan.geo_s.bits, BSH,
      return chain
          ? launch(fused_kernel<BR, BD, BSH, kTokensNorm>, p, grid, smem, stream, false, true)
          : launch(fused_kernel<BR, BD, BSH, kTokens>, p, grid, smem, stream, false, true)));
  return cudaErrorInvalidValue;
}

template <int BR>
cudaError_t launch_grouped_family(const StackParams &p, int grid, size_t smem,
                                  cudaStream_t stream) {
  MOE_BITS_SWITCH(p.plan.geo_b.bits_r, BD, MOE_BITS_SWITCH(p.plan.geo_s.bits, BSH,
      return launch(fused_kernel<BR, BD, BSH, kGrouped>, p, grid, smem, stream, false, true)));
  return cudaErrorInvalidValue;
}

template <int BR>
cudaError_t launch_gate_up_family(const GateUpParams &p, int grid, cudaStream_t stream,
                                  bool pdl) {
  MOE_BITS_SWITCH(p.plan.geo_s.bits, BS,
      return p.v != nullptr
                 ? launch(gate_up_kernel<BR, BS, true>, p, grid, p.plan.smem, stream, pdl, false)
                 : launch(gate_up_kernel<BR, BS, false>, p, grid, p.plan.smem, stream, pdl, false));
  return cudaErrorInvalidValue;
}

template <int BD>
cudaError_t launch_down_family(const DownParams &p, int grid, cudaStream_t stream, bool pdl) {
  MOE_BITS_SWITCH(p.plan.geo_b.bits_s, BSD,
      return launch(down_kernel<BD, BSD>, p, grid, p.plan.smem, stream, pdl, false));
  return cudaErrorInvalidValue;
}

// Sets the dynamic shared-memory limit of a kernel to the most the device allows next to its
// static shared memory (the attribute is global to a kernel instance, so one handle can never
// lower it below what another handle launches with); *lim becomes the smallest such limit.
inline cudaError_t set_smem_limit(const void *fn, int smem_optin, int *lim) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return e;
  const int dyn = smem_optin - static_cast<int>(fa.sharedSizeBytes);
  if (dyn < *lim) *lim = dyn;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

// The kernels of width BR that a config with (bits_d, bits_sh) may launch: kernel A (both
// inputs) and the fused token kernels (both modes), or (down) the down kernels of width BR.
template <int BR>
cudaError_t prepare_family(int smem_optin, int bits_d, int bits_sh, bool down, int *lim) {
  cudaError_t e = cudaSuccess;
  auto set = [&](const void *fn) {
    if (e == cudaSuccess) e = set_smem_limit(fn, smem_optin, lim);
  };
  if (down) {
    MOE_BITS_SWITCH(bits_sh, BSD, set(reinterpret_cast<const void *>(down_kernel<BR, BSD>)));
    return e;
  }
  MOE_BITS_SWITCH(bits_sh, BS,
      set(reinterpret_cast<const void *>(gate_up_kernel<BR, BS, false>));
      set(reinterpret_cast<const void *>(gate_up_kernel<BR, BS, true>)));
  MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sh, BSH,
      set(reinterpret_cast<const void *>(fused_kernel<BR, BD, BSH, kTokens>));
      set(reinterpret_cast<const void *>(fused_kernel<BR, BD, BSH, kTokensNorm>))));
  return e;
}

template <int BR>
cudaError_t prepare_grouped_family(int smem_optin, int bits_d, int bits_sh, int *lim) {
  cudaError_t e = cudaSuccess;
  MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sh, BSH,
      e = set_smem_limit(reinterpret_cast<const void *>(fused_kernel<BR, BD, BSH, kGrouped>),
                         smem_optin, lim)));
  return e;
}

// CTAs per SM of the fused kernels of a mode set with smem dynamic bytes (the smallest).
template <int BR, int MODE>
cudaError_t fused_occupancy_mode(int bits_d, int bits_sh, size_t smem, int *per_sm) {
  cudaError_t e = cudaSuccess;
  int n = 0;
  MOE_BITS_SWITCH(bits_d, BD, MOE_BITS_SWITCH(bits_sh, BSH,
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_kernel<BR, BD, BSH, MODE>,
                                                        kThreads, smem)));
  if (n < *per_sm) *per_sm = n;
  return e;
}

// The non-template entry points, defined once per width in moe_kernels_g<B>.cu ...
#define MOE_KERNEL_FAMILY(B)                                                                     \
  cudaError_t launch_fused_g##B(const StackParams &p, int grid, size_t smem,                     \
                                cudaStream_t stream) {                                           \
    return launch_fused_family<B>(p, grid, smem, stream);                                        \
  }                                                                                              \
  cudaError_t launch_gate_up_g##B(const GateUpParams &p, int grid, cudaStream_t stream,          \
                                  bool pdl) {                                                    \
    return launch_gate_up_family<B>(p, grid, stream, pdl);                                       \
  }                                                                                              \
  cudaError_t launch_down_g##B(const DownParams &p, int grid, cudaStream_t stream, bool pdl) {   \
    return launch_down_family<B>(p, grid, stream, pdl);                                          \
  }                                                                                              \
  cudaError_t prepare_g##B(int smem_optin, int bits_d, int bits_sh, bool down, int *lim) {       \
    return prepare_family<B>(smem_optin, bits_d, bits_sh, down, lim);                            \
  }                                                                                              \
  cudaError_t fused_occupancy_g##B(int bits_d, int bits_sh, size_t smem, int *per_sm) {          \
    cudaError_t e = fused_occupancy_mode<B, kTokens>(bits_d, bits_sh, smem, per_sm);             \
    return e == cudaSuccess ? fused_occupancy_mode<B, kTokensNorm>(bits_d, bits_sh, smem, per_sm) \
                            : e;                                                                 \
  }

// ... and in moe_grouped_g<B>.cu.
#define MOE_GROUPED_FAMILY(B)                                                                    \
  cudaError_t launch_grouped_g##B(const StackParams &p, int grid, size_t smem,                   \
                                  cudaStream_t stream) {                                         \
    return launch_grouped_family<B>(p, grid, smem, stream);                                      \
  }                                                                                              \
  cudaError_t prepare_grouped_g##B(int smem_optin, int bits_d, int bits_sh, int *lim) {          \
    return prepare_grouped_family<B>(smem_optin, bits_d, bits_sh, lim);                          \
  }                                                                                              \
  cudaError_t grouped_occupancy_g##B(int bits_d, int bits_sh, size_t smem, int *per_sm) {        \
    return fused_occupancy_mode<B, kGrouped>(bits_d, bits_sh, smem, per_sm);                     \
  }

}  // namespace moe
