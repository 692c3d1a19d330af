// moe_api.cu -- the C ABI of include/moe_decode.h: validation, prepared handles, the layer-stack
// CUDA-graph driver and the host-buffer step.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "moe_decode.h"
#include "moe_kernels.cuh"
#include "moe_mma.cuh"
#include "moe_timeline.cuh"

namespace {

bool bits_ok(int b) { return b == 4 || b == 6 || b == 8; }
// The column-split kernel serves both column modes (strict layer order, or ids known ahead).
bool cols_mode(int kernel_mode) {
  return kernel_mode == MOE_KERNELS_COLUMNS || kernel_mode == MOE_KERNELS_COLUMNS_AHEAD;
}
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool proj_ok(const moe_proj &p) {
  return p.codes && p.scales && p.biases && aligned(p.codes, 16) && aligned(p.scales, 16) &&
         aligned(p.biases, 16);
}

int validate_config(const moe_decode_config *c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->din <= 0 || c->din % 64 || c->dff <= 0 || c->dff % 64) return MOE_ERR_INVALID_ARG;
  if (c->n_experts < 1 || c->top_k < 0 || c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (c->max_tokens < 1) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > 4) return MOE_ERR_INVALID_ARG;
  if (c->top_k + c->n_shared < 1) return MOE_ERR_INVALID_ARG;
  if (c->n_shared > 0 && (c->dff_shared <= 0 || c->dff_shared % 64)) return MOE_ERR_INVALID_ARG;
  if (!bits_ok(c->bits_gate) || !bits_ok(c->bits_up) || !bits_ok(c->bits_down))
    return MOE_ERR_UNSUPPORTED;
  if (c->n_shared > 0 && !bits_ok(c->bits_shared)) return MOE_ERR_UNSUPPORTED;
  if (c->bits_gate != c->bits_up) return MOE_ERR_UNSUPPORTED;
  if (c->shared_gate != 0 && c->shared_gate != 1) return MOE_ERR_INVALID_ARG;
  if (c->resid_dtype != MOE_DTYPE_BF16 && c->resid_dtype != MOE_DTYPE_F32)
    return MOE_ERR_INVALID_ARG;
  if (c->out_dtype != MOE_DTYPE_BF16 && c->out_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
  if (c->kernel_mode != MOE_KERNELS_FUSED && c->kernel_mode != MOE_KERNELS_SEPARATE &&
      c->kernel_mode != MOE_KERNELS_POOL && c->kernel_mode != MOE_KERNELS_MMA &&
      !cols_mode(c->kernel_mode))
    return MOE_ERR_INVALID_ARG;
  // int32 indexing of the activation vector and of one expert's rows
  const int64_t act = (int64_t)c->top_k * c->dff + (int64_t)c->n_shared * c->dff_shared;
  if (act > (1 << 24) || (int64_t)c->din * c->dff > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int validate_weights(const moe_decode_config *c, const moe_layer_weights *w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (c->top_k > 0 && (!proj_ok(w->gate) || !proj_ok(w->up) || !proj_ok(w->down)))
    return MOE_ERR_INVALID_ARG;
  if (c->n_shared > 0 && (!proj_ok(w->sh_gate) || !proj_ok(w->sh_up) || !proj_ok(w->sh_down)))
    return MOE_ERR_INVALID_ARG;
  if (c->n_shared > 0 && c->shared_gate == 1 && (!w->gate_vec || !aligned(w->gate_vec, 2)))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe::ProjDev dev(const moe_proj &p) {
  return moe::ProjDev{static_cast<const uint8_t *>(p.codes),
                      static_cast<const __half *>(p.scales), static_cast<const __half *>(p.biases)};
}

moe::LayerPtrs layer_ptrs(const moe_decode_config &c, const moe_layer_weights &w) {
  moe::LayerPtrs p;
  p.gate = dev(w.gate);
  p.up = dev(w.up);
  p.down = dev(w.down);
  p.sh_gate = dev(w.sh_gate);
  p.sh_up = dev(w.sh_up);
  p.sh_down = dev(w.sh_down);
  p.gate_vec = (c.n_shared > 0 && c.shared_gate == 1) ? static_cast<const uint16_t *>(w.gate_vec)
                                                      : nullptr;
  return p;
}

// What every launch of a given shape needs, resolved once at create time.
struct Prepared {
  moe_decode_config cfg;
  moe::LayerShape shape;
  moe::Plan plan;
  int bits_sh;       // shared-expert code width as the kernels see it
  int grid_sep;      // CTAs of the separate kernels
  int grid_fused;    // CTAs of the fused kernel (all resident)
  bool grouped_ok;   // m > 1 forwards stream each selected expert once (fused mode)
  moe::GroupPlan gplan;
  // column-split mode
  moe::Plan col_plan;
  moe::ColPlan cplan;
  int grid_cols = 0;
};

int prepare(const moe_decode_config *c, Prepared &P) {
  int rc = validate_config(c);
  if (rc != MOE_OK) return rc;
  P.cfg = *c;
  P.shape = moe::LayerShape{c->din, c->dff, c->top_k, c->n_experts, c->n_shared, c->dff_shared};
  P.bits_sh = c->n_shared > 0 ? c->bits_shared : c->bits_down;
  if (!moe::make_plan(P.shape, c->bits_gate, c->bits_down, P.bits_sh, &P.plan))
    return MOE_ERR_UNSUPPORTED;
  int device = 0, sms = 0, smem_optin = 0, major = 0, minor = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  int dyn_limit = 0;
  if (moe::prepare_kernels(smem_optin, c->bits_gate, c->bits_down, P.bits_sh, &dyn_limit) !=
      cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (P.plan.smem > (size_t)dyn_limit) return MOE_ERR_UNSUPPORTED;
  // Batches of tokens run grouped by expert when the shape allows it; otherwise token by token.
  // The pool mode always runs the grouped kernel (a plan for at least two tokens also serves one).
  const bool pool = c->kernel_mode == MOE_KERNELS_POOL;
  P.grouped_ok = ((c->max_tokens > 1 && c->kernel_mode == MOE_KERNELS_FUSED) || pool) &&
                 moe::make_group_plan(P.shape, c->bits_gate, c->bits_down, P.bits_sh,
                                      c->max_tokens > 1 ? c->max_tokens : 2, &P.gplan) &&
                 P.gplan.smem <= (size_t)dyn_limit;
  if (pool && !P.grouped_ok) return MOE_ERR_UNSUPPORTED;
  // the tensor-core batch kernels group at most kMaxPairs slots of kMaxGroupTokens tokens
  if (c->kernel_mode == MOE_KERNELS_MMA &&
      (c->max_tokens > moe::kMaxGroupTokens || c->max_tokens * c->top_k > moe::kMaxPairs ||
       c->n_experts > moe::kMaxGroupExperts))
    return MOE_ERR_UNSUPPORTED;
  P.grid_sep = sms;
  const int lim = moe::fused_grid_limit(P.plan, c->bits_gate, c->bits_down, P.bits_sh);
  P.grid_fused = lim < sms ? lim : sms;
  const bool fused_grid = c->kernel_mode == MOE_KERNELS_FUSED || pool;
  if (fused_grid && P.grid_fused < 1) return MOE_ERR_UNSUPPORTED;
  const int grid = fused_grid ? P.grid_fused : P.grid_sep;
  if ((c->din + grid - 1) / grid > moe::kMaxRowsB) return MOE_ERR_UNSUPPORTED;
  if (cols_mode(c->kernel_mode)) {
    if (c->max_tokens != 1) return MOE_ERR_UNSUPPORTED;
    int lim = 0;
    if (moe::prepare_cols(smem_optin, moe::col_gu_bits(c->bits_gate),
                          moe::col_down_bits(c->bits_down), moe::col_down_bits(P.bits_sh),
                          &lim) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_UNSUPPORTED;  // no column-split kernel for these code widths
    }
    const int ring = lim < moe::kRingBytes ? lim : moe::kRingBytes;
    if (!moe::make_col_plan(P.shape, c->bits_gate, c->bits_down, P.bits_sh, sms, ring, &P.cplan,
                            &P.col_plan))
      return MOE_ERR_UNSUPPORTED;
    const int per = moe::cols_grid_limit(P.col_plan.smem, moe::col_gu_bits(c->bits_gate),
                                         moe::col_down_bits(c->bits_down),
                                         moe::col_down_bits(P.bits_sh));
    if (per < sms) return MOE_ERR_UNSUPPORTED;  // one CTA per SM, all resident
    P.grid_cols = sms;
  }
  return MOE_OK;
}

size_t act_floats(const moe_decode_config &c) {
  return (size_t)c.top_k * c.dff + (size_t)c.n_shared * c.dff_shared;
}

size_t dtype_bytes(int dt) { return dt == MOE_DTYPE_F32 ? 4 : 2; }

// Kernel A's input when the previous layer's RMSNorm is folded in: x = RMSNorm(v) with weight
// gamma, v fp32 [m][din] (v null: kernel A reads x).
struct NormIn {
  const float *v = nullptr;
  const uint16_t *gamma = nullptr;
  float eps = 0.f;
};

// Separate kernels: kernel A then kernel B for each token of one layer.
cudaError_t enqueue_separate(const Prepared &P, const moe::LayerPtrs &w, float *act,
                             int32_t *err, const void *x, int m, const int32_t *ids,
                             const float *scores, const void *resid, int resid_dtype, void *out,
                             int out_dtype, cudaStream_t stream, int parts,
                             const NormIn &norm = NormIn{}, int32_t *ids_used = nullptr) {
  const moe_decode_config &c = P.cfg;
  for (int t = 0; t < m; ++t) {
    const int32_t *it = ids ? ids + (size_t)t * c.top_k : nullptr;
    moe::GateUpParams a;
    a.s = P.shape;
    a.w = w;
    a.plan = P.plan;
    a.x = norm.v ? nullptr : static_cast<const uint16_t *>(x) + (size_t)t * c.din;
    a.v = norm.v ? norm.v + (size_t)t * c.din : nullptr;
    a.gamma = norm.gamma;
    a.eps = norm.eps;
    a.ids = it;
    a.scores = scores ? scores + (size_t)t * c.top_k : nullptr;
    a.act = act;
    a.err = err;
    a.ids_used = ids_used ? ids_used + (size_t)t * c.top_k : nullptr;
    cudaError_t e = cudaSuccess;
    if (parts & MOE_PART_GATE_UP) e = moe::launch_gate_up(a, P.grid_sep, stream, true);
    if (e != cudaSuccess) return e;
    moe::DownParams b;
    b.s = P.shape;
    b.w = w;
    b.plan = P.plan;
    b.ids = it;
    b.act = act;
    b.resid = static_cast<const char *>(resid) + (size_t)t * c.din * dtype_bytes(resid_dtype);
    b.out = static_cast<char *>(out) + (size_t)t * c.din * dtype_bytes(out_dtype);
    b.resid_f32 = resid_dtype == MOE_DTYPE_F32;
    b.out_f32 = out_dtype == MOE_DTYPE_F32;
    b.err = err;
    if (parts & MOE_PART_DOWN) e = moe::launch_down(b, P.grid_sep, stream, true);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Fused kernel over L layers (device array `layers`) and m tokens.
cudaError_t enqueue_fused(const Prepared &P, const moe::LayerPtrs *layers, int L, float *act,
                          float *y, int32_t *err, uint32_t *bar, float *ping0, float *ping1,
                          const void *x, int m, const int32_t *ids, const float *scores,
                          const void *resid0, int resid_dtype, void *out, int out_dtype,
                          cudaStream_t stream, const uint16_t *norm_w = nullptr,
                          float norm_eps = 0.f, int32_t *ids_used = nullptr) {
  cudaError_t e = cudaMemsetAsync(bar, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  moe::StackParams p;
  p.s = P.shape;
  p.plan = P.plan;
  p.layers = layers;
  p.L = L;
  p.m = m;
  p.x = static_cast<const uint16_t *>(x);
  p.norm_w = norm_w;
  p.norm_eps = norm_eps;
  p.ids = ids;
  p.scores = scores;
  p.resid0 = resid0;
  p.resid0_f32 = resid_dtype == MOE_DTYPE_F32;
  p.ping0 = ping0;
  p.ping1 = ping1;
  p.out = out;
  p.out_f32 = out_dtype == MOE_DTYPE_F32;
  p.act = act;
  p.err = err;
  p.bar = bar;
  p.pool = P.cfg.kernel_mode == MOE_KERNELS_POOL;
  // the grouped path reads x only; the pool mode is always grouped
  p.grouped = (m > 1 && P.grouped_ok && norm_w == nullptr) || p.pool;
  p.ids_used = ids_used;
  p.gp = P.gplan;
  p.y = y;
  p.act_stride = static_cast<int>(act_floats(P.cfg));
  return moe::launch_fused(p, P.grid_fused, stream);
}

int read_and_clear_error(int32_t *err, int32_t *out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(err, 0, sizeof v) != cudaSuccess) return MOE_ERR_CUDA;
  *out = (v & 4) ? MOE_ERR_PLAN : (v & 2) ? MOE_ERR_TIMEOUT : (v & 1) ? MOE_ERR_BAD_ID : MOE_OK;
  return MOE_OK;
}

// Column-split launch over L layers (m = 1): see moe_cols.cuh.
cudaError_t enqueue_cols(const Prepared &P, const moe::LayerPtrs *layers,
                         const moe::ColPtrs *cols, int L, float *slab, int32_t *err,
                         uint32_t *bar, const void *x, const int32_t *ids, const float *scores,
                         const void *resid0, int resid_dtype, void *out, int out_dtype,
                         cudaStream_t stream, unsigned long long *tl = nullptr,
                         int32_t *ids_used = nullptr) {
  cudaError_t e = cudaMemsetAsync(bar, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  moe::StackParams p;
  std::memset(&p, 0, sizeof p);
  p.s = P.shape;
  p.plan = P.col_plan;
  p.layers = layers;
  p.L = L;
  p.m = 1;
  p.x = static_cast<const uint16_t *>(x);
  p.ids = ids;
  p.scores = scores;
  p.resid0 = resid0;
  p.resid0_f32 = resid_dtype == MOE_DTYPE_F32;
  p.out = out;
  p.out_f32 = out_dtype == MOE_DTYPE_F32;
  p.err = err;
  p.bar = bar;
  p.cols = cols;
  p.cp = P.cplan;
  p.slab = slab;
  p.ahead = P.cfg.kernel_mode == MOE_KERNELS_COLUMNS_AHEAD;
  p.tl = tl;
  p.ids_used = ids_used;
  return moe::launch_cols(p, P.grid_cols, stream);
}

// The column-block-major copies of every layer's down projections (column-split mode), owned by
// a handle or a stack.
struct ColWeights {
  std::vector<void *> bufs;
  moe::ColPtrs *dev = nullptr;  // device array [L]

  bool repack(int experts, int din, int dff, int bits, const moe_proj &p, moe::ColDownDev *out) {
    const size_t words = (size_t)experts * (dff * moe::col_down_bits(bits) / 32) * din;
    const size_t pairs = (size_t)experts * (dff / 64) * din;
    void *c = nullptr, *b = nullptr;
    if (cudaMalloc(&c, words * 4) != cudaSuccess) return false;
    bufs.push_back(c);
    if (cudaMalloc(&b, pairs * 4) != cudaSuccess) return false;
    bufs.push_back(b);
    out->codes = static_cast<const uint32_t *>(c);
    out->sb = static_cast<const __half2 *>(b);
    return moe::launch_repack_down(static_cast<const uint8_t *>(p.codes),
                                   static_cast<const __half *>(p.scales),
                                   static_cast<const __half *>(p.biases), experts, din, dff, bits,
                                   static_cast<uint32_t *>(c), static_cast<__half2 *>(b),
                                   nullptr) == cudaSuccess;
  }
  bool records(int experts, int rows, int din, int bits, const moe_proj &g, const moe_proj &u,
               const uint8_t **out) {
    void *b = nullptr;
    const size_t bytes = (size_t)experts * rows * moe::col_record_bytes(din, moe::col_gu_bits(bits));
    if (cudaMalloc(&b, bytes) != cudaSuccess) return false;
    bufs.push_back(b);
    *out = static_cast<const uint8_t *>(b);
    return moe::launch_repack_gate_up(
               static_cast<const uint8_t *>(g.codes), static_cast<const __half *>(g.scales),
               static_cast<const __half *>(g.biases), static_cast<const uint8_t *>(u.codes),
               static_cast<const __half *>(u.scales), static_cast<const __half *>(u.biases),
               experts, rows, din, bits, static_cast<uint8_t *>(b), nullptr) == cudaSuccess;
  }
  // MOE_OK, MOE_ERR_OOM or MOE_ERR_CUDA.
  int build(const moe_decode_config &c, const moe_layer_weights *w, int L) {
    // the caller's weights may still be written by work on other streams
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    std::vector<moe::ColPtrs> host(L);
    for (int l = 0; l < L; ++l) {
      moe::ColPtrs cp;
      std::memset(&cp, 0, sizeof cp);
      if (c.top_k > 0 && !repack(c.n_experts, c.din, c.dff, c.bits_down, w[l].down, &cp.r)) {
        cudaGetLastError();
        return MOE_ERR_OOM;
      }
      if (c.n_shared > 0 &&
          !repack(c.n_shared, c.din, c.dff_shared, c.bits_shared, w[l].sh_down, &cp.s)) {
        cudaGetLastError();
        return MOE_ERR_OOM;
      }
      if (c.top_k > 0 &&
          !records(c.n_experts, c.dff, c.din, c.bits_gate, w[l].gate, w[l].up, &cp.gu_r)) {
        cudaGetLastError();
        return MOE_ERR_OOM;
      }
      if (c.n_shared > 0 && !records(c.n_shared, c.dff_shared, c.din, c.bits_shared, w[l].sh_gate,
                                     w[l].sh_up, &cp.gu_s)) {
        cudaGetLastError();
        return MOE_ERR_OOM;
      }
      host[l] = cp;
    }
    if (cudaMalloc(&dev, sizeof(moe::ColPtrs) * L) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_OOM;
    }
    if (cudaMemcpy(dev, host.data(), sizeof(moe::ColPtrs) * L, cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  void release() {
    for (void *b : bufs) cudaFree(b);
    bufs.clear();
    cudaFree(dev);
    dev = nullptr;
  }
};

size_t slab_floats(const Prepared &P) {
  return cols_mode(P.cfg.kernel_mode)
             ? (size_t)2 * P.grid_cols * P.cfg.din
             : 0;
}

// Device workspace of a handle or a stack.
struct Workspace {
  float *act = nullptr;
  float *y = nullptr;
  int32_t *err = nullptr;
  uint32_t *bar = nullptr;
  moe::LayerPtrs *layers = nullptr;
  float *slab = nullptr;  // column-split mode: [2][grid][din] partial outputs
  int32_t *ids_used = nullptr;  // handles: [max_tokens][top_k] ids the last forward's kernels read
  int32_t *route = nullptr;     // tensor-core batch mode: the batch's route (kMmaRouteInts)
  float *sscal = nullptr;       // tensor-core batch mode: [max_tokens] shared scalars

  // Grouped forwards (and the tensor-core batch mode) keep every token's activations and
  // per-slot partial outputs at once.
  bool alloc(const moe_decode_config &c, int n_layers, bool grouped, size_t nslab = 0) {
    const size_t na = act_floats(c) * (grouped ? c.max_tokens : 1);
    const size_t ny = grouped ? (size_t)c.max_tokens * (c.top_k + c.n_shared) * c.din : 1;
    bool ok = cudaMalloc(&act, (na > 0 ? na : 1) * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&y, ny * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&err, sizeof(int32_t)) == cudaSuccess &&
              cudaMemset(err, 0, sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&bar, sizeof(uint32_t)) == cudaSuccess &&
              cudaMalloc(&layers, sizeof(moe::LayerPtrs) * n_layers) == cudaSuccess &&
              (nslab == 0 || cudaMalloc(&slab, nslab * sizeof(float)) == cudaSuccess) &&
              cudaMalloc(&ids_used, (size_t)c.max_tokens * (c.top_k > 0 ? c.top_k : 1) *
                                        sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&route, moe::kMmaRouteInts * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&sscal, (size_t)c.max_tokens * sizeof(float)) == cudaSuccess;
    if (!ok) cudaGetLastError();
    return ok;
  }
  void release() {
    cudaFree(act);
    cudaFree(y);
    cudaFree(err);
    cudaFree(bar);
    cudaFree(layers);
    cudaFree(slab);
    cudaFree(ids_used);
    cudaFree(route);
    cudaFree(sscal);
  }
};

// The tensor-core batch mode's own state: each layer's tile-group copy (moe_mma.cuh) and the
// batch workspace, owned by a handle or a stack.
struct MmaState {
  std::vector<void *> bufs;
  std::vector<moe::MmaLayerDev> layers;
  int32_t *nc = nullptr;
  float *xsum = nullptr, *xinv = nullptr, *ainv = nullptr, *asum = nullptr;
  __half *x16 = nullptr, *a16 = nullptr;
  float2 *gu_part = nullptr;
  float *y_part = nullptr;
  float *zero = nullptr;

  template <class T>
  bool grab(T **p, size_t bytes) {
    void *b = nullptr;
    if (cudaMalloc(&b, bytes > 0 ? bytes : 16) != cudaSuccess) return false;
    bufs.push_back(b);
    *p = static_cast<T *>(b);
    return true;
  }
  // MOE_OK, MOE_ERR_OOM or MOE_ERR_CUDA.
  int build(const moe_decode_config &c, const moe_layer_weights *w, int L) {
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    const size_t M = c.max_tokens, gx = c.din / 64, act = act_floats(c), ga = act / 64;
    const size_t ny = c.top_k + c.n_shared;
    bool ok = grab(&nc, 2 * sizeof(int32_t)) && grab(&xsum, M * gx * 4) &&
              grab(&xinv, M * gx * 4) && grab(&x16, M * gx * 128 * 2) &&
              grab(&gu_part, (size_t)moe::kMmaMaxChunks * M * act * 8) &&
              grab(&a16, M * ga * 128 * 2) && grab(&ainv, M * ga * 4) &&
              grab(&asum, M * ga * 4) &&
              grab(&y_part, (size_t)moe::kMmaMaxChunks * M * ny * c.din * 4) &&
              grab(&zero, 256) && cudaMemset(zero, 0, 256) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return MOE_ERR_OOM;
    }
    const int bsh = c.n_shared > 0 ? c.bits_shared : c.bits_down;
    layers.resize(L);
    for (int l = 0; l < L; ++l) {
      moe::MmaLayerDev d{};
      const moe_layer_weights &x = w[l];
      uint8_t *b = nullptr;
      if (c.top_k > 0) {
        if (!grab(&b, (size_t)c.n_experts * (c.dff / 16) * (c.din / 64) *
                          moe::mma_gu_block(c.bits_gate)))
          return MOE_ERR_OOM;
        d.gu_r = b;
        if (moe::launch_repack_mma_gu(
                static_cast<const uint8_t *>(x.gate.codes), static_cast<const __half *>(x.gate.scales),
                static_cast<const __half *>(x.gate.biases), static_cast<const uint8_t *>(x.up.codes),
                static_cast<const __half *>(x.up.scales), static_cast<const __half *>(x.up.biases),
                c.n_experts, c.dff, c.din, c.bits_gate, b, nullptr) != cudaSuccess)
          return MOE_ERR_CUDA;
        if (!grab(&b, (size_t)c.n_experts * (c.din / 16) * (c.dff / 64) *
                          moe::mma_dn_block(c.bits_down)))
          return MOE_ERR_OOM;
        d.dn_r = b;
        if (moe::launch_repack_mma_down(static_cast<const uint8_t *>(x.down.codes),
                                        static_cast<const __half *>(x.down.scales),
                                        static_cast<const __half *>(x.down.biases), c.n_experts,
                                        c.din, c.dff, c.bits_down, b, nullptr) != cudaSuccess)
          return MOE_ERR_CUDA;
      }
      if (c.n_shared > 0) {
        if (!grab(&b, (size_t)c.n_shared * (c.dff_shared / 16) * (c.din / 64) *
                          moe::mma_gu_block(bsh)))
          return MOE_ERR_OOM;
        d.gu_s = b;
        if (moe::launch_repack_mma_gu(
                static_cast<const uint8_t *>(x.sh_gate.codes),
                static_cast<const __half *>(x.sh_gate.scales),
                static_cast<const __half *>(x.sh_gate.biases),
                static_cast<const uint8_t *>(x.sh_up.codes),
                static_cast<const __half *>(x.sh_up.scales),
                static_cast<const __half *>(x.sh_up.biases), c.n_shared, c.dff_shared, c.din, bsh,
                b, nullptr) != cudaSuccess)
          return MOE_ERR_CUDA;
        if (!grab(&b, (size_t)c.n_shared * (c.din / 16) * (c.dff_shared / 64) *
                          moe::mma_dn_block(bsh)))
          return MOE_ERR_OOM;
        d.dn_s = b;
        if (moe::launch_repack_mma_down(static_cast<const uint8_t *>(x.sh_down.codes),
                                        static_cast<const __half *>(x.sh_down.scales),
                                        static_cast<const __half *>(x.sh_down.biases), c.n_shared,
                                        c.din, c.dff_shared, bsh, b, nullptr) != cudaSuccess)
          return MOE_ERR_CUDA;
      }
      layers[l] = d;
    }
    return cudaDeviceSynchronize() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  void release() {
    for (void *b : bufs) cudaFree(b);
    bufs.clear();
    layers.clear();
  }
};

// Tensor-core batch kernels (moe_mma.cu) for the m tokens of layer l.
cudaError_t enqueue_mma(const Prepared &P, const moe::LayerPtrs &w, const MmaState &ms, int l,
                        const Workspace &ws, const void *x, int m, const int32_t *ids,
                        const float *scores, const void *resid, int resid_dtype, void *out,
                        int out_dtype, cudaStream_t stream, int32_t *ids_used = nullptr) {
  const moe_decode_config &c = P.cfg;
  moe::MmaParams p;
  std::memset(&p, 0, sizeof p);
  p.s = P.shape;
  p.w = w;
  p.t = ms.layers[l];
  p.bits_r = c.bits_gate;
  p.bits_s = P.bits_sh;
  p.bits_dr = c.bits_down;
  p.bits_ds = P.bits_sh;
  p.m = m;
  p.x = static_cast<const uint16_t *>(x);
  p.ids = ids;
  p.scores = scores;
  p.resid = resid;
  p.out = out;
  p.resid_f32 = resid_dtype == MOE_DTYPE_F32;
  p.out_f32 = out_dtype == MOE_DTYPE_F32;
  p.act_stride = static_cast<int>(act_floats(c));
  p.route = ws.route;
  p.nc = ms.nc;
  p.sscal = ws.sscal;
  p.xsum = ms.xsum;
  p.xinv = ms.xinv;
  p.x16 = ms.x16;
  p.gu_part = ms.gu_part;
  p.a16 = ms.a16;
  p.ainv = ms.ainv;
  p.asum = ms.asum;
  p.y_part = ms.y_part;
  p.zero = ms.zero;
  p.err = ws.err;
  p.ids_used = ids_used;
  return moe::launch_mma_layer(p, stream);
}

}  // namespace

// ====================================================================== single layer
struct moe_decode {
  Prepared P;
  moe::LayerPtrs w;
  Workspace ws;
  ColWeights cw;
  MmaState mma;
  int last_m = 0;  // tokens of the last forward (moe_decode_routes)
};

extern "C" int moe_decode_create(const moe_decode_config *cfg, const moe_layer_weights *weights,
                                 moe_decode_t **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc != MOE_OK) return rc;
  rc = validate_weights(cfg, weights);
  if (rc != MOE_OK) return rc;
  moe_decode *h = new (std::nothrow) moe_decode();
  if (!h) return MOE_ERR_OOM;
  rc = prepare(cfg, h->P);
  if (rc != MOE_OK) {
    delete h;
    return rc;
  }
  h->w = layer_ptrs(*cfg, *weights);
  if (!h->ws.alloc(*cfg, 1, h->P.grouped_ok, slab_floats(h->P))) {
    h->ws.release();
    delete h;
    return MOE_ERR_OOM;
  }
  if (cols_mode(cfg->kernel_mode)) {
    rc = h->cw.build(*cfg, weights, 1);
    if (rc != MOE_OK) {
      h->cw.release();
      h->ws.release();
      delete h;
      return rc;
    }
  }
  if (cfg->kernel_mode == MOE_KERNELS_MMA) {
    rc = h->mma.build(*cfg, weights, 1);
    if (rc != MOE_OK) {
      h->mma.release();
      h->ws.release();
      delete h;
      return rc;
    }
  }
  if (cudaMemcpy(h->ws.layers, &h->w, sizeof h->w, cudaMemcpyHostToDevice) != cudaSuccess) {
    h->ws.release();
    delete h;
    return MOE_ERR_CUDA;
  }
  *out = h;
  return MOE_OK;
}

extern "C" int moe_decode_forward(moe_decode_t *h, const void *x, int32_t m, const int32_t *ids,
                                  const float *scores, const void *resid, void *out,
                                  void *stream) {
  if (!h || !x || !resid || !out) return MOE_ERR_INVALID_ARG;
  const moe_decode_config &c = h->P.cfg;
  if (m < 1 || m > c.max_tokens) return MOE_ERR_INVALID_ARG;
  if (c.top_k > 0 && (!ids || !scores)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(resid, dtype_bytes(c.resid_dtype)) ||
      !aligned(out, dtype_bytes(c.out_dtype)) || (ids && !aligned(ids, 4)) ||
      (scores && !aligned(scores, 4)))
    return MOE_ERR_INVALID_ARG;
  if (x == out) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  int32_t *used = c.top_k > 0 ? h->ws.ids_used : nullptr;
  if (cols_mode(c.kernel_mode))
    e = enqueue_cols(h->P, h->ws.layers, h->cw.dev, 1, h->ws.slab, h->ws.err, h->ws.bar, x, ids,
                     scores, resid, c.resid_dtype, out, c.out_dtype, st, nullptr, used);
  else if (c.kernel_mode == MOE_KERNELS_MMA)
    e = enqueue_mma(h->P, h->w, h->mma, 0, h->ws, x, m, ids, scores, resid, c.resid_dtype, out,
                    c.out_dtype, st, used);
  else if (c.kernel_mode == MOE_KERNELS_FUSED || c.kernel_mode == MOE_KERNELS_POOL)
    e = enqueue_fused(h->P, h->ws.layers, 1, h->ws.act, h->ws.y, h->ws.err, h->ws.bar, nullptr,
                      nullptr, x, m, ids, scores, resid, c.resid_dtype, out, c.out_dtype, st,
                      nullptr, 0.f, used);
  else
    e = enqueue_separate(h->P, h->w, h->ws.act, h->ws.err, x, m, ids, scores, resid,
                         c.resid_dtype, out, c.out_dtype, st,
                         MOE_PART_GATE_UP | MOE_PART_DOWN, NormIn{}, used);
  if (e == cudaSuccess) h->last_m = m;
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_decode_routes(moe_decode_t *h, int32_t *ids_used, void *slot_out,
                                 void *stream) {
  if (!h || (!ids_used && !slot_out)) return MOE_ERR_INVALID_ARG;
  const moe_decode_config &c = h->P.cfg;
  if (h->last_m < 1) return MOE_ERR_INVALID_ARG;  // no forward yet
  if (slot_out && c.kernel_mode != MOE_KERNELS_POOL) return MOE_ERR_UNSUPPORTED;
  if ((ids_used && !aligned(ids_used, 4)) || (slot_out && !aligned(slot_out, 4)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t m = h->last_m;
  if (ids_used && c.top_k > 0 &&
      cudaMemcpyAsync(ids_used, h->ws.ids_used, m * c.top_k * sizeof(int32_t),
                      cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (slot_out &&
      cudaMemcpyAsync(slot_out, h->ws.y, m * (c.top_k + c.n_shared) * c.din * sizeof(float),
                      cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" int moe_decode_get_error(moe_decode_t *h, int32_t *device_error) {
  if (!h) return MOE_ERR_INVALID_ARG;
  return read_and_clear_error(h->ws.err, device_error);
}

extern "C" void moe_decode_destroy(moe_decode_t *h) {
  if (!h) return;
  h->cw.release();
  h->mma.release();
  h->ws.release();
  delete h;
}

// ====================================================================== one layer, no allocation
namespace {

// The activations between kernel A and kernel B of moe_decode_forward_noalloc, and the error word
// of calls that pass none.  Static storage: zero at module load, never allocated or freed.
static __device__ __align__(256) float g_noalloc_act[MOE_NOALLOC_MAX_ACT_FLOATS];
static __device__ __align__(256) int32_t g_noalloc_err[64];

constexpr int kNoallocDevices = 64;

constexpr int kNoallocPlans = 8;

struct NoallocPlan {
  bool valid = false;
  moe_decode_config cfg{};  // the config `prep` was made for
  Prepared prep{};
};

struct NoallocDevice {
  bool ready = false;
  float *act = nullptr;
  int32_t *err = nullptr;
  NoallocPlan plans[kNoallocPlans];  // the last configs seen on this device
  int next = 0;                      // the entry the next new config replaces
};

NoallocDevice g_noalloc[kNoallocDevices];
std::mutex g_noalloc_mu;

// Scratch addresses and the prepared launch plan of the current device: the addresses are looked
// up once per device, a plan once per config (the last kNoallocPlans configs are kept).
int noalloc_setup(const moe_decode_config *cfg, float **act, int32_t **err, Prepared *P) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kNoallocDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocDevice &d = g_noalloc[dev];
  if (!d.ready) {
    void *a = nullptr, *e = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_act) != cudaSuccess ||
        cudaGetSymbolAddress(&e, g_noalloc_err) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    d.act = static_cast<float *>(a);
    d.err = static_cast<int32_t *>(e);
    d.ready = true;
  }
  NoallocPlan *hit = nullptr;
  for (NoallocPlan &p : d.plans)
    if (p.valid && std::memcmp(&p.cfg, cfg, sizeof *cfg) == 0) hit = &p;
  if (!hit) {
    hit = &d.plans[d.next];
    d.next = (d.next + 1) % kNoallocPlans;
    hit->valid = false;
    const int rc = prepare(cfg, hit->prep);
    if (rc != MOE_OK) return rc;
    hit->cfg = *cfg;
    hit->valid = true;
  }
  *act = d.act;
  *err = d.err;
  *P = hit->prep;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_forward_noalloc(const moe_decode_config *cfg,
                                          const moe_layer_weights *weights, const void *x,
                                          int32_t m, const int32_t *ids, const float *scores,
                                          const void *resid, void *out, int32_t *device_error,
                                          void *stream) {
  int rc = validate_config(cfg);
  if (rc != MOE_OK) return rc;
  if (cfg->kernel_mode != MOE_KERNELS_SEPARATE) return MOE_ERR_UNSUPPORTED;
  if (act_floats(*cfg) > (size_t)MOE_NOALLOC_MAX_ACT_FLOATS) return MOE_ERR_UNSUPPORTED;
  rc = validate_weights(cfg, weights);
  if (rc != MOE_OK) return rc;
  if (!x || !resid || !out) return MOE_ERR_INVALID_ARG;
  if (m < 1 || m > cfg->max_tokens) return MOE_ERR_INVALID_ARG;
  if (cfg->top_k > 0 && (!ids || !scores)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(resid, dtype_bytes(cfg->resid_dtype)) ||
      !aligned(out, dtype_bytes(cfg->out_dtype)) || (ids && !aligned(ids, 4)) ||
      (scores && !aligned(scores, 4)) || (device_error && !aligned(device_error, 4)))
    return MOE_ERR_INVALID_ARG;
  if (x == out) return MOE_ERR_INVALID_ARG;
  float *act = nullptr;
  int32_t *err = nullptr;
  Prepared P;
  rc = noalloc_setup(cfg, &act, &err, &P);
  if (rc != MOE_OK) return rc;
  const cudaError_t e = enqueue_separate(
      P, layer_ptrs(*cfg, *weights), act, device_error ? device_error : err, x, m, ids, scores,
      resid, cfg->resid_dtype, out, cfg->out_dtype, static_cast<cudaStream_t>(stream),
      MOE_PART_GATE_UP | MOE_PART_DOWN);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ====================================================================== stack of layers
namespace {
struct GraphEntry {
  const void *x, *ids, *scores, *resid0, *out;
  int m, parts;
  cudaGraphExec_t exec;
  uint64_t last_use;
};
constexpr size_t kMaxGraphs = 16;
}  // namespace

struct moe_stack {
  Prepared P;
  std::vector<moe::LayerPtrs> layers;
  Workspace ws;
  ColWeights cw;
  MmaState mma;
  float *ping[2] = {nullptr, nullptr};
  cudaStream_t cap = nullptr;
  std::vector<GraphEntry> graphs;
  uint64_t clock = 0;
  // the next layer's RMSNorm folded in (moe_stack_create_chained): bf16 [L - 1][din] weights
  const uint16_t *norm_w = nullptr;
  float norm_eps = 0.f;
  // device staging for moe_stack_step_host
  void *x_dev = nullptr, *resid_dev = nullptr;
  int32_t *ids_dev = nullptr;
  float *scores_dev = nullptr, *out_dev = nullptr;
  unsigned long long *tl = nullptr;  // timeline builds: the column-split kernel's time stamps
};

extern "C" void moe_stack_destroy(moe_stack_t *s) {
  if (!s) return;
  for (auto &g : s->graphs) cudaGraphExecDestroy(g.exec);
  if (s->cap) cudaStreamDestroy(s->cap);
  s->cw.release();
  s->mma.release();
  s->ws.release();
  cudaFree(s->ping[0]);
  cudaFree(s->ping[1]);
  cudaFree(s->x_dev);
  cudaFree(s->resid_dev);
  cudaFree(s->ids_dev);
  cudaFree(s->scores_dev);
  cudaFree(s->out_dev);
  cudaFree(s->tl);
  delete s;
}

namespace {
int stack_create(const moe_decode_config *cfg, int32_t n_layers, const moe_layer_weights *layers,
                 const void *norm_weight, float eps, moe_stack_t **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !layers || n_layers < 1) return MOE_ERR_INVALID_ARG;
  int rc = validate_config(cfg);
  if (rc != MOE_OK) return rc;
  if (cfg->out_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
  if (norm_weight && (cols_mode(cfg->kernel_mode) || cfg->kernel_mode == MOE_KERNELS_MMA))
    return MOE_ERR_UNSUPPORTED;
  for (int l = 0; l < n_layers; ++l) {
    rc = validate_weights(cfg, &layers[l]);
    if (rc != MOE_OK) return rc;
  }
  moe_stack *s = new (std::nothrow) moe_stack();
  if (!s) return MOE_ERR_OOM;
  rc = prepare(cfg, s->P);
  if (rc != MOE_OK) {
    delete s;
    return rc;
  }
  if (norm_weight) {
    s->norm_w = static_cast<const uint16_t *>(norm_weight);
    s->norm_eps = eps;
    s->P.grouped_ok = false;  // batches run token by token: the grouped path reads x only
  }
  s->layers.resize(n_layers);
  for (int l = 0; l < n_layers; ++l) s->layers[l] = layer_ptrs(*cfg, layers[l]);
  const size_t M = cfg->max_tokens, din = cfg->din, K = cfg->top_k;
  bool ok = s->ws.alloc(*cfg, n_layers, s->P.grouped_ok, slab_floats(s->P)) &&
            cudaMalloc(&s->ping[0], M * din * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&s->ping[1], M * din * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&s->x_dev, (size_t)n_layers * M * din * 2) == cudaSuccess &&
            cudaMalloc(&s->resid_dev, M * din * dtype_bytes(cfg->resid_dtype)) == cudaSuccess &&
            cudaMalloc(&s->ids_dev, (size_t)n_layers * M * (K > 0 ? K : 1) * 4) == cudaSuccess &&
            cudaMalloc(&s->scores_dev, (size_t)n_layers * M * (K > 0 ? K : 1) * 4) ==
                cudaSuccess &&
            cudaMalloc(&s->out_dev, M * din * sizeof(float)) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    moe_stack_destroy(s);
    return MOE_ERR_OOM;
  }
  if (cudaMemcpy(s->ws.layers, s->layers.data(), sizeof(moe::LayerPtrs) * n_layers,
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking) != cudaSuccess) {
    moe_stack_destroy(s);
    return MOE_ERR_CUDA;
  }
  if (cfg->kernel_mode == MOE_KERNELS_MMA) {
    rc = s->mma.build(*cfg, layers, n_layers);
    if (rc != MOE_OK) {
      moe_stack_destroy(s);
      return rc;
    }
  }
  if (cols_mode(cfg->kernel_mode)) {
    rc = s->cw.build(*cfg, layers, n_layers);
    if (rc != MOE_OK) {
      moe_stack_destroy(s);
      return rc;
    }
#ifdef MOE_TIMELINE
    const size_t n_tl = (size_t)s->P.grid_cols * n_layers * moe::kTlPoints;
    if (cudaMalloc(&s->tl, n_tl * 8) != cudaSuccess || cudaMemset(s->tl, 0, n_tl * 8) != cudaSuccess) {
      moe_stack_destroy(s);
      return MOE_ERR_OOM;
    }
#endif
  }
  *out = s;
  return MOE_OK;
}
}  // namespace

extern "C" int moe_stack_create(const moe_decode_config *cfg, int32_t n_layers,
                                const moe_layer_weights *layers, moe_stack_t **out) {
  return stack_create(cfg, n_layers, layers, nullptr, 0.f, out);
}

extern "C" int moe_stack_create_chained(const moe_decode_config *cfg, int32_t n_layers,
                                        const moe_layer_weights *layers,
                                        const void *norm_weight, float eps, moe_stack_t **out) {
  if (out) *out = nullptr;
  if (!norm_weight || !aligned(norm_weight, 16) || !(eps >= 0.f) || eps > 1.f)
    return MOE_ERR_INVALID_ARG;
  return stack_create(cfg, n_layers, layers, norm_weight, eps, out);
}

namespace {

cudaError_t enqueue_stack(moe_stack *s, const void *x, int m, const int32_t *ids,
                          const float *scores, const void *resid0, void *out, cudaStream_t st,
                          int parts) {
  const int L = (int)s->layers.size();
  const moe_decode_config &c = s->P.cfg;
  if (cols_mode(c.kernel_mode))
    return enqueue_cols(s->P, s->ws.layers, s->cw.dev, L, s->ws.slab, s->ws.err, s->ws.bar, x, ids,
                        scores, resid0, c.resid_dtype, out, MOE_DTYPE_F32, st, s->tl);
  if (c.kernel_mode == MOE_KERNELS_FUSED && parts == (MOE_PART_GATE_UP | MOE_PART_DOWN))
    return enqueue_fused(s->P, s->ws.layers, L, s->ws.act, s->ws.y, s->ws.err, s->ws.bar,
                         s->ping[0], s->ping[1], x, m, ids, scores, resid0, c.resid_dtype, out,
                         MOE_DTYPE_F32, st, s->norm_w, s->norm_eps);
  const size_t din = c.din, K = c.top_k;
  if (c.kernel_mode == MOE_KERNELS_MMA) {
    for (int l = 0; l < L; ++l) {
      const void *xl = static_cast<const uint16_t *>(x) + (size_t)l * m * din;
      const int32_t *il = ids ? ids + (size_t)l * m * K : nullptr;
      const float *sl = scores ? scores + (size_t)l * m * K : nullptr;
      const void *rl = l == 0 ? resid0 : s->ping[(l - 1) & 1];
      void *ol = l == L - 1 ? out : s->ping[l & 1];
      cudaError_t e = enqueue_mma(s->P, s->layers[l], s->mma, l, s->ws, xl, m, il, sl, rl,
                                  l == 0 ? c.resid_dtype : MOE_DTYPE_F32, ol, MOE_DTYPE_F32, st);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  for (int l = 0; l < L; ++l) {
    NormIn norm;
    if (s->norm_w && l > 0) {
      norm.v = s->ping[(l - 1) & 1];
      norm.gamma = s->norm_w + (size_t)(l - 1) * din;
      norm.eps = s->norm_eps;
    }
    const void *xl = static_cast<const uint16_t *>(x) + (s->norm_w ? 0 : (size_t)l * m * din);
    const int32_t *il = ids ? ids + (size_t)l * m * K : nullptr;
    const float *sl = scores ? scores + (size_t)l * m * K : nullptr;
    const void *rl = l == 0 ? resid0 : s->ping[(l - 1) & 1];
    const int rdt = l == 0 ? c.resid_dtype : MOE_DTYPE_F32;
    void *ol = l == L - 1 ? out : s->ping[l & 1];
    cudaError_t e = enqueue_separate(s->P, s->layers[l], s->ws.act, s->ws.err, xl, m, il, sl, rl,
                                     rdt, ol, MOE_DTYPE_F32, st, parts, norm);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int capture(moe_stack *s, const void *x, int m, const int32_t *ids, const float *scores,
            const void *resid0, void *out, int parts, cudaGraphExec_t *exec) {
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaError_t e = enqueue_stack(s, x, m, ids, scores, resid0, out, s->cap, parts);
  cudaError_t e2 = cudaStreamEndCapture(s->cap, &graph);
  if (e != cudaSuccess || e2 != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  e = cudaGraphInstantiate(exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

extern "C" int moe_stack_step_parts(moe_stack_t *s, int32_t parts, const void *x, int32_t m,
                                    const int32_t *ids, const float *scores, const void *resid0,
                                    void *out, void *stream) {
  if (!s || !x || !resid0 || !out) return MOE_ERR_INVALID_ARG;
  if (parts < 1 || parts > (MOE_PART_GATE_UP | MOE_PART_DOWN)) return MOE_ERR_INVALID_ARG;
  if ((cols_mode(s->P.cfg.kernel_mode) || s->P.cfg.kernel_mode == MOE_KERNELS_MMA) &&
      parts != (MOE_PART_GATE_UP | MOE_PART_DOWN))
    return MOE_ERR_UNSUPPORTED;
  if (m < 1 || m > s->P.cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (s->P.cfg.top_k > 0 && (!ids || !scores)) return MOE_ERR_INVALID_ARG;
  if (!aligned(out, 4) || !aligned(x, 16) || !aligned(resid0, dtype_bytes(s->P.cfg.resid_dtype)))
    return MOE_ERR_INVALID_ARG;
  GraphEntry *hit = nullptr;
  for (auto &g : s->graphs)
    if (g.x == x && g.ids == ids && g.scores == scores && g.resid0 == resid0 && g.out == out &&
        g.m == m && g.parts == parts)
      hit = &g;
  if (!hit) {
    cudaGraphExec_t exec = nullptr;
    int rc = capture(s, x, m, ids, scores, resid0, out, parts, &exec);
    if (rc != MOE_OK) return rc;
    if (s->graphs.size() >= kMaxGraphs) {
      size_t lru = 0;
      for (size_t i = 1; i < s->graphs.size(); ++i)
        if (s->graphs[i].last_use < s->graphs[lru].last_use) lru = i;
      cudaGraphExecDestroy(s->graphs[lru].exec);
      s->graphs.erase(s->graphs.begin() + lru);
    }
    s->graphs.push_back(GraphEntry{x, ids, scores, resid0, out, m, parts, exec, 0});
    hit = &s->graphs.back();
  }
  hit->last_use = ++s->clock;
  return cudaGraphLaunch(hit->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

extern "C" int moe_stack_step(moe_stack_t *s, const void *x, int32_t m, const int32_t *ids,
                              const float *scores, const void *resid0, void *out, void *stream) {
  return moe_stack_step_parts(s, MOE_PART_GATE_UP | MOE_PART_DOWN, x, m, ids, scores, resid0, out,
                              stream);
}

extern "C" int moe_stack_step_host(moe_stack_t *s, const void *x_host, int32_t m,
                                   const int32_t *ids_host, const float *scores_host,
                                   const void *resid0_host, float *out_host, void *stream) {
  if (!s || !x_host || !resid0_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (m < 1 || m > s->P.cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  const size_t L = s->layers.size(), din = s->P.cfg.din, K = s->P.cfg.top_k;
  if (K > 0 && (!ids_host || !scores_host)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t x_layers = s->norm_w ? 1 : L;  // a chained stack reads layer 0's x only
  bool ok =
      cudaMemcpyAsync(s->x_dev, x_host, x_layers * m * din * 2, cudaMemcpyHostToDevice, st) ==
          cudaSuccess &&
      cudaMemcpyAsync(s->resid_dev, resid0_host, m * din * dtype_bytes(s->P.cfg.resid_dtype),
                      cudaMemcpyHostToDevice, st) == cudaSuccess;
  if (ok && K > 0)
    ok = cudaMemcpyAsync(s->ids_dev, ids_host, L * m * K * 4, cudaMemcpyHostToDevice, st) ==
             cudaSuccess &&
         cudaMemcpyAsync(s->scores_dev, scores_host, L * m * K * 4, cudaMemcpyHostToDevice, st) ==
             cudaSuccess;
  if (!ok) return MOE_ERR_CUDA;
  int rc = moe_stack_step(s, s->x_dev, m, K > 0 ? s->ids_dev : nullptr,
                          K > 0 ? s->scores_dev : nullptr, s->resid_dev, s->out_dev, stream);
  if (rc != MOE_OK) return rc;
  if (cudaMemcpyAsync(out_host, s->out_dev, m * din * sizeof(float), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

#ifdef MOE_TIMELINE
extern "C" int moe_stack_timeline(moe_stack_t *s, void *host, int64_t bytes, int32_t *grid) {
  if (!s || !host || !grid) return MOE_ERR_INVALID_ARG;
  if (!s->tl) return MOE_ERR_UNSUPPORTED;
  const size_t need = (size_t)s->P.grid_cols * s->layers.size() * moe::kTlPoints * 8;
  if (bytes < (int64_t)need) return MOE_ERR_INVALID_ARG;
  *grid = s->P.grid_cols;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  return cudaMemcpy(host, s->tl, need, cudaMemcpyDeviceToHost) == cudaSuccess ? MOE_OK
                                                                               : MOE_ERR_CUDA;
}
#endif

extern "C" int moe_stack_get_error(moe_stack_t *s, int32_t *device_error) {
  if (!s) return MOE_ERR_INVALID_ARG;
  return read_and_clear_error(s->ws.err, device_error);
}

// ====================================================================== debug unpack
extern "C" int moe_unpack_codes_device(const void *packed, int64_t rows, int64_t cols,
                                       int32_t bits, uint8_t *codes, void *stream) {
  if (!packed || !codes || rows < 0 || cols < 0 || cols % 64) return MOE_ERR_INVALID_ARG;
  if (!bits_ok(bits)) return MOE_ERR_UNSUPPORTED;
  if (!aligned(packed, 16)) return MOE_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MOE_OK;
  return moe::launch_unpack(static_cast<const uint8_t *>(packed), rows, cols, bits, codes,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// ====================================================================== debug route inversion
extern "C" int moe_route_invert_device(const int32_t *ids, int32_t m, int32_t k,
                                       int32_t n_experts, int32_t *out, void *stream) {
  if (!ids || !out || m < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if ((int64_t)m * k > moe::kMaxPairs || n_experts < 1 || n_experts > moe::kMaxGroupExperts)
    return MOE_ERR_UNSUPPORTED;
  if (!aligned(ids, 4) || !aligned(out, 4)) return MOE_ERR_INVALID_ARG;
  return moe::launch_route_invert(ids, m, k, n_experts, out, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// ====================================================================== bounded-wait check
extern "C" int moe_debug_wait_timeout(int32_t kind, int32_t *scratch, int32_t *device_error,
                                      void *stream) {
  if ((kind != 0 && kind != 1) || !scratch || !device_error) return MOE_ERR_INVALID_ARG;
  if (!aligned(scratch, 4) || !aligned(device_error, 4)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  // about 0.1 s at GB300 clocks
  return moe::launch_wait_timeout(kind, reinterpret_cast<uint32_t *>(scratch), device_error,
                                  200000000LL, st) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// ====================================================================== router
extern "C" int moe_router_topk(const float *logits, int32_t m, int32_t n_experts, int32_t top_k,
                               int32_t *ids, float *scores, void *stream) {
  if (!logits || !ids || !scores || m < 1 || n_experts < 1 || top_k < 1 || top_k > n_experts)
    return MOE_ERR_INVALID_ARG;
  if (n_experts > 1024 || top_k > moe::kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(scores, 4)) return MOE_ERR_INVALID_ARG;
  return moe::launch_router(logits, m, n_experts, top_k, ids, scores,
                            static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// ====================================================================== column-split plan (host)
extern "C" int moe_debug_col_pieces(int32_t top_k, int32_t dff, int32_t n_shared,
                                    int32_t dff_shared, int32_t bits_down, int32_t bits_shared,
                                    int32_t u0, int32_t u1, int32_t *out, int32_t max_pieces) {
  if (!out || u0 < 0 || u1 < u0 || top_k < 0 || n_shared < 0 || max_pieces < 0)
    return MOE_ERR_INVALID_ARG;
  if (top_k + n_shared < 1 || (top_k > 0 && (dff <= 0 || dff % 64)) ||
      (n_shared > 0 && (dff_shared <= 0 || dff_shared % 64)))
    return MOE_ERR_INVALID_ARG;
  bits_down = moe::col_down_bits(bits_down);     // 6-bit down codes are stored as bytes
  bits_shared = moe::col_down_bits(bits_shared);
  if ((bits_down != 4 && bits_down != 8) || (n_shared > 0 && bits_shared != 4 && bits_shared != 8))
    return MOE_ERR_UNSUPPORTED;
  const int64_t U = (int64_t)top_k * dff + (int64_t)n_shared * dff_shared;
  if (U > (1 << 24)) return MOE_ERR_UNSUPPORTED;
  if (u1 > U) return MOE_ERR_INVALID_ARG;
  if (u1 - u0 > moe::kMaxColsCta) return MOE_ERR_UNSUPPORTED;  // beyond the kernel's buffers
  moe::ColPiece pc[moe::kMaxColPieces];
  int nbk = 0;
  const int cb_r = 32 / bits_down, cb_s = n_shared > 0 ? 32 / bits_shared : cb_r;
  const int np = moe::col_pieces(top_k, dff, n_shared, dff_shared, cb_r, cb_s, u0, u1, pc, &nbk);
  if (np < 0 || np > max_pieces) return MOE_ERR_UNSUPPORTED;
  for (int q = 0; q < np; ++q) {
    const int32_t v[8] = {pc[q].seg, pc[q].j0, pc[q].j1, pc[q].a0,
                          pc[q].blk0, pc[q].nb, pc[q].pb, pc[q].grp};
    std::memcpy(out + 8 * q, v, sizeof v);
  }
  return np;
}

extern "C" int moe_debug_col_plan(const moe_decode_config *cfg, int32_t grid, int32_t ring_bytes,
                                  int32_t *out, int32_t *bounds) {
  if (!out || grid < 1 || ring_bytes < 1) return MOE_ERR_INVALID_ARG;
  const int rc = validate_config(cfg);
  if (rc != MOE_OK) return rc;
  const moe::LayerShape shape{cfg->din, cfg->dff, cfg->top_k, cfg->n_experts, cfg->n_shared,
                              cfg->dff_shared};
  const int bits_sh = cfg->n_shared > 0 ? cfg->bits_shared : cfg->bits_down;
  moe::ColPlan cp;
  moe::Plan plan;
  std::memset(&cp, 0, sizeof cp);
  std::memset(&plan, 0, sizeof plan);
  if (!moe::make_col_plan(shape, cfg->bits_gate, cfg->bits_down, bits_sh, grid, ring_bytes, &cp,
                          &plan))
    return MOE_ERR_UNSUPPORTED;
  const int32_t v[10] = {plan.nst, plan.stage_bytes, cp.nbs, cp.ro, cp.cb_r,
                         cp.cb_s, plan.geo_r.R, plan.geo_s.R, cp.pack, cp.prefetch};
  std::memcpy(out, v, sizeof v);
  if (bounds) std::memcpy(bounds, cp.bounds, sizeof(int32_t) * (grid + 1));
  return MOE_OK;
}
