// moe_api.cu -- the C ABI of include/moe_decode.h: validation, prepared handles, the layer-stack
// CUDA-graph driver and the host-buffer step.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "moe_decode.h"
#include "moe_kernels.cuh"

namespace {

using moe::DownParams;
using moe::GateUpParams;
using moe::ProjDev;

bool bits_ok(int b) { return b == 4 || b == 6 || b == 8; }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool proj_ok(const moe_proj &p) {
  return p.codes && p.scales && p.biases && aligned(p.codes, 16) && aligned(p.scales, 2) &&
         aligned(p.biases, 2);
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
  if (c->warps_per_block < 0) return MOE_ERR_INVALID_ARG;
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

ProjDev dev(const moe_proj &p) {
  return ProjDev{static_cast<const uint8_t *>(p.codes), static_cast<const __half *>(p.scales),
                 static_cast<const __half *>(p.biases)};
}

// Everything a layer launch needs, resolved once.
struct Layer {
  moe_decode_config cfg;
  moe_layer_weights w;
  int bits_s, bits_sd;      // shared-class bits (routed bits when there is no shared expert)
  size_t smem_a, smem_b;
  int grid_a, grid_b;
};

int prepare_layer(const moe_decode_config *c, const moe_layer_weights *w, Layer &L) {
  int rc = validate_config(c);
  if (rc != MOE_OK) return rc;
  rc = validate_weights(c, w);
  if (rc != MOE_OK) return rc;
  L.cfg = *c;
  L.w = *w;
  L.bits_s = c->n_shared > 0 ? c->bits_shared : c->bits_gate;
  L.bits_sd = c->n_shared > 0 ? c->bits_shared : c->bits_down;
  L.smem_a = moe::gate_up_smem_bytes(c->din, c->bits_gate, L.bits_s, c->n_shared);
  L.smem_b = moe::down_smem_bytes(c->dff, c->top_k, c->n_shared, c->dff_shared, c->bits_down,
                                  L.bits_sd);
  int device = 0, sms = 0, smem_optin = 0, major = 0, minor = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
  const size_t static_reserve = 2048;  // the kernels' static shared memory
  if (L.smem_a + static_reserve > (size_t)smem_optin || L.smem_b + static_reserve > (size_t)smem_optin)
    return MOE_ERR_UNSUPPORTED;
  if (moe::prepare_kernels(smem_optin - (int)static_reserve, c->bits_gate, L.bits_s, c->bits_down,
                           L.bits_sd) != cudaSuccess)
    return MOE_ERR_CUDA;
  L.grid_a = sms;
  L.grid_b = sms;
  return MOE_OK;
}

size_t act_floats(const moe_decode_config &c) {
  return (size_t)c.top_k * c.dff + (size_t)c.n_shared * c.dff_shared;
}

size_t dtype_bytes(int dt) { return dt == MOE_DTYPE_F32 ? 4 : 2; }

// Enqueues one layer for m tokens (kernel A then kernel B per token).
cudaError_t enqueue_layer(const Layer &L, float *act, int32_t *err, const void *x, int m,
                          const int32_t *ids, const float *scores, const void *resid,
                          int resid_dtype, void *out, int out_dtype, cudaStream_t stream,
                          bool pdl, int parts = MOE_PART_GATE_UP | MOE_PART_DOWN) {
  const moe_decode_config &c = L.cfg;
  for (int t = 0; t < m; ++t) {
    GateUpParams a;
    a.gate = dev(L.w.gate);
    a.up = dev(L.w.up);
    a.sh_gate = dev(L.w.sh_gate);
    a.sh_up = dev(L.w.sh_up);
    a.x = static_cast<const uint16_t *>(x) + (size_t)t * c.din;
    a.ids = ids ? ids + (size_t)t * c.top_k : nullptr;
    a.scores = scores ? scores + (size_t)t * c.top_k : nullptr;
    a.gate_vec = (c.n_shared > 0 && c.shared_gate == 1)
                     ? static_cast<const uint16_t *>(L.w.gate_vec)
                     : nullptr;
    a.act = act;
    a.err = err;
    a.din = c.din;
    a.dff = c.dff;
    a.top_k = c.top_k;
    a.n_experts = c.n_experts;
    a.n_shared = c.n_shared;
    a.dff_shared = c.dff_shared;
    cudaError_t e = cudaSuccess;
    if (parts & MOE_PART_GATE_UP)
      e = moe::launch_gate_up(a, c.bits_gate, L.bits_s, L.grid_a, L.smem_a, stream, pdl);
    if (e != cudaSuccess) return e;

    DownParams b;
    b.down = dev(L.w.down);
    b.sh_down = dev(L.w.sh_down);
    b.ids = a.ids;
    b.act = act;
    b.resid = static_cast<const char *>(resid) + (size_t)t * c.din * dtype_bytes(resid_dtype);
    b.out = static_cast<char *>(out) + (size_t)t * c.din * dtype_bytes(out_dtype);
    b.err = err;
    b.resid_f32 = resid_dtype == MOE_DTYPE_F32;
    b.out_f32 = out_dtype == MOE_DTYPE_F32;
    b.din = c.din;
    b.dff = c.dff;
    b.top_k = c.top_k;
    b.n_experts = c.n_experts;
    b.n_shared = c.n_shared;
    b.dff_shared = c.dff_shared;
    if (parts & MOE_PART_DOWN)
      e = moe::launch_down(b, c.bits_down, L.bits_sd, L.grid_b, L.smem_b, stream, pdl);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int read_and_clear_error(int32_t *err, int32_t *out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(err, 0, sizeof v) != cudaSuccess) return MOE_ERR_CUDA;
  *out = v ? MOE_ERR_BAD_ID : MOE_OK;
  return MOE_OK;
}

}  // namespace

// ====================================================================== single layer
struct moe_decode {
  Layer layer;
  float *act = nullptr;
  int32_t *err = nullptr;
};

extern "C" int moe_decode_create(const moe_decode_config *cfg, const moe_layer_weights *weights,
                                 moe_decode_t **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_decode *h = new (std::nothrow) moe_decode();
  if (!h) return MOE_ERR_OOM;
  int rc = prepare_layer(cfg, weights, h->layer);
  if (rc != MOE_OK) {
    delete h;
    return rc;
  }
  const size_t n = act_floats(*cfg) * cfg->max_tokens;
  if (cudaMalloc(&h->act, (n > 0 ? n : 1) * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&h->err, sizeof(int32_t)) != cudaSuccess ||
      cudaMemset(h->err, 0, sizeof(int32_t)) != cudaSuccess) {
    cudaFree(h->act);
    cudaFree(h->err);
    delete h;
    cudaGetLastError();
    return MOE_ERR_OOM;
  }
  *out = h;
  return MOE_OK;
}

extern "C" int moe_decode_forward(moe_decode_t *h, const void *x, int32_t m, const int32_t *ids,
                                  const float *scores, const void *resid, void *out,
                                  void *stream) {
  if (!h || !x || !resid || !out) return MOE_ERR_INVALID_ARG;
  const moe_decode_config &c = h->layer.cfg;
  if (m < 1 || m > c.max_tokens) return MOE_ERR_INVALID_ARG;
  if (c.top_k > 0 && (!ids || !scores)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 2) || !aligned(resid, dtype_bytes(c.resid_dtype)) ||
      !aligned(out, dtype_bytes(c.out_dtype)) || (ids && !aligned(ids, 4)) ||
      (scores && !aligned(scores, 4)))
    return MOE_ERR_INVALID_ARG;
  if (x == out) return MOE_ERR_INVALID_ARG;
  cudaError_t e = enqueue_layer(h->layer, h->act, h->err, x, m, ids, scores, resid, c.resid_dtype,
                                out, c.out_dtype, static_cast<cudaStream_t>(stream), true);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_decode_get_error(moe_decode_t *h, int32_t *device_error) {
  if (!h) return MOE_ERR_INVALID_ARG;
  return read_and_clear_error(h->err, device_error);
}

extern "C" void moe_decode_destroy(moe_decode_t *h) {
  if (!h) return;
  cudaFree(h->act);
  cudaFree(h->err);
  delete h;
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
  std::vector<Layer> layers;       // layers[0] reads resid0 in cfg.resid_dtype, the rest fp32
  moe_decode_config cfg;
  float *act = nullptr;
  int32_t *err = nullptr;
  float *ping[2] = {nullptr, nullptr};
  cudaStream_t cap = nullptr;
  std::vector<GraphEntry> graphs;
  uint64_t clock = 0;
  bool pdl = true;
  // device staging for moe_stack_step_host
  void *x_dev = nullptr, *resid_dev = nullptr;
  int32_t *ids_dev = nullptr;
  float *scores_dev = nullptr, *out_dev = nullptr;
};

extern "C" void moe_stack_destroy(moe_stack_t *s) {
  if (!s) return;
  for (auto &g : s->graphs) cudaGraphExecDestroy(g.exec);
  if (s->cap) cudaStreamDestroy(s->cap);
  cudaFree(s->act);
  cudaFree(s->err);
  cudaFree(s->ping[0]);
  cudaFree(s->ping[1]);
  cudaFree(s->x_dev);
  cudaFree(s->resid_dev);
  cudaFree(s->ids_dev);
  cudaFree(s->scores_dev);
  cudaFree(s->out_dev);
  delete s;
}

extern "C" int moe_stack_create(const moe_decode_config *cfg, int32_t n_layers,
                                const moe_layer_weights *layers, moe_stack_t **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !layers || n_layers < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->out_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
  moe_stack *s = new (std::nothrow) moe_stack();
  if (!s) return MOE_ERR_OOM;
  s->cfg = *cfg;
  s->layers.resize(n_layers);
  for (int l = 0; l < n_layers; ++l) {
    moe_decode_config c = *cfg;
    if (l > 0) c.resid_dtype = MOE_DTYPE_F32;
    int rc = prepare_layer(&c, &layers[l], s->layers[l]);
    if (rc != MOE_OK) {
      moe_stack_destroy(s);
      return rc;
    }
  }
  const size_t M = cfg->max_tokens, din = cfg->din, K = cfg->top_k;
  const size_t na = act_floats(*cfg);
  bool ok = cudaMalloc(&s->act, (na > 0 ? na : 1) * sizeof(float)) == cudaSuccess &&
            cudaMalloc(&s->err, sizeof(int32_t)) == cudaSuccess &&
            cudaMemset(s->err, 0, sizeof(int32_t)) == cudaSuccess &&
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
  if (cudaStreamCreateWithFlags(&s->cap, cudaStreamNonBlocking) != cudaSuccess) {
    moe_stack_destroy(s);
    return MOE_ERR_CUDA;
  }
  *out = s;
  return MOE_OK;
}

namespace {

cudaError_t enqueue_stack(moe_stack *s, const void *x, int m, const int32_t *ids,
                          const float *scores, const void *resid0, void *out, cudaStream_t st,
                          bool pdl, int parts) {
  const int L = (int)s->layers.size();
  const size_t din = s->cfg.din, K = s->cfg.top_k;
  for (int l = 0; l < L; ++l) {
    const void *xl = static_cast<const uint16_t *>(x) + (size_t)l * m * din;
    const int32_t *il = ids ? ids + (size_t)l * m * K : nullptr;
    const float *sl = scores ? scores + (size_t)l * m * K : nullptr;
    const void *rl = l == 0 ? resid0 : s->ping[(l - 1) & 1];
    const int rdt = l == 0 ? s->cfg.resid_dtype : MOE_DTYPE_F32;
    void *ol = l == L - 1 ? out : s->ping[l & 1];
    cudaError_t e = enqueue_layer(s->layers[l], s->act, s->err, xl, m, il, sl, rl, rdt, ol,
                                  MOE_DTYPE_F32, st, pdl, parts);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int capture(moe_stack *s, const void *x, int m, const int32_t *ids, const float *scores,
            const void *resid0, void *out, bool pdl, int parts, cudaGraphExec_t *exec) {
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(s->cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaError_t e = enqueue_stack(s, x, m, ids, scores, resid0, out, s->cap, pdl, parts);
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
  if (m < 1 || m > s->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (s->cfg.top_k > 0 && (!ids || !scores)) return MOE_ERR_INVALID_ARG;
  if (!aligned(out, 4) || !aligned(x, 2) || !aligned(resid0, dtype_bytes(s->cfg.resid_dtype)))
    return MOE_ERR_INVALID_ARG;
  GraphEntry *hit = nullptr;
  for (auto &g : s->graphs)
    if (g.x == x && g.ids == ids && g.scores == scores && g.resid0 == resid0 && g.out == out &&
        g.m == m && g.parts == parts)
      hit = &g;
  if (!hit) {
    cudaGraphExec_t exec = nullptr;
    int rc = capture(s, x, m, ids, scores, resid0, out, s->pdl, parts, &exec);
    if (rc != MOE_OK && s->pdl) {  // a driver without programmatic edges in graphs
      s->pdl = false;
      rc = capture(s, x, m, ids, scores, resid0, out, false, parts, &exec);
    }
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
  if (m < 1 || m > s->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  const size_t L = s->layers.size(), din = s->cfg.din, K = s->cfg.top_k;
  if (K > 0 && (!ids_host || !scores_host)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool ok =
      cudaMemcpyAsync(s->x_dev, x_host, L * m * din * 2, cudaMemcpyHostToDevice, st) ==
          cudaSuccess &&
      cudaMemcpyAsync(s->resid_dev, resid0_host, m * din * dtype_bytes(s->cfg.resid_dtype),
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

extern "C" int moe_stack_get_error(moe_stack_t *s, int32_t *device_error) {
  if (!s) return MOE_ERR_INVALID_ARG;
  return read_and_clear_error(s->err, device_error);
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
