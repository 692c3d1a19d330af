/*
 * moe_decode.h -- C ABI of the GB300 (sm_103a) decode MoE expert block.
 *
 * The block (one token; M tokens are M independent copies of it):
 *
 *   w       = scale * q + bias                     per group of 64 codes along a row; q is an
 *                                                  unsigned 4-, 6- or 8-bit code, scale and bias fp16
 *   act_k   = silu(W_gate,k . x) * (W_up,k . x)    for each routed slot k and each shared expert
 *   out     = resid + (sum_k score_k * W_down,k . act_k  +  scalar * sum_s W_down,s . act_s)
 *   scalar  = sigmoid(x . g) with a gate vector g, else 1
 *
 * Sources: "two-kernel decode-MoE that beats gather_qmm" (What changed, step 2: kernel A computes
 * gate/up + swiglu into act_g[K, Dff], kernel B computes down * score summed over K; Scope /
 * flags: 4/8-bit affine codes; Next: 6-bit and mixed bits per projection) and "Red Lite dev39 --
 * fused expert tail" (Change: one dispatch computes the weighted sum over the pool, then
 * x = resid + (routed + shared * scalar), then writes the layer output).
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device pointers of the current device; "host" pointers
 *     are ordinary host memory.  Streams are cudaStream_t passed as void* (NULL = legacy stream).
 *   - Weights are borrowed: the caller keeps them alive and unchanged until destroy.
 *   - Host-detectable errors return a negative moe_status and enqueue nothing.  Errors the GPU
 *     finds (an expert id outside [0, n_experts)) set a sticky device error word that
 *     moe_decode_get_error / moe_stack_get_error read; the offending slot contributes zero.
 *     No kernel traps or asserts.
 *   - A handle is not thread-safe: calls on one handle must not run concurrently on the host, and
 *     forwards enqueued on different streams must not overlap on the GPU (they share workspace).
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer, bad enum */
  MOE_ERR_UNSUPPORTED = -2,  /* valid but not built: bits not in {4,6,8}, gate bits != up bits,
                                shared memory needs above the device limit, wrong GPU */
  MOE_ERR_CUDA = -3,         /* a CUDA runtime call failed (launch, copy, graph) */
  MOE_ERR_OOM = -4,          /* device or pinned allocation failed */
  MOE_ERR_BAD_ID = -5,       /* device error word: an expert id was outside [0, n_experts) */
  MOE_ERR_TIMEOUT = -6,      /* device error word: a pipeline wait gave up after about two seconds
                                (a bug, never expected); the kernel returned without its result */
  MOE_ERR_PLAN = -7          /* device error word: a kernel found its launch plan inconsistent with
                                the shape (a bug, never expected: create checks every CTA's part);
                                the kernel skipped its work */
} moe_status;

enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 };

/* Shapes and formats of one layer, fixed at create time. */
typedef struct moe_decode_config {
  int32_t din;             /* hidden size; a multiple of 64 */
  int32_t dff;             /* routed expert width; a multiple of 64 */
  int32_t n_experts;       /* E >= 1 */
  int32_t top_k;           /* K routed slots per token, 0 <= K (K + n_shared >= 1) */
  int32_t max_tokens;      /* largest M a forward may pass, >= 1 */
  int32_t bits_gate;       /* 4, 6 or 8; must equal bits_up */
  int32_t bits_up;
  int32_t bits_down;       /* 4, 6 or 8, independent of gate/up */
  int32_t n_shared;        /* shared experts, 0..4 */
  int32_t dff_shared;      /* shared expert width; a multiple of 64 when n_shared > 0 */
  int32_t bits_shared;     /* 4, 6 or 8: gate, up and down of every shared expert */
  int32_t shared_gate;     /* 0: scalar 1;  1: scalar = sigmoid(x . gate_vec) */
  int32_t resid_dtype;     /* MOE_DTYPE_BF16 or MOE_DTYPE_F32 */
  int32_t out_dtype;       /* MOE_DTYPE_F32 (default) or MOE_DTYPE_BF16 (rounded to nearest) */
  int32_t kernel_mode;     /* MOE_KERNELS_FUSED (default), _SEPARATE, _COLUMNS, _COLUMNS_AHEAD,
                              _POOL, _MMA */
} moe_decode_config;

/* How a layer is launched.  FUSED: one cooperative persistent kernel per forward (or per stack
 * step) runs the gate/up phase, a device-wide barrier, then the down phase, streaming the down
 * weights into shared memory while the gate/up phase computes.  SEPARATE: kernel A then kernel B
 * per layer with programmatic dependent launch (the unfused form, kept for comparison).
 * COLUMNS: one cooperative persistent kernel per forward or stack step in which each CTA carries
 * a contiguous range of activation columns through gate/up, SwiGLU and the matching columns of
 * the down projection (the same sums as kernel A and kernel B of "two-kernel decode-MoE that
 * beats gather_qmm", What changed, step 2, and the tail of "Red Lite dev39 -- fused expert tail",
 * Change), writing per-CTA partial outputs that the row owners sum in a fixed order: one
 * device-wide barrier per layer.  Requires max_tokens == 1, gate/up codes of 4 or 8 bits,
 * bits_down (and bits_shared when n_shared > 0) of 4 or 8, din <= 4096; create returns
 * MOE_ERR_UNSUPPORTED otherwise.  Create copies every projection into the kernel's own layout
 * (owned by the handle, about the size of the layer's weights: gate and up rows interleaved with
 * their scales and biases, the down projection column-block-major) and allocates a partial-sum
 * buffer; after create the kernel reads only those copies and gate_vec.  The chained stack and
 * moe_stack_step_parts (one phase) do not take this mode.  Results are deterministic (fixed summation order) and equal
 * the other modes within the parity bound, not bit for bit (the sums associate differently).
 * COLUMNS_AHEAD: the same kernel and arithmetic (results byte-identical to COLUMNS) for steps
 * whose expert ids are all inputs known before the step, as when ids are drawn per layer from a
 * seed: the weight stream of layer l + 1 starts as soon as the CTA's consumers are done with
 * layer l's gate/up phase instead of after layer l's device-wide barrier.  It is not the decode
 * dependency (there a router needs layer l's output to pick layer l + 1's experts); it measures
 * how far the stream itself goes when that dependency is lifted. */
/* POOL: the pool-and-tail form of "Red Lite dev39 -- fused expert tail" (Change) kept apart, for
 * any m: one cooperative persistent kernel groups the m tokens' slots by expert, computes every
 * routed slot's and shared expert's down output WITHOUT its coefficient into a workspace buffer
 * (device-wide barrier), then a tail forms
 *   out = resid + (sum_k score_k * y_k  +  scalar * sum_s y_s),  k in slot order,
 * exactly the page's association.  moe_decode_routes copies the per-slot outputs out.  It is the
 * unfused counterpart of the other modes, which fold the score or the scalar into the activation
 * and sum routed and shared terms in one accumulation; results agree within the parity bound. */
/* MMA: the batch form on tensor cores, for a few to a few dozen tokens.  The m tokens' slots are
 * grouped by expert (distinct ids ascending, pairs in (token, slot) order); each selected expert's
 * gate/up and down rows are read once for all the tokens that name it, in tiles of 16 rows x 8
 * (token, slot) pairs on mma.sync bf16 instructions (codes enter exactly as bf16 integers, 8-bit
 * codes as two nibble tiles; x exactly; the fp32 activation as a bf16 high part plus a bf16
 * remainder; fp32 accumulation; the group scale and bias applied per 64 codes).  Four launches
 * per layer: route and shared scalars, gate/up, down, tail (out = resid + the valid slots in slot
 * order + the shared experts).  Requires max_tokens <= 64, max_tokens * top_k <= 256,
 * n_experts <= 1024; the chained stack and moe_stack_step_parts (one phase) do not take it.
 * Deterministic; equal to the other modes within the parity bound. */
enum {
  MOE_KERNELS_FUSED = 0,
  MOE_KERNELS_SEPARATE = 1,
  MOE_KERNELS_COLUMNS = 2,
  MOE_KERNELS_COLUMNS_AHEAD = 3,
  MOE_KERNELS_POOL = 4,
  MOE_KERNELS_MMA = 5
};

/*
 * One projection of every expert of a class, canonical packed layout, all device pointers:
 *   codes  [experts][rows][cols*bits/8] bytes: per row a little-endian bit stream, code c at bits
 *          [c*bits, c*bits + bits), LSB first (8 codes per uint32 at 4 bits, 4 at 8 bits,
 *          16 per 3 uint32 at 6 bits); 16-byte aligned
 *   scales [experts][rows][cols/64] fp16, biases likewise; 16-byte aligned
 * gate and up have rows = dff, cols = din; down has rows = din, cols = dff.
 */
typedef struct moe_proj {
  const void *codes;
  const void *scales;
  const void *biases;
} moe_proj;

typedef struct moe_layer_weights {
  moe_proj gate, up, down;          /* routed experts, [n_experts] stacked */
  moe_proj sh_gate, sh_up, sh_down; /* shared experts, [n_shared] stacked (ignored if none) */
  const void *gate_vec;             /* bf16 [din] device, required when shared_gate == 1 */
} moe_layer_weights;

typedef struct moe_decode moe_decode_t;
typedef struct moe_stack moe_stack_t;

/* Prepares one layer: validates the config and weight pointers, picks the kernels, allocates the
 * workspace (fp32 activations [max_tokens][K*dff + n_shared*dff_shared] and the error word).
 * The prepared handle is the "prepared executor" form: nothing is set up per forward.
 * Returns MOE_OK and *out, or an error and *out = NULL. */
int moe_decode_create(const moe_decode_config *cfg, const moe_layer_weights *weights,
                      moe_decode_t **out);

/* Enqueues the block for m tokens on `stream` (asynchronous, allocation-free).
 *   x      bf16 [m][din] device, 16-byte aligned token activations
 *   ids    int32 [m][top_k] device              routed expert ids, slot order as given
 *   scores fp32 [m][top_k] device               router weights of the slots
 *   resid  [m][din] device, cfg->resid_dtype    residual added in the tail
 *   out    [m][din] device, cfg->out_dtype      result; may alias resid, must not alias x
 * Kernel A (gate/up + SwiGLU, scaled by the slot's score or the shared scalar) writes the
 * workspace; kernel B (down GEMV, summed over slots and shared experts, plus resid) writes out.
 * Both launch with programmatic dependent launch so B streams its weights while A finishes. */
int moe_decode_forward(moe_decode_t *h, const void *x, int32_t m, const int32_t *ids,
                       const float *scores, const void *resid, void *out, void *stream);

/* Synchronises the device, returns the sticky device error word in *device_error (MOE_OK,
 * MOE_ERR_BAD_ID or MOE_ERR_TIMEOUT) and clears it. */
int moe_decode_get_error(moe_decode_t *h, int32_t *device_error);

/* The route the last moe_decode_forward of this handle took, for checking it (no counterpart
 * beyond the page's tmp-buffer accessor of "Red Lite dev39 -- fused expert tail", Change).
 *   ids_used  int32 [m][top_k] device or NULL: the expert ids the kernels read, in the order
 *             they read them (slot order), as written by the kernels themselves
 *   slot_out  fp32 [m][top_k + n_shared][din] device or NULL (MOE_KERNELS_POOL only): each routed
 *             slot's down output W_down[id] . act (before its score) and each shared expert's
 *             (before the scalar); rows of a slot with an invalid id are unspecified
 * m is the last forward's token count.  Asynchronous on `stream`, ordered after that forward when
 * both use the same stream.  Returns MOE_ERR_INVALID_ARG for a null handle, both pointers null, a
 * misaligned pointer or no forward yet, MOE_ERR_UNSUPPORTED for slot_out outside the pool mode. */
int moe_decode_routes(moe_decode_t *h, int32_t *ids_used, void *slot_out, void *stream);

void moe_decode_destroy(moe_decode_t *h);

/* ---- one layer without a handle and without device allocation -------------------------------
 * The pages have no counterpart of this call: their kernels always run inside an engine that owns
 * its buffers.  It exists for callers that may not allocate device memory at all (an allocator
 * that is frozen while graphs are captured, a memory pool with a hard budget): it runs the same
 * two kernels as MOE_KERNELS_SEPARATE, kernel A then kernel B per token, with the activation vector
 * kept in a fixed scratch array of the library instead of a handle's workspace.
 *
 *   cfg, weights   as for moe_decode_create; cfg->kernel_mode must be MOE_KERNELS_SEPARATE and
 *                  K*dff + n_shared*dff_shared must not exceed MOE_NOALLOC_MAX_ACT_FLOATS
 *                  (else MOE_ERR_UNSUPPORTED); weights are borrowed for the call
 *   x, ids, scores, resid, out, m, stream   as for moe_decode_forward (m <= cfg->max_tokens)
 *   device_error   int32 device word the kernels OR error bits into (bit 0: an expert id outside
 *                  [0, n_experts), that slot contributed zero; bit 1: a wait gave up).  It must
 *                  hold 0 before the first call and is never cleared by the library.  NULL sends
 *                  the bits to a library word that no call reads.
 *
 * Scratch: a file-scope device array of MOE_NOALLOC_MAX_ACT_FLOATS floats (256 KiB) per device,
 * whose address is looked up once per device (with the lookup's return code checked).  Nothing is
 * allocated, freed or zeroed by the call; the scratch needs no initial value because kernel A
 * writes every activation before kernel B reads it.
 * Races: every call on a device shares that one array.  Calls on one device must be ordered on
 * the GPU (one stream, or streams joined by events); two calls that overlap on the GPU corrupt
 * each other's activations.
 * Capture: the first call on a device looks the scratch up, and the first call with a given config
 * sets the kernels' shared-memory limits (the last 8 configs per device are remembered); make those
 * calls outside stream capture.  Later calls with a remembered config only enqueue two kernels per
 * token and may be captured into a CUDA graph.
 * Returns MOE_OK, or a negative status with nothing enqueued. */
#define MOE_NOALLOC_MAX_ACT_FLOATS 65536
int moe_decode_forward_noalloc(const moe_decode_config *cfg, const moe_layer_weights *weights,
                               const void *x, int32_t m, const int32_t *ids, const float *scores,
                               const void *resid, void *out, int32_t *device_error,
                               void *stream);

/* ---- a stack of layers replayed as one CUDA graph ------------------------------------------
 * Layer l reads x_l = x + l*m*din, ids_l = ids + l*m*top_k, scores_l likewise; its residual is
 * resid0 (cfg->resid_dtype) for l = 0 and the fp32 output of layer l-1 after that; the last
 * layer writes `out` (fp32 [m][din]).  No layer reads its ids before the previous layer's output
 * is complete: every kernel waits on its predecessor before touching token data, and only
 * weight prefetch runs ahead.  cfg->out_dtype must be MOE_DTYPE_F32. */
int moe_stack_create(const moe_decode_config *cfg, int32_t n_layers,
                     const moe_layer_weights *layers, moe_stack_t **out);

/* The same stack with the next layer's RMSNorm folded in: layer l >= 1 does not read x_l but
 * normalises the previous layer's fp32 output,
 *   x_l[c] = bf16( gamma_l[c] * (out_{l-1}[c] * r) ),  r = 1 / sqrt(mean_c out_{l-1}[c]^2 + eps)
 * "Red Lite dev39 -- fused expert tail" (Measurements) records a tail that also folded in the
 * next layer's RMSNorm and names the step without a formula; this is the usual RMSNorm.  Every
 * CTA of layer l's first phase computes r itself: the squares summed in fp64 in a fixed order, r
 * rounded once to fp32, the two products in fp32, the result rounded to the nearest bf16 (ties
 * to even), so the fused and the separate kernel modes give identical bytes.
 *   norm_weight  bf16 [n_layers - 1][din] device, 16-byte aligned, borrowed for the stack's life:
 *                row l - 1 is gamma_l
 *   eps          in [0, 1]
 * moe_stack_step then reads x as [m][din] (layer 0 only; moe_stack_step_host copies m*din
 * values).  Batches (m > 1) run token by token.  Other arguments and returns as for
 * moe_stack_create (MOE_ERR_INVALID_ARG also for a null or misaligned norm_weight or an eps
 * outside [0, 1]). */
int moe_stack_create_chained(const moe_decode_config *cfg, int32_t n_layers,
                             const moe_layer_weights *layers, const void *norm_weight, float eps,
                             moe_stack_t **out);

/* Enqueues one decode step of the whole stack on `stream` (device pointers as above).  The first
 * call with a given (x, ids, scores, resid0, out, m) captures and instantiates a CUDA graph
 * (not asynchronous, allocates); later calls with the same pointers only launch it. */
int moe_stack_step(moe_stack_t *s, const void *x, int32_t m, const int32_t *ids,
                   const float *scores, const void *resid0, void *out, void *stream);

/* Measurement aid: the same step with only some kernels of every layer in the graph.
 * parts = MOE_PART_GATE_UP (kernel A of each layer), MOE_PART_DOWN (kernel B of each layer, reading
 * whatever activations the workspace holds) or both (identical to moe_stack_step).  Replaying one
 * part times that kernel's launches back to back with the same launch configuration. */
enum { MOE_PART_GATE_UP = 1, MOE_PART_DOWN = 2 };
int moe_stack_step_parts(moe_stack_t *s, int32_t parts, const void *x, int32_t m,
                         const int32_t *ids, const float *scores, const void *resid0, void *out,
                         void *stream);

/* One decode step from HOST buffers: copies x, ids, scores and resid0 (best from pinned memory)
 * into the stack's device staging buffers, replays the graph, copies out back, and synchronises
 * the stream before returning. */
int moe_stack_step_host(moe_stack_t *s, const void *x_host, int32_t m, const int32_t *ids_host,
                        const float *scores_host, const void *resid0_host, float *out_host,
                        void *stream);

int moe_stack_get_error(moe_stack_t *s, int32_t *device_error);
void moe_stack_destroy(moe_stack_t *s);

/* ---- dense bf16 decode GEMV ------------------------------------------------------------------
 * The q/k/v/o attention projections that "Measure attention projections instead of serving
 * them, and record the amortisation trap" measures beside the block at 1, 8 and 32 rows.  For
 * each of n_mats weight matrices r:
 *   y[r][t][o] = sum_i W[r][o][i] * x_r[t][i]          (bf16 products, fp32 accumulation)
 *   W        bf16 [n_mats][n_out][n_in] device, 16-byte aligned; n_in a multiple of 8
 *   x        bf16 device, 16-byte aligned: x_r = x + r * x_stride elements is [m][n_in]
 *            (x_stride 0: one input for every matrix; otherwise a multiple of 8)
 *   y        fp32 [n_mats][m][n_out] device
 *   m        rows (tokens), 1..32.  Up to 4 rows CUDA cores stream W (the product is HBM-bound);
 *            from 5 rows bf16 tensor-core tiles (16 weight rows x 8 tokens) take the products.
 * One launch covers every matrix, so a caller can stream far more than L2 per launch (the page's
 * rule against timing cache-resident weights).  The sum order is fixed: repeat calls give
 * identical bytes.  Asynchronous on `stream`.  Returns MOE_OK, MOE_ERR_INVALID_ARG on a size or
 * alignment outside the above (nothing enqueued), or MOE_ERR_CUDA if the launch fails. */
int moe_gemv_bf16(const void *W, const void *x, int64_t x_stride, float *y, int32_t n_mats,
                  int32_t m, int32_t n_out, int32_t n_in, void *stream);

/* ---- canonical packing (host) ---------------------------------------------------------------
 * codes: uint8 [rows][cols], one code per byte, each < 2^bits; packed: [rows][cols*bits/8].
 * cols must be a multiple of 64.  Returns MOE_ERR_INVALID_ARG on a code out of range. */
int moe_pack_codes(const uint8_t *codes, int64_t rows, int64_t cols, int32_t bits, void *packed);
int moe_unpack_codes(const void *packed, int64_t rows, int64_t cols, int32_t bits, uint8_t *codes);

/* Debug: unpacks packed device codes on the GPU with the kernels' own window/mask decoding, one
 * code per output byte (device [rows][cols]); for checking the decoding bit for bit. */
int moe_unpack_codes_device(const void *packed, int64_t rows, int64_t cols, int32_t bits,
                            uint8_t *codes, void *stream);

/* ---- synthetic weights in HBM (input generation, not the block) ------------------------------
 * Fill device buffers with the counter-based generator defined in the Python module
 * quantized_moe_expert_dequant_gb300.synth, bit for bit: element i of expert e (e counted from
 * expert0) is derived from mix64(key + G*(((e << 40) | i) + 1)).
 *   codes : n_experts * words_per_expert uint64 words
 *   scales: n_experts * per_expert fp16 values, about U(0.005, 0.02)
 *   biases: fp16, about -2^(bits-1) * scale, from the scales already in `scales` */
int moe_synth_codes(void *dst, uint64_t key, int32_t expert0, int32_t n_experts,
                    int64_t words_per_expert, void *stream);
int moe_synth_scales(void *dst, uint64_t key, int32_t expert0, int32_t n_experts,
                     int64_t per_expert, void *stream);
int moe_synth_biases(void *dst, const void *scales, uint64_t key, int32_t expert0,
                     int32_t n_experts, int64_t per_expert, int32_t bits, void *stream);

/* Route inversion of a batch of tokens, as the grouped kernels compute it (a debug export, so the
 * integer result can be compared bit for bit with an independent implementation).  ids is int32
 * [m][k] device; out is int32 device with room for 2 + 2*m*k + m*k values and receives U (the
 * number of distinct ids in [0, n_experts)), then those ids ascending (uniq[U]), then offs[U + 1]
 * and then the pairs p = token * k + slot grouped by expert, ascending within each (the pairs
 * of uniq[u] are at offs[u] .. offs[u + 1] - 1).  Asynchronous on stream.  Limits: m * k <= 256,
 * n_experts <= 1024 (MOE_ERR_UNSUPPORTED beyond).  The pages group the routers' top-k pools by
 * expert only implicitly ("Red Lite dev39 -- fused expert tail", Change). */
int moe_route_invert_device(const int32_t *ids, int32_t m, int32_t k, int32_t n_experts,
                            int32_t *out, void *stream);

/* The router step before the block: for each of m tokens, the top_k of n_experts fp32 logits
 * (larger first; between equal logits the lower expert id first) and the softmax of the chosen
 * logits over those top_k -- the top-k pool with weights that "Red Lite dev39 -- fused expert tail"
 * (Change) feeds to the expert tail in GPU-routed decode.
 *   logits  fp32 [m][n_experts] device (no NaN)
 *   ids     int32 [m][top_k] device: expert ids in pool order
 *   scores  fp32 [m][top_k] device: weights in the same order, summing to 1 (fp32 rounding)
 * Asynchronous on stream.  Limits: 1 <= top_k <= min(64, n_experts), n_experts <= 1024
 * (MOE_ERR_UNSUPPORTED beyond).  The pages give the pool and its weights, not the selection rule;
 * ties to the lower id is this implementation's. */
int moe_router_topk(const float *logits, int32_t m, int32_t n_experts, int32_t top_k,
                    int32_t *ids, float *scores, void *stream);

/* Exercises the bounded-wait path of the kernels without any fault: one thread waits, with the
 * kernels' own wait functions and a limit of about 0.1 s, on a condition nothing satisfies --
 * kind 0 a grid-barrier count (in scratch, which the call zeroes; int32 device, 4-byte aligned),
 * kind 1 an mbarrier stage that no producer fills.  The wait gives up, ORs the time-out bit (2)
 * into device_error (int32 device) and the kernel returns; the context stays usable.  Asynchronous
 * on stream.  No counterpart on the pages: it checks this implementation's guarantee that no
 * wait runs forever. */
int moe_debug_wait_timeout(int32_t kind, int32_t *scratch, int32_t *device_error, void *stream);

/* The column split's cut of a CTA's activation columns [u0, u1) into pieces, exactly as the
 * MOE_KERNELS_COLUMNS kernel computes it on the device (host only, no CUDA call: a debug export so
 * that the decomposition can be checked on a machine without a GPU).  The activation columns are
 * the flattened routed-then-shared rows of the gate/up projections (top_k * dff routed, then
 * n_shared * dff_shared); the plan gives each CTA its range (moe_debug_col_plan's bounds), and the
 * range is cut at every segment (routed slot or shared expert) and every group of 64 columns.
 *   bits_down, bits_shared  4 or 8: the down projection's code width (32 / bits codes per word)
 *   out   int32 host, room for 8 * max_pieces values: per piece seg (slot, or top_k + shared
 *         index), j0, j1 (columns inside the expert), a0 (index of j0 in the CTA's range), blk0
 *         (first 32-bit column block), nb (blocks), pb (index of the first block in the CTA's
 *         block list), grp (j0 / 64)
 * Returns the piece count (>= 0), MOE_ERR_UNSUPPORTED when the range holds more columns, pieces or
 * blocks than the kernel holds (or more pieces than max_pieces), MOE_ERR_INVALID_ARG for bad
 * arguments (a range outside [0, U]).  No counterpart on the pages: the split by columns is this
 * implementation's. */
int moe_debug_col_pieces(int32_t top_k, int32_t dff, int32_t n_shared, int32_t dff_shared,
                         int32_t bits_down, int32_t bits_shared, int32_t u0, int32_t u1,
                         int32_t *out, int32_t max_pieces);

/* The column split's launch plan for a config on a grid of `grid` CTAs with `ring_bytes` of
 * dynamic shared memory, exactly as moe_decode_create makes it (host only, no CUDA call: a debug
 * export for checks without a GPU).  cfg's kernel_mode is ignored.  out (int32 host, 10 values)
 * receives: stages in the ring, bytes per stage, column blocks per down stage (nbs), rows per
 * owner in the partial-sum slab (ro), the routed and the shared down projection's codes per
 * 32-bit word, the gate/up rows per routed and per shared phase-A stage, whether down stages are
 * packed across pieces, whether the stages past the first ring-full are prefetched into L2.
 * bounds (int32 host, grid + 1 values, or NULL) receives the CTAs' column ranges: CTA c owns the
 * activation columns [bounds[c], bounds[c + 1]), bounds[0] = 0 and bounds[grid] = U.  An
 * unpacked plan starts from the even split (U c / grid) and moves each inner boundary at most 16
 * columns so that the CTA with the most stages has as few as possible, then the fewest bytes,
 * then the total bytes are least; a packed plan keeps the even split.  Returns MOE_OK, or MOE_ERR_UNSUPPORTED when the column split does not take the config
 * (or the grid), MOE_ERR_INVALID_ARG for an invalid config.  No counterpart on the pages. */
int moe_debug_col_plan(const moe_decode_config *cfg, int32_t grid, int32_t ring_bytes,
                       int32_t *out, int32_t *bounds);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
