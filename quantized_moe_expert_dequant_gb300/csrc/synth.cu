// synth.cu -- synthetic weights drawn directly in HBM (input generation, not the MoE block).
//
// Implements, bit for bit, the counter-based definitions of the Python module
// quantized_moe_expert_dequant_gb300.synth so that a multi-GB stack can be drawn on the device
// and any one expert recomputed on the host: SplitMix64's output function (Steele, Lea and Flood,
// OOPSLA 2014) applied to key + G*(((e << 40) | i) + 1), and fp32 arithmetic rounded to nearest
// at every step (explicit __fmul_rn/__fadd_rn, so nothing is contracted into an FMA).
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_decode.h"

namespace {

constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t element_hash(uint64_t key, int64_t expert, int64_t i) {
  const uint64_t idx = (static_cast<uint64_t>(expert) << 40) | static_cast<uint64_t>(i);
  return mix64(key + kG * (idx + 1));
}

__global__ void codes_kernel(uint64_t *dst, uint64_t key, int expert0, int64_t total,
                             int64_t per_expert) {
  for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n < total;
       n += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = n / per_expert, i = n - e * per_expert;
    dst[n] = element_hash(key, expert0 + e, i);
  }
}

__global__ void scales_kernel(__half *dst, uint64_t key, int expert0, int64_t total,
                              int64_t per_expert) {
  for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n < total;
       n += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = n / per_expert, i = n - e * per_expert;
    const uint32_t u = static_cast<uint32_t>(element_hash(key, expert0 + e, i) >> 40);
    float v = __fmul_rn(__uint2float_rn(u), 5.9604644775390625e-08f);  // * 2^-24, exact
    v = __fmul_rn(v, 0.015f);
    v = __fadd_rn(v, 0.005f);
    dst[n] = __float2half_rn(v);
  }
}

__global__ void biases_kernel(__half *dst, const __half *scales, uint64_t key, int expert0,
                              int64_t total, int64_t per_expert, float half_range) {
  for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n < total;
       n += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = n / per_expert, i = n - e * per_expert;
    const uint32_t u = static_cast<uint32_t>(element_hash(key, expert0 + e, i) >> 40);
    const float t = __fsub_rn(__fmul_rn(__uint2float_rn(u), 5.9604644775390625e-08f), 0.5f);
    const float c = __fadd_rn(half_range, t);
    const float m = __fmul_rn(__half2float(scales[n]), c);
    dst[n] = __float2half_rn(-m);
  }
}

int grid_for(int64_t total) {
  int64_t g = (total + 255) / 256;
  return static_cast<int>(g < 1 ? 1 : (g > 4096 ? 4096 : g));
}

}  // namespace

extern "C" int moe_synth_codes(void *dst, uint64_t key, int32_t expert0, int32_t n_experts,
                               int64_t words_per_expert, void *stream) {
  if (!dst || expert0 < 0 || n_experts < 0 || words_per_expert < 0) return MOE_ERR_INVALID_ARG;
  const int64_t total = (int64_t)n_experts * words_per_expert;
  if (total == 0) return MOE_OK;
  codes_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t *>(dst), key, expert0, total, words_per_expert);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_synth_scales(void *dst, uint64_t key, int32_t expert0, int32_t n_experts,
                                int64_t per_expert, void *stream) {
  if (!dst || expert0 < 0 || n_experts < 0 || per_expert < 0) return MOE_ERR_INVALID_ARG;
  const int64_t total = (int64_t)n_experts * per_expert;
  if (total == 0) return MOE_OK;
  scales_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<__half *>(dst), key, expert0, total, per_expert);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_synth_biases(void *dst, const void *scales, uint64_t key, int32_t expert0,
                                int32_t n_experts, int64_t per_expert, int32_t bits,
                                void *stream) {
  if (!dst || !scales || expert0 < 0 || n_experts < 0 || per_expert < 0) return MOE_ERR_INVALID_ARG;
  if (bits != 4 && bits != 6 && bits != 8) return MOE_ERR_UNSUPPORTED;
  const int64_t total = (int64_t)n_experts * per_expert;
  if (total == 0) return MOE_OK;
  biases_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<__half *>(dst), static_cast<const __half *>(scales), key, expert0, total,
      per_expert, static_cast<float>(1 << (bits - 1)));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
