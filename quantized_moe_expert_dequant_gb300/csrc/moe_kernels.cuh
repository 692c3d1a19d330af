// moe_kernels.cuh -- parameters and launchers of the decode MoE kernels (host-visible).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

struct ProjDev {
  const uint8_t *codes;   // [experts][rows][cols*bits/8]
  const __half *scales;   // [experts][rows][cols/64]
  const __half *biases;   // [experts][rows][cols/64]
};

// Kernel A: act[u] = coef_u * silu(gate_u . x) * (up_u . x) for every row pair u of the routed
// slots (coef = the slot's score) and of the shared experts (coef = the shared scalar).
struct GateUpParams {
  ProjDev gate, up, sh_gate, sh_up;
  const uint16_t *x;         // bf16 [din]
  const int32_t *ids;        // [top_k]
  const float *scores;       // [top_k]
  const uint16_t *gate_vec;  // bf16 [din] or nullptr (shared scalar 1)
  float *act;                // [top_k*dff + n_shared*dff_shared]
  int32_t *err;              // sticky error word
  int din, dff, top_k, n_experts, n_shared, dff_shared;
};

// Kernel B: out[i] = resid[i] + sum over slots and shared experts of W_down[i, :] . act_segment.
struct DownParams {
  ProjDev down, sh_down;
  const int32_t *ids;        // [top_k]
  const float *act;          // [top_k*dff + n_shared*dff_shared], from kernel A
  const void *resid;         // [din] bf16 or fp32
  void *out;                 // [din] fp32 or bf16
  int32_t *err;
  int resid_f32, out_f32;
  int din, dff, top_k, n_experts, n_shared, dff_shared;
};

constexpr int kMaxTopK = 64;
constexpr int kAThreads = 512;
constexpr int kBThreads = 256;
constexpr int kBRows = 2;  // output rows per warp item in kernel B

size_t gate_up_smem_bytes(int din, int bits_r, int bits_s, int n_shared);
size_t down_smem_bytes(int dff, int top_k, int n_shared, int dff_shared, int bits_d, int bits_sd);

// Both return a cudaError_t; `pdl` launches with programmatic stream serialisation.
cudaError_t launch_gate_up(const GateUpParams &p, int bits_r, int bits_s, int grid, size_t smem,
                           cudaStream_t stream, bool pdl);
cudaError_t launch_down(const DownParams &p, int bits_d, int bits_sd, int grid, size_t smem,
                        cudaStream_t stream, bool pdl);
cudaError_t prepare_kernels(int smem_optin, int bits_r, int bits_s, int bits_d, int bits_sd);
cudaError_t launch_unpack(const uint8_t *packed, int64_t rows, int64_t cols, int bits,
                          uint8_t *codes, cudaStream_t stream);

}  // namespace moe
