// gemv.cu -- dense bf16 decode GEMV: the q/k/v/o attention projections that "Measure attention
// projections instead of serving them, and record the amortisation trap" measures at 1, 8 and 32
// rows.  For each of n_mats weight matrices r:
//
//   y[r][t][o] = sum_i W[r][o][i] * x_r[t][i]        (bf16 inputs, fp32 accumulation)
//
// Two kernels, chosen by the number of rows m (tokens):
//   gemv_cc_kernel<MT>   m <= 4: the product is HBM-bound, so CUDA cores do it while the weights
//                        stream once: a warp owns 4 weight rows, each lane 8 columns per 256-column
//                        step (one 16-byte streaming load per row), x comes through L1.
//   gemv_mma_kernel<NT>  5 <= m <= 32: a dense contraction with up to 32 columns of x, on bf16
//                        tensor-core tiles (mma.sync m16n8k16, fp32 accumulate): a warp owns 16
//                        weight rows; per 32-column chunk each lane loads 16 contiguous bytes of
//                        two rows straight into A fragments, and the k order inside the chunk is
//                        permuted identically for x (a sum does not depend on its order).
// The weights are read once (streaming loads); one launch covers every matrix, so a caller can
// move more than a gigabyte per launch, the page's rule against timing cache-resident weights.
// Partial sums are combined in a fixed order: repeat runs give identical bytes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_decode.h"

namespace gemv {

constexpr int kThreads = 256;  // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kRowsCC = 4;     // weight rows per warp task, CUDA-core kernel
constexpr int kRowsMMA = 16;   // weight rows per warp task, tensor-core kernel

struct Params {
  const uint16_t *W;  // bf16 [n_mats][n_out][n_in]
  const uint16_t *x;  // bf16 [m][n_in] of matrix r at x + r * x_stride
  float *y;           // fp32 [n_mats][m][n_out]
  int64_t x_stride;
  int n_mats, m, n_out, n_in;
  int row_tiles;      // tasks per matrix
  int64_t tasks;      // n_mats * row_tiles
};

__device__ __forceinline__ uint4 ld_weights(const uint16_t *p) {  // read once: streaming
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ uint4 ld_input(const uint16_t *p) {  // shared by every warp: cached
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Sums V values over the 32 lanes: log2(V) exchange steps halve the values a lane holds, a
// butterfly finishes.  Lane l returns the sum of value (l >> (5 - log2 V)) & (V - 1).
template <int V>
__device__ __forceinline__ float lanes_transpose_sum(float (&v)[V], int lane) {
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

template <int V>
struct Log2 {
  static constexpr int v = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : -1;
};

// ------------------------------------------------------------------ m <= 4: CUDA cores
template <int MT>
__global__ void __launch_bounds__(kThreads) gemv_cc_kernel(const Params p) {
  constexpr int R = kRowsCC, V = R * MT;
  const int lane = threadIdx.x & 31;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
       task < p.tasks; task += nw) {
    const int mat = static_cast<int>(task / p.row_tiles);
    const int r0 = static_cast<int>(task - static_cast<int64_t>(mat) * p.row_tiles) * R;
    const uint16_t *Wm = p.W + static_cast<int64_t>(mat) * p.n_out * p.n_in;
    const uint16_t *xm = p.x + static_cast<int64_t>(mat) * p.x_stride;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int c = lane * 8; c < p.n_in; c += 256) {
      uint4 w[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        w[r] = r0 + r < p.n_out ? ld_weights(Wm + static_cast<int64_t>(r0 + r) * p.n_in + c)
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const uint4 xv = t < p.m ? ld_input(xm + static_cast<int64_t>(t) * p.n_in + c)
                                 : make_uint4(0, 0, 0, 0);
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
          float a = acc[r * MT + t];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            a = fmaf(lo_bf16(ws[h]), lo_bf16(xs[h]), a);
            a = fmaf(hi_bf16(ws[h]), hi_bf16(xs[h]), a);
          }
          acc[r * MT + t] = a;
        }
      }
    }
    const float s = lanes_transpose_sum<V>(acc, lane);
    const int idx = (lane >> (5 - Log2<V>::v)) & (V - 1);
    const int r = idx / MT, t = idx - r * MT;
    if ((lane & ((32 / V) - 1)) == 0 && t < p.m && r0 + r < p.n_out)
      p.y[(static_cast<int64_t>(mat) * p.m + t) * p.n_out + r0 + r] = s;
  }
}

// ------------------------------------------------------------------ 5 <= m <= 32: tensor cores
// D[16 x 8] += A[16 x 16] B[16 x 8], bf16 inputs, fp32 accumulation.  A is row-major: lane
// (g = lane / 4, q = lane % 4) holds rows g and g + 8 at k slots 2q, 2q + 1 (registers 0, 1)
// and 2q + 8, 2q + 9 (registers 2, 3); B holds k slots 2q, 2q + 1 and 2q + 8, 2q + 9 of column
// g; D holds rows g and g + 8 at columns 2q, 2q + 1.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT>
__global__ void __launch_bounds__(kThreads) gemv_mma_kernel(const Params p) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t task = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
       task < p.tasks; task += nw) {
    const int mat = static_cast<int>(task / p.row_tiles);
    const int r0 = static_cast<int>(task - static_cast<int64_t>(mat) * p.row_tiles) * kRowsMMA;
    const uint16_t *Wm = p.W + static_cast<int64_t>(mat) * p.n_out * p.n_in;
    const uint16_t *xm = p.x + static_cast<int64_t>(mat) * p.x_stride;
    const bool ok_a = r0 + g < p.n_out, ok_b = r0 + g + 8 < p.n_out;
    const uint16_t *wa = Wm + static_cast<int64_t>(r0 + g) * p.n_in;
    const uint16_t *wb = wa + 8 * static_cast<int64_t>(p.n_in);
    float d[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
    // Each lane owns columns c .. c + 7 of a 32-column chunk; inside the chunk the two MMAs take
    // columns (c, c+1 | c+2, c+3) and (c+4, c+5 | c+6, c+7) as k slots (2q, 2q+1 | 2q+8, 2q+9),
    // for A and B alike.  The chunk loop is the same for every lane (the MMAs are warp-wide);
    // columns past n_in (a multiple of 8) read as zeros.
#pragma unroll 4
    for (int k0 = 0; k0 < p.n_in; k0 += 32) {
      const int c = k0 + 8 * q;
      const bool ok_c = c < p.n_in;
      const uint4 za = make_uint4(0, 0, 0, 0);
      const uint4 a = ok_a && ok_c ? ld_weights(wa + c) : za;
      const uint4 b = ok_b && ok_c ? ld_weights(wb + c) : za;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int t = 8 * j + g;
        const uint4 xv =
            t < p.m && ok_c ? ld_input(xm + static_cast<int64_t>(t) * p.n_in + c) : za;
        mma_bf16(d[j], a.x, b.x, a.y, b.y, xv.x, xv.y);
        mma_bf16(d[j], a.z, b.z, a.w, b.w, xv.z, xv.w);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int t0 = 8 * j + 2 * q;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int t = t0 + (h & 1), row = r0 + g + (h >> 1) * 8;
        if (t < p.m && row < p.n_out)
          p.y[(static_cast<int64_t>(mat) * p.m + t) * p.n_out + row] = d[j][h];
      }
    }
  }
}

template <typename K>
static cudaError_t launch(K kern, Params p, int rows_per_task, cudaStream_t stream) {
  p.row_tiles = (p.n_out + rows_per_task - 1) / rows_per_task;
  p.tasks = static_cast<int64_t>(p.n_mats) * p.row_tiles;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // Tasks are equal, so the launch takes as many rounds as the resident warps need, and the grid
  // shrinks until every warp has the same number of tasks (no partly filled last round).
  const int64_t resident = static_cast<int64_t>(sms) * per_sm * kWarps;
  const int64_t rounds = (p.tasks + resident - 1) / resident;
  const int64_t warps = (p.tasks + rounds - 1) / rounds;
  const int64_t grid = (warps + kWarps - 1) / kWarps;
  kern<<<static_cast<int>(grid), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gemv

extern "C" int moe_gemv_bf16(const void *W, const void *x, int64_t x_stride, float *y,
                             int32_t n_mats, int32_t m, int32_t n_out, int32_t n_in,
                             void *stream) {
  auto aligned = [](const void *ptr, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
  };
  if (!W || !x || !y || n_mats < 1 || m < 1 || m > 32 || n_out < 1 || n_in < 8 || n_in % 8 ||
      x_stride < 0 || x_stride % 8 || !aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4))
    return MOE_ERR_INVALID_ARG;
  gemv::Params p;
  p.W = static_cast<const uint16_t *>(W);
  p.x = static_cast<const uint16_t *>(x);
  p.y = y;
  p.x_stride = x_stride;
  p.n_mats = n_mats;
  p.m = m;
  p.n_out = n_out;
  p.n_in = n_in;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  using namespace gemv;
  if (m == 1)
    e = launch(gemv_cc_kernel<1>, p, kRowsCC, st);
  else if (m == 2)
    e = launch(gemv_cc_kernel<2>, p, kRowsCC, st);
  else if (m <= 4)
    e = launch(gemv_cc_kernel<4>, p, kRowsCC, st);
  else if (m <= 8)
    e = launch(gemv_mma_kernel<1>, p, kRowsMMA, st);
  else if (m <= 16)
    e = launch(gemv_mma_kernel<2>, p, kRowsMMA, st);
  else if (m <= 24)
    e = launch(gemv_mma_kernel<3>, p, kRowsMMA, st);
  else
    e = launch(gemv_mma_kernel<4>, p, kRowsMMA, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
