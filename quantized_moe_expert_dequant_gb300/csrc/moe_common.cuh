// moe_common.cuh -- device building blocks of the decode MoE kernels (sm_103a).
//
// Decoding packed codes without integer-to-float conversions
// ----------------------------------------------------------
// A 32-bit pattern below 2^24 read as an IEEE binary32 value is exactly  pattern * 2^-149
// (a subnormal, or the smallest normal binade, whose value is linear in the bits).  So a code q
// that sits at bit offset o of a word, with o + bits <= 24, becomes the exact float q * 2^(o-149)
// with ONE bitwise AND, and one FMA multiplies it into the dot product if the activation it
// meets was pre-scaled by 2^(149 - S - o).  The product is q * x * 2^-S; the step's sum is
// rescaled by 2^S once, together with the group scale.  fp32 subnormals are kept (this code is
// built without flush-to-zero), and S is chosen per vector from its largest magnitude so that no
// pre-scaled activation overflows.
//
// Code windows per format (a "step" is the unit one lane decodes at a time):
//   4-bit  step = 16 B  = 32 codes: nibbles 0..5 of a word masked in place (o = 0,4,..,20);
//                                   nibbles 6, 7 from word >> 8 (o = 16, 20)
//   8-bit  step = 16 B  = 16 codes: bytes 0..2 in place (o = 0, 8, 16); byte 3 from word >> 8
//   6-bit  step = 48 B  = 64 codes: each 3-word triple (96 bits, 16 codes) is cut into four
//                                   24-bit windows by funnel shifts; codes at o = 0, 6, 12, 18
// Every step lies inside one group of 64 codes, so one (scale, bias) pair applies to it:
//   sum_c (s q_c + b) x_c = s * sum_c q_c x_c + b * sum_c x_c.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

constexpr int kGroup = 64;

// ------------------------------------------------------------------ programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ float bf16_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40);  // NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// 2^k as a float for k in [-126, 127]
__device__ __forceinline__ float pow2f(int k) {
  return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// S for a vector whose largest magnitude is maxabs: pre-scaled values stay below 2^127.
__device__ __forceinline__ int choose_shift(float maxabs) {
  const int e = static_cast<int>((__float_as_uint(maxabs) >> 23) & 255u) - 127;
  int s = e + 24;
  s = s < 22 ? 22 : s;
  return s > 127 ? 127 : s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ packed formats
template <int BITS>
struct Fmt;
template <>
struct Fmt<4> {
  static constexpr int kVecs = 1;   // uint4 vectors per step
  static constexpr int kCodes = 32; // codes per step
};
template <>
struct Fmt<8> {
  static constexpr int kVecs = 1;
  static constexpr int kCodes = 16;
};
template <>
struct Fmt<6> {
  static constexpr int kVecs = 3;
  static constexpr int kCodes = 64;
};

// Bit offset o (inside its 24-bit window) of the code at column c of a row.
template <int BITS>
__host__ __device__ __forceinline__ int code_offset(int c) {
  if (BITS == 4) {
    const int n = c & 7;
    return n < 6 ? 4 * n : (n == 6 ? 16 : 20);
  } else if (BITS == 8) {
    const int n = c & 3;
    return n < 3 ? 8 * n : 16;
  } else {
    return 6 * (c & 3);
  }
}

// Masked code words of one step, code j of the step in m[j]: each m[j] < 2^24, equal to
// q_j << code_offset(j).
template <int BITS>
__device__ __forceinline__ void step_masks(const uint4 *v, uint32_t (&m)[Fmt<BITS>::kCodes]) {
  if constexpr (BITS == 4) {
    const uint32_t w[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t = w[i] >> 8;
      m[8 * i + 0] = w[i] & 0x0000000fu;
      m[8 * i + 1] = w[i] & 0x000000f0u;
      m[8 * i + 2] = w[i] & 0x00000f00u;
      m[8 * i + 3] = w[i] & 0x0000f000u;
      m[8 * i + 4] = w[i] & 0x000f0000u;
      m[8 * i + 5] = w[i] & 0x00f00000u;
      m[8 * i + 6] = t & 0x000f0000u;
      m[8 * i + 7] = t & 0x00f00000u;
    }
  } else if constexpr (BITS == 8) {
    const uint32_t w[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[4 * i + 0] = w[i] & 0x000000ffu;
      m[4 * i + 1] = w[i] & 0x0000ff00u;
      m[4 * i + 2] = w[i] & 0x00ff0000u;
      m[4 * i + 3] = __byte_perm(w[i], 0u, 0x4344u);  // byte 3 moved to byte 2, rest zero
    }
  } else {
    const uint32_t w[12] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y,
                            v[1].z, v[1].w, v[2].x, v[2].y, v[2].z, v[2].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t w0 = w[3 * t], w1 = w[3 * t + 1], w2 = w[3 * t + 2];
      const uint32_t win[4] = {w0, __funnelshift_r(w0, w1, 24), __funnelshift_r(w1, w2, 16),
                               w2 >> 8};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        m[16 * t + 4 * q + 0] = win[q] & 0x0000003fu;
        m[16 * t + 4 * q + 1] = win[q] & 0x00000fc0u;
        m[16 * t + 4 * q + 2] = win[q] & 0x0003f000u;
        m[16 * t + 4 * q + 3] = win[q] & 0x00fc0000u;
      }
    }
  }
}

// ------------------------------------------------------------------ integer dot products
// For 4- and 8-bit codes the activations of a step become 23-bit two's-complement fixed point
// with one binary exponent per step, f_i = rint(v_i * 2^(22 - E)) with max|v| < 2^E, split into
// three byte planes f = h * 2^16 + m * 2^8 + l (l, m unsigned, h signed, |h| <= 64).  dp4a then
// multiplies four unsigned code bytes by four plane bytes and accumulates exactly in 32 bits, so
// a step's sum_c q_c * f_c is exact; it is rounded once to fp32 and scaled by 2^(E - 22).  The
// only approximation is the rounding of each activation to 23 bits below the step's largest one,
// the same relative size as one fp32 rounding.  8-bit codes need no masking at all; 4-bit codes
// need one AND for the low nibbles and one for the high nibbles (kept 16x, undone at the end).

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// E with max|v| < 2^E (clamped so that both 2^(22 - E) and 2^(E - 26) are normal floats).
__device__ __forceinline__ int fixed_exponent(float maxabs) {
  const int e = static_cast<int>((__float_as_uint(maxabs) >> 23) & 255u) - 126;
  return e < -100 ? -100 : (e > 126 ? 126 : e);
}

// Byte planes of four fixed-point values (value k in byte k of each plane).
__device__ __forceinline__ void byte_planes(int f0, int f1, int f2, int f3, uint32_t &pl,
                                            uint32_t &pm, uint32_t &ph) {
  pl = __byte_perm(__byte_perm(f0, f1, 0x0040), __byte_perm(f2, f3, 0x0040), 0x5410);
  pm = __byte_perm(__byte_perm(f0, f1, 0x0051), __byte_perm(f2, f3, 0x0051), 0x5410);
  ph = __byte_perm(__byte_perm(f0, f1, 0x0062), __byte_perm(f2, f3, 0x0062), 0x5410);
}

// A thread's activations for one step of BITS-bit codes, ready for that format's dot product:
// dot(codes) * unit = sum_c q_c * v_c, and sum = sum_c v_c (for the bias term).
template <int BITS>
struct Operand;

template <>
struct Operand<8> {
  static constexpr int C = 16;
  uint32_t pl[4], pm[4], ph[4];
  float unit, sum;
  __device__ __forceinline__ void set(const float (&v)[C]) {
    float mx = 0.f, sm = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      mx = fmaxf(mx, fabsf(v[c]));
      sm += v[c];
    }
    const int E = fixed_exponent(mx);
    const float sc = pow2f(22 - E);
    unit = pow2f(E - 22);
    sum = sm;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      byte_planes(__float2int_rn(v[4 * j] * sc), __float2int_rn(v[4 * j + 1] * sc),
                  __float2int_rn(v[4 * j + 2] * sc), __float2int_rn(v[4 * j + 3] * sc), pl[j],
                  pm[j], ph[j]);
  }
  __device__ __forceinline__ float dot(const uint4 *c) const {
    const uint32_t w[4] = {c[0].x, c[0].y, c[0].z, c[0].w};
    uint32_t dl = 0, dm = 0;
    int dh = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      dl = dp4a_uu(w[j], pl[j], dl);
      dm = dp4a_uu(w[j], pm[j], dm);
      dh = dp4a_us(w[j], ph[j], dh);
    }
    // dl, dm <= 16 * 255 * 255, so dm * 256 + dl < 2^31; |dh| <= 16 * 255 * 64
    return fmaf(static_cast<float>(dh), 65536.f, static_cast<float>(dm * 256u + dl));
  }
};

template <>
struct Operand<4> {
  static constexpr int C = 32;
  uint32_t el[4], em[4], eh[4];  // even codes of word j (low nibbles)
  uint32_t ol[4], om[4], oh[4];  // odd codes of word j (high nibbles, read as 16 * q)
  float unit, sum;
  __device__ __forceinline__ void set(const float (&v)[C]) {
    float mx = 0.f, sm = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      mx = fmaxf(mx, fabsf(v[c]));
      sm += v[c];
    }
    const int E = fixed_exponent(mx);
    const float sc = pow2f(22 - E);
    unit = pow2f(E - 26);  // the dot below is 16 * sum q f
    sum = sm;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      byte_planes(__float2int_rn(v[8 * j] * sc), __float2int_rn(v[8 * j + 2] * sc),
                  __float2int_rn(v[8 * j + 4] * sc), __float2int_rn(v[8 * j + 6] * sc), el[j],
                  em[j], eh[j]);
      byte_planes(__float2int_rn(v[8 * j + 1] * sc), __float2int_rn(v[8 * j + 3] * sc),
                  __float2int_rn(v[8 * j + 5] * sc), __float2int_rn(v[8 * j + 7] * sc), ol[j],
                  om[j], oh[j]);
    }
  }
  __device__ __forceinline__ float dot(const uint4 *c) const {
    const uint32_t w[4] = {c[0].x, c[0].y, c[0].z, c[0].w};
    uint32_t l0 = 0, m0 = 0, l1 = 0, m1 = 0;
    int h0 = 0, h1 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = w[j] & 0x0f0f0f0fu, hi = w[j] & 0xf0f0f0f0u;
      l0 = dp4a_uu(lo, el[j], l0);
      m0 = dp4a_uu(lo, em[j], m0);
      h0 = dp4a_us(lo, eh[j], h0);
      l1 = dp4a_uu(hi, ol[j], l1);
      m1 = dp4a_uu(hi, om[j], m1);
      h1 = dp4a_us(hi, oh[j], h1);
    }
    // 16 * sum q f: the even sums scaled by 16 join the odd ones (read as 16 * q already);
    // l, m <= 2 * 16 * 240 * 255, so m * 256 + l < 2^31
    const uint32_t l = l0 * 16u + l1, m = m0 * 16u + m1;
    const int h = h0 * 16 + h1;
    return fmaf(static_cast<float>(h), 65536.f, static_cast<float>(m * 256u + l));
  }
};

// 6-bit codes keep the float decoding above (three words per 16 codes do not fall on bytes).
template <>
struct Operand<6> {
  static constexpr int C = 64;
  float xs[C];
  float unit, sum;
  __device__ __forceinline__ void set(const float (&v)[C]) {
    float mx = 0.f, sm = 0.f;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      mx = fmaxf(mx, fabsf(v[c]));
      sm += v[c];
    }
    const int S = choose_shift(mx);
    unit = pow2f(S);
    sum = sm;
#pragma unroll
    for (int c = 0; c < C; ++c) xs[c] = v[c] * pow2f(149 - S - code_offset<6>(c));
  }
  __device__ __forceinline__ float dot(const uint4 *c) const {
    uint32_t m[C];
    step_masks<6>(c, m);
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < C; j += 4) {
      a0 = __ffma2_rn(make_float2(__uint_as_float(m[j + 0]), __uint_as_float(m[j + 1])),
                      make_float2(xs[j + 0], xs[j + 1]), a0);
      a1 = __ffma2_rn(make_float2(__uint_as_float(m[j + 2]), __uint_as_float(m[j + 3])),
                      make_float2(xs[j + 2], xs[j + 3]), a1);
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
  }
};

}  // namespace moe
