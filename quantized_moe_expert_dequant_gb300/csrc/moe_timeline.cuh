// moe_timeline.cuh -- per-CTA, per-layer time stamps of the column-split kernel.
//
// Compiled in only when MOE_TIMELINE is defined (the library's timeline build,
// libmoe_decode_timeline.so); the product build contains none of it.  Slot k of (CTA, layer) in
// StackParams::tl receives clock64() (k < kTlClockPoints, the SM's cycle counter: differences
// within one CTA) or %globaltimer in ns (k >= kTlClockPoints: alignment across CTAs) when the
// kernel passes point k.  Points 0..15 are listed where the column-split kernel stamps them;
// for ring stage i < kTlStages of the layer, 16 + i is when consumer warp 0 found it full,
// 28 + i when the producer issued it and 40 + i when consumer warp 0 began to wait for it.
#pragma once

#include <cstdint>

namespace moe {

constexpr int kTlPoints = 64;
constexpr int kTlClockPoints = 56;
constexpr int kTlStages = 12;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

#ifdef MOE_TIMELINE
// Stamps from inside shared phase code: the kernel points these at the current (CTA, layer) row
// (consumer thread 0, producer lane 0) and records the ring's stage count at the layer's start.
__device__ __forceinline__ unsigned long long *&tl_hook_row() {
  __shared__ unsigned long long *row;
  return row;
}
__device__ __forceinline__ unsigned long long *&tl_hook_row_p() {
  __shared__ unsigned long long *row;
  return row;
}
__device__ __forceinline__ int &tl_stage_base() {
  __shared__ int base;
  return base;
}
__device__ __forceinline__ int &tl_stage_base_p() {
  __shared__ int base;
  return base;
}
#define MOE_TL_AT(row, k)                                                                    \
  do {                                                                                       \
    if ((row) != nullptr)                                                                    \
      (row)[k] = (k) < ::moe::kTlClockPoints ? static_cast<unsigned long long>(clock64())     \
                                             : ::moe::global_ns();                           \
  } while (0)
#define MOE_TL_ROW(tl, L, l) \
  ((tl) != nullptr ? (tl) + (static_cast<size_t>(blockIdx.x) * (L) + (l)) * ::moe::kTlPoints : nullptr)
#define MOE_TL_HOOK(k) MOE_TL_AT(::moe::tl_hook_row(), k)
#define MOE_TL_SET_HOOK(row) (::moe::tl_hook_row() = (row))
#define MOE_TL_SET_HOOK_P(row) (::moe::tl_hook_row_p() = (row))
#define MOE_TL_STAGE_BASE(used) (::moe::tl_stage_base() = (used))
#define MOE_TL_STAGE_BASE_P(used) (::moe::tl_stage_base_p() = (used))
#define MOE_TL_STAGE_C(used)                                                                 \
  do {                                                                                       \
    const int i_ = (used) - ::moe::tl_stage_base();                                          \
    if (i_ >= 0 && i_ < ::moe::kTlStages) MOE_TL_AT(::moe::tl_hook_row(), 16 + i_);          \
  } while (0)
#define MOE_TL_STAGE_WAIT(used)                                                              \
  do {                                                                                       \
    const int i_ = (used) - ::moe::tl_stage_base();                                          \
    if (i_ >= 0 && i_ < ::moe::kTlStages) MOE_TL_AT(::moe::tl_hook_row(), 40 + i_);          \
  } while (0)
#define MOE_TL_STAGE_P(used)                                                                 \
  do {                                                                                       \
    const int i_ = (used) - ::moe::tl_stage_base_p();                                        \
    if (i_ >= 0 && i_ < ::moe::kTlStages) MOE_TL_AT(::moe::tl_hook_row_p(), 28 + i_);        \
  } while (0)
#else
#define MOE_TL_AT(row, k) ((void)0)
#define MOE_TL_ROW(tl, L, l) (static_cast<unsigned long long *>(nullptr))
#define MOE_TL_HOOK(k) ((void)0)
#define MOE_TL_SET_HOOK(row) ((void)0)
#define MOE_TL_SET_HOOK_P(row) ((void)0)
#define MOE_TL_STAGE_BASE(used) ((void)0)
#define MOE_TL_STAGE_BASE_P(used) ((void)0)
#define MOE_TL_STAGE_C(used) ((void)0)
#define MOE_TL_STAGE_WAIT(used) ((void)0)
#define MOE_TL_STAGE_P(used) ((void)0)
#endif

}  // namespace moe
