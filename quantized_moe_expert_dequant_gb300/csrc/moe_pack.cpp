// moe_pack.cpp -- host packing to and from the canonical layout of include/moe_decode.h:
// per row a little-endian bit stream, code c at bits [c*bits, c*bits + bits), LSB first.
// Affine 4- and 8-bit codes are in "two-kernel decode-MoE that beats gather_qmm" (Scope / flags);
// 6-bit and mixed widths are that page's planned next step (Next: step 2c).
#include <cstdint>
#include <cstring>

#include "moe_decode.h"

static bool bits_ok(int b) { return b == 4 || b == 6 || b == 8; }

extern "C" int moe_pack_codes(const uint8_t *codes, int64_t rows, int64_t cols, int32_t bits,
                              void *packed) {
  if (!codes || !packed || rows < 0 || cols < 0 || cols % 64) return MOE_ERR_INVALID_ARG;
  if (!bits_ok(bits)) return MOE_ERR_UNSUPPORTED;
  const uint32_t limit = 1u << bits;
  const int64_t rb = cols * bits / 8;
  uint8_t *dst = static_cast<uint8_t *>(packed);
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t *src = codes + r * cols;
    uint8_t *row = dst + r * rb;
    std::memset(row, 0, (size_t)rb);
    // accumulate codes into a 64-bit window and flush whole bytes, low bits first
    uint64_t acc = 0;
    int nbits = 0;
    int64_t o = 0;
    for (int64_t c = 0; c < cols; ++c) {
      if (src[c] >= limit) return MOE_ERR_INVALID_ARG;
      acc |= (uint64_t)src[c] << nbits;
      nbits += bits;
      while (nbits >= 8) {
        row[o++] = (uint8_t)(acc & 0xffu);
        acc >>= 8;
        nbits -= 8;
      }
    }
  }
  return MOE_OK;
}

extern "C" int moe_unpack_codes(const void *packed, int64_t rows, int64_t cols, int32_t bits,
                                uint8_t *codes) {
  if (!codes || !packed || rows < 0 || cols < 0 || cols % 64) return MOE_ERR_INVALID_ARG;
  if (!bits_ok(bits)) return MOE_ERR_UNSUPPORTED;
  const int64_t rb = cols * bits / 8;
  const uint8_t *src = static_cast<const uint8_t *>(packed);
  const uint32_t mask = (1u << bits) - 1;
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t *row = src + r * rb;
    uint64_t acc = 0;
    int nbits = 0;
    int64_t i = 0;
    for (int64_t c = 0; c < cols; ++c) {
      while (nbits < bits) {
        acc |= (uint64_t)row[i++] << nbits;
        nbits += 8;
      }
      codes[r * cols + c] = (uint8_t)(acc & mask);
      acc >>= bits;
      nbits -= bits;
    }
  }
  return MOE_OK;
}
