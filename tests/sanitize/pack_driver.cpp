// pack_driver.cpp -- runs the library's host packer (moe_pack_codes / moe_unpack_codes,
// quantized_moe_expert_dequant_gb300/csrc/moe_pack.cpp) in a build with AddressSanitizer and
// UndefinedBehaviorSanitizer (tests/test_sanitizers.py compiles the two together): round trips at
// every code width with buffers of exactly the packed size, and the argument checks.  Any
// out-of-bounds access or undefined operation aborts the run.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "moe_decode.h"

#define CHECK(c)                                                      \
  do {                                                                \
    if (!(c)) {                                                       \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      return 1;                                                       \
    }                                                                 \
  } while (0)

int main() {
  uint64_t s = 0x9ACCull;
  auto next = [&s]() {
    s = s * 6364136223846793005ull + 1442695040888963407ull;
    return static_cast<uint32_t>(s >> 32);
  };
  for (int bits : {4, 6, 8}) {
    for (int64_t rows : {1, 3, 7}) {
      for (int64_t cols : {64, 192, 448}) {
        // heap buffers of exactly the sizes the format needs, so that ASan sees any overrun
        uint8_t *codes = static_cast<uint8_t *>(std::malloc(rows * cols));
        uint8_t *packed = static_cast<uint8_t *>(std::malloc(rows * cols * bits / 8));
        uint8_t *back = static_cast<uint8_t *>(std::malloc(rows * cols));
        CHECK(codes && packed && back);
        for (int64_t i = 0; i < rows * cols; ++i) codes[i] = next() & ((1u << bits) - 1u);
        CHECK(moe_pack_codes(codes, rows, cols, bits, packed) == MOE_OK);
        CHECK(moe_unpack_codes(packed, rows, cols, bits, back) == MOE_OK);
        for (int64_t i = 0; i < rows * cols; ++i) CHECK(back[i] == codes[i]);
        codes[rows * cols - 1] = static_cast<uint8_t>(1u << bits);  // out of range: refused
        if (bits < 8) CHECK(moe_pack_codes(codes, rows, cols, bits, packed) == MOE_ERR_INVALID_ARG);
        std::free(codes);
        std::free(packed);
        std::free(back);
      }
    }
  }
  uint8_t one[64] = {0};
  uint8_t out[64];
  CHECK(moe_pack_codes(one, 1, 64, 5, out) == MOE_ERR_UNSUPPORTED);
  CHECK(moe_pack_codes(one, 1, 65, 4, out) == MOE_ERR_INVALID_ARG);
  CHECK(moe_pack_codes(nullptr, 1, 64, 4, out) == MOE_ERR_INVALID_ARG);
  CHECK(moe_unpack_codes(out, -1, 64, 4, one) == MOE_ERR_INVALID_ARG);
  CHECK(moe_pack_codes(one, 0, 64, 4, out) == MOE_OK);  // no rows: nothing written
  std::printf("packer sanitizer run ok\n");
  return 0;
}
