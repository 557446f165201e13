// Test-only shim: exposes ATen's header-only Philox4_32 engine (used as a
// black box) through a C function, so the tests can cross-check the two
// independent Philox4x32-10 implementations of this repository against a
// library implementation.
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdint>

extern "C" void aten_philox_words(uint64_t seed, uint64_t subsequence, uint64_t offset,
                                  uint32_t out[4]) {
  at::Philox4_32 engine(seed, subsequence, offset);
  for (int i = 0; i < 4; ++i) out[i] = engine();
}
