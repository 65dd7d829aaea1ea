// Host-side check of the kernels' division by launch-invariant divisors
// (kda::make_fastdiv / kda::fdiv): for every divisor 1..4096, every 2^k - 1,
// 2^k, 2^k + 1 below 2^31 and 16000 random divisors, the quotient of edge
// numerators (0, 1, d - 1, d, d + 1, 2d - 1, multiples of d and their
// predecessors, 2^30 - 1, 2^30, 2^31 - 2, 2^31 - 1) and of random numerators
// below 2^31 must equal the exact integer quotient.  Prints "ok <count>".
#include <cstdint>
#include <cstdio>

#include "kda_kernel.cuh"

int main() {
  uint64_t state = 0x9E3779B97F4A7C15ull;  // xorshift64
  auto rnd = [&]() {
    state ^= state << 13;
    state ^= state >> 7;
    state ^= state << 17;
    return state;
  };
  long long checked = 0;
  auto check = [&](uint32_t x, uint32_t d, const kda::FastDiv& f) {
    if (x > 0x7fffffffu) return true;
    ++checked;
    if (kda::fdiv(x, f) == x / d) return true;
    std::printf("FAIL d=%u x=%u got %u\n", d, x, kda::fdiv(x, f));
    return false;
  };
  for (int trial = 0; trial < 4096 + 93 + 16000; ++trial) {
    uint32_t d;
    if (trial < 4096) {
      d = trial + 1;
    } else if (trial < 4096 + 93) {
      const int k = (trial - 4096) / 3, o = (trial - 4096) % 3 - 1;
      const uint64_t dd = (1ull << k) + o;
      if (dd == 0 || dd >= (1ull << 31)) continue;
      d = static_cast<uint32_t>(dd);
    } else {
      d = static_cast<uint32_t>(rnd() % 0x7fffffffull) + 1;
    }
    const kda::FastDiv f = kda::make_fastdiv(d);
    const uint32_t edge[] = {0u, 1u, d - 1, d, d + 1, 2 * d - 1, 0x3fffffffu, 0x40000000u,
                             0x7ffffffeu, 0x7fffffffu};
    for (uint32_t x : edge)
      if (!check(x, d, f)) return 1;
    for (int r = 0; r < 64; ++r) {
      uint32_t x;
      if (r < 16) {  // a multiple of d or its predecessor
        const uint64_t q = rnd() % (0x7fffffffull / d + 1);
        const uint64_t v = q * d + ((r & 1) ? d - 1 : 0);
        if (v > 0x7fffffffull) continue;
        x = static_cast<uint32_t>(v);
      } else {
        x = static_cast<uint32_t>(rnd() & 0x7fffffffu);
      }
      if (!check(x, d, f)) return 1;
    }
  }
  std::printf("ok %lld\n", checked);
  return 0;
}
