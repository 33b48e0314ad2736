// Host check of the descriptor-word arithmetic the MMA issue loops use: a
// shared-memory matrix descriptor split into a low word (start address and
// leading byte offset) and a constant high word (stride byte offset, version,
// 128-byte swizzle), stepped through a tile by adding offset / 16 to the low
// word. For every 16-byte aligned start address a of one CTA's shared window
// (below 2^18 bytes: at most 227 KB of dynamic shared memory plus the 1 KB the
// hardware reserves) and every aligned offset that stays inside it, the
// stepped words must equal the descriptor built from a + offset. The fields
// are also decoded back from a full descriptor and compared with the
// addresses they were built from.
#include <cstdio>
#include <cstdint>

#include "sdesc.cuh"

using fa::sdesc_hi;
using fa::sdesc_lo;
using fa::sdesc_sw128;

static int fail(const char *what, uint32_t a, uint32_t off, uint32_t lbo) {
  std::printf("mismatch (%s): start %u offset %u lbo %u\n", what, a, off, lbo);
  return 1;
}

int main() {
  const uint32_t kWindow = 1u << 18;
  const uint32_t lbos[2] = {16u, 16384u};  // K-major operands; MN-major operands of 64-element chunks
  for (uint32_t li = 0; li < 2; ++li) {
    const uint32_t lbo = lbos[li];
    const uint64_t hi = static_cast<uint64_t>(sdesc_hi(1024)) << 32;
    for (uint32_t a = 0; a < kWindow; a += 16) {
      const uint32_t lo = sdesc_lo(a, lbo);
      if ((hi | lo) != sdesc_sw128(a, lbo, 1024)) return fail("split", a, 0, lbo);
      // every offset from a that stays in the window, in 16-byte steps
      for (uint32_t off = 16; a + off < kWindow; off += 16)
        if ((hi | (lo + off / 16)) != sdesc_sw128(a + off, lbo, 1024)) return fail("step", a, off, lbo);
    }
  }
  // decoded fields of a full descriptor
  for (uint32_t a = 0; a < kWindow; a += 1040) {
    const uint32_t a16 = a & ~15u;
    const uint64_t d = sdesc_sw128(a16, 16384, 1024);
    const uint32_t start = static_cast<uint32_t>(d & 0x3FFFu) << 4;
    const uint32_t lbo = static_cast<uint32_t>((d >> 16) & 0x3FFFu) << 4;
    const uint32_t sbo = static_cast<uint32_t>((d >> 32) & 0x3FFFu) << 4;
    const uint32_t version = static_cast<uint32_t>((d >> 46) & 3u);
    const uint32_t base_off = static_cast<uint32_t>((d >> 49) & 7u);
    const uint32_t layout = static_cast<uint32_t>(d >> 61);
    if (start != a16 || lbo != 16384u || sbo != 1024u || version != 1u || base_off != 0u || layout != 2u)
      return fail("fields", a16, 0, 16384u);
    // bits outside the fields stay clear
    const uint64_t fields = 0x3FFFull | (0x3FFFull << 16) | (0x3FFFull << 32) | (3ull << 46) | (7ull << 49) |
                            (7ull << 61);
    if (d & ~fields) return fail("reserved bits", a16, 0, 16384u);
  }
  std::printf("ok\n");
  return 0;
}
