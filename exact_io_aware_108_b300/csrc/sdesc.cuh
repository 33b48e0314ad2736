// sdesc.cuh -- shared-memory matrix descriptors of tcgen05.mma operands
// (128-byte swizzle), usable on the host too so that the arithmetic the
// issue loops rely on can be checked on the CPU (tests/sdesc_check.cu).
#pragma once
#include <cstdint>

namespace fa {

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   K-major operand (rows of 64 16-bit elements = 128 B, 8-row atoms of 1 KB):
//     lbo unused (16), sbo = 1024 (next 8-row group); step K by 16 elements
//     by adding 32 bytes to the start address.
//   MN-major operand (rows = K index, 64 MN elements per 128-B row):
//     lbo = byte distance between 64-element MN chunks, sbo = 1024 (next
//     8 K-rows); step K by 16 by adding 2048 bytes.
// Bits: [0,14) start>>4, [16,30) lbo>>4, [32,46) sbo>>4, [46,48) version 1,
// [49,52) base offset 0 (atoms are 1 KB aligned), [61,64) layout 2 = SW128.
__host__ __device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// The same descriptor as two 32-bit words, for issue loops that step the
// start address: lo = start >> 4 | (LBO >> 4) << 16, hi = SBO >> 4 | the
// version and swizzle bits. The descriptor of start + off (off a multiple of
// 16) is {lo + off / 16, hi}: the start-address field is 14 bits wide and
// shared-memory addresses stay below 2^18, so the add never carries into
// the LBO field.
__host__ __device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
}  // namespace fa
