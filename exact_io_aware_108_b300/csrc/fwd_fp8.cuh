// fwd_fp8.cuh -- V^T for the 8-bit forward.
//
// The kind::f8f6f4 product O += P V reads its B operand (V, N = d rows by
// K = keys) K-major: each row of the shared-memory tile holds 128 consecutive
// keys of one channel. This kernel writes V [B*Hkv][N][d] (e4m3 bytes) as
// V^T [B*Hkv][d][Npad] (Npad = N rounded up to 128; the pad is zero), one
// 128-key x 128-channel tile per CTA through shared memory: 16-byte loads of
// key rows, 16-byte stores of channel rows.
#pragma once
#include <cstdint>

namespace fa {

__global__ void __launch_bounds__(256) fwd_fp8_vt_kernel(const uint8_t *__restrict__ v, uint8_t *__restrict__ vt,
                                                         int N, int Npad) {
  constexpr int D = 128;
  __shared__ uint32_t tile[128][D / 4 + 1];  // [key][4 channels], padded row
  const int kt = blockIdx.x;
  const size_t head = blockIdx.y;
  const uint8_t *src = v + head * static_cast<size_t>(N) * D;
  uint8_t *dst = vt + head * static_cast<size_t>(D) * Npad;
  // load: 128 keys x 8 uint4 per key
  for (int i = threadIdx.x; i < 128 * 8; i += 256) {
    const int key = i >> 3, c16 = i & 7;
    const int n = kt * 128 + key;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (n < N) w = *reinterpret_cast<const uint4 *>(src + static_cast<size_t>(n) * D + c16 * 16);
    tile[key][c16 * 4 + 0] = w.x;
    tile[key][c16 * 4 + 1] = w.y;
    tile[key][c16 * 4 + 2] = w.z;
    tile[key][c16 * 4 + 3] = w.w;
  }
  __syncthreads();
  // store: channel c, keys 16g .. 16g+15 -> one uint4
  for (int i = threadIdx.x; i < D * 8; i += 256) {
    const int c = i >> 3, g = i & 7;
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t r = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t word = tile[16 * g + 4 * q + e][c >> 2];
        r |= ((word >> (8 * (c & 3))) & 0xFFu) << (8 * e);
      }
      out[q] = r;
    }
    *reinterpret_cast<uint4 *>(dst + static_cast<size_t>(c) * Npad + kt * 128 + 16 * g) =
        make_uint4(out[0], out[1], out[2], out[3]);
  }
}

}  // namespace fa
