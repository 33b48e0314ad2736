// softmax_row.cuh -- the online-softmax update of one query row over one
// 128-key tile, shared by the forward kernels so that every forward path
// performs exactly the same arithmetic (dense and block-sparse results are
// then bitwise comparable).
//
// In base 2 ("Flash Attention: revolutionizing transformer efficiency",
// section "The Math Behind Flash Attention": softmax decomposition and
// merger): x_c = s_c * scale * log2(e); the running max m moves to
// max(m, max_c x_c); p_c = 2^(x_c - m_new); alpha = 2^(m_old - m_new); the
// caller updates l <- alpha l + sum_c p_c and O <- alpha O + P V. The max is
// exact, so the largest probability of a row is exactly 1 when it is rounded
// to 16 bits for the P V product (a lagging max rounds the dominant
// probability too: for sharp bf16 softmax that doubled the error of O).
#pragma once
#include "ptx.cuh"

namespace fa {

// Masks entries c >= limit of s (the 128 raw scores of this row) and
// moves the running max: returns -m_use, the offset of the exponent, and
// sets m_new and alpha = 2^(m - m_new).
__device__ __forceinline__ float softmax_max(float (&s)[128], int limit, float sl2, float m,
                                             float &m_new, float &alpha) {
  if (limit < 128) {
#pragma unroll
    for (int c = 0; c < 128; ++c)
      if (c >= limit) s[c] = -INFINITY;
  }
  float mx0 = fmax3(s[0], s[1], s[2]), mx1 = fmax3(s[3], s[4], s[5]);
  float mx2 = fmax3(s[6], s[7], s[8]), mx3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
  for (int c = 12; c < 124; c += 8) {
    mx0 = fmax3(mx0, s[c], s[c + 1]);
    mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
    mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
    mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
  }
  mx0 = fmax3(mx0, s[124], s[125]);
  mx1 = fmax3(mx1, s[126], s[127]);
  const float mxs = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
  m_new = fmaxf(m, mxs);
  const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
  alpha = ex2_approx(m - m_use);
  return -m_use;
}

// p_c = 2^(s_c * sl2 + nm) in place for columns [C0, C1) (a multiple of 4
// wide), added into the four partial sums acc in a fixed order.
template <int C0, int C1>
__device__ __forceinline__ void softmax_exp(float (&s)[128], float sl2, float nm, float (&acc)[4]) {
#pragma unroll
  for (int c = C0; c < C1; c += 4) {
    ffma2(s[c], s[c + 1], s[c], s[c + 1], sl2, sl2, nm, nm);
    ffma2(s[c + 2], s[c + 3], s[c + 2], s[c + 3], sl2, sl2, nm, nm);
    s[c] = ex2_approx(s[c]);
    s[c + 1] = ex2_approx(s[c + 1]);
    s[c + 2] = ex2_approx(s[c + 2]);
    s[c + 3] = ex2_approx(s[c + 3]);
    fadd2(acc[0], acc[1], acc[0], acc[1], s[c], s[c + 1]);
    fadd2(acc[2], acc[3], acc[2], acc[3], s[c + 2], s[c + 3]);
  }
}

__device__ __forceinline__ float softmax_sum(const float (&acc)[4]) {
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// The whole row update: on return s holds p (fp32); returns the tile's sum
// of p. Same arithmetic as softmax_max + softmax_exp<0, 128> + softmax_sum.
__device__ __forceinline__ float softmax_row(float (&s)[128], int limit, float sl2, float m,
                                             float &m_new, float &alpha) {
  const float nm = softmax_max(s, limit, sl2, m, m_new, alpha);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  softmax_exp<0, 128>(s, sl2, nm, acc);
  return softmax_sum(acc);
}

// Packs p (fp32) of columns c0 .. c0+31 into 16 16-bit pairs.
template <bool BF16>
__device__ __forceinline__ void pack_p32(const float (&s)[128], int c0, uint32_t (&hi)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) hi[i] = pack2<BF16>(s[c0 + 2 * i], s[c0 + 2 * i + 1]);
}

// O row chunk (32 fp32 values) *= alpha.
__device__ __forceinline__ void scale32(uint32_t (&o)[32], float alpha) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float x0, x1;
    fmul2(x0, x1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha);
    o[i] = __float_as_uint(x0);
    o[i + 1] = __float_as_uint(x1);
  }
}

}  // namespace fa
