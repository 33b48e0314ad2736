// bwd_kernel.cuh -- backward attention kernels for sm_103a.
//
// The backward recomputes the probabilities tile by tile from Q, K and the
// forward's log-sum-exp instead of storing them ("Flash Attention:
// revolutionizing transformer efficiency", key idea 2, Recomputation). For
// a key tile j and a query tile i, with P = exp(scale Q_i K_j^T - LSE_i):
//   dV_j += P^T dO_i            dP = dO_i V_j^T
//   dS    = P o (dP - D_i),     D_i = rowsum(dO_i o O_i)
//   dK_j += scale dS^T Q_i      dQ_i += scale dS K_j
//
// Precision. All five products take fp16 operands, whatever the input type:
// P and dS are rounded to fp16 (11 significant bits) before their products,
// not to bf16 (8 bits). With sharp bf16 softmax at d = 128 (logit std 4) the
// bf16 rounding of dS alone puts rare dQ and dK elements past a 2e-2
// absolute error (dS rows sum to zero, so a dQ element can be much smaller
// than the terms whose rounding errors it collects). For bf16 inputs the
// operands are converted to fp16:
//   Q, K, V   unscaled. The conversion is exact for 2^-17 <= |x| <= 65504
//             (smaller values are rounded to fp16's subnormal grid, an
//             absolute change of at most 2^-25); larger values are clamped
//             to 65504 and reported through the device error word.
//   dO        scaled by 2^-e_do, e_do chosen from max |dO| so that the
//             largest element lands in [2^14, 2^15): gradients of any
//             magnitude keep fp16's full precision. dP and dV are
//             multiplied back by 2^e_do in fp32 (exact).
//   dS        stored as dS * scale * 2^-e_s, one e_s per call from the
//             bound |dS| <= |dP| + |D| <= d max|dO| max|V| + max|D| so the
//             largest possible value stays below 2^15; dK is multiplied back
//             by 2^e_s in its epilogue, dQ when its fp32 accumulator is
//             converted to 16 bits (both exact).
// For fp16 inputs only the dS scaling applies.
//
// Kernels:
//   bwd_pre_kernel   -D_i and -LSE_i * log2(e) per query row (padded
//                    to whole 128-row tiles; pad rows get D = 0, LSE = +inf so
//                    P = 0), zeroes the fp32 dQ accumulator, and records
//                    max |dO|, max |D| and max |V| for the scaling above. D_i = dO_i .
//                    O_i uses O plus its rounding residual when the forward
//                    wrote one: with bf16 O alone the rounding of O moves D_i
//                    by up to ~0.05 at d = 128, which reaches dQ and dK.
//   bwd_cvt_kernel   (bf16 inputs) Q -> fp16 and dO -> fp16 * 2^-e_do into
//                    the workspace, read by the main kernel's tensor maps.
//   bwd_main_kernel  persistent, one CTA per SM; its work items are the
//                    128-key tiles j of each (batch, key/value head). Per
//                    item K_j, V_j stay in shared memory (converted there to
//                    fp16 for bf16 inputs), dK_j and dV_j stay in TMEM, and the
//                    CTA loops over the query tiles that see key tile j, of
//                    every query head that reads this key/value head (one
//                    head unless the attention is grouped-query).
//                    The scores are computed transposed (keys on TMEM lanes)
//                    so P^T and dS^T are row-local to one thread per key.
//   bwd_dq_kernel    dQ accumulator (fp32) -> dQ (fp16/bf16).
//
// Main-kernel roles (512 threads; setmaxnreg moves registers from
// warpgroup 0 to the other three):
//   warp 0 lane 0   work items (from the counter, handed to the other roles
//                   through two shared-memory slots); TMA: K_j, V_j once per
//                   item; Q_i, dO_i tiles and the LSE/D rows of query tile i
//                   through a two-stage ring.
//   warp 1          TMEM allocation; lane 0 issues every tcgen05.mma.
//   warpgroups 1, 2 at the start of an item: K_j, V_j -> fp16 in place (bf16
//                   inputs).
//   warpgroups 1, 2 one 64-query half h of the tile each: P^T -> TMEM
//                   (fp16), dS^T -> shared memory (fp16, scale and 2^-e_s
//                   folded in, computed from the fp32 P). A thread holds 4
//                   keys x 16 queries (16-lane TMEM shapes), so it reads only
//                   16 of the half's per-query LSE and D values; at the end
//                   of an item warpgroup 1 writes dK, warpgroup 2 writes dV
//                   (one key row per thread).
//   warpgroup 3     reads the dQ partial from TMEM and adds it to the fp32
//                   accumulator (d = 128: thread r owns head-dim
//                   channel r of the transposed partial; d = 64: thread r
//                   owns query r).
// The MMA issue order per query tile i is dP_i, dV_i, dQ_i, S_{i+1}, dK_i
// for d = 128: the next score tile is computed before dK_i, so the P phase
// of tile i+1 overlaps the dK_i product and the dQ_i read-out, while the Q
// stage of tile i+1 still has most of a tile's time to land (its load
// latency grows to several thousand cycles under the dQ reduction traffic).
// For d = 64 (smaller tiles, shorter loads) S_{i+1} goes right after dV_i.
// TMEM columns: dK [0,D), dV [D,2D), S^T [2D,2D+128) (half h's P^T aliases
// columns [64h, 64h+32) of it), dP^T [2D+128, 2D+256); the dQ partial reuses
// the dP^T columns for d = 128 and has its own 64 columns for d = 64.
#pragma once
#include "common.cuh"
#include "schedule.cuh"

namespace fa {

struct BwdArgs {
  void *dq, *dk, *dv;
  const void *o, *dout;
  const void *o_res;  // rounding residual of O (same 16-bit type) or null
  const float *lse;
  float *lse_l2;    // [BH, nqt*128]  -LSE * log2(e)
  float *delta;     // [BH, nqt*128]  -D
  float *dq_acc;    // [BH, nqt*128, D]
  const int32_t *kv_len;
  const uint8_t *block_mask;
  // bf16 inputs: the fp16 copies of Q and of dO * 2^-e_do ([B*H, N, D],
  // written by bwd_cvt_kernel) and the sources they are made from
  const void *q;
  void *q16, *do16;
  // [0] max |dO|, [1] max |D|, [2] max |V| as fp32 bit patterns
  // (non-negative floats order like their bits), zeroed before
  // bwd_pre_kernel; [3] the dS exponent e_s, written by the main kernel for
  // the dQ conversion
  unsigned int *stats;
  const void *v;     // V, read by bwd_pre_kernel for max |V|
  long long n_v16;   // 16-byte chunks of V
  const void *k;      // K, prefetched into L2 one work item ahead
  unsigned int *work;  // work-item counter of the main kernel, zeroed before its launch
  int n_items;         // work items: B * Hkv * nkt
  int H, N, nqt, nkt;
  int hgroup;    // heads per scheduling group (causal launch order, see below)
  int Hkv;       // key/value heads (grouped-query attention: H = Hkv * kv_group)
  int kv_group;  // query heads per key/value head
  float scale, scale_log2;
  // [B*H] index of query head g of the group that reads key/value head bkv
  __device__ __forceinline__ int q_head(int bkv, int g) const { return q_head_of(bkv, g, H, Hkv); }
};

// 1-D bulk copy global -> shared, completion as transaction bytes on bar.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// 2^e as an fp32 value, e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// e such that x * 2^-e lies in [2^(top-1), 2^top) for finite x > 0; 0
// otherwise. Clamped to [-120, 120] so both 2^e and 2^-e are normal floats.
__device__ __forceinline__ int scale_exponent(float x, int top) {
  if (!(x > 0.f) || !(x <= 3.0e38f)) return 0;
  int e;
  frexpf(x, &e);  // x = m 2^e, m in [0.5, 1): x < 2^e
  e -= top;
  return e < -120 ? -120 : (e > 120 ? 120 : e);
}

// Exponent of the dO scaling: max |dO| * 2^-e_do in [2^14, 2^15).
__device__ __forceinline__ int do_exponent(const unsigned int *stats) {
  return scale_exponent(__uint_as_float(stats[0]), 15);
}

// Exponent of the dS scaling (dS is stored as dS * scale * 2^-e_s): from
// |dS| <= |dP| + |D| <= d max|dO| max|V| + max|D|, the largest possible
// stored value stays below 2^15. One value for the whole call, so the fp32
// dQ accumulator holds dQ * 2^-e_s and the conversion to 16 bits multiplies
// it back. Clamped values are at most 65504, so the bound stays finite for
// finite inputs.
__device__ __forceinline__ int ds_exponent(const unsigned int *stats, float scale, int d) {
  const float amax_do = __uint_as_float(stats[0]), amax_d = __uint_as_float(stats[1]);
  const float amax_v = fminf(__uint_as_float(stats[2]), 65504.f);
  return scale_exponent(scale * (static_cast<float>(d) * amax_do * amax_v + amax_d), 15);
}

// Eight bf16 values (16 bytes) -> eight fp16 values, rounded to nearest and
// clamped to +-65504; amax takes the largest magnitude seen.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w, float &amax) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float lo = __uint_as_float(in[k] << 16), hi = __uint_as_float(in[k] & 0xFFFF0000u);
    amax = fmax3(amax, fabsf(lo), fabsf(hi));
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(out[k]) : "f"(hi), "f"(lo));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Largest magnitude of eight 16-bit values.
template <bool BF16>
__device__ __forceinline__ float amax16x8(uint4 w) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) m = fmax3(m, fabsf(unpack_lo<BF16>(in[k])), fabsf(unpack_hi<BF16>(in[k])));
  return m;
}

// Block-wide max of a non-negative value, then one atomicMax on its bits.
__device__ __forceinline__ void block_max_to(unsigned int *dst, float v, float *red) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
    atomicMax(dst, __float_as_uint(m));
  }
}

// ----------------------------------------------------------------- pre
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdArgs a, long long rows_pad) {
  constexpr int LPR = D / 8;         // lanes per row (8 elements each)
  constexpr int RPW = 32 / LPR;      // rows per warp step
  __shared__ float red[3][8];
  const int lane = threadIdx.x & 31;
  const int sub = lane % LPR, grp = lane / LPR;
  const long long tile_rows = static_cast<long long>(a.nqt) * 128;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long w0 = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  float amax_do = 0.f, amax_d = 0.f;
  for (long long base = w0 * RPW; base < rows_pad; base += warps * RPW) {
    const long long row = base + grp;
    const bool live = row < rows_pad;
    float acc = 0.f;
    long long bh = 0, i = 0;
    if (live) {
      bh = row / tile_rows;
      i = row % tile_rows;
      if (i < a.N) {
        const size_t off = (static_cast<size_t>(bh) * a.N + i) * D + sub * 8;
        const uint4 o4 = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.o) + off);
        const uint4 g4 =
            *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.dout) + off);
        uint4 r4 = make_uint4(0u, 0u, 0u, 0u);
        if (a.o_res != nullptr)
          r4 = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.o_res) + off);
        const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w};
        const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
        const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc = fmaf(unpack_lo<BF16>(ow[k]) + unpack_lo<BF16>(rw[k]), unpack_lo<BF16>(gw[k]), acc);
          acc = fmaf(unpack_hi<BF16>(ow[k]) + unpack_hi<BF16>(rw[k]), unpack_hi<BF16>(gw[k]), acc);
        }
        amax_do = fmaxf(amax_do, amax16x8<BF16>(g4));
      }
      float4 *z = reinterpret_cast<float4 *>(a.dq_acc + row * D + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int s = LPR / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (live && sub == 0) {
      // stored negated so the main kernel forms P = 2^(s * scale * log2 e +
      // nl) and dS = P * (dP * scale - scale * D) with one packed FMA per
      // pair (the scale is applied there: the prepare phase does not take it)
      a.delta[row] = -acc;
      amax_d = fmaxf(amax_d, fabsf(acc));
      float nl = -INFINITY;
      if (i < a.N) {
        const float l = a.lse[static_cast<size_t>(bh) * a.N + i];
        if (l != -INFINITY) nl = -l * 1.4426950408889634f;
      }
      a.lse_l2[row] = nl;
    }
  }
  // max |V| (bf16 V is converted to fp16 by the main kernel; either type
  // needs it for the dS exponent)
  float amax_v = 0.f;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < a.n_v16;
       g += static_cast<long long>(gridDim.x) * blockDim.x)
    amax_v = fmaxf(amax_v, amax16x8<BF16>(reinterpret_cast<const uint4 *>(a.v)[g]));
  block_max_to(a.stats + 0, amax_do, red[0]);
  block_max_to(a.stats + 1, amax_d, red[1]);
  block_max_to(a.stats + 2, amax_v, red[2]);
}

// ----------------------------------------------------------------- fp16 copies
// bf16 inputs: Q -> fp16 (unscaled) and dO -> fp16 * 2^-e_do, 16 bytes per
// thread step, grid-stride over [B*H, N, D] (n16 groups of 8 elements).
__global__ void __launch_bounds__(256) bwd_cvt_kernel(const BwdArgs a, long long n16) {
  const float f_do = exp2i(-do_exponent(a.stats));
  float amax_q = 0.f;
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n16;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 q = reinterpret_cast<const uint4 *>(a.q)[g];
    reinterpret_cast<uint4 *>(a.q16)[g] = bf16x8_to_f16x8(q, amax_q);
    const uint4 w = reinterpret_cast<const uint4 *>(a.dout)[g];
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(in[k] << 16) * f_do, hi = __uint_as_float(in[k] & 0xFFFF0000u) * f_do;
      asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(out[k]) : "f"(hi), "f"(lo));
    }
    reinterpret_cast<uint4 *>(a.do16)[g] = make_uint4(out[0], out[1], out[2], out[3]);
  }
  if (amax_q > 65504.f) atomicOr(&g_fa_device_error, kDevErrRange);
}

// ----------------------------------------------------------------- dq convert
// dQ accumulator (fp32, dQ * 2^-e_s as the main kernel recorded e_s) -> dQ
// (16-bit). Eight channels per thread (two 16-byte loads, one 16-byte
// store); heads run along grid.y and rows along grid.x, so the per-head
// padding of the accumulator's rows needs no division.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const BwdArgs a, int BH) {
  constexpr int kLanes = D / 8;          // threads per row
  constexpr int kRows = 256 / kLanes;    // rows per block step
  const long long tile_rows = static_cast<long long>(a.nqt) * 128;
  const float u_s = exp2i(static_cast<int>(a.stats[3]));
  const int sub = static_cast<int>(threadIdx.x) % kLanes, r0 = static_cast<int>(threadIdx.x) / kLanes;
  for (int bh = static_cast<int>(blockIdx.y); bh < BH; bh += static_cast<int>(gridDim.y)) {
    const float *acc = a.dq_acc + static_cast<size_t>(bh) * tile_rows * D + sub * 8;
    uint16_t *out = static_cast<uint16_t *>(a.dq) + static_cast<size_t>(bh) * a.N * D + sub * 8;
    for (int i = static_cast<int>(blockIdx.x) * kRows + r0; i < a.N; i += static_cast<int>(gridDim.x) * kRows) {
      const float4 *src = reinterpret_cast<const float4 *>(acc + static_cast<size_t>(i) * D);
      const float4 v0 = src[0], v1 = src[1];
      uint4 o;
      o.x = pack2<BF16>(v0.x * u_s, v0.y * u_s);
      o.y = pack2<BF16>(v0.z * u_s, v0.w * u_s);
      o.z = pack2<BF16>(v1.x * u_s, v1.y * u_s);
      o.w = pack2<BF16>(v1.z * u_s, v1.w * u_s);
      *reinterpret_cast<uint4 *>(out + static_cast<size_t>(i) * D) = o;
    }
  }
}

// ----------------------------------------------------------------- main
template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kKB = D / 64;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;         // 2 stages
  static constexpr int kdOOff = kQOff + 2 * kTileBytes;    // 2 stages
  static constexpr int kdSOff = kdOOff + 2 * kTileBytes;   // 128 keys x 128 queries bf16
  static constexpr int kLseOff = kdSOff + 32768;           // 2 stages x 128 fp32
  static constexpr int kDeltaOff = kLseOff + 1024;         // 2 stages x 128 fp32
  static constexpr int kBarOff = kDeltaOff + 1024;
  // Barriers. Per query tile (phase = the CTA's running tile count): Q/dO
  // stage full/empty, S^T, dP^T, P^T halves, dV issued, dS^T, dQ full/empty,
  // dS^T read. Per work item (phase = the CTA's running count of items with
  // work): K landed, V landed, K and V in fp16 (256 arrivals), all products
  // done, dK/dV read out of TMEM (256 arrivals). Item slots: full (the
  // producer) and empty (13 consumer arrivals: the MMA thread and the warps
  // of the three compute warpgroups). kBEND: the MMA thread's final drain.
  static constexpr int kBKL = 0, kBQF = 1 /* x2 */, kBQE = 3 /* x2 */, kBSF = 5, kBDPF = 6,
                       kBPR = 7 /* x2 */, kBDV = 9, kBDSR = 10, kBDQF = 11, kBDQE = 12, kBFIN = 13,
                       kBDSF = 14, kBCK = 15, kBCV = 16, kBVL = 17, kBACC = 18, kBITF = 19 /* x2 */,
                       kBITE = 21 /* x2 */, kBEND = 23, kNumBars = 24;
  static constexpr int kItemConsumers = 1 + 12;
  // d = 128: the dQ partial is computed transposed (dQ^T = K^T dS^T, TMEM
  // lane = head-dim channel, column = query) so one warp's reduction into
  // the fp32 accumulator covers 32 consecutive channels of a row: a whole
  // 128-byte line per instruction instead of 32 scattered 16-byte pieces.
  static constexpr bool kDqT = (D == 128);
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // misc: [0] TMEM address, [1] abort flag, [2..3] work item slots
  static constexpr int kSmemBytes = kMiscOff + 16;
  static constexpr uint32_t kColDK = 0, kColDV = D, kColS = 2 * D, kColDP = 2 * D + 128;
  static constexpr uint32_t kColDQ = kDqT ? kColDP : 2 * D + 256;
  static constexpr uint32_t kTmemCols = 512;
  // MMA order: S_{i+1} right after dV_i (d = 64) or after dQ_i (d = 128,
  // where the Q load of tile i+1 needs the longer window); both measured.
  static constexpr bool kSAfterDV = (D == 64);
  // d = 128: the two dO stages and the dS^T buffer are three 32 KB buffers
  // in a row whose roles rotate: dO of tile u goes to buffer u % 3 and dS^T
  // of tile u to buffer (u + 2) % 3, the one that held dO of tile u - 1
  // (its readers, dP and dV of tile u - 1, are done once dP of tile u is:
  // a commit covers every earlier product). So writing dS^T never waits for
  // the previous tile's dQ and dK products, which read the third buffer;
  // a buffer goes dO(u) -> dS^T(u + 1) -> dO(u + 3), refilled once dK of
  // tile u + 1 is done, which is the Q stage's release. (At d = 64 a dO tile
  // is 16 KB and dS^T 32 KB, so d = 64 keeps one dS^T buffer.)
  static constexpr bool kRotDS = (D == 128);
  // byte offsets of the dO tile and of the dS^T buffer of running tile u
  __device__ static __forceinline__ uint32_t do_off(int u) {
    return kdOOff + (kRotDS ? static_cast<unsigned>(u) % 3u : static_cast<unsigned>(u) & 1u) * kTileBytes;
  }
  __device__ static __forceinline__ uint32_t ds_off(int u) {
    return kRotDS ? kdOOff + (static_cast<unsigned>(u) + 2u) % 3u * kTileBytes : kdSOff;
  }
  static_assert(kColDP + 128 <= kTmemCols && kColDQ + (kDqT ? 128 : D) <= kTmemCols, "TMEM budget");
  static_assert(!kRotDS || (kTileBytes == 32768 && kdSOff == kdOOff + 2 * kTileBytes), "rotation layout");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // setmaxnreg split: launch with 128 registers x 512 threads; warpgroup 0
  // (producer, MMA issuer) gives registers to the three compute warpgroups.
  static constexpr int kThreads = 512;
  static constexpr int kLaunchRegs = 128, kRegsLow = 56, kRegsHigh = 152;
  static_assert(kRegsLow * 128 + kRegsHigh * 384 <= kLaunchRegs * kThreads, "register split");
};

// Next kept query tile >= from for key tile kt (block-sparse column scan).
__device__ __forceinline__ int next_kept(const uint8_t *mask, int nkt, int nqt, int kt, int from) {
  int i = from;
  while (i < nqt && mask[static_cast<size_t>(i) * nkt + kt] == 0) ++i;
  return i;
}

// Work item of the backward: one key tile of one key/value head, and the
// (query head, query tile) pairs of its group that see it.
struct BwdItem {
  int bkv;      // [B*Hkv] key/value head
  int kt;       // key tile
  int kvl;      // keys of this batch entry (kv_len clamped to [0, N])
  int n_iter;   // (query head, query tile) pairs walked
  int q_first;  // first query tile walked for each query head
};

template <bool CAUSAL, bool SPARSE>
__device__ __forceinline__ BwdItem bwd_item(const BwdArgs &a, int w) {
  const WorkItem wi = grouped_item(w, a.n_items / a.nkt, a.nkt, a.hgroup, false);
  BwdItem it;
  it.bkv = wi.bh;
  it.kt = wi.tile;
  int kvl = a.N;
  if (a.kv_len != nullptr) {
    const int v = a.kv_len[it.bkv / a.Hkv];
    kvl = v < 0 ? 0 : (v > a.N ? a.N : v);
  }
  it.kvl = kvl;
  // query tiles that see this key tile: [q_begin, nqt), filtered by the mask
  const int q_begin = CAUSAL ? it.kt : 0;
  int n = 0;
  if (it.kt * 128 < kvl) {
    if (SPARSE) {
      for (int i = 0; i < a.nqt; ++i) n += a.block_mask[static_cast<size_t>(i) * a.nkt + it.kt] != 0;
    } else {
      n = a.nqt - q_begin;
    }
  }
  // grouped-query attention: every query head of the group, (g, qi) in order
  it.n_iter = n * a.kv_group;
  it.q_first = SPARSE ? next_kept(a.block_mask, a.nkt, a.nqt, it.kt, 0) : q_begin;
  return it;
}

// Persistent backward: one CTA per SM takes work items (key tile, key/value
// head) from a counter, in the grouped order of grouped_item: groups of
// hgroup heads, key tile major inside a group, so the heaviest items
// (causal: low key tiles see the most query tiles) start first while the
// heads that run concurrently stay few enough for their Q and dO to stay in
// L2. Between two items the next item's V and K loads start as soon as the
// last dP^T and dQ products of the previous item have read them, and the
// dK/dV epilogue and the last dQ reductions of the previous item overlap
// the next item's start.
template <int D, bool BF16, bool CAUSAL, bool SPARSE>
__global__ void __launch_bounds__(512, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (sbase & 1023u) {  // the swizzled tiles need a 1 KB aligned base
    if (tid == 0) atomicOr(&g_fa_device_error, kDevErrSmemAlign);
    return;
  }
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile uint32_t *abort_flag = misc + 1;
  volatile int *item_slot = reinterpret_cast<volatile int *>(misc + 2);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };
  auto advance = [&](const BwdItem &it, int &g, int &qi) {
    qi = SPARSE ? next_kept(a.block_mask, a.nkt, a.nqt, it.kt, qi + 1) : qi + 1;
    if (qi >= a.nqt) {
      ++g;
      qi = it.q_first;
    }
  };
  // consumer side of the item slots: item k of this CTA (-1: no more work);
  // one arrival per consumer warp (the MMA thread arrives alone)
  // (after a stop the roles keep taking items: the compute warpgroups write
  // zeros for them)
  auto take_item = [&](int k, bool whole_warp, int &w) -> bool {
    const int s = k & 1;
    bool got = mbar_wait_handoff(bar(C::kBITF + s), (k >> 1) & 1, abort_flag);
    if (whole_warp) got = __all_sync(0xffffffffu, got);
    if (!got) return false;
    w = item_slot[s];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(bar(C::kBITE + s));
    return true;
  };

  if (blockIdx.x == 0 && tid == 0) a.stats[3] = static_cast<unsigned int>(ds_exponent(a.stats, a.scale, D));
  if (tid == 0) {
    mbar_init(bar(C::kBKL), 1);
    mbar_init(bar(C::kBVL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kBQF + s), 1);
      mbar_init(bar(C::kBQE + s), 1);
      mbar_init(bar(C::kBPR + s), 128);
      mbar_init(bar(C::kBITF + s), 1);
      mbar_init(bar(C::kBITE + s), C::kItemConsumers);
    }
    mbar_init(bar(C::kBSF), 1);
    mbar_init(bar(C::kBDPF), 1);
    mbar_init(bar(C::kBDV), 1);
    mbar_init(bar(C::kBDSR), 256);
    mbar_init(bar(C::kBDQF), 1);
    mbar_init(bar(C::kBDQE), 128);
    mbar_init(bar(C::kBFIN), 1);
    mbar_init(bar(C::kBDSF), 1);
    mbar_init(bar(C::kBCK), 256);
    mbar_init(bar(C::kBCV), 256);
    mbar_init(bar(C::kBACC), 256);
    mbar_init(bar(C::kBEND), 1);
    *abort_flag = 0u;
    fence_barrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const long long tile_rows = static_cast<long long>(a.nqt) * 128;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsLow));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      int U = 0;                        // Q/dO tiles issued
      int u_last = -1;                  // last tile of the previous item with work
      int k_issued = 0, v_issued = 0;   // K and V loads issued
      bool ok = true;
      int w = static_cast<int>(blockIdx.x);  // the grid never exceeds the item count
      item_slot[0] = w;
      mbar_arrive(bar(C::kBITF));
      for (int k = 0; w >= 0; ++k) {
        // after a stop, or with the test switch (every wait then runs out),
        // the items are handed on without loads
        const BwdItem it = bwd_item<CAUSAL, SPARSE>(a, w);
        ok = !*abort_flag && !pipelines_starved();
        int g = 0, qi = it.q_first;
        for (int u = 0; ok && u < it.n_iter; ++u) {
          const int st = U & 1;
          if (!mbar_wait(bar(C::kBQE + st), ((U >> 1) & 1) ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(C::kBQF + st), 2 * C::kTileBytes + 1024);
          const int qh = a.q_head(it.bkv, g);
          for (int kb = 0; kb < C::kKB; ++kb) {
            tma_load_3d_hint(sbase + C::kQOff + st * C::kTileBytes + kb * 16384, &tm_q, bar(C::kBQF + st),
                             kb * 64, qi * 128, qh, pol_q);
            tma_load_3d_hint(sbase + C::do_off(U) + kb * 16384, &tm_do, bar(C::kBQF + st), kb * 64, qi * 128,
                             qh, pol_q);
          }
          const long long r0 = qh * tile_rows + static_cast<long long>(qi) * 128;
          bulk_load(sbase + C::kLseOff + st * 512, a.lse_l2 + r0, 512, bar(C::kBQF + st));
          bulk_load(sbase + C::kDeltaOff + st * 512, a.delta + r0, 512, bar(C::kBQF + st));
          ++U;
          advance(it, g, qi);
          if (u == 0) {
            // this item's V once the previous item's last dP^T product has
            // read V, its K once the last dQ product has read K
            if (u_last >= 0 && !mbar_wait(bar(C::kBDPF), u_last & 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(bar(C::kBVL), C::kTileBytes);
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d_hint(sbase + C::kVOff + kb * 16384, &tm_v, bar(C::kBVL), kb * 64, it.kt * 128, it.bkv,
                               pol_kv);
            ++v_issued;
            if (u_last >= 0 && !mbar_wait(bar(C::kBDQF), u_last & 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(bar(C::kBKL), C::kTileBytes);
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d_hint(sbase + C::kKOff + kb * 16384, &tm_k, bar(C::kBKL), kb * 64, it.kt * 128, it.bkv,
                               pol_kv);
            ++k_issued;
          }
        }
        if (ok && it.n_iter > 0) u_last = U - 1;
        // the next item goes to the other slot once every consumer has read
        // the item before it; its K and V are pulled into L2 meanwhile
        const int s1 = (k + 1) & 1;
        if (k >= 1 && !mbar_wait_handoff(bar(C::kBITE + s1), (((k + 1) >> 1) - 1) & 1, abort_flag)) break;
        int w1 = static_cast<int>(gridDim.x) + static_cast<int>(atomicAdd(a.work, 1u));
        if (w1 >= a.n_items) w1 = -1;
        item_slot[s1] = w1;
        mbar_arrive(bar(C::kBITF + s1));
        if (w1 >= 0 && !*abort_flag) {
          const WorkItem nx = grouped_item(w1, a.n_items / a.nkt, a.nkt, a.hgroup, false);
          const uint32_t bytes = static_cast<uint32_t>(min(128, a.N - nx.tile * 128)) * D * 2;
          const size_t off = (static_cast<size_t>(nx.bh) * a.N + static_cast<size_t>(nx.tile) * 128) * D * 2;
          bulk_prefetch_l2(static_cast<const uint8_t *>(a.k) + off, bytes);
          bulk_prefetch_l2(static_cast<const uint8_t *>(a.v) + off, bytes);
        }
        w = w1;
      }
      if (*abort_flag) {
        // let the copies in flight land before the CTA exits
        if (k_issued > 0) mbar_wait_drain(bar(C::kBKL), (k_issued - 1) & 1, abort_flag);
        if (v_issued > 0) mbar_wait_drain(bar(C::kBVL), (v_issued - 1) & 1, abort_flag);
        for (int t = max(0, U - 2); t < U; ++t) mbar_wait_drain(bar(C::kBQF + (t & 1)), (t >> 1) & 1, abort_flag);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // every operand is fp16 (bf16 inputs are converted; see the top)
      constexpr uint32_t kIdSS = idesc_f16(false, 128, 128, false, false);   // S^T, dP^T
      constexpr uint32_t kIdKV = idesc_f16(false, 128, D, false, true);      // dK, dV
      constexpr uint32_t kIdQ = C::kDqT ? idesc_f16(false, 128, 128, true, true)  // dQ^T
                                        : idesc_f16(false, 128, D, true, true);   // dQ
      // Shared-memory descriptors as 32-bit low words (the high word, SBO =
      // 1024 and the 128-byte swizzle, is the same for all): K-major tiles
      // (LBO 16) and MN-major tiles (LBO 16384, the distance between
      // 64-column blocks); a step of off bytes adds off / 16. Kept few and
      // cheap: this thread shares its sub-partition with three busy warps,
      // and every instruction it issues delays the next product.
      // (The words are derived per tile from an opaque copy of the shared
      // base, so the compiler does not hoist every step out of the loops
      // into this thread's few registers.)
      constexpr uint32_t kHi = sdesc_hi(1024);
      constexpr uint32_t kStageStep = C::kTileBytes >> 4;
      // S^T = K_j Q_i^T for the query tile in stage st
      auto issue_s = [&](int st) {
        const uint32_t sb = opaque_u32(sbase);
        const uint32_t k_k = sdesc_lo(sb + C::kKOff, 16);
        const uint32_t q_k = sdesc_lo(sb + C::kQOff, 16) + st * kStageStep;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t o = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
          mma_ss_w(tmem + C::kColS, k_k + o, q_k + o, kHi, kIdSS, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBSF));
      };
      int U = 0;   // query tiles processed
      int kl = 0;  // items with work processed
      for (int k = 0;; ++k) {
        int w;
        if (!take_item(k, false, w) || w < 0) break;
        if (*abort_flag) continue;
        const BwdItem it = bwd_item<CAUSAL, SPARSE>(a, w);
        if (it.n_iter == 0) continue;
        bool ok;
        // K landed (and, bf16 inputs, converted), the first Q stage landed,
        // and the previous tile's dV products are done reading P^T from the
        // S^T columns
        ok = mbar_wait(bar(C::kBKL), kl & 1, abort_flag) && mbar_wait(bar(C::kBCK), kl & 1, abort_flag) &&
             mbar_wait(bar(C::kBQF + (U & 1)), (U >> 1) & 1, abort_flag) &&
             (U == 0 || mbar_wait(bar(C::kBDV), (U - 1) & 1, abort_flag));
        if (!ok) continue;
        tc_fence_after();
        issue_s(U & 1);
        for (int u = 0; u < it.n_iter; ++u, ++U) {
          const int st = U & 1;
          const uint32_t sb = opaque_u32(sbase);
          const uint32_t do_k = sdesc_lo(sb + C::do_off(U), 16);
          // d = 128: the dP^T columns hold the previous dQ partial until read out
          if (C::kDqT && U > 0 && !mbar_wait(bar(C::kBDQE), (U - 1) & 1, abort_flag)) { ok = false; break; }
          // the first dP^T of an item needs its V (in fp16)
          if (u == 0 && !(mbar_wait(bar(C::kBVL), kl & 1, abort_flag) && mbar_wait(bar(C::kBCV), kl & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {  // dP^T = V_j dO_i^T
            const uint32_t o = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            mma_ss_w(tmem + C::kColDP, sdesc_lo(sb + C::kVOff, 16) + o, do_k + o, kHi, kIdSS, ks > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBDPF));
          // the first dV product of an item overwrites the accumulators: the
          // previous item's dK and dV must have been read out of TMEM
          if (u == 0 && kl > 0 && !mbar_wait(bar(C::kBACC), (kl - 1) & 1, abort_flag)) { ok = false; break; }
          // dV_j += P^T dO_i, P^T read from TMEM, one 64-query half at a time
          for (int h = 0; ok && h < 2; ++h) {
            if (!mbar_wait(bar(C::kBPR + h), U & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t do_mn = sdesc_lo(opaque_u32(sbase) + C::do_off(U), 16384);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ts_w(tmem + C::kColDV, tmem + C::kColS + 64 * h + 8 * ks, do_mn + (4 * h + ks) * 128, kHi,
                       kIdKV, (u > 0 || h > 0 || ks > 0) ? 1u : 0u);
          }
          if (!ok) break;
          mma_commit(bar(C::kBDV));
          if (C::kSAfterDV && u + 1 < it.n_iter) {
            // next score tile: its Q stage must have landed, and the S^T
            // columns are free once this tile's dV products have read P^T
            if (!mbar_wait(bar(C::kBQF + (st ^ 1)), ((U + 1) >> 1) & 1, abort_flag) ||
                !mbar_wait(bar(C::kBDV), U & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_s(st ^ 1);
          }
          if (!mbar_wait(bar(C::kBDSR), U & 1, abort_flag)) { ok = false; break; }
          // d = 64: the dQ columns hold the previous partial until read out
          if (!C::kDqT && U > 0 && !mbar_wait(bar(C::kBDQE), (U - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // dQ first, so its read-out overlaps the next S^T and the dK MMA
          const uint32_t sb2 = opaque_u32(sbase);
          const uint32_t k_mn = sdesc_lo(sb2 + C::kKOff, 16384), ds_mn = sdesc_lo(sb2 + C::ds_off(U), 16384);
          if constexpr (C::kDqT) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // dQ_i^T = K_j^T dS^T (both MN-major in smem)
              mma_ss_w(tmem + C::kColDQ, k_mn + ks * 128, ds_mn + ks * 128, kHi, kIdQ, ks > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // dQ_i = dS K_j (dS read MN-major from the dS^T buffer)
              mma_ss_w(tmem + C::kColDQ, ds_mn + ks * 128, k_mn + ks * 128, kHi, kIdQ, ks > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBDQF));
          if (!C::kSAfterDV && u + 1 < it.n_iter) {
            // next score tile: its Q stage must have landed, and the S^T
            // columns are free once this tile's dV products have read P^T
            if (!mbar_wait(bar(C::kBQF + (st ^ 1)), ((U + 1) >> 1) & 1, abort_flag) ||
                !mbar_wait(bar(C::kBDV), U & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_s(st ^ 1);
          }
          const uint32_t sb3 = opaque_u32(sbase);
          const uint32_t ds_k = sdesc_lo(sb3 + C::ds_off(U), 16);
          const uint32_t q_mn = sdesc_lo(sb3 + C::kQOff, 16384) + st * kStageStep;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // dK_j += dS^T Q_i (dS^T K-major in smem)
            mma_ss_w(tmem + C::kColDK, ds_k + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), q_mn + ks * 128, kHi,
                     kIdKV, (u > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar(C::kBDSF));
          mma_commit(bar(C::kBQE + st));
        }
        if (!ok) continue;
        mma_commit(bar(C::kBFIN));
        ++kl;
      }
      // every issued product completes before TMEM is released
      mma_commit(bar(C::kBEND));
      mbar_wait_drain(bar(C::kBEND), 0, abort_flag);
    }
  }
    // teardown of warpgroup 0 (the two register regions do not rejoin)
    tc_fence_before();
    named_bar_sync(1, C::kThreads);
    if (warp == 1) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, C::kTmemCols);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int e_s = ds_exponent(a.stats, a.scale, D);
    const int e_do = BF16 ? do_exponent(a.stats) : 0;
    if (warp < 12) {
    // ------------------------------------------------------------ P^T and dS^T, one query half
    const int h = (warp >> 2) - 1;  // query half: columns [64h, 64h+64) of the tile
    const int r = tid & 127;         // key row of this thread's lane (epilogue)
    const float sl2 = a.scale_log2;
    const float f_s = exp2i(-e_s);
    const float sc_dp = a.scale * f_s * exp2i(e_do);  // multiplies dP16
    const float sc_d = a.scale * f_s;                 // multiplies -D
    // TMEM is read and written in 16-lane blocks j = 0, 1 of the warp's
    // quadrant (16x256b loads, 16x128b stores): in block j this thread holds
    // lanes t4 and t4 + 8, i.e. the keys 32 (warp & 3) + 16 j + 8 i + t4
    // (i = 0, 1) of the tile, and for each column group b = 0..7 the query
    // pair 8 b + 2 c4, +1 of this half. It therefore needs only 16 of the
    // half's 64 per-query LSE and D values, read as 8 float2 each.
    const int t4 = lane >> 2, c4 = lane & 3;
    const uint32_t tq = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    int U = 0, kl = 0;
    for (int k = 0;; ++k) {
      int w;
      if (!take_item(k, true, w) || w < 0) break;
      const BwdItem it = bwd_item<CAUSAL, SPARSE>(a, w);
      const int kt = it.kt, kvl = it.kvl;
      bool ok = !*abort_flag, have = false;
      // dK carries 2^-e_s (from dS), dV carries 2^-e_do (from dO); read
      // again per item rather than kept in a register through the tile loop
      float f_out = 1.f;
      if (ok && it.n_iter > 0) {
        // ---- bf16 inputs: K_j, then V_j -> fp16 in place. The first S^T
        // needs only K; the first dP^T waits for V.
        constexpr int kChunks = C::kTileBytes / 16;  // 16-byte chunks per tile
        float amax = 0.f;
        const bool k_in = !BF16 || mbar_wait_warp(bar(C::kBKL), kl & 1, abort_flag);
        if (BF16 && k_in) {
          uint4 *k16 = reinterpret_cast<uint4 *>(smem + C::kKOff);
          for (int c = tid - 128; c < kChunks; c += 256) k16[c] = bf16x8_to_f16x8(k16[c], amax);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bar(C::kBCK));
        const bool v_in = k_in && (!BF16 || mbar_wait_warp(bar(C::kBVL), kl & 1, abort_flag));
        if (BF16 && v_in) {
          uint4 *v16 = reinterpret_cast<uint4 *>(smem + C::kVOff);
          for (int c = tid - 128; c < kChunks; c += 256) v16[c] = bf16x8_to_f16x8(v16[c], amax);
          if (amax > 65504.f) atomicOr(&g_fa_device_error, kDevErrRange);
          fence_proxy_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bar(C::kBCV));
        ok = v_in;
        int g = 0, qi = it.q_first;
        for (const int u_end = U + it.n_iter; ok && U < u_end; ++U) {
          const int st = U & 1;
          const float2 *nl2 = reinterpret_cast<const float2 *>(smem + C::kLseOff + st * 512 + h * 256) + c4;
          const float2 *nd2 = reinterpret_cast<const float2 *>(smem + C::kDeltaOff + st * 512 + h * 256) + c4;
          if (!mbar_wait_warp(bar(C::kBQF + st), (U >> 1) & 1, abort_flag)) { ok = false; break; }
          if (!mbar_wait_warp(bar(C::kBSF), U & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // p[j][4b + 2i + e]: key (j, i), query 8b + 2c4 + e of this half, fp32,
          // kept in registers for dS
          float p[2][32];
          {
            uint32_t sv[2][32];
            tmem_ld_16x256b_x8(tq + C::kColS + 64 * h, sv[0]);
            tmem_ld_16x256b_x8(tq + (16u << 16) + C::kColS + 64 * h, sv[1]);
            tmem_wait_ld();
            reg_fence_32(sv[0]);
            reg_fence_32(sv[1]);
#pragma unroll
            for (int b = 0; b < 8; ++b) {
              const float2 nl = nl2[4 * b];
#pragma unroll
              for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  const int e = 4 * b + 2 * i;
                  ffma2(p[j][e], p[j][e + 1], __uint_as_float(sv[j][e]), __uint_as_float(sv[j][e + 1]), sl2,
                        sl2, nl.x, nl.y);
                  p[j][e] = ex2_approx(p[j][e]);
                  p[j][e + 1] = ex2_approx(p[j][e + 1]);
                }
            }
            // causal: query c of this tile sees key k iff qi*128 + c >= kt*128 + k;
            // a dead key sees nothing. Local column 8b + 2c4 + e is query
            // 64h + 8b + 2c4 + e of the tile.
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                const int kk = kt * 128 + 32 * (warp & 3) + 16 * j + 8 * i + t4;
                const int cmin = (kk >= kvl ? 128 : (CAUSAL ? (kk - qi * 128) : -1)) - 64 * h;
                if (cmin > 0) {
#pragma unroll
                  for (int b = 0; b < 8; ++b)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                      if (8 * b + 2 * c4 + e < cmin) p[j][4 * b + 2 * i + e] = 0.f;
                }
              }
          }
          // P^T (16-bit pairs, column = query pair) into the first 32 columns of
          // this half's S^T columns (already read)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t pw[16];
#pragma unroll
            for (int b = 0; b < 8; ++b) {
              pw[2 * b] = pack2<false>(p[j][4 * b], p[j][4 * b + 1]);
              pw[2 * b + 1] = pack2<false>(p[j][4 * b + 2], p[j][4 * b + 3]);
            }
            tmem_st_16x128b_x8(tq + (static_cast<uint32_t>(16 * j) << 16) + C::kColS + 64 * h, pw);
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(C::kBPR + h));
          if (!mbar_wait_warp(bar(C::kBDPF), U & 1, abort_flag)) { ok = false; break; }
          // d = 64: the previous dQ/dK MMAs must be done reading dS before it
          // is rewritten (d = 128 writes the rotated buffer, see BwdCfg)
          if (!C::kRotDS && U > 0 && !mbar_wait_warp(bar(C::kBDSF), (U - 1) & 1, abort_flag)) { ok = false; break; }
          const uint32_t sDS = sbase + C::ds_off(U) + h * 16384;
          tc_fence_after();
          uint32_t dv[2][32];
          tmem_ld_16x256b_x8(tq + C::kColDP + 64 * h, dv[0]);
          tmem_ld_16x256b_x8(tq + (16u << 16) + C::kColDP + 64 * h, dv[1]);
          tmem_wait_ld();
          reg_fence_32(dv[0]);
          reg_fence_32(dv[1]);
          // ds[j][i][b]: key (j, i), queries 8b + 2c4, +1 of this half, as a
          // 16-bit pair; for fixed (j, i, b) the warp holds one 8 x 8 block of
          // dS^T (rows = 8 keys, columns = 8 queries) in the m8n8 fragment
          // layout (row lane / 4, column pair lane % 4)
          uint32_t ds[2][2][8];
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            float2 nd = nd2[4 * b];
            fmul2(nd.x, nd.y, nd.x, nd.y, sc_d, sc_d);
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                // dS * scale * 2^-e_s = P * (dP16 * scale * 2^(e_do - e_s) - scale * D * 2^-e_s)
                const int e = 4 * b + 2 * i;
                float t0, t1;
                ffma2(t0, t1, __uint_as_float(dv[j][e]), __uint_as_float(dv[j][e + 1]), sc_dp, sc_dp, nd.x,
                      nd.y);
                fmul2(t0, t1, t0, t1, p[j][e], p[j][e + 1]);
                ds[j][i][b] = pack2<false>(t0, t1);
              }
          }
          // four blocks per stmatrix: blocks b = 4q .. 4q + 3 of key rows
          // 32 (warp & 3) + 16 j + 8 i + 0..7; lane l gives the address of
          // row l % 8 of block l / 8: 16-byte chunk b of the row's 128 bytes
          // in region h, swizzled by (row & 7)
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const int rr = lane & 7, bb = 4 * q + (lane >> 3);
                const uint32_t addr = sDS + (32 * (warp & 3) + 16 * j + 8 * i + rr) * 128 + ((bb ^ rr) << 4);
                stmatrix_x4(addr, ds[j][i][4 * q], ds[j][i][4 * q + 1], ds[j][i][4 * q + 2], ds[j][i][4 * q + 3]);
              }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(bar(C::kBDSR));
          advance(it, g, qi);
        }
        // the output factor's global load overlaps the wait
        f_out = exp2i(h == 0 ? ds_exponent(a.stats, a.scale, D) : (BF16 ? do_exponent(a.stats) : 0));
        have = ok && mbar_wait_warp(bar(C::kBFIN), kl & 1, abort_flag);
        if (have) tc_fence_after();
        ++kl;
      }
      // ---- dK (warpgroup 1) or dV (warpgroup 2) out of TMEM; the next
      // item's first dV product waits until both are read
      const uint32_t acc_col = tmem + lane_addr + (h == 0 ? C::kColDK : C::kColDV);
      if (have) {
        // 64 channels at a time: each thread puts its key row's channels into
        // this warp's 4 KB slice of a staging box (its 32 rows of 128 bytes,
        // 16-byte chunks swizzled by the row, so neither pass has bank
        // conflicts), then the warp writes its rows out eight threads per
        // 128-byte row piece: four whole lines per warp instruction. Rows
        // past N are not written. The slice lies in this half's part of the
        // buffer the next dS^T goes to, in the rows this warp writes there:
        // the products that read it last (dS^T of the item's last tile at
        // d = 64, dO of that tile at d = 128) are done (kBFIN), and no other
        // warp touches it, so the warps need not wait for one another.
        // Stores straight from registers (a 16-byte piece of each of 32 rows
        // per warp instruction) kept the memory pipeline busy for longer
        // than a tile and held up the next item's start.
        const uint32_t slice = sbase + C::ds_off(U) + h * 16384 + (warp & 3) * 4096;
#pragma unroll 1
        for (int c64 = 0; c64 < D; c64 += 64) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(acc_col + c64 + c0, v);
            tmem_wait_ld();
            reg_fence_32(v);
            uint32_t pw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0, x1;
              fmul2(x0, x1, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), f_out, f_out);
              pw[i] = pack2<BF16>(x0, x1);
            }
            // channels c0 .. c0 + 31 are 16-byte chunks c0 / 8 .. +3 of the row
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(slice + lane * 128 + (static_cast<uint32_t>((c0 / 8 + q) ^ (lane & 7)) << 4), pw[4 * q],
                           pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
          }
          if (c64 + 64 == D) {  // every accumulator column has been read
            tc_fence_before();
            mbar_arrive(bar(C::kBACC));
          }
          __syncwarp();
          const int rows = min(32, a.N - kt * 128 - 32 * (warp & 3));  // this warp's rows inside N
          const int cc = lane & 7;  // 16-byte chunk of the write-out pass
          uint16_t *out = static_cast<uint16_t *>(h == 0 ? a.dk : a.dv) +
                          (static_cast<size_t>(it.bkv) * a.N + static_cast<size_t>(kt) * 128 + 32 * (warp & 3)) * D +
                          c64 + cc * 8;
#pragma unroll 4
          for (int i = 0; i < 8; ++i) {
            const int row = 4 * i + (lane >> 3);
            const uint4 w = ld_shared_v4(slice + row * 128 + (static_cast<uint32_t>(cc ^ (row & 7)) << 4));
            if (row < rows) *reinterpret_cast<uint4 *>(out + static_cast<size_t>(row) * D) = w;
          }
          __syncwarp();  // the slice has been read before it is written again
        }
      } else {
        // zeros (an item without work, or after a stop), row by row
        const int key = kt * 128 + r;
        if (key < a.N) {
          uint4 *d4 = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(h == 0 ? a.dk : a.dv) +
                                                (static_cast<size_t>(it.bkv) * a.N + static_cast<size_t>(key)) * D);
          for (int q = 0; q < D / 8; ++q) d4[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    } else {
    // ------------------------------------------------------------ dQ partials
    const int r = tid & 127;  // d = 128: head-dim channel; d = 64: query row
    int U = 0;
    for (int k = 0;; ++k) {
      int w;
      if (!take_item(k, true, w) || w < 0) break;
      if (*abort_flag) continue;
      const BwdItem it = bwd_item<CAUSAL, SPARSE>(a, w);
      int g = 0, qi = it.q_first;
      for (int u = 0; u < it.n_iter; ++u, ++U) {
        if (!mbar_wait_warp(bar(C::kBDQF), U & 1, abort_flag)) break;
        tc_fence_after();
        // read the whole partial into registers, release the TMEM columns
        // (the next dP^T or dQ MMA may overwrite them), then reduce into the
        // accumulator
        constexpr int kCols = C::kDqT ? 128 : D;
        uint32_t v[kCols / 32][32];
#pragma unroll
        for (int j = 0; j < kCols / 32; ++j) tmem_ld_32x32b_x32(tmem + lane_addr + C::kColDQ + j * 32, v[j]);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kCols / 32; ++j) reg_fence_32(v[j]);
        tc_fence_before();
        mbar_arrive(bar(C::kBDQE));
        if constexpr (C::kDqT) {
          // thread r holds channel r of the 128 queries of this tile. The L2
          // takes the reductions more slowly than the warps issue them; a short
          // pause after every 16 keeps the sub-partition's memory-instruction
          // queue from filling, so the softmax warpgroups' shared-memory
          // accesses behind it are not held up. The pause is a nanosleep, not
          // a spin on the clock: a spinning warp takes issue slots from the
          // softmax warps of its sub-partition, whose exponentials are the
          // longest step of each tile (measured 4-7 % faster than a 120-cycle
          // spin; 128-192 ns sleep alike, 96 ns or a pause every 32 slower,
          // 256 ns or more, or every 8, much slower).
          float *acc = a.dq_acc + (a.q_head(it.bkv, g) * tile_rows + static_cast<long long>(qi) * 128) * D + r;
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              atomicAdd(acc + (j * 32 + i) * D, __uint_as_float(v[j][i]));
              if ((i & 15) == 15) __nanosleep(160);
            }
        } else {
          float *acc = a.dq_acc + (a.q_head(it.bkv, g) * tile_rows + static_cast<long long>(qi) * 128 + r) * D;
#pragma unroll
          for (int j = 0; j < D / 32; ++j)
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              atomicAdd(reinterpret_cast<float4 *>(acc + j * 32 + i),
                        make_float4(__uint_as_float(v[j][i]), __uint_as_float(v[j][i + 1]),
                                    __uint_as_float(v[j][i + 2]), __uint_as_float(v[j][i + 3])));
        }
        advance(it, g, qi);
      }
    }
    }
    // teardown of the compute warpgroups
    tc_fence_before();
    named_bar_sync(1, C::kThreads);
  }
}

}  // namespace fa
