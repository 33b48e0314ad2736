// fwd2_kernel.cuh -- forward attention for sm_103a, two query tiles per CTA.
//
// The block loop of "Flash Attention: revolutionizing transformer
// efficiency" (query blocks outer, key/value blocks inner, running max m and
// sum l), as in fwd_kernel.cuh, but each CTA owns two 128-row query tiles A
// and B of the same (batch, head) and one softmax warpgroup per tile. The MMA
// thread alternates between the tiles -- S_A = Q_A K_j^T, S_B = Q_B K_j^T,
// O_A += P_A V_j, O_B += P_B V_j -- so while one warpgroup runs its softmax
// the tensor cores work on the other tile. K_j and V_j are loaded once for
// both tiles. The MMA issue order per key tile t is P_A V_t, S_A(t+1),
// P_B V_t, S_B(t+1): each tile's next scores follow its own P V, so the
// chain of one tile never waits for the other tile's softmax.
//
// Roles (384 threads; setmaxnreg moves registers from warpgroup 0 to the two
// softmax warpgroups):
//   warp 0 lane 0  TMA producer (Q_A, Q_B once; K/V ring)
//   warp 1         TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 4..7     softmax of tile A (thread r = query row r)
//   warps 8..11    softmax of tile B
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B after it.
// P (16-bit pairs) is written into the first 64 columns of its own, already
// read S buffer. QK^T of the next key tile into that buffer waits for the
// P V that reads it.
//
// Online softmax: softmax_row (softmax_row.cuh), the same arithmetic as
// fwd_kernel.cuh.
//
// FP8 (d = 128 only): Q, K and V are e4m3 with per-tensor dequantisation
// factors (low-precision forward of the FlashAttention-3 section of "Flash
// Attention: revolutionizing transformer efficiency"). Both products run as
// kind::f8f6f4 (K = 32 per instruction): S = Q K^T with K-major Q and K, and
// O += P V^T-fed, where V arrives already transposed ([d][keys], written by
// fwd_fp8_vt_kernel) so that its tile is K-major too. P is scaled by 2^8
// before it is rounded to e4m3 (p' = 2^(x - m + 8) <= 256 < 448, and small
// probabilities keep their mantissa down to 2^-14 instead of 2^-6); l sums
// the unrounded p', so O = (P' V) / l' needs no correction and
// LSE = (m + log2 l' - 8) ln 2. P takes 32 TMEM columns, four keys per column.
#pragma once
#include "common.cuh"
#include "fwd_kernel.cuh"
#include "schedule.cuh"

namespace fa {

template <int D, bool FP8 = false>
struct Fwd2Cfg {
  static_assert(!FP8 || D == 128, "the 8-bit forward is built for d = 128");
  static constexpr int kTileBytes = 128 * D * (FP8 ? 1 : 2);
  static constexpr int kStages = FP8 ? 4 : ((D == 64) ? 3 : 2);
  static constexpr int kKB = FP8 ? 1 : D / 64;   // 128-byte TMA boxes per tile row
  static constexpr int kBoxElems = FP8 ? 128 : 64;
  static constexpr int kQOff = 0;                          // Q_A, Q_B
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kBQ = 0;
  static constexpr int kBKF = 1;
  static constexpr int kBVF = kBKF + kStages;
  static constexpr int kBKE = kBVF + kStages;
  static constexpr int kBVE = kBKE + kStages;
  static constexpr int kBSF = kBVE + kStages;  // [2] S_X ready
  static constexpr int kBPF = kBSF + 2;        // [2][2] half h of P_X in TMEM (128 arrivals)
  static constexpr int kBOR = kBPF + 4;        // [2] P_X V done
  static constexpr int kBDR = kBOR + 2;
  static constexpr int kNumBars = kBDR + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  __host__ __device__ static constexpr uint32_t col_s(int x) { return x ? 128u : 0u; }
  static constexpr uint32_t kColO0 = 256;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColO0 + 2 * D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // setmaxnreg split: launch with 168 registers x 384 threads; warpgroup 0
  // gives back to 56, the two softmax warpgroups take 224 (sum unchanged).
  static constexpr int kLaunchRegs = 168, kRegsLow = 56, kRegsHigh = 224;
  static_assert(kRegsLow * 128 + kRegsHigh * 256 <= kLaunchRegs * 384, "register split");
};

// tm_o, tm_r: O and its rounding residual as [B*H][N][D] 16-bit tensors
// with the same 64 x 128 x 1 boxes as Q (tm_r is only used when a.o_res is
// set; the 8-bit forward stores O directly).
template <int D, bool BF16, bool CAUSAL, bool FP8 = false>
__global__ void __launch_bounds__(384, 1)
    fwd2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const __grid_constant__ CUtensorMap tm_r, const FwdArgs a) {
  static_assert(!FP8 || BF16, "8-bit inputs give bf16 O");
  using C = Fwd2Cfg<D, FP8>;
  extern __shared__ uint8_t smem_raw2[];
  const uint32_t raw = smem_u32(smem_raw2);
  const uint32_t sbase = align_up_1024(raw);
  uint8_t *smem = smem_raw2 + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile uint32_t *abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };

  // ---- work item: 256 query rows (tiles 2qb, 2qb+1) of one head
  // Launch order: groups of hgroup heads; within a group query-block
  // major, heaviest first (causal: the last blocks see the most key tiles),
  // while the heads that run concurrently stay few enough for their K and V
  // to stay in L2.
  const int nqb = (a.nqt + 1) >> 1;
  const WorkItem item =
      grouped_item(static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x) / nqb, nqb, a.hgroup, CAUSAL);
  const int bh = item.bh, qb = item.tile;
  const int b = bh / a.H;
  const int kvh = a.kv_head(bh);
  int kvl = a.N;
  if (a.kv_len != nullptr) {
    const int v = a.kv_len[b];
    kvl = v < 0 ? 0 : (v > a.N ? a.N : v);
  }
  const int nkt_eff = (kvl + 127) >> 7;
  int n_tile[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int qt = 2 * qb + x;
    n_tile[x] = (qt < a.nqt) ? (CAUSAL ? min(qt + 1, nkt_eff) : nkt_eff) : 0;
  }
  const int n_max = max(n_tile[0], n_tile[1]);
  const bool has_b = (2 * qb + 1) < a.nqt;

  if (tid == 0) {
    mbar_init(bar(C::kBQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBKF + s), 1);
      mbar_init(bar(C::kBVF + s), 1);
      mbar_init(bar(C::kBKE + s), 1);
      mbar_init(bar(C::kBVE + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::kBSF + x), 1);
      mbar_init(bar(C::kBPF + 2 * x), 128);
      mbar_init(bar(C::kBPF + 2 * x + 1), 128);
      mbar_init(bar(C::kBOR + x), 1);
    }
    mbar_init(bar(C::kBDR), 1);
    *abort_flag = 0u;
    fence_barrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsLow));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_max > 0 && !pipelines_starved()) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(bar(C::kBQ), C::kTileBytes * (has_b ? 2 : 1));
      for (int x = 0; x < (has_b ? 2 : 1); ++x)
        for (int kb = 0; kb < C::kKB; ++kb)
          tma_load_3d_hint(sbase + C::kQOff + x * C::kTileBytes + kb * 16384, &tm_q, bar(C::kBQ),
                           kb * C::kBoxElems, (2 * qb + x) * 128, bh, pol_q);
      int nk = 0, nv = 0;
      for (int t = 0; t < n_max; ++t) {
        const int st = t % C::kStages;
        const uint32_t ph = (t / C::kStages) & 1;
        if (!mbar_wait(bar(C::kBKE + st), ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBKF + st), C::kTileBytes);
        for (int kb = 0; kb < C::kKB; ++kb)
          tma_load_3d_hint(sbase + C::kKOff + st * C::kTileBytes + kb * 16384, &tm_k,
                           bar(C::kBKF + st), kb * C::kBoxElems, t * 128, kvh, pol_kv);
        nk = t + 1;
        if (!mbar_wait(bar(C::kBVE + st), ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBVF + st), C::kTileBytes);
        if constexpr (FP8)  // V^T: 128 keys (x) of all 128 rows d
          tma_load_3d_hint(sbase + C::kVOff + st * C::kTileBytes, &tm_v, bar(C::kBVF + st), t * 128, 0,
                           kvh, pol_kv);
        else
          for (int kb = 0; kb < C::kKB; ++kb)
            tma_load_3d_hint(sbase + C::kVOff + st * C::kTileBytes + kb * 16384, &tm_v,
                             bar(C::kBVF + st), kb * 64, t * 128, kvh, pol_kv);
        nv = t + 1;
      }
      if (*abort_flag) {
        mbar_wait_drain(bar(C::kBQ), 0, abort_flag);
        for (int t = max(0, nk - C::kStages); t < nk; ++t)
          mbar_wait_drain(bar(C::kBKF + t % C::kStages), (t / C::kStages) & 1, abort_flag);
        for (int t = max(0, nv - C::kStages); t < nv; ++t)
          mbar_wait_drain(bar(C::kBVF + t % C::kStages), (t / C::kStages) & 1, abort_flag);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_max > 0) {
      // (for 8-bit inputs the e4m3 format code is f16's, 0: the same descriptor)
      constexpr uint32_t kIdQK = idesc_f16(BF16 && !FP8, 128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_f16(BF16 && !FP8, 128, D, false, !FP8);
      // S_x(t) = Q_x K_t^T into TMEM; the caller has waited for K_t
      auto issue_qk = [&](int x, int t) {
        const uint32_t sb = opaque_u32(sbase);
        const uint32_t kbase = sb + C::kKOff + (t % C::kStages) * C::kTileBytes;
        const uint32_t qbase = sb + C::kQOff + x * C::kTileBytes;
        if constexpr (FP8) {
          // 32 e4m3 elements = 32 B of the single 128-byte column block per step
          const uint32_t q_k = sdesc_lo(qbase, 16), k_k = sdesc_lo(kbase, 16);
#pragma unroll
          for (int ks = 0; ks < D / 32; ++ks)
            mma_ss_f8_w(tmem + C::col_s(x), q_k + ks * 2, k_k + ks * 2, sdesc_hi(1024), kIdQK, ks > 0 ? 1u : 0u);
        } else {
          // descriptors as 32-bit words stepped by adds (sdesc_lo): this
          // thread shares its sub-partition with the softmax warps, and
          // every instruction it issues delays the next product
          const uint32_t q_k = sdesc_lo(qbase, 16), k_k = sdesc_lo(kbase, 16);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t o = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
            mma_ss_w(tmem + C::col_s(x), q_k + o, k_k + o, sdesc_hi(1024), kIdQK, ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(C::kBSF + x));
      };
      // Per key tile t and query tile x: O_x += P_x V_t, then, once that
      // product has read P_x out of S_x, S_x = Q_x K_{t+1}^T. Tile x's next
      // scores do not wait for the other tile's softmax.
      bool ok = mbar_wait(bar(C::kBQ), 0, abort_flag) && mbar_wait(bar(C::kBKF), 0, abort_flag);
      if (ok) {
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (n_tile[x] > 0) issue_qk(x, 0);
        mma_commit(bar(C::kBKE));
      }
      for (int t = 0; ok && t < n_max; ++t) {
        const int st = t % C::kStages;
        const uint32_t ph = (t / C::kStages) & 1;
        const int st1 = (t + 1) % C::kStages;
        const uint32_t ph1 = ((t + 1) / C::kStages) & 1;
        if (!mbar_wait(bar(C::kBVF + st), ph, abort_flag)) { ok = false; break; }
        const uint32_t vbase = opaque_u32(sbase) + C::kVOff + st * C::kTileBytes;
        bool k_next = false;  // K_{t+1} waited for
#pragma unroll 1
        for (int x = 0; x < 2; ++x) {
          if (t >= n_tile[x]) continue;
          const uint32_t ocol = tmem + C::kColO0 + x * D;
          const uint32_t pcol = tmem + C::col_s(x);
          // P_x arrives in two halves of 64 keys; each half's products start
          // as soon as it is in TMEM
          for (int h = 0; h < 2; ++h) {
            if (!mbar_wait(bar(C::kBPF + 2 * x + h), t & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            if constexpr (FP8) {
              // A = P (4 keys per TMEM column, 8 columns per step); B = V^T
              // K-major, 32 keys = 32 B per step
              const uint32_t v_k = sdesc_lo(vbase, 16);
#pragma unroll
              for (int ks = 2 * h; ks < 2 * h + 2; ++ks)
                mma_ts_f8_w(ocol, pcol + ks * 8, v_k + ks * 2, sdesc_hi(1024), kIdPV, (t > 0 || ks > 0) ? 1u : 0u);
            } else {
              const uint32_t v_mn = sdesc_lo(vbase, 16384);
#pragma unroll
              for (int ks = 4 * h; ks < 4 * h + 4; ++ks)
                mma_ts_w(ocol, pcol + ks * 8, v_mn + ks * 128, sdesc_hi(1024), kIdPV, (t > 0 || ks > 0) ? 1u : 0u);
            }
          }
          if (!ok) break;
          mma_commit(bar(C::kBOR + x));
          if (t + 1 < n_tile[x]) {
            // S_x holds P_x until this tile's P V is done
            if ((!k_next && !mbar_wait(bar(C::kBKF + st1), ph1, abort_flag)) ||
                !mbar_wait(bar(C::kBOR + x), t & 1, abort_flag)) { ok = false; break; }
            k_next = true;
            tc_fence_after();
            issue_qk(x, t + 1);
          }
        }
        if (!ok) break;
        if (k_next) mma_commit(bar(C::kBKE + st1));
        mma_commit(bar(C::kBVE + st));
      }
      mma_commit(bar(C::kBDR));
      mbar_wait_drain(bar(C::kBDR), 0, abort_flag);
    }
  }
    // teardown of warpgroup 0 (the two register regions do not rejoin)
    tc_fence_before();
    named_bar_sync(1, 384);
    if (warp == 1) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, C::kTmemCols);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
    // ------------------------------------------------------------ softmax of tile x
    const int x = (warp - 4) >> 2;
    const int row = (tid - 128) & 127;
    const int qt = 2 * qb + x;
    const int n = n_tile[x];
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t scol = tmem + lane_addr + C::col_s(x);
    const uint32_t ocol = tmem + lane_addr + C::kColO0 + x * D;
    const int q_row = qt * 128 + row;
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      if (!mbar_wait_warp(bar(C::kBSF + x), t & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[128];
      {
        uint32_t r0[32], r1[32], r2[32], r3[32];
        tmem_ld_32x32b_x32(scol + 0, r0);
        tmem_ld_32x32b_x32(scol + 32, r1);
        tmem_ld_32x32b_x32(scol + 64, r2);
        tmem_ld_32x32b_x32(scol + 96, r3);
        tmem_wait_ld();
        reg_fence_32(r0);
        reg_fence_32(r1);
        reg_fence_32(r2);
        reg_fence_32(r3);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
          s[64 + c] = __uint_as_float(r2[c]);
          s[96 + c] = __uint_as_float(r3[c]);
        }
      }
      int limit = kvl - t * 128;
      if (CAUSAL && t == qt) limit = min(limit, row + 1);
      float m_new, alpha;
      const float nm = softmax_max(s, limit, sl2, m, m_new, alpha);
      // rescale O_x first, so the P V of this tile can start right after the
      // first half of P. S_x(t) complete implies P_x V of tile t - 1 is done:
      // that product was finished before S_x(t) was issued.
      if (t > 0 && __any_sync(0xffffffffu, m_new != m)) {
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(ocol + 32 * j, o);
          tmem_wait_ld();
          reg_fence_32(o);
          scale32(o, alpha);
          tmem_st_32x32b_x32(ocol + 32 * j, o);
        }
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      // 8-bit P: exponent offset +8 (p' = 2^8 p), keys 4c..4c+3 in column c
      const float nmx = FP8 ? nm + 8.f : nm;
      softmax_exp<0, 64>(s, sl2, nmx, acc);
      if constexpr (FP8) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_e4m3x4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
        tmem_st_32x32b_x16(scol, w);
      } else {
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t hi[16];
          pack_p32<BF16>(s, c0, hi);
          tmem_st_32x32b_x16(scol + c0 / 2, hi);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBPF + 2 * x));
      softmax_exp<64, 128>(s, sl2, nmx, acc);
      if constexpr (FP8) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_e4m3x4(s[64 + 4 * i], s[64 + 4 * i + 1], s[64 + 4 * i + 2], s[64 + 4 * i + 3]);
        tmem_st_32x32b_x16(scol + 16, w);
      } else {
#pragma unroll
        for (int c0 = 64; c0 < 128; c0 += 32) {
          uint32_t hi[16];
          pack_p32<BF16>(s, c0, hi);
          tmem_st_32x32b_x16(scol + c0 / 2, hi);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBPF + 2 * x + 1));
      l = l * alpha + softmax_sum(acc);
      m = m_new;
    }
    // ---- epilogue: O / l and LSE (rows of a missing tile B are skipped)
    bool have_o = ok && n > 0;
    if (have_o) {
      have_o = mbar_wait_warp(bar(C::kBOR + x), (n - 1) & 1, abort_flag);
      tc_fence_after();
    }
    if (qt < a.nqt) {
      // 8-bit inputs: O carries V's dequantisation factor
      const float inv_l = (l > 0.f) ? (FP8 ? a.o_scale : 1.f) / l : 0.f;
      uint32_t oall[D / 32][32];
      if (have_o) {
#pragma unroll
        for (int j = 0; j < D / 32; ++j) tmem_ld_32x32b_x32(ocol + 32 * j, oall[j]);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < D / 32; ++j) reg_fence_32(oall[j]);
      } else {
#pragma unroll
        for (int j = 0; j < D / 32; ++j)
#pragma unroll
          for (int i = 0; i < 32; ++i) oall[j][i] = 0u;
      }
      if constexpr (FP8) {
        uint16_t *orow = static_cast<uint16_t *>(a.o) +
                         (static_cast<size_t>(bh) * a.N + static_cast<size_t>(q_row)) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          const uint32_t (&o)[32] = oall[c0 / 32];
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          if (q_row < a.N) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
      } else {
        // O (then its residual) goes through the Q_x tile, free once the last
        // P_x V is done (every S_x product was issued before it), in the
        // 128-byte-swizzled box layout of the tensor map, and leaves by TMA
        // stores: the CTA waits only until the boxes are read, not written.
        // Rows past N are outside the tensor and are not written.
        const uint32_t stage = sbase + C::kQOff + x * C::kTileBytes;
        const bool res = a.o_res != nullptr;
        for (int pass = 0; pass < (res ? 2 : 1); ++pass) {
          if (pass == 1) {  // the O boxes must have been read before the residual overwrites them
            if (row == 0) bulk_wait_read0();
            named_bar_sync(2 + x, 128);
          }
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            const uint32_t (&o)[32] = oall[c0 / 32];
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float x0 = __uint_as_float(o[2 * i]) * inv_l, x1 = __uint_as_float(o[2 * i + 1]) * inv_l;
              const uint32_t pk = pack2<BF16>(x0, x1);
              w[i] = pass == 0 ? pk : pack2<BF16>(x0 - unpack_lo<BF16>(pk), x1 - unpack_hi<BF16>(pk));
            }
            // columns c0 .. c0 + 31 are 16-byte chunks 4 (c0 % 64) / 32 .. +3
            // of this row in box c0 / 64
            const uint32_t rbase = stage + (c0 / 64) * 16384 + row * 128;
            const int ch0 = (c0 % 64) / 8;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                               rbase + (static_cast<uint32_t>((ch0 + v) ^ (row & 7)) << 4)),
                           "r"(w[4 * v]), "r"(w[4 * v + 1]), "r"(w[4 * v + 2]), "r"(w[4 * v + 3])
                           : "memory");
          }
          fence_proxy_async_smem();
          named_bar_sync(2 + x, 128);
          if (row == 0) {
#pragma unroll
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_store_3d(pass == 0 ? &tm_o : &tm_r, stage + kb * 16384, kb * 64, qt * 128, bh);
            bulk_commit();
          }
        }
        if (row == 0) bulk_wait_read0();
      }
      if (q_row < a.N)
        a.lse[static_cast<size_t>(bh) * a.N + q_row] =
            (l > 0.f) ? (m + log2f(l) - (FP8 ? 8.f : 0.f)) * 0.69314718055994530942f : -INFINITY;
    }
    // teardown of the softmax warpgroups
    tc_fence_before();
    named_bar_sync(1, 384);
  }
}

}  // namespace fa
