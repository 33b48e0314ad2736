// fwd_small_kernel.cuh -- forward attention for short sequences, sm_103a.
//
// The block loop of "Flash Attention: revolutionizing transformer
// efficiency" (query blocks outer, key/value blocks inner, running max m and
// sum l; softmax_row.cuh), one 128-row query tile per CTA, sized so that two
// CTAs share each SM. With few key tiles per query tile (N <= 2048) a CTA's
// start-up (barrier set-up, TMEM allocation, first Q/K/V latency) and its
// epilogue are a large part of its life; a second resident CTA runs its
// tiles meanwhile. 256 threads launched with 128 registers each, 256 TMEM
// columns (S, into which P is written once S is read, then O), one K and
// one V stage.
//
// Roles (setmaxnreg moves registers from warpgroup 1 to warpgroup 0):
//   warps 0..3     softmax, one query row per thread (TMEM lanes 0..127)
//   warp 4 lane 0  TMA producer (Q once; K/V ring)
//   warp 5         TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 6, 7     idle
// Per key tile t the MMA thread issues S = Q K_t^T once P(t-1) V(t-1) is
// done (S holds P), then O += P(t) V(t) once P(t) and V(t) are in place.
// The arithmetic per row and the P V product order (two 64-key halves) are
// those of the two-tile kernel.
#pragma once
#include "common.cuh"
#include "fwd_kernel.cuh"
#include "softmax_row.cuh"

namespace fa {

template <int D>
struct SmallCfg {
  static constexpr int kKB = D / 64;               // 128-byte column blocks
  static constexpr int kTileBytes = 128 * D * 2;   // one 128-row tile
  // d = 64: P gets TMEM columns of its own and K, V get two stages each, so
  // the next Q K^T waits only until the softmax has read S, not for P V;
  // d = 128: P is written over S (the 256 columns hold S and O), one stage.
  static constexpr bool kSepP = (D == 64);
  static constexpr int kKStages = kSepP ? 2 : 1;
  static constexpr int kVStages = kSepP ? 2 : 1;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kBQ = 0;
  static constexpr int kBKF = 1;                   // [kKStages]
  static constexpr int kBKE = kBKF + kKStages;     // [kKStages]
  static constexpr int kBVF = kBKE + kKStages;     // [kVStages]
  static constexpr int kBVE = kBVF + kVStages;     // [kVStages]
  static constexpr int kBSF = kBVE + kVStages;     // S(t) in TMEM
  static constexpr int kBSR = kBSF + 1;            // S(t) read by the softmax (128 arrivals; d = 64)
  static constexpr int kBPF = kBSR + 1;            // [2] half h of P(t) in TMEM (128 arrivals)
  static constexpr int kBOR = kBPF + 2;            // P(t) V(t) done
  static constexpr int kBDR = kBOR + 1;            // drain
  static constexpr int kNumBars = kBDR + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag, list count
  static constexpr int kListOff = kMiscOff + 16;            // block-sparse: kept key tiles
  static constexpr int kMaxList = 2048;                     // nkt <= 2048
  static constexpr int kSmemBytes = kListOff + kMaxList * 2 + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0, kColP = kSepP ? 128 : 0, kColO = kSepP ? 192 : 128;
  static constexpr uint32_t kTmemCols = 256;
  static_assert(kColO + D <= kTmemCols && (!kSepP || kColP + 64 <= kColO), "TMEM budget");
  // setmaxnreg split: launch with 128 registers x 256 threads (two CTAs per
  // SM); warpgroup 1 gives back to 48, the softmax warpgroup takes 208.
  static constexpr int kLaunchRegs = 128, kRegsLow = 48, kRegsHigh = 208;
  static_assert(kRegsLow * 128 + kRegsHigh * 128 <= kLaunchRegs * 256, "register split");
  // two CTAs per SM: 228 KB per SM, 1 KB reserved per CTA
  static_assert(2 * (kSmemBytes + 1024) <= 233472, "shared memory for two CTAs per SM");
};

template <int D, bool BF16, bool CAUSAL, bool SPARSE = false, bool SPLIT = false>
__global__ void __launch_bounds__(256, 2)
    fwd_small_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using C = SmallCfg<D>;
  extern __shared__ uint8_t smem_small[];
  const uint32_t raw = smem_u32(smem_small);
  const uint32_t sbase = align_up_1024(raw);
  uint8_t *smem = smem_small + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile uint32_t *abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };

  // ---- work item: heads are contiguous in the grid so concurrent CTAs share
  // K/V in L2; causal rows run heaviest tile first.
  const WorkItem item = tile_item(static_cast<int>(blockIdx.x), a.nqt, CAUSAL);
  const int bh = item.bh, qt = item.tile;
  const int b = bh / a.H;
  const int kvh = a.kv_head(bh);
  int kvl = a.N;
  if (a.kv_len != nullptr) {
    const int v = a.kv_len[b];
    kvl = v < 0 ? 0 : (v > a.N ? a.N : v);
  }
  const int nkt_eff = (kvl + 127) >> 7;
  uint16_t *list = reinterpret_cast<uint16_t *>(smem + C::kListOff);

  if (tid == 0) {
    mbar_init(bar(C::kBQ), 1);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(bar(C::kBKF + i), 1);
      mbar_init(bar(C::kBKE + i), 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(bar(C::kBVF + i), 1);
      mbar_init(bar(C::kBVE + i), 1);
    }
    mbar_init(bar(C::kBSF), 1);
    mbar_init(bar(C::kBSR), 128);
    mbar_init(bar(C::kBPF), 128);
    mbar_init(bar(C::kBPF + 1), 128);
    mbar_init(bar(C::kBOR), 1);
    mbar_init(bar(C::kBDR), 1);
    *abort_flag = 0u;
    fence_barrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 5) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  if (SPARSE && warp == 6) {
    // kept key tiles of this query tile, in increasing order (block-sparse)
    const uint8_t *mrow = a.block_mask + static_cast<size_t>(qt) * a.nkt;
    int cnt = 0;
    for (int j0 = 0; j0 < nkt_eff; j0 += 32) {
      const int j = j0 + lane;
      const bool keep = (j < nkt_eff) && (mrow[j] != 0);
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (keep) list[cnt + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(j);
      cnt += __popc(bal);
    }
    if (lane == 0) misc[2] = static_cast<uint32_t>(cnt);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int n_all = SPARSE ? static_cast<int>(misc[2]) : (CAUSAL ? min(qt + 1, nkt_eff) : nkt_eff);
  // split-KV: this CTA's contiguous share [t_lo, t_lo + n_tiles) of the tiles
  const int split = SPLIT ? static_cast<int>(blockIdx.y) : 0;
  int t_lo = 0, n_tiles = n_all;
  if constexpr (SPLIT) split_share(n_all, split, a.num_splits, &t_lo, &n_tiles);

  if (warp >= 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsLow));
  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0 && !pipelines_starved()) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(bar(C::kBQ), C::kTileBytes);
      for (int kb = 0; kb < C::kKB; ++kb)
        tma_load_3d_hint(sbase + C::kQOff + kb * 16384, &tm_q, bar(C::kBQ), kb * 64, qt * 128, bh, pol_q);
      int nk = 0, nv = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int ks = t % C::kKStages, vs = t % C::kVStages;
        const uint32_t kph = (t / C::kKStages) & 1, vph = (t / C::kVStages) & 1;
        const int kt = SPARSE ? list[t_lo + t] : t_lo + t;
        if (!mbar_wait(bar(C::kBKE + ks), kph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBKF + ks), C::kTileBytes);
        for (int kb = 0; kb < C::kKB; ++kb)
          tma_load_3d_hint(sbase + C::kKOff + ks * C::kTileBytes + kb * 16384, &tm_k, bar(C::kBKF + ks),
                           kb * 64, kt * 128, kvh, pol_kv);
        nk = t + 1;
        if (!mbar_wait(bar(C::kBVE + vs), vph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBVF + vs), C::kTileBytes);
        for (int kb = 0; kb < C::kKB; ++kb)
          tma_load_3d_hint(sbase + C::kVOff + vs * C::kTileBytes + kb * 16384, &tm_v, bar(C::kBVF + vs),
                           kb * 64, kt * 128, kvh, pol_kv);
        nv = t + 1;
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA exits
        mbar_wait_drain(bar(C::kBQ), 0, abort_flag);
        for (int t = max(0, nk - C::kKStages); t < nk; ++t)
          mbar_wait_drain(bar(C::kBKF + t % C::kKStages), (t / C::kKStages) & 1, abort_flag);
        for (int t = max(0, nv - C::kVStages); t < nv; ++t)
          mbar_wait_drain(bar(C::kBVF + t % C::kVStages), (t / C::kVStages) & 1, abort_flag);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdQK = idesc_f16(BF16, 128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_f16(BF16, 128, D, false, true);
      bool ok = mbar_wait(bar(C::kBQ), 0, abort_flag);
      // S(t) = Q K(t)^T into the S columns
      auto issue_qk = [&](int t) {
        const uint32_t sb = opaque_u32(sbase);
        // descriptors as 32-bit words stepped by adds (sdesc_lo): few
        // instructions per product for this thread
        const uint32_t q_k = sdesc_lo(sb + C::kQOff, 16);
        const uint32_t k_k = sdesc_lo(sb + C::kKOff + (t % C::kKStages) * C::kTileBytes, 16);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          // A = Q, B = K_j, both K-major: 16 channels = 32 B per step
          const uint32_t o = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
          mma_ss_w(tmem + C::kColS, q_k + o, k_k + o, sdesc_hi(1024), kIdQK, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBSF));
        mma_commit(bar(C::kBKE + t % C::kKStages));
      };
      if constexpr (C::kSepP) {
        // P has its own columns: S(t + 1) only waits until the softmax has
        // read S(t), so it runs while the softmax of tile t works
        if (ok && mbar_wait(bar(C::kBKF), 0, abort_flag)) {
          tc_fence_after();
          issue_qk(0);
        } else {
          ok = false;
        }
      }
      for (int t = 0; ok && t < n_tiles; ++t) {
        const uint32_t ph = t & 1;
        if constexpr (C::kSepP) {
          if (t + 1 < n_tiles) {
            if (!mbar_wait(bar(C::kBKF + (t + 1) % C::kKStages), ((t + 1) / C::kKStages) & 1, abort_flag) ||
                !mbar_wait(bar(C::kBSR), ph, abort_flag)) { ok = false; break; }
            tc_fence_after();
            issue_qk(t + 1);
          }
        } else {
          if (!mbar_wait(bar(C::kBKF), ph, abort_flag)) { ok = false; break; }
          // S holds P(t-1) until P(t-1) V(t-1) is done
          if (t > 0 && !mbar_wait(bar(C::kBOR), (t - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          issue_qk(t);
        }
        const int vs = t % C::kVStages;
        if (!mbar_wait(bar(C::kBVF + vs), (t / C::kVStages) & 1, abort_flag)) { ok = false; break; }
        const uint32_t v_mn = sdesc_lo(opaque_u32(sbase) + C::kVOff + vs * C::kTileBytes, 16384);
        // O += P(t) V(t) in two halves of 64 keys
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(bar(C::kBPF + h), ph, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int k = 4 * h; k < 4 * h + 4; ++k)
            // B = V_j, MN-major: 16 keys per step = 16 rows of 128 B
            mma_ts_w(tmem + C::kColO, tmem + C::kColP + k * 8, v_mn + k * 128, sdesc_hi(1024), kIdPV,
                     (t > 0 || k > 0) ? 1u : 0u);
        }
        if (!ok) break;
        mma_commit(bar(C::kBVE + vs));
        mma_commit(bar(C::kBOR));
      }
      // every issued MMA must finish before TMEM is released
      mma_commit(bar(C::kBDR));
      mbar_wait_drain(bar(C::kBDR), 0, abort_flag);
    }
  }
    // teardown of warpgroup 1 (the two register regions do not rejoin)
    tc_fence_before();
    named_bar_sync(1, 256);
    if (warp == 5) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, C::kTmemCols);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsHigh));
    // ------------------------------------------------------------ softmax
    const int row = tid;  // 0 .. 127
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t scol = tmem + lane_addr + C::kColS;
    const uint32_t pcol = tmem + lane_addr + C::kColP;
    const uint32_t ocol = tmem + lane_addr + C::kColO;
    const int q_row = qt * 128 + row;
    const float sl2 = a.scale_log2;
    // a warp whose rows all lie past N keeps only the barriers' counts in
    // step (d = 128: S(t) complete implies their previous phase completed)
    const bool pad_warp = qt * 128 + warp * 32 >= a.N;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait_warp(bar(C::kBSF), t & 1, abort_flag)) { ok = false; break; }
      if (pad_warp) {
        if constexpr (C::kSepP) {
          mbar_arrive(bar(C::kBSR));
          // S(t + 1) may start before P(t) is written, so a warp without rows
          // would run ahead into tile t + 1 and arrive on the P barriers for
          // it while tile t's phase still waits for the other warps: it
          // waits for P(t-1) V(t-1), which completes every earlier phase
          if (t > 0 && !mbar_wait_warp(bar(C::kBOR), (t - 1) & 1, abort_flag)) { ok = false; break; }
        }
        mbar_arrive(bar(C::kBPF));
        mbar_arrive(bar(C::kBPF + 1));
        continue;
      }
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
        if constexpr (C::kSepP) {  // S is in registers: the next Q K^T may overwrite it
          tc_fence_before();
          mbar_arrive(bar(C::kBSR));
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
          s[64 + c] = __uint_as_float(r2[c]);
          s[96 + c] = __uint_as_float(r3[c]);
        }
      }
      // mask: keys past kv_len / N, and keys after the query on the diagonal
      const int kt = SPARSE ? list[t_lo + t] : t_lo + t;
      int limit = kvl - kt * 128;
      if (CAUSAL && kt == qt) limit = min(limit, row + 1);
      float m_new, alpha;
      const float nm = softmax_max(s, limit, sl2, m, m_new, alpha);
      // O holds every earlier tile once P(t-1) V(t-1) is done (d = 128: S(t)
      // waited for it; d = 64: wait here, which also frees the P columns)
      if (C::kSepP && t > 0) {
        if (!mbar_wait_warp(bar(C::kBOR), (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
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
      softmax_exp<0, 64>(s, sl2, nm, acc);
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t hi[16];
        pack_p32<BF16>(s, c0, hi);
        tmem_st_32x32b_x16(pcol + c0 / 2, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBPF));
      softmax_exp<64, 128>(s, sl2, nm, acc);
#pragma unroll
      for (int c0 = 64; c0 < 128; c0 += 32) {
        uint32_t hi[16];
        pack_p32<BF16>(s, c0, hi);
        tmem_st_32x32b_x16(pcol + c0 / 2, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBPF + 1));
      l = l * alpha + softmax_sum(acc);
      m = m_new;
    }
    // ---- epilogue: O / l, its rounding residual, and LSE of the real rows
    if (!pad_warp) {
      bool have_o = ok && n_tiles > 0;
      if (have_o) {
        have_o = mbar_wait_warp(bar(C::kBOR), (n_tiles - 1) & 1, abort_flag);
        tc_fence_after();
      }
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      uint16_t *orow = static_cast<uint16_t *>(a.o) + (static_cast<size_t>(bh) * a.N + q_row) * D;
      // split-KV partial (rows < N only; the merge reads no others): O / l in
      // fp32 and this share's LSE, in the layout fwd_merge_kernel reads
      const size_t prow = static_cast<size_t>(split) * a.nqt * 128 * (gridDim.x / a.nqt) +
                          static_cast<size_t>(bh) * a.nqt * 128 + static_cast<size_t>(q_row);
#pragma unroll 1
      for (int j = 0; j < D / 32; ++j) {
        uint32_t o[32];
        if (have_o) {
          tmem_ld_32x32b_x32(ocol + 32 * j, o);
          tmem_wait_ld();
          reg_fence_32(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if constexpr (SPLIT) {
          if (q_row < a.N) {
            float4 *dst = reinterpret_cast<float4 *>(a.o_part + prow * D + 32 * j);
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              dst[i / 4] = make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                       __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
          }
        } else {
          uint32_t pk[16], rk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x0 = __uint_as_float(o[2 * i]) * inv_l, x1 = __uint_as_float(o[2 * i + 1]) * inv_l;
            pk[i] = pack2<BF16>(x0, x1);
            rk[i] = pack2<BF16>(x0 - unpack_lo<BF16>(pk[i]), x1 - unpack_hi<BF16>(pk[i]));
          }
          if (q_row < a.N) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * j);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            if (a.o_res != nullptr) {
              uint4 *dr = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.o_res) +
                                                    (orow - static_cast<uint16_t *>(a.o)) + 32 * j);
#pragma unroll
              for (int v = 0; v < 4; ++v) dr[v] = make_uint4(rk[4 * v], rk[4 * v + 1], rk[4 * v + 2], rk[4 * v + 3]);
            }
          }
        }
      }
      if (q_row < a.N)
        (SPLIT ? a.lse_part[prow] : a.lse[static_cast<size_t>(bh) * a.N + q_row]) =
            (l > 0.f) ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
    // teardown of the softmax warpgroup
    tc_fence_before();
    named_bar_sync(1, 256);
  }
}

}  // namespace fa
