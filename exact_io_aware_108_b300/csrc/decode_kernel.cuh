// decode_kernel.cuh -- attention of a few new tokens per sequence against a
// paged key/value cache, for sm_103a.
//
// The cache is a pool of pages [num_pages * Hkv][page_size][D] ("Enhancing
// Transformer Models: Innovations in Attention Mechanisms and Performance
// Optimization", section "From FlashAttention to PagedAttention": attention
// data moved between HBM and on-chip memory page by page); key tile kt of
// the sequence of batch b gathers the pool pages block_table[b *
// pages_per_seq + kt * 128 / page_size + p], one TMA box per page and
// 64-channel half, into the dense 128-key tile layout. The arithmetic per
// row is the online softmax of the forward (softmax_row.cuh).
//
// One CTA per (sequence, key/value head, query tile of 64 rows, share of the
// key tiles). The 64 query rows are the dec_nq new tokens of the H / Hkv
// query heads of one key/value head (row r sees keys j <= kv_len[b] - dec_nq
// + r % dec_nq); the M = 128 products read rows 64..127 of "Q" from the
// memory after the Q tile, which only feeds TMEM lanes 64..127 of S and O,
// never read.
//
// The key walk is bound by HBM, and one CTA's chain per key tile (S -> the
// softmax -> P V, with the V refill waiting for P V) leaves the load latency
// exposed; so the kernel is sized for two CTAs per SM, whose chains overlap:
// 128 threads, 256 TMEM columns (S with P aliased into its first 64 columns
// once read, then O), about 83 KB of shared memory (Q, one K stage, one V
// stage at d = 128).
//
// Roles:
//   warps 0, 1     softmax, one query row per thread (TMEM lanes 0..63)
//   warp 2 lane 0  TMA producer (Q once; K and V tiles, block table one tile
//                  ahead); then the whole warp zeroes the V rows past kv_len
//                  of the sequence's last tile (stale cache slots must not
//                  reach P V as 0 * non-finite)
//   warp 3         TMEM allocation; lane 0 issues every tcgen05.mma
#pragma once
#include "common.cuh"
#include "fwd_kernel.cuh"
#include "softmax_row.cuh"

namespace fa {

template <int D>
struct DecCfg {
  static constexpr int kQRows = 64;
  static constexpr int kKB = D / 64;               // 128-byte column blocks
  static constexpr int kQColBlock = kQRows * 128;  // bytes of one Q column block
  static constexpr int kQBytes = kQColBlock * kKB;
  static constexpr int kTileBytes = 128 * D * 2;   // one 128-key K or V tile
  static constexpr int kKStages = 1;
  static constexpr int kVStages = (D == 64) ? 2 : 1;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kBQ = 0;
  static constexpr int kBKF = 1;
  static constexpr int kBKE = kBKF + kKStages;
  static constexpr int kBVF = kBKE + kKStages;
  static constexpr int kBVE = kBVF + kVStages;
  static constexpr int kBSF = kBVE + kVStages;  // S(t) in TMEM
  static constexpr int kBPF = kBSF + 1;         // P(t) in TMEM (64 arrivals)
  static constexpr int kBOR = kBPF + 1;         // P(t) V(t) done
  static constexpr int kBVL = kBOR + 1;         // last V tile landed (single use)
  static constexpr int kBVZ = kBVL + 1;         // its tail rows zeroed (single use)
  static constexpr int kBDR = kBVZ + 1;         // drain
  static constexpr int kNumBars = kBDR + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0, kColO = 128, kTmemCols = 256;
  // two CTAs per SM: 228 KB per SM, 1 KB reserved per CTA
  static_assert(2 * (kSmemBytes + 1024) <= 233472, "shared memory for two CTAs per SM");
};

template <int D, bool BF16>
__global__ void __launch_bounds__(128, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_dec[];
  const uint32_t raw = smem_u32(smem_dec);
  const uint32_t sbase = align_up_1024(raw);
  uint8_t *smem = smem_dec + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile uint32_t *abort_flag = misc + 1;
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8u * static_cast<uint32_t>(i); };

  // ---- work item (a.H holds Hkv: the grid runs over key/value heads)
  const int bh = static_cast<int>(blockIdx.x) / a.nqt;
  const int qt = static_cast<int>(blockIdx.x) % a.nqt;
  const int b = bh / a.Hkv, kvh = bh % a.Hkv;
  const int kv_cap = a.pages_per_seq * a.page_size;
  int kvl = kv_cap;
  if (a.kv_len != nullptr) {
    const int v = a.kv_len[b];
    kvl = v < 0 ? 0 : (v > kv_cap ? kv_cap : v);
  }
  const int n_all = (kvl + 127) >> 7;
  const int split = static_cast<int>(blockIdx.y);
  const int t_lo = static_cast<int>(static_cast<long long>(n_all) * split / a.num_splits);
  const int n_tiles = static_cast<int>(static_cast<long long>(n_all) * (split + 1) / a.num_splits) - t_lo;
  const bool zero_tail = n_tiles > 0 && t_lo + n_tiles == n_all && (kvl & 127) != 0;

  if (tid == 0) {
    mbar_init(bar(C::kBQ), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(bar(C::kBKF + s), 1);
      mbar_init(bar(C::kBKE + s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(bar(C::kBVF + s), 1);
      mbar_init(bar(C::kBVE + s), 1);
    }
    mbar_init(bar(C::kBSF), 1);
    mbar_init(bar(C::kBPF), 64);
    mbar_init(bar(C::kBOR), 1);
    mbar_init(bar(C::kBVL), 1);
    mbar_init(bar(C::kBVZ), 1);
    mbar_init(bar(C::kBDR), 1);
    *abort_flag = 0u;
    fence_barrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  if (warp == 3) {
    tmem_alloc(sbase + C::kMiscOff, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0 && !pipelines_starved()) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_first();  // every cache page is read once
      mbar_arrive_expect_tx(bar(C::kBQ), C::kQBytes);
      for (int kb = 0; kb < C::kKB; ++kb)
        tma_load_3d_hint(sbase + C::kQOff + kb * C::kQColBlock, &tm_q, bar(C::kBQ), kb * 64, qt * C::kQRows, bh,
                         pol_q);
      const int ppt = 128 / a.page_size;
      const int32_t *bt_row = a.block_table + static_cast<size_t>(b) * a.pages_per_seq;
      auto pages_of = [&](int kt) { return min(ppt, (kvl - kt * 128 + a.page_size - 1) / a.page_size); };
      // pool coordinates of the next tile's pages, read one tile ahead
      int zc_next[8];
      {
        const int np0 = pages_of(t_lo);
#pragma unroll
        for (int p = 0; p < 8; ++p) zc_next[p] = (p < np0) ? bt_row[t_lo * ppt + p] * a.Hkv + kvh : 0;
      }
      const uint32_t rowb = static_cast<uint32_t>(a.page_size * 128);
      int nk = 0, nv = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int kt = t_lo + t;
        const int npg = pages_of(kt);
        int zc[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) zc[p] = zc_next[p];
        if (t + 1 < n_tiles) {
          const int np1 = pages_of(kt + 1);
#pragma unroll
          for (int p = 0; p < 8; ++p) zc_next[p] = (p < np1) ? bt_row[(kt + 1) * ppt + p] * a.Hkv + kvh : 0;
        }
        const uint32_t bytes = static_cast<uint32_t>(npg * a.page_size * D * 2);
        const int ks = t % C::kKStages, vs = t % C::kVStages;
        if (!mbar_wait(bar(C::kBKE + ks), ((t / C::kKStages) & 1) ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBKF + ks), bytes);
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < npg)
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d_hint(sbase + C::kKOff + ks * C::kTileBytes + kb * 16384 + p * rowb, &tm_k,
                               bar(C::kBKF + ks), kb * 64, 0, zc[p], pol_kv);
        nk = t + 1;
        if (!mbar_wait(bar(C::kBVE + vs), ((t / C::kVStages) & 1) ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBVF + vs), bytes);
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < npg)
            for (int kb = 0; kb < C::kKB; ++kb)
              tma_load_3d_hint(sbase + C::kVOff + vs * C::kTileBytes + kb * 16384 + p * rowb, &tm_v,
                               bar(C::kBVF + vs), kb * 64, 0, zc[p], pol_kv);
        nv = t + 1;
      }
      // the last V tile: waited here by the thread that loaded it (its phase is
      // unambiguous), then handed to the whole warp for the tail zeroing
      if (zero_tail && nv == n_tiles &&
          mbar_wait(bar(C::kBVF + (n_tiles - 1) % C::kVStages), ((n_tiles - 1) / C::kVStages) & 1, abort_flag))
        mbar_arrive(bar(C::kBVL));
      if (*abort_flag) {
        mbar_wait_drain(bar(C::kBQ), 0, abort_flag);
        for (int t = max(0, nk - C::kKStages); t < nk; ++t)
          mbar_wait_drain(bar(C::kBKF + t % C::kKStages), (t / C::kKStages) & 1, abort_flag);
        for (int t = max(0, nv - C::kVStages); t < nv; ++t)
          mbar_wait_drain(bar(C::kBVF + t % C::kVStages), (t / C::kVStages) & 1, abort_flag);
      }
    }
    __syncwarp();
    if (zero_tail && mbar_wait_warp(bar(C::kBVL), 0, abort_flag)) {
      const int t = n_tiles - 1;
      const int valid = kvl - (t_lo + t) * 128;  // 1 .. 127 keys of the tile are real
      // whole 128-byte rows: the swizzle only permutes 16-byte chunks within a row
      uint8_t *vt = smem + C::kVOff + (t % C::kVStages) * C::kTileBytes;
      for (int kb = 0; kb < C::kKB; ++kb)
        for (int i = lane; i < (128 - valid) * 8; i += 32)
          *reinterpret_cast<uint4 *>(vt + kb * 16384 + (valid + (i >> 3)) * 128 + (i & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::kBVZ));
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdQK = idesc_f16(BF16, 128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_f16(BF16, 128, D, false, true);
      bool ok = mbar_wait(bar(C::kBQ), 0, abort_flag);
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int ks = t % C::kKStages, vs = t % C::kVStages;
        if (!mbar_wait(bar(C::kBKF + ks), (t / C::kKStages) & 1, abort_flag)) { ok = false; break; }
        // S holds P(t-1) until P(t-1) V(t-1) is done
        if (t > 0 && !mbar_wait(bar(C::kBOR), (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sb = opaque_u32(sbase);
        const uint32_t kbase = sb + C::kKOff + ks * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          // A = Q, B = K_j, both K-major: 16 channels = 32 B per step
          const uint32_t qoff = (k >> 2) * C::kQColBlock + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
          mma_ss(tmem + C::kColS, sdesc_sw128(sb + C::kQOff + qoff, 16, 1024), sdesc_sw128(kbase + koff, 16, 1024),
                 kIdQK, k > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBSF));
        mma_commit(bar(C::kBKE + ks));
        // O += P(t) V(t): P as 16-bit pairs in the first 64 columns of S
        if (!mbar_wait(bar(C::kBPF), t & 1, abort_flag)) { ok = false; break; }
        if (zero_tail && t == n_tiles - 1) {
          if (!mbar_wait(bar(C::kBVZ), 0, abort_flag)) { ok = false; break; }
        } else if (!mbar_wait(bar(C::kBVF + vs), (t / C::kVStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vbase = sb + C::kVOff + vs * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          // B = V_j, MN-major: 16 keys per step = 16 rows of 128 B
          mma_ts(tmem + C::kColO, tmem + C::kColS + k * 8, sdesc_sw128(vbase + k * 2048, 16384, 1024), kIdPV,
                 (t > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(C::kBVE + vs));
        mma_commit(bar(C::kBOR));
      }
      // every issued MMA must finish before TMEM is released
      mma_commit(bar(C::kBDR));
      mbar_wait_drain(bar(C::kBDR), 0, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = tid;  // 0 .. 63
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t scol = tmem + lane_addr + C::kColS;
    const uint32_t ocol = tmem + lane_addr + C::kColO;
    const int q_row = qt * C::kQRows + row;
    const float sl2 = a.scale_log2;
    // a warp whose rows all lie past N keeps only the P barrier's count in
    // step (S(t) complete implies the barrier's previous phase completed)
    const bool pad_warp = qt * C::kQRows + warp * 32 >= a.N;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait_warp(bar(C::kBSF), t & 1, abort_flag)) { ok = false; break; }
      if (pad_warp) {
        mbar_arrive(bar(C::kBPF));
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
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s[c] = __uint_as_float(r0[c]);
          s[32 + c] = __uint_as_float(r1[c]);
          s[64 + c] = __uint_as_float(r2[c]);
          s[96 + c] = __uint_as_float(r3[c]);
        }
      }
      const int kt = t_lo + t;
      const int limit = (q_row < a.N) ? kvl - kt * 128 - a.dec_nq + 1 + q_row % a.dec_nq : 0;
      float m_new, alpha;
      const float nm = softmax_max(s, limit, sl2, m, m_new, alpha);
      // S(t) complete implies P(t-1) V(t-1) is done (S(t) waited for it): O
      // is final for tile t - 1 and can be rescaled
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
      softmax_exp<0, 128>(s, sl2, nm, acc);
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t hi[16];
        pack_p32<BF16>(s, c0, hi);
        tmem_st_32x32b_x16(scol + c0 / 2, hi);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBPF));
      l = l * alpha + softmax_sum(acc);
      m = m_new;
    }
    // ---- epilogue: O / l and LSE of the real rows
    if (!pad_warp) {
      bool have_o = ok && n_tiles > 0;
      if (have_o) {
        have_o = mbar_wait_warp(bar(C::kBOR), (n_tiles - 1) & 1, abort_flag);
        tc_fence_after();
      }
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const float lse_row = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
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
      if (q_row < a.N) {
        if (a.num_splits > 1) {
          // this share's O / l in fp32 and its LSE, merged by fwd_merge_kernel
          const size_t prow = static_cast<size_t>(split) * a.nqt * 128 * (gridDim.x / a.nqt) +
                              static_cast<size_t>(bh) * a.nqt * 128 + static_cast<size_t>(q_row);
          float4 *dst = reinterpret_cast<float4 *>(a.o_part + prow * D);
#pragma unroll
          for (int j = 0; j < D / 32; ++j)
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              dst[(32 * j + i) / 4] =
                  make_float4(__uint_as_float(oall[j][i]) * inv_l, __uint_as_float(oall[j][i + 1]) * inv_l,
                              __uint_as_float(oall[j][i + 2]) * inv_l, __uint_as_float(oall[j][i + 3]) * inv_l);
          a.lse_part[prow] = lse_row;
        } else {
          uint16_t *orow = static_cast<uint16_t *>(a.o) + (static_cast<size_t>(bh) * a.N + q_row) * D;
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack2<BF16>(__uint_as_float(oall[j][2 * i]) * inv_l, __uint_as_float(oall[j][2 * i + 1]) * inv_l);
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * j);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
          a.lse[static_cast<size_t>(bh) * a.N + q_row] = lse_row;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 3) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
