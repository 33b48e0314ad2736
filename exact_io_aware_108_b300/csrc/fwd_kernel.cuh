// fwd_kernel.cuh -- forward attention kernel for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, head): the block
// loop of "Flash Attention: revolutionizing transformer efficiency" (sections
// "The Flash Attention Algorithm" and "Implementation Details": query block
// outer, key/value blocks inner, running row max m and row sum l), with the
// output kept unnormalised in TMEM and divided by l once at the end.
//
// Roles (256 threads):
//   warp 0, lane 0  TMA producer: Q tile once, then K_j / V_j tiles through a
//                   ring of shared-memory stages (128-byte swizzle).
//   warp 1          allocates TMEM; lane 0 issues every tcgen05.mma:
//                   S_j = Q K_j^T into one of two TMEM score buffers, and
//                   O += P_j V_j with P_j read from TMEM.
//   warp 2          builds the kept-tile list of a block-sparse row.
//   warps 4..7      softmax: thread r owns query row r (TMEM lane r). Reads
//                   S_j, applies the mask, updates m and l, writes P_j as
//                   16-bit values to TMEM, rescales the O row when m grows,
//                   and finally writes O / l and LSE.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,256+D), P0 and P1 (64
// columns each, two 16-bit probabilities per column) after O.
//
// Online softmax in base 2: x = s * scale * log2(e); p = 2^(x - m);
// l <- 2^(m_old - m) l + sum p; O <- 2^(m_old - m) O + P V
// (softmax decomposition and merger, section "The Math Behind Flash
// Attention"; the per-row update is softmax_row in softmax_row.cuh). m is the
// exact running row max, so the largest probability of a row is exactly 1
// when it is rounded to 16 bits for the P V product, and O is rescaled in
// TMEM whenever any row of the warp sees a new max.
#pragma once
#include "common.cuh"
#include "schedule.cuh"
#include "softmax_row.cuh"

namespace fa {

struct FwdArgs {
  void *o;
  void *o_res;               // [B,H,N,D] rounding residual of O, or null
  float *lse;
  const int32_t *kv_len;     // [B] or null
  const uint8_t *block_mask; // [nkt, nkt] or null
  int H, N, nqt, nkt;
  int hgroup;    // heads per scheduling group of the two-tile kernel's causal launch order
  int Hkv;       // key/value heads (grouped-query attention: H = Hkv * kv_group)
  int kv_group;  // query heads per key/value head
  // split-KV (single-tile kernel only): grid.y = num_splits CTAs share the
  // key tiles of a query tile; each writes O / l (fp32) of its share into
  // o_part [num_splits][BH*nqt*128][D] and its LSE into lse_part
  // [num_splits][BH*nqt*128]; fwd_merge_kernel combines them.
  int num_splits;
  float *o_part;
  float *lse_part;
  float scale_log2;
  float o_scale;  // 8-bit forward: V's dequantisation factor, applied to O
  // paged key/value cache (decode_kernel.cuh): K and V are pools of pages
  // [num_pages * Hkv][page_size][D]; page p of key tile kt of the sequence
  // of batch b is block_table[b * pages_per_seq + kt * 128 / page_size + p];
  // dec_nq new tokens per sequence and query head.
  const int32_t *block_table;
  int page_size, pages_per_seq, dec_nq;

  // [B*Hkv] index of the key/value head that query head bh ([B*H] index) reads
  __device__ __forceinline__ int kv_head(int bh) const { return kv_head_of(bh, H, Hkv); }
};

template <int D>
struct FwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;    // one 128-row tile, 16-bit
  static constexpr int kStages = (D == 64) ? 4 : 2; // K/V ring depth
  static constexpr int kKB = D / 64;                // 128-byte column blocks
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // barriers: Q, K full/empty, V full/empty, S full x2, P full x2, O ready, drain
  static constexpr int kBQ = 0;
  static constexpr int kBKF = 1;
  static constexpr int kBVF = kBKF + kStages;
  static constexpr int kBKE = kBVF + kStages;
  static constexpr int kBVE = kBKE + kStages;
  static constexpr int kBSF = kBVE + kStages;
  static constexpr int kBPF = kBSF + 2;
  static constexpr int kBOR = kBPF + 2;
  static constexpr int kBDR = kBOR + 1;
  static constexpr int kNumBars = kBDR + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort, list count
  static constexpr int kListOff = kMiscOff + 16;
  static constexpr int kMaxList = 2048;                     // block-sparse: nkt <= 2048
  static constexpr int kSmemBytes = kListOff + kMaxList * 2 + 1024;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
  static constexpr uint32_t kColP0 = 256 + D, kColP1 = 256 + D + 64;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kColP1 + 64 <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, bool BF16, bool CAUSAL, bool SPARSE>
__global__ void __launch_bounds__(256, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = align_up_1024(raw);
  uint8_t *smem = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
  volatile uint32_t *abort_flag = misc + 1;
  uint16_t *list = reinterpret_cast<uint16_t *>(smem + C::kListOff);
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

  if (tid == 0) {
    mbar_init(bar(C::kBQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBKF + s), 1);
      mbar_init(bar(C::kBVF + s), 1);
      mbar_init(bar(C::kBKE + s), 1);
      mbar_init(bar(C::kBVE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(C::kBSF + s), 1);
      mbar_init(bar(C::kBPF + s), 128);
    }
    mbar_init(bar(C::kBOR), 1);
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
  if (SPARSE && warp == 2) {
    // kept key tiles of this query tile, in increasing order
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
  const int split = static_cast<int>(blockIdx.y);
  int t_lo, n_tiles;
  split_share(n_all, split, a.num_splits, &t_lo, &n_tiles);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0 && !pipelines_starved()) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      mbar_arrive_expect_tx(bar(C::kBQ), C::kTileBytes);
      for (int kb = 0; kb < C::kKB; ++kb)
        tma_load_3d_hint(sbase + C::kQOff + kb * 16384, &tm_q, bar(C::kBQ), kb * 64, qt * 128, bh,
                         pol_q);
      int nk = 0, nv = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % C::kStages;
        const uint32_t ph = (t / C::kStages) & 1;
        const int kt = SPARSE ? list[t_lo + t] : t_lo + t;
        if (!mbar_wait(bar(C::kBKE + st), ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBKF + st), C::kTileBytes);
        for (int kb = 0; kb < C::kKB; ++kb)
          tma_load_3d_hint(sbase + C::kKOff + st * C::kTileBytes + kb * 16384, &tm_k,
                           bar(C::kBKF + st), kb * 64, kt * 128, kvh, pol_kv);
        nk = t + 1;
        if (!mbar_wait(bar(C::kBVE + st), ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(bar(C::kBVF + st), C::kTileBytes);
        for (int kb = 0; kb < C::kKB; ++kb)
          tma_load_3d_hint(sbase + C::kVOff + st * C::kTileBytes + kb * 16384, &tm_v,
                           bar(C::kBVF + st), kb * 64, kt * 128, kvh, pol_kv);
        nv = t + 1;
      }
      if (*abort_flag) {
        // let every copy still in flight land before the CTA exits
        mbar_wait_drain(bar(C::kBQ), 0, abort_flag);
        for (int t = max(0, nk - C::kStages); t < nk; ++t)
          mbar_wait_drain(bar(C::kBKF + t % C::kStages), (t / C::kStages) & 1, abort_flag);
        for (int t = max(0, nv - C::kStages); t < nv; ++t)
          mbar_wait_drain(bar(C::kBVF + t % C::kStages), (t / C::kStages) & 1, abort_flag);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdQK = idesc_f16(BF16, 128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_f16(BF16, 128, D, false, true);
      bool ok = mbar_wait(bar(C::kBQ), 0, abort_flag);
      tc_fence_after();
      auto issue_pv = [&](int u) -> bool {
        const int st = u % C::kStages;
        const uint32_t ph = (u / C::kStages) & 1;
        const int pb = u & 1;
        if (!mbar_wait(bar(C::kBPF + pb), (u >> 1) & 1, abort_flag)) return false;
        if (!mbar_wait(bar(C::kBVF + st), ph, abort_flag)) return false;
        tc_fence_after();
        const uint32_t vbase = sbase + C::kVOff + st * C::kTileBytes;
        const uint32_t pcol = tmem + (pb ? C::kColP1 : C::kColP0);
        {
          // two halves of 64 keys, high then low part of each (the product
          // order of the two-tile kernel, so both round O identically)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int ks = 4 * h; ks < 4 * h + 4; ++ks) {
              // B = V_j, MN-major: 16 keys per step = 16 rows of 128 B
              mma_ts_w(tmem + C::kColO, pcol + ks * 8, sdesc_lo(vbase, 16384) + ks * 128, sdesc_hi(1024), kIdPV,
                       (u > 0 || ks > 0) ? 1u : 0u);
            }
          }
        }
        mma_commit(bar(C::kBVE + st));
        mma_commit(bar(C::kBOR));
        return true;
      };
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int st = t % C::kStages;
        const uint32_t ph = (t / C::kStages) & 1;
        const int sb = t & 1;
        if (!mbar_wait(bar(C::kBKF + st), ph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kbase = sbase + C::kKOff + st * C::kTileBytes;
        const uint32_t scol = tmem + (sb ? C::kColS1 : C::kColS0);
        const uint32_t q_k = sdesc_lo(sbase + C::kQOff, 16), k_k = sdesc_lo(kbase, 16);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // A = Q, B = K_j, both K-major: 16 head-dim elements = 32 B per step
          const uint32_t o = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
          mma_ss_w(scol, q_k + o, k_k + o, sdesc_hi(1024), kIdQK, ks > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::kBSF + sb));
        mma_commit(bar(C::kBKE + st));
        if (t > 0 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(n_tiles - 1);
      // every issued MMA must finish before TMEM is released
      mma_commit(bar(C::kBDR));
      mbar_wait_drain(bar(C::kBDR), 0, abort_flag);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int row = tid - 128;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int q_row = qt * 128 + row;
    const float sl2 = a.scale_log2;
    // every row of this warp lies past N (the last query tile; the padding of
    // a decode block): its P rows feed only O rows that are never stored, so
    // it skips the softmax and only keeps the P barrier's count in step.
    // S(t) complete implies the P barrier's previous phase of this buffer
    // completed (S(t) overwrote S(t-2) after P(t-2) arrived).
    const bool pad_warp = qt * 128 + (warp & 3) * 32 >= a.N;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int sb = t & 1;
      const int kt = SPARSE ? list[t_lo + t] : t_lo + t;
      if (!mbar_wait_warp(bar(C::kBSF + sb), (t >> 1) & 1, abort_flag)) { ok = false; break; }
      if (pad_warp) {
        mbar_arrive(bar(C::kBPF + sb));
        continue;
      }
      tc_fence_after();
      float s[128];
      {
        const uint32_t scol = tmem + lane_addr + (sb ? C::kColS1 : C::kColS0);
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
      // mask: keys past kv_len / N, and keys after the query on the diagonal
      int limit = kvl - kt * 128;
      if (CAUSAL && kt == qt) limit = min(limit, row + 1);
      float m_new, alpha;
      const float rs = softmax_row(s, limit, sl2, m, m_new, alpha);
      l = l * alpha + rs;
      {
        const uint32_t pcol = tmem + lane_addr + (sb ? C::kColP1 : C::kColP0);
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t hi[16];
          pack_p32<BF16>(s, c0, hi);
          tmem_st_32x32b_x16(pcol + c0 / 2, hi);
        }
      }
      if (t > 0) {
        // O holds P_{t-1} V_{t-1} only once that MMA is done
        if (!mbar_wait_warp(bar(C::kBOR), (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, m_new != m)) {
          // all of the row in one TMEM round trip (a wait::ld costs ~600 cycles)
          uint32_t o[D / 32][32];
#pragma unroll
          for (int j = 0; j < D / 32; ++j) tmem_ld_32x32b_x32(tmem + lane_addr + C::kColO + 32 * j, o[j]);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {
            reg_fence_32(o[j]);
            scale32(o[j], alpha);
            tmem_st_32x32b_x32(tmem + lane_addr + C::kColO + 32 * j, o[j]);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::kBPF + sb));
      m = m_new;
    }
    // ---- epilogue: O / l and LSE
    if (!pad_warp) {
    bool have_o = ok && n_tiles > 0;
    if (have_o) {
      have_o = mbar_wait_warp(bar(C::kBOR), (n_tiles - 1) & 1, abort_flag);
      tc_fence_after();
    }
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    const float lse_row = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    uint16_t *orow = static_cast<uint16_t *>(a.o) +
                     (static_cast<size_t>(bh) * a.N + static_cast<size_t>(q_row)) * D;
    uint32_t oall[D / 32][32];
    if (have_o) {
#pragma unroll
      for (int j = 0; j < D / 32; ++j) tmem_ld_32x32b_x32(tmem + lane_addr + C::kColO + 32 * j, oall[j]);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < D / 32; ++j) reg_fence_32(oall[j]);
    } else {
#pragma unroll
      for (int j = 0; j < D / 32; ++j)
#pragma unroll
        for (int i = 0; i < 32; ++i) oall[j][i] = 0u;
    }
    if (a.num_splits > 1 && q_row < a.N) {
      // split-KV partial: O / l in fp32 and this share's LSE (the merge
      // reads only rows < N)
      const size_t prow = static_cast<size_t>(split) * a.nqt * 128 * (gridDim.x / a.nqt) +
                          static_cast<size_t>(bh) * a.nqt * 128 + static_cast<size_t>(q_row);
      float4 *dst = reinterpret_cast<float4 *>(a.o_part + prow * D);
#pragma unroll
      for (int j = 0; j < D / 32; ++j)
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          dst[(32 * j + i) / 4] = make_float4(__uint_as_float(oall[j][i]) * inv_l, __uint_as_float(oall[j][i + 1]) * inv_l,
                                              __uint_as_float(oall[j][i + 2]) * inv_l, __uint_as_float(oall[j][i + 3]) * inv_l);
      a.lse_part[prow] = lse_row;
    } else if (a.num_splits == 1) {
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      const uint32_t (&o)[32] = oall[c0 / 32];
      uint32_t pk[16], rk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x0 = __uint_as_float(o[2 * i]) * inv_l, x1 = __uint_as_float(o[2 * i + 1]) * inv_l;
        pk[i] = pack2<BF16>(x0, x1);
        rk[i] = pack2<BF16>(x0 - unpack_lo<BF16>(pk[i]), x1 - unpack_hi<BF16>(pk[i]));
      }
      if (q_row < a.N) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        if (a.o_res != nullptr) {
          uint4 *dr = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.o_res) +
                                                (orow - static_cast<uint16_t *>(a.o)) + c0);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dr[v] = make_uint4(rk[4 * v], rk[4 * v + 1], rk[4 * v + 2], rk[4 * v + 3]);
        }
      }
    }
    if (q_row < a.N) a.lse[static_cast<size_t>(bh) * a.N + q_row] = lse_row;
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------- split-KV merge
// Combines the num_splits partial results of each query row with the softmax
// merge identity ("Flash Attention: revolutionizing transformer efficiency",
// section "The Math Behind Flash Attention": for the scores split x u y,
// LSE(x u y) = log(e^LSE(x) + e^LSE(y)) and softmax(x u y) V is the
// e^(LSE(part) - LSE) weighted sum of the parts' results):
//   M = max_s LSE_s, w_s = e^(LSE_s - M), LSE = M + log sum_s w_s,
//   O = sum_s w_s O_s / sum_s w_s.
// A row whose parts all have LSE = -inf (no key) gets O = 0, LSE = -inf.
// One thread per 4 channels of a row.
template <bool BF16>
__global__ void __launch_bounds__(256) fwd_merge_kernel(const FwdArgs a, long long rows, int D) {
  const long long per_row = D / 4;
  const long long tile_rows = static_cast<long long>(a.nqt) * 128;
  const long long part_rows = tile_rows * (rows / a.N);  // BH * nqt * 128
  for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < rows * per_row;
       g += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = g / per_row, c = (g % per_row) * 4;
    const long long bh = row / a.N, i = row % a.N;
    const long long prow = bh * tile_rows + i;
    float mx = -INFINITY;
    for (int sp = 0; sp < a.num_splits; ++sp) mx = fmaxf(mx, a.lse_part[sp * part_rows + prow]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (mx != -INFINITY) {
      for (int sp = 0; sp < a.num_splits; ++sp) {
        const float ls = a.lse_part[sp * part_rows + prow];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - mx);
        const float4 o = *reinterpret_cast<const float4 *>(a.o_part + (sp * part_rows + prow) * D + c);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
        wsum += w;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const float x[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
    uint2 pk, rk;
    pk.x = pack2<BF16>(x[0], x[1]);
    pk.y = pack2<BF16>(x[2], x[3]);
    rk.x = pack2<BF16>(x[0] - unpack_lo<BF16>(pk.x), x[1] - unpack_hi<BF16>(pk.x));
    rk.y = pack2<BF16>(x[2] - unpack_lo<BF16>(pk.y), x[3] - unpack_hi<BF16>(pk.y));
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.o) + row * D + c) = pk;
    if (a.o_res != nullptr) *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.o_res) + row * D + c) = rk;
    if (c == 0) a.lse[row] = (mx == -INFINITY) ? -INFINITY : mx + logf(wsum);
  }
}

}  // namespace fa
