// fa_lib.cu -- the C ABI of libfa.so (declared in include/fa.h): argument
// checks, TMA tensor-map encoding, kernel dispatch and the device error flag.
// All device code is included here so the library is one translation unit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>

#include "fa.h"
#include "fwd_kernel.cuh"
#include "fwd2_kernel.cuh"
#include "fwd_fp8.cuh"
#include "decode_kernel.cuh"
#include "fwd_small_kernel.cuh"
#include "bwd_kernel.cuh"

namespace {

thread_local std::string g_last_error;

fa_status fail(fa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

fa_status ok() {
  g_last_error.clear();
  return FA_OK;
}

fa_status cuda_fail(cudaError_t e, const char *what) {
  return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [B*H, N, d] 16-bit tensor viewed as a 3-D TMA map with 64 x 128 x 1 boxes
// (one 128-byte-wide column block of a 128-row tile), 128-byte swizzle.
// Rows past N read as zero.
fa_status make_tile_map(CUtensorMap *m, const void *ptr, fa_dtype dt, int N, long long BH, int d,
                        const char *name, unsigned box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, dt == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return FA_OK;
}

// 8-bit tensor [rows_outer, rows, inner] (inner bytes contiguous, row pitch
// `pitch` bytes, a multiple of 16) as a 3-D TMA map with 128 x 128 x 1 boxes
// (128 bytes wide), 128-byte swizzle. Elements past `inner` or `rows` read
// as zero.
fa_status make_tile_map8(CUtensorMap *m, const void *ptr, long long inner, long long pitch, int rows,
                         long long outer, const char *name) {
  auto fn = encode_fn();
  if (!fn) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch),
                           static_cast<cuuint64_t>(pitch) * static_cast<cuuint64_t>(rows)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return FA_OK;
}

// Heads per scheduling group of the causal launch order: CTAs of a group
// run heaviest first; the group's two streamed 16-bit tensors (K and V in
// the forward, Q and dO in the backward) are kept to about 48 MB so they
// stay in the 126 MB L2 while the group runs. Non-causal grids keep one
// head per group (equal work per CTA).
int head_group(int N, int d, bool causal) {
  if (!causal) return 1;
  const long long per_head = static_cast<long long>(N) * d * 2 * 2;
  long long g = (48ll << 20) / per_head;
  return static_cast<int>(g < 1 ? 1 : (g > 16 ? 16 : g));
}

// The two-tile forward's group: the largest power of two heads within the
// 48 MB rule and at most 8. Measured on the long-context sweep (B * N =
// 32768, H = 16, d = 128): groups of 8 against the rule's 16 / 12 / 6 heads
// at N = 4096 / 8192 / 16384 ran equal / 2 % / 4 % faster; a group size
// that leaves a short last group costs.
int fwd_head_group(int N, int d, bool causal) {
  const int g = head_group(N, d, causal);
  int p = 1;
  while (p * 2 <= g && p * 2 <= 8) p *= 2;
  return p;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Shape {
  int B, H, N, d;
  long long BH;
  int nqt;
};

fa_status check_common(int B, int H, int N, int d, float scale, fa_dtype dt, Shape *s) {
  if (B < 1 || H < 1 || N < 1) return fail(FA_ERR_INVALID_ARG, "B, H, N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (d < 1) return fail(FA_ERR_INVALID_ARG, "d must be >= 1 (got %d)", d);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d not built (64 or 128)", d);
  if (dt != FA_F16 && dt != FA_BF16) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  s->B = B;
  s->H = H;
  s->N = N;
  s->d = d;
  s->BH = static_cast<long long>(B) * H;
  s->nqt = (N + 127) / 128;
  if (s->BH * s->nqt > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B*H*ceil(N/128) exceeds 2^31-1");
  if (s->BH > INT_MAX / 2) return fail(FA_ERR_INVALID_ARG, "B*H too large");
  return FA_OK;
}

fa_status check_ptrs(std::initializer_list<std::pair<const void *, const char *>> ps) {
  for (auto &p : ps) {
    if (p.first == nullptr) return fail(FA_ERR_INVALID_ARG, "%s is null", p.second);
    if (!aligned16(p.first)) return fail(FA_ERR_INVALID_ARG, "%s is not 16-byte aligned", p.second);
  }
  return FA_OK;
}

// cudaFuncSetAttribute once per (kernel, device).
cudaError_t set_smem(const void *kernel, int bytes) {
  static std::mutex mu;
  static std::map<const void *, unsigned long long> done;  // kernel -> bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> g(mu);
  unsigned long long &bits = done[kernel];
  if (dev < 64 && ((bits >> dev) & 1ull)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev < 64) bits |= 1ull << dev;
  return e;
}

template <int D, bool BF16, bool CAUSAL, bool SPARSE>
fa_status launch_fwd_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const fa::FwdArgs &a, int grid, cudaStream_t st) {
  auto kern = fa::fwd_kernel<D, BF16, CAUSAL, SPARSE>;
  constexpr int smem = fa::FwdCfg<D>::kSmemBytes;
  cudaError_t e = set_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(fwd)");
  kern<<<dim3(grid, a.num_splits), 256, smem, st>>>(tq, tk, tv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "fwd launch");
  return FA_OK;
}

// Two-query-tile kernel; it relies on setmaxnreg shifting registers between
// warpgroups, which is only safe when the kernel was built with exactly the
// register count the split assumes (checked once per kernel and device).
// Returns false (nothing launched) when that check fails.
template <int D, bool BF16, bool CAUSAL, bool FP8 = false>
bool try_launch_fwd2(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                     const CUtensorMap &to, const CUtensorMap &tr, const fa::FwdArgs &a, int nqb_grid,
                     cudaStream_t st, fa_status *r) {
  auto kern = fa::fwd2_kernel<D, BF16, CAUSAL, FP8>;
  using C2 = fa::Fwd2Cfg<D, FP8>;
  static std::mutex mu;
  static int usable[64] = {};  // 0 unknown, 1 yes, -1 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> g(mu);
    if (usable[dev] == 0) {
      cudaFuncAttributes at;
      usable[dev] = (cudaFuncGetAttributes(&at, reinterpret_cast<const void *>(kern)) == cudaSuccess &&
                     at.numRegs == C2::kLaunchRegs)
                        ? 1
                        : -1;
    }
    if (usable[dev] < 0) return false;
  }
  constexpr int smem = C2::kSmemBytes;
  cudaError_t e = set_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) {
    *r = cuda_fail(e, "cudaFuncSetAttribute(fwd2)");
    return true;
  }
  kern<<<nqb_grid, 384, smem, st>>>(tq, tk, tv, to, tr, a);
  e = cudaGetLastError();
  *r = (e != cudaSuccess) ? cuda_fail(e, "fwd2 launch") : FA_OK;
  return true;
}

// Short-sequence forward: one query tile per CTA, two CTAs per SM; used up
// to this many 128-row query tiles (N <= 2048), and at any length when the
// two-tile kernel's grid (one CTA per pair of query tiles) would leave SMs
// idle: it then runs twice as many CTAs (measured: one head of N = 8192,
// 344 against 263 TFLOP/s; with 128 heads of N = 4096 the two-tile kernel
// stays ahead, 1043 against 1016).
constexpr int kSmallMaxTiles = 16;
int sm_count();

// Short-sequence forward: one query tile per CTA, two CTAs per SM. Like the
// two-tile kernel it relies on setmaxnreg, so it runs only when built with
// exactly the register count its split assumes (checked once per kernel and
// device); returns false (nothing launched) otherwise.
template <int D, bool BF16, bool CAUSAL, bool SPARSE = false, bool SPLIT = false>
bool try_launch_fwd_small(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const fa::FwdArgs &a, int grid, cudaStream_t st, fa_status *r) {
  auto kern = fa::fwd_small_kernel<D, BF16, CAUSAL, SPARSE, SPLIT>;
  static std::mutex mu;
  static int usable[64] = {};  // 0 unknown, 1 yes, -1 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  {
    std::lock_guard<std::mutex> g(mu);
    if (usable[dev] == 0) {
      cudaFuncAttributes at;
      usable[dev] = (cudaFuncGetAttributes(&at, reinterpret_cast<const void *>(kern)) == cudaSuccess &&
                     at.numRegs == fa::SmallCfg<D>::kLaunchRegs)
                        ? 1
                        : -1;
    }
    if (usable[dev] < 0) return false;
  }
  constexpr int smem = fa::SmallCfg<D>::kSmemBytes;
  cudaError_t e = set_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) {
    *r = cuda_fail(e, "cudaFuncSetAttribute(fwd small)");
    return true;
  }
  kern<<<dim3(grid, SPLIT ? a.num_splits : 1), 256, smem, st>>>(tq, tk, tv, a);
  e = cudaGetLastError();
  *r = (e != cudaSuccess) ? cuda_fail(e, "fwd small launch") : FA_OK;
  return true;
}

// Paged decode: two CTAs per SM (128 threads, DecCfg<D>::kSmemBytes each).
template <int D, bool BF16>
fa_status launch_decode(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const fa::FwdArgs &a, int grid, cudaStream_t st) {
  auto kern = fa::decode_kernel<D, BF16>;
  constexpr int smem = fa::DecCfg<D>::kSmemBytes;
  cudaError_t e = set_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode)");
  kern<<<dim3(grid, a.num_splits), 128, smem, st>>>(tq, tk, tv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return FA_OK;
}

// Split-KV merge: one thread per 4 channels of a query row.
template <bool BF16>
fa_status launch_merge(const fa::FwdArgs &a, long long rows, int d, cudaStream_t st) {
  const long long threads = rows * (d / 4);
  const long long blocks = std::min<long long>((threads + 255) / 256, 148ll * 16);
  fa::fwd_merge_kernel<BF16><<<static_cast<int>(blocks), 256, 0, st>>>(a, rows, d);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? cuda_fail(e, "split-KV merge launch") : FA_OK;
}

template <int D, bool BF16>
fa_status launch_fwd_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &to, const CUtensorMap &tr, const fa::FwdArgs &a, int grid,
                       bool causal, bool sparse, cudaStream_t st) {
  fa_status r = FA_OK;
  if (sparse) {
    // block-sparse: one query tile per CTA, two CTAs per SM, each walking
    // its own row's kept key tiles
    if (try_launch_fwd_small<D, BF16, false, true>(tq, tk, tv, a, grid, st, &r)) return r;
    return launch_fwd_t<D, BF16, false, true>(tq, tk, tv, a, grid, st);
  }
  if (a.num_splits > 1) {
    // split-KV: one-tile kernel over (query tile, split), then the merge. At
    // d = 64 the shares run two CTAs per SM (measured 7 % faster than one);
    // at d = 128 the one-CTA-per-SM kernel is faster (660 against 617
    // TFLOP/s on one 8192-row head)
    bool small = false;
    if constexpr (D == 64)
      small = causal ? try_launch_fwd_small<D, BF16, true, false, true>(tq, tk, tv, a, grid, st, &r)
                     : try_launch_fwd_small<D, BF16, false, false, true>(tq, tk, tv, a, grid, st, &r);
    if (!small)
      r = causal ? launch_fwd_t<D, BF16, true, false>(tq, tk, tv, a, grid, st)
                 : launch_fwd_t<D, BF16, false, false>(tq, tk, tv, a, grid, st);
    if (r != FA_OK) return r;
    return launch_merge<BF16>(a, static_cast<long long>(grid / a.nqt) * a.N, D, st);
  }
  // short sequences: one query tile per CTA, two CTAs per SM (the start-up
  // and epilogue of one CTA overlap the other's tiles)
  if ((a.nqt <= kSmallMaxTiles || (grid / a.nqt) * ((a.nqt + 1) / 2) < sm_count()) &&
      (causal ? try_launch_fwd_small<D, BF16, true>(tq, tk, tv, a, grid, st, &r)
              : try_launch_fwd_small<D, BF16, false>(tq, tk, tv, a, grid, st, &r)))
    return r;
  // dense / causal / key padding: two query tiles per CTA
  const long long bh = grid / a.nqt;
  const int grid2 = static_cast<int>(bh * ((a.nqt + 1) / 2));
  if (causal ? try_launch_fwd2<D, BF16, true>(tq, tk, tv, to, tr, a, grid2, st, &r)
             : try_launch_fwd2<D, BF16, false>(tq, tk, tv, to, tr, a, grid2, st, &r))
    return r;
  if (causal) return launch_fwd_t<D, BF16, true, false>(tq, tk, tv, a, grid, st);
  return launch_fwd_t<D, BF16, false, false>(tq, tk, tv, a, grid, st);
}


// Hkv: key/value heads (0 = H); H must be a multiple of it (grouped-query
// attention: query head h reads key/value head h / (H / Hkv)).
fa_status check_kv_heads(int H, int *Hkv, bool sparse) {
  if (*Hkv == 0) *Hkv = H;
  if (*Hkv < 1 || *Hkv > H || H % *Hkv != 0)
    return fail(FA_ERR_INVALID_ARG, "Hkv=%d must divide H=%d", *Hkv, H);
  if (sparse && *Hkv != H) return fail(FA_ERR_UNSUPPORTED, "block-sparse attention needs Hkv == H");
  return FA_OK;
}

// SMs of the current device (148 on B300; that figure when the query fails).
int sm_count() {
  static std::mutex mu;
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> g(mu);
  if (n[dev] == 0) {
    int v = 0;
    n[dev] = (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) ? v : 148;
  }
  return n[dev];
}

constexpr int kMaxSplits = 256;

// Split-KV factor: the request when it is >= 1, else the S in [1, min(64,
// key tiles)] that minimises the modelled time ceil(ctas * S / SMs) waves of
// (ceil(T / S) + 1) tile times each (T = key tiles of an average row; the
// +1 stands for the CTA's prologue, epilogue and its share of the merge);
// ties go to the smaller S. The CTA slots are the SMs times the CTAs per SM
// of the kernel that runs the shares: two at d = 64, one at d = 128.
int resolve_splits(long long ctas, int nkt, int d, bool causal, int requested) {
  if (requested >= 1) return requested;
  const int T = causal ? (nkt + 1) / 2 : nkt;
  const long long sms = (d == 64 ? 2ll : 1ll) * sm_count();
  int best = 1;
  double best_cost = 0.0;
  for (int S = 1; S <= std::min(64, std::max(1, T)); ++S) {
    const double waves = static_cast<double>((ctas * S + sms - 1) / sms);
    const double cost = waves * (static_cast<double>((T + S - 1) / S) + 1.0);
    if (S == 1 || cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

// Decode split factor: the request when it is >= 1; else, with 2 * SMs CTA
// slots (the decode kernel runs two CTAs per SM), as many shares as fill one
// wave of slots when that is at least 2, otherwise about two waves' worth,
// with at least 16 key tiles of the longest sequence per share and at most
// 64 shares. The key walk is bound by HBM; a share that is too short pays
// its start-up (first K/V latency) and partial-result traffic too often, and
// a partly filled last wave leaves SMs idle (measured: 4, 8, 16, 32 and 128
// sequences of 16K-32K, 2K-8K and 1K-2K keys).
int resolve_decode_splits(long long ctas, int nkt_max, int requested) {
  if (requested >= 1) return requested;
  const long long slots = 2ll * sm_count();
  const long long one_wave = slots / ctas;
  const long long want = one_wave >= 2 ? one_wave : std::max(1ll, 2 * slots / ctas);
  const long long cap = std::max(1, std::min(64, nkt_max / 16));
  return static_cast<int>(std::max(1ll, std::min(want, cap)));
}

// Split-KV workspace: fp32 O / l [S][R][d] then fp32 LSE [S][R], R = B*H*nqt*128.
size_t splitkv_ws_bytes(long long BH, int nqt, int d, int S) {
  if (S <= 1) return 0;
  const size_t R = static_cast<size_t>(BH) * nqt * 128;
  return static_cast<size_t>(S) * R * (static_cast<size_t>(d) + 1) * 4;
}

fa_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int N, int d, float scale, int causal, fa_dtype dt, const int32_t *kv_len,
                   const uint8_t *block_mask, bool sparse, void *o_res, void *stream, int Hkv = 0,
                   int num_splits = 1, void *workspace = nullptr, size_t ws_bytes = 0) {
  Shape s;
  fa_status r = check_common(B, H, N, d, scale, dt, &s);
  if (r != FA_OK) return r;
  if ((r = check_kv_heads(H, &Hkv, sparse)) != FA_OK) return r;
  if (num_splits > kMaxSplits) return fail(FA_ERR_INVALID_ARG, "num_splits=%d exceeds %d", num_splits, kMaxSplits);
  const int S = resolve_splits(s.BH * s.nqt, s.nqt, d, causal != 0, num_splits);
  if (S > 1) {
    const size_t need = splitkv_ws_bytes(s.BH, s.nqt, d, S);
    if (workspace == nullptr) return fail(FA_ERR_INVALID_ARG, "workspace is null (num_splits=%d)", S);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(FA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    if (ws_bytes < need) return fail(FA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  }
  const long long BHkv = static_cast<long long>(B) * Hkv;
  r = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}});
  if (r != FA_OK) return r;
  if (sparse) {
    if (block_mask == nullptr) return fail(FA_ERR_INVALID_ARG, "block_mask is null");
    if (s.nqt > fa::FwdCfg<64>::kMaxList)
      return fail(FA_ERR_UNSUPPORTED, "block-sparse needs ceil(N/128) <= %d", fa::FwdCfg<64>::kMaxList);
  }
  if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u))
    return fail(FA_ERR_INVALID_ARG, "kv_len is not 4-byte aligned");
  if (o_res != nullptr && !aligned16(o_res))
    return fail(FA_ERR_INVALID_ARG, "o_res is not 16-byte aligned");
  CUtensorMap tq, tk, tv;
  if ((r = make_tile_map(&tq, q, dt, N, s.BH, d, "q")) != FA_OK) return r;
  if ((r = make_tile_map(&tk, k, dt, N, BHkv, d, "k")) != FA_OK) return r;
  if ((r = make_tile_map(&tv, v, dt, N, BHkv, d, "v")) != FA_OK) return r;
  // O and its residual, stored by the two-tile kernel through TMA
  CUtensorMap to, tr;
  if ((r = make_tile_map(&to, o, dt, N, s.BH, d, "o")) != FA_OK) return r;
  if ((r = make_tile_map(&tr, o_res != nullptr ? o_res : o, dt, N, s.BH, d, "o_res")) != FA_OK) return r;
  fa::FwdArgs a;
  a.o = o;
  a.o_res = o_res;
  a.lse = lse;
  a.kv_len = kv_len;
  a.block_mask = block_mask;
  a.H = H;
  a.N = N;
  a.nqt = s.nqt;
  a.nkt = s.nqt;
  a.hgroup = fwd_head_group(N, d, causal != 0);
  a.Hkv = Hkv;
  a.kv_group = H / Hkv;
  a.num_splits = S;
  a.block_table = nullptr;
  a.page_size = a.pages_per_seq = a.dec_nq = 0;
  a.o_part = S > 1 ? static_cast<float *>(workspace) : nullptr;
  a.lse_part = S > 1 ? a.o_part + static_cast<size_t>(S) * s.BH * s.nqt * 128 * d : nullptr;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o_scale = 1.f;
  const int grid = static_cast<int>(s.BH * s.nqt);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool c = causal != 0;
  if (d == 64)
    r = dt == FA_BF16 ? launch_fwd_d<64, true>(tq, tk, tv, to, tr, a, grid, c, sparse, st)
                      : launch_fwd_d<64, false>(tq, tk, tv, to, tr, a, grid, c, sparse, st);
  else
    r = dt == FA_BF16 ? launch_fwd_d<128, true>(tq, tk, tv, to, tr, a, grid, c, sparse, st)
                      : launch_fwd_d<128, false>(tq, tk, tv, to, tr, a, grid, c, sparse, st);
  if (r != FA_OK) return r;
  return ok();
}

// Workspace: LSE*log2(e) and D per query row, padded to whole 128-row tiles,
// then the fp32 dQ accumulator over the same padded rows.
size_t padded_rows(int B, int H, int N) {
  return static_cast<size_t>(B) * H * static_cast<size_t>((N + 127) / 128) * 128;
}
size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Then a 256-byte block of statistics (max |dO|, max |D|) and, for bf16
// inputs, the fp16 copies of Q and of the scaled dO ([B, H, N, d] each; the
// space is reserved for either input type).
size_t fa_bwd_ws_bytes(int B, int H, int N, int d) {
  const size_t rows = padded_rows(B, H, N);
  const size_t elems = static_cast<size_t>(B) * H * static_cast<size_t>(N) * d;
  return 2 * up256(rows * 4) + up256(rows * static_cast<size_t>(d) * 4) + 256 + 2 * up256(elems * 2);
}

template <int D, bool BF16, bool CAUSAL, bool SPARSE>
fa_status launch_bwd_main_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const fa::BwdArgs &a, int grid, cudaStream_t st) {
  auto kern = fa::bwd_main_kernel<D, BF16, CAUSAL, SPARSE>;
  constexpr int smem = fa::BwdCfg<D>::kSmemBytes;
  // The kernel moves registers between warpgroups with setmaxnreg; the split
  // only fits when it was built with exactly the register count it assumes.
  static std::mutex mu;
  static int usable[64] = {};  // 0 unknown, 1 yes, -1 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fail(FA_ERR_CUDA, "bwd: cannot query the current device");
  {
    std::lock_guard<std::mutex> g(mu);
    if (usable[dev] == 0) {
      cudaFuncAttributes at;
      usable[dev] = (cudaFuncGetAttributes(&at, reinterpret_cast<const void *>(kern)) == cudaSuccess &&
                     at.numRegs == fa::BwdCfg<D>::kLaunchRegs)
                        ? 1
                        : -1;
    }
    if (usable[dev] < 0)
      return fail(FA_ERR_CUDA, "bwd: kernel register count differs from its warpgroup split");
  }
  cudaError_t e = set_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd)");
  kern<<<grid, fa::BwdCfg<D>::kThreads, smem, st>>>(tq, tk, tv, tdo, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bwd launch");
  return FA_OK;
}

enum BwdPhase : unsigned { kPrepare = 1u, kMain = 2u, kFinish = 4u, kAll = 7u };

template <int D, bool BF16>
fa_status launch_bwd_d(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const fa::BwdArgs &a, long long rows_pad,
                       long long n_vec4, int grid, bool causal, bool sparse, unsigned phases,
                       cudaStream_t st) {
  cudaError_t e;
  if (phases & kPrepare) {
    e = cudaMemsetAsync(a.stats, 0, 4 * sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_fail(e, "bwd statistics reset");
    constexpr int rows_per_block = 8 * (32 / (D / 8));
    long long pre_blocks = (rows_pad + rows_per_block - 1) / rows_per_block;
    if (pre_blocks > 148 * 16) pre_blocks = 148 * 16;
    fa::bwd_pre_kernel<D, BF16><<<static_cast<int>(pre_blocks), 256, 0, st>>>(a, rows_pad);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "bwd prepare launch");
    if (BF16) {
      // fp16 copies of Q and of dO * 2^-e_do for the main kernel's products
      // (e_do comes from the max |dO| the prepare kernel just recorded)
      const long long n16 = n_vec4 / 2;
      long long cvt_blocks = (n16 + 255) / 256;
      if (cvt_blocks > 148 * 16) cvt_blocks = 148 * 16;
      fa::bwd_cvt_kernel<<<static_cast<int>(cvt_blocks), 256, 0, st>>>(a, n16);
      e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "bwd conversion launch");
    }
  }
  if (phases & kMain) {
    // the persistent main kernel takes its work items from this counter
    e = cudaMemsetAsync(a.work, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return cuda_fail(e, "bwd work counter reset");
    fa_status r;
    if (sparse)
      r = launch_bwd_main_t<D, BF16, false, true>(tq, tk, tv, tdo, a, grid, st);
    else if (causal)
      r = launch_bwd_main_t<D, BF16, true, false>(tq, tk, tv, tdo, a, grid, st);
    else
      r = launch_bwd_main_t<D, BF16, false, false>(tq, tk, tv, tdo, a, grid, st);
    if (r != FA_OK) return r;
  }
  if (phases & kFinish) {
    // heads along y, rows along x: about 16 blocks of 256 threads per SM
    const long long bh = n_vec4 * 4 / (static_cast<long long>(a.N) * D);
    const int gy = static_cast<int>(std::min<long long>(bh, 65535));
    constexpr int kRows = 256 / (D / 8);
    const long long rows_x = (a.N + kRows - 1) / kRows;
    const int gx = static_cast<int>(std::max<long long>(1, std::min<long long>(rows_x, (148ll * 16 + gy - 1) / gy)));
    fa::bwd_dq_kernel<BF16, D><<<dim3(gx, gy), 256, 0, st>>>(a, static_cast<int>(bh));
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "bwd finish launch");
  }
  return FA_OK;
}

fa_status bwd_impl(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                   float scale, int causal, fa_dtype dt, const int32_t *kv_len,
                   const uint8_t *block_mask, bool sparse, const void *o_res, void *workspace,
                   size_t ws_bytes, void *stream, unsigned phases = kAll, int Hkv = 0) {
  Shape s;
  fa_status r = check_common(B, H, N, d, scale, dt, &s);
  if (r != FA_OK) return r;
  if ((r = check_kv_heads(H, &Hkv, sparse)) != FA_OK) return r;
  const long long BHkv = static_cast<long long>(B) * Hkv;
  // each phase reads/writes only some of the tensors
  if (phases & kPrepare) {
    r = check_ptrs({{q, "q"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {dout, "dout"}});
    if (r != FA_OK) return r;
  }
  if (phases & kMain) {
    r = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {dout, "dout"}, {dk, "dk"}, {dv, "dv"}});
    if (r != FA_OK) return r;
  }
  if (phases & kFinish) {
    r = check_ptrs({{dq, "dq"}});
    if (r != FA_OK) return r;
  }
  r = check_ptrs({{workspace, "workspace"}});
  if (r != FA_OK) return r;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(FA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = fa_bwd_ws_bytes(B, H, N, d);
  if (ws_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  if (sparse && block_mask == nullptr) return fail(FA_ERR_INVALID_ARG, "block_mask is null");
  // no forward computes block-sparse attention with key padding, so its
  // gradient is not offered either
  if (sparse && kv_len != nullptr)
    return fail(FA_ERR_INVALID_ARG, "kv_len cannot be combined with a block mask");
  if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u))
    return fail(FA_ERR_INVALID_ARG, "kv_len is not 4-byte aligned");
  if (o_res != nullptr && !aligned16(o_res))
    return fail(FA_ERR_INVALID_ARG, "o_res is not 16-byte aligned");
  const size_t rows = padded_rows(B, H, N);
  const size_t elems = static_cast<size_t>(s.BH) * static_cast<size_t>(N) * d;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  unsigned int *stats =
      reinterpret_cast<unsigned int *>(ws + 2 * up256(rows * 4) + up256(rows * static_cast<size_t>(d) * 4));
  void *q16 = reinterpret_cast<uint8_t *>(stats) + 256;
  void *do16 = static_cast<uint8_t *>(q16) + up256(elems * 2);
  CUtensorMap tq, tk, tv, tdo;
  if (phases & kMain) {
    // bf16 inputs: the products read the fp16 copies of Q and dO (K and V
    // are converted in shared memory)
    const bool cv = dt == FA_BF16;
    if ((r = make_tile_map(&tq, cv ? q16 : q, cv ? FA_F16 : dt, N, s.BH, d, "q")) != FA_OK) return r;
    if ((r = make_tile_map(&tk, k, dt, N, BHkv, d, "k")) != FA_OK) return r;
    if ((r = make_tile_map(&tv, v, dt, N, BHkv, d, "v")) != FA_OK) return r;
    if ((r = make_tile_map(&tdo, cv ? do16 : dout, cv ? FA_F16 : dt, N, s.BH, d, "dout")) != FA_OK)
      return r;
  }
  fa::BwdArgs a;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.o = o;
  a.o_res = o_res;
  a.dout = dout;
  a.lse = lse;
  a.lse_l2 = reinterpret_cast<float *>(ws);
  a.delta = reinterpret_cast<float *>(ws + up256(rows * 4));
  a.q = q;
  a.q16 = q16;
  a.do16 = do16;
  a.stats = stats;
  a.v = v;
  a.n_v16 = BHkv * static_cast<long long>(N) * d / 8;
  a.dq_acc = reinterpret_cast<float *>(ws + 2 * up256(rows * 4));
  a.kv_len = kv_len;
  a.block_mask = block_mask;
  a.k = k;
  a.work = stats + 8;
  a.n_items = static_cast<int>(BHkv * s.nqt);
  a.H = H;
  a.N = N;
  a.nqt = s.nqt;
  a.nkt = s.nqt;
  a.Hkv = Hkv;
  a.kv_group = H / Hkv;
  // a CTA streams the Q and dO of all kv_group query heads of its group
  a.hgroup = std::max(1, head_group(N, d, causal != 0) / a.kv_group);
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  const long long rows_pad = static_cast<long long>(rows);
  const long long n_vec4 = s.BH * static_cast<long long>(N) * d / 4;
  // persistent: one CTA per SM (at most one per work item)
  const int grid = static_cast<int>(std::min<long long>(BHkv * s.nqt, sm_count()));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool c = causal != 0;
  if (d == 64)
    r = dt == FA_BF16 ? launch_bwd_d<64, true>(tq, tk, tv, tdo, a, rows_pad, n_vec4, grid, c, sparse, phases, st)
                      : launch_bwd_d<64, false>(tq, tk, tv, tdo, a, rows_pad, n_vec4, grid, c, sparse, phases, st);
  else
    r = dt == FA_BF16 ? launch_bwd_d<128, true>(tq, tk, tv, tdo, a, rows_pad, n_vec4, grid, c, sparse, phases, st)
                      : launch_bwd_d<128, false>(tq, tk, tv, tdo, a, rows_pad, n_vec4, grid, c, sparse, phases, st);
  if (r != FA_OK) return r;
  return ok();
}

// ------------------------------------------------------------------------
// Fixed scratch for fa_bwd_noalloc: callers that may not allocate device
// memory get the backward's workspace from this array instead. It is part of
// the library's device image, so every GPU that loads the library holds it
// until the process exits. Every call shares it.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device and context (host code may not use the symbol itself as a
// pointer). The context is part of the key: after a device reset the
// primary context is recreated, the module is loaded again and the array
// may sit at a new address.
fa_status noalloc_scratch(void **out) {
  using CtxGetCurrent = CUresult (*)(CUcontext *);
  static CtxGetCurrent ctx_get = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      ctx_get = reinterpret_cast<CtxGetCurrent>(p);
  });
  static std::mutex mu;
  static void *addr[64] = {};
  static CUcontext ctx_of[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
  if (ctx_get == nullptr) return fail(FA_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
  // no current context yet (first CUDA call of this thread): the lookup
  // below makes the device's primary context current
  CUcontext ctx = nullptr;
  if (ctx_get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (addr[dev] == nullptr || ctx == nullptr || ctx_of[dev] != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    if (ctx_get(&ctx) != CUDA_SUCCESS || ctx == nullptr)
      return fail(FA_ERR_CUDA, "cannot query the current CUDA context");
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                 int N, int d, float scale, int causal, fa_dtype dtype, void *stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, nullptr, nullptr, false,
                  nullptr, stream);
}

fa_status fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                    int N, int d, float scale, int causal, fa_dtype dtype, const int32_t *kv_len,
                    void *o_res, void *stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, kv_len, nullptr, false,
                  o_res, stream);
}

fa_status fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float scale, fa_dtype dtype,
                             const uint8_t *block_mask, void *o_res, void *stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, 0, dtype, nullptr, block_mask, true, o_res,
                  stream);
}

fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int Hkv, int N, int d, float scale, int causal, fa_dtype dtype,
                     const int32_t *kv_len, void *o_res, void *stream) {
  if (Hkv < 1) return fail(FA_ERR_INVALID_ARG, "Hkv=%d must be >= 1", Hkv);
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, kv_len, nullptr, false,
                  o_res, stream, Hkv);
}

int fa_fwd_splitkv_num_splits(int B, int H, int N, int d, int causal, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || num_splits > kMaxSplits) return 0;
  const int nqt = (N + 127) / 128;
  return resolve_splits(static_cast<long long>(B) * H * nqt, nqt, d, causal != 0, num_splits);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int causal, int num_splits) {
  const int S = fa_fwd_splitkv_num_splits(B, H, N, d, causal, num_splits);
  if (S < 1) return 0;
  return splitkv_ws_bytes(static_cast<long long>(B) * H, (N + 127) / 128, d, S);
}

fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int H, int Hkv, int N, int d, float scale, int causal, fa_dtype dtype,
                         const int32_t *kv_len, void *o_res, int num_splits, void *workspace,
                         size_t workspace_bytes, void *stream) {
  if (Hkv < 1) return fail(FA_ERR_INVALID_ARG, "Hkv=%d must be >= 1", Hkv);
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, kv_len, nullptr, false,
                  o_res, stream, Hkv, num_splits, workspace, workspace_bytes);
}

// Paged decode: rows per (batch, key/value head) block and its query tiles.
struct DecodeShape {
  long long BHkv;
  int R, nqt, nkt_max;
};

fa_status check_decode(int B, int H, int Hkv, int Nq, int d, int page_size, int num_pages,
                       int pages_per_seq, float scale, fa_dtype dt, DecodeShape *s) {
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1)
    return fail(FA_ERR_INVALID_ARG, "B, H, Hkv, Nq must be >= 1 (got %d, %d, %d, %d)", B, H, Hkv, Nq);
  if (H % Hkv != 0 || Hkv > H) return fail(FA_ERR_INVALID_ARG, "Hkv=%d must divide H=%d", Hkv, H);
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d not built (64 or 128)", d);
  if (dt != FA_F16 && dt != FA_BF16) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dt);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return fail(FA_ERR_UNSUPPORTED, "page_size %d not built (16, 32, 64 or 128)", page_size);
  if (num_pages < 1 || pages_per_seq < 1)
    return fail(FA_ERR_INVALID_ARG, "num_pages and pages_per_seq must be >= 1");
  if (static_cast<long long>(num_pages) * Hkv > INT_MAX / 2)
    return fail(FA_ERR_INVALID_ARG, "num_pages * Hkv too large");
  if (static_cast<long long>(pages_per_seq) * page_size > (1ll << 30))
    return fail(FA_ERR_INVALID_ARG, "pages_per_seq * page_size too large");
  const long long R = static_cast<long long>(H / Hkv) * Nq;
  if (R > (1 << 20)) return fail(FA_ERR_INVALID_ARG, "(H / Hkv) * Nq too large");
  s->BHkv = static_cast<long long>(B) * Hkv;
  s->R = static_cast<int>(R);
  s->nqt = static_cast<int>((R + fa::DecCfg<64>::kQRows - 1) / fa::DecCfg<64>::kQRows);
  s->nkt_max = static_cast<int>((static_cast<long long>(pages_per_seq) * page_size + 127) / 128);
  if (s->BHkv * s->nqt > INT_MAX) return fail(FA_ERR_INVALID_ARG, "grid too large");
  return FA_OK;
}

size_t fa_fwd_fp8_workspace_size(int B, int Hkv, int N, int d) {
  if (B < 1 || Hkv < 1 || N < 1 || d != 128) return 0;
  const size_t npad = static_cast<size_t>((N + 127) / 128) * 128;
  return static_cast<size_t>(B) * Hkv * d * npad;
}

fa_status fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                     int Hkv, int N, int d, float scale, int causal, float q_descale, float k_descale,
                     float v_descale, const int32_t *kv_len, void *workspace, size_t workspace_bytes,
                     void *stream) {
  Shape s;
  fa_status r = check_common(B, H, N, d, scale, FA_BF16, &s);
  if (r != FA_OK) return r;
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "the 8-bit forward is built for d = 128 (got %d)", d);
  if (Hkv < 1) return fail(FA_ERR_INVALID_ARG, "Hkv=%d must be >= 1", Hkv);
  if ((r = check_kv_heads(H, &Hkv, false)) != FA_OK) return r;
  for (float f : {q_descale, k_descale, v_descale})
    if (!(f > 0.f) || !std::isfinite(f))
      return fail(FA_ERR_INVALID_ARG, "dequantisation factors must be finite and > 0");
  if (!std::isfinite(scale * q_descale * k_descale))
    return fail(FA_ERR_INVALID_ARG, "scale * q_descale * k_descale overflows");
  r = check_ptrs({{q, "q"}, {k, "k"}, {v, "v"}, {o, "o"}, {lse, "lse"}, {workspace, "workspace"}});
  if (r != FA_OK) return r;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(FA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t need = fa_fwd_fp8_workspace_size(B, Hkv, N, d);
  if (workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  if (kv_len != nullptr && (reinterpret_cast<uintptr_t>(kv_len) & 3u))
    return fail(FA_ERR_INVALID_ARG, "kv_len is not 4-byte aligned");
  const long long BHkv = static_cast<long long>(B) * Hkv;
  const int npad = s.nqt * 128;
  CUtensorMap tq, tk, tv;
  if ((r = make_tile_map8(&tq, q, d, d, N, s.BH, "q")) != FA_OK) return r;
  if ((r = make_tile_map8(&tk, k, d, d, N, BHkv, "k")) != FA_OK) return r;
  if ((r = make_tile_map8(&tv, workspace, N, npad, d, BHkv, "v^T")) != FA_OK) return r;
  if (BHkv > 65535) return fail(FA_ERR_UNSUPPORTED, "B*Hkv=%lld exceeds 65535", BHkv);
  fa::FwdArgs a{};
  a.o = o;
  a.o_res = nullptr;
  a.lse = lse;
  a.kv_len = kv_len;
  a.block_mask = nullptr;
  a.H = H;
  a.N = N;
  a.nqt = s.nqt;
  a.nkt = s.nqt;
  a.hgroup = head_group(N, d, causal != 0) * 2;  // 8-bit K and V: half the bytes per head
  a.Hkv = Hkv;
  a.kv_group = H / Hkv;
  a.num_splits = 1;
  a.scale_log2 = scale * q_descale * k_descale * 1.4426950408889634f;
  a.o_scale = v_descale;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  fa::fwd_fp8_vt_kernel<<<dim3(s.nqt, static_cast<unsigned>(BHkv)), 256, 0, st>>>(
      static_cast<const uint8_t *>(v), static_cast<uint8_t *>(workspace), N, npad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "V^T launch");
  const int grid2 = static_cast<int>(s.BH * ((s.nqt + 1) / 2));
  // (the 8-bit instance stores O with plain stores; its O map is not read)
  const bool launched = causal ? try_launch_fwd2<128, true, true, true>(tq, tk, tv, tq, tq, a, grid2, st, &r)
                               : try_launch_fwd2<128, true, false, true>(tq, tk, tv, tq, tq, a, grid2, st, &r);
  if (!launched) return fail(FA_ERR_CUDA, "8-bit forward: kernel register count differs from its warpgroup split");
  if (r != FA_OK) return r;
  return ok();
}

int fa_decode_paged_num_splits(int B, int H, int Hkv, int Nq, int d, int page_size,
                               int pages_per_seq, int num_splits) {
  DecodeShape s;
  if (num_splits > kMaxSplits ||
      check_decode(B, H, Hkv, Nq, d, page_size, 1, pages_per_seq, 1.f, FA_BF16, &s) != FA_OK)
    return 0;
  return resolve_decode_splits(s.BHkv * s.nqt, s.nkt_max, num_splits);
}

size_t fa_decode_paged_workspace_size(int B, int H, int Hkv, int Nq, int d, int page_size,
                                      int pages_per_seq, int num_splits) {
  const int S = fa_decode_paged_num_splits(B, H, Hkv, Nq, d, page_size, pages_per_seq, num_splits);
  if (S < 1) return 0;
  DecodeShape s;
  check_decode(B, H, Hkv, Nq, d, page_size, 1, pages_per_seq, 1.f, FA_BF16, &s);
  return splitkv_ws_bytes(s.BHkv, s.nqt, d, S);
}

fa_status fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_table, const int32_t *seq_len, void *o, float *lse,
                          int B, int H, int Hkv, int Nq, int d, int page_size, int num_pages,
                          int pages_per_seq, float scale, fa_dtype dtype, int num_splits,
                          void *workspace, size_t workspace_bytes, void *stream) {
  DecodeShape s;
  fa_status r = check_decode(B, H, Hkv, Nq, d, page_size, num_pages, pages_per_seq, scale, dtype, &s);
  if (r != FA_OK) return r;
  r = check_ptrs({{q, "q"}, {k_cache, "k_cache"}, {v_cache, "v_cache"}, {o, "o"}, {lse, "lse"}});
  if (r != FA_OK) return r;
  for (auto p : {std::make_pair(static_cast<const void *>(block_table), "block_table"),
                 std::make_pair(static_cast<const void *>(seq_len), "seq_len")}) {
    if (p.first == nullptr) return fail(FA_ERR_INVALID_ARG, "%s is null", p.second);
    if (reinterpret_cast<uintptr_t>(p.first) & 3u) return fail(FA_ERR_INVALID_ARG, "%s is not 4-byte aligned", p.second);
  }
  if (num_splits > kMaxSplits) return fail(FA_ERR_INVALID_ARG, "num_splits=%d exceeds %d", num_splits, kMaxSplits);
  const int S = resolve_decode_splits(s.BHkv * s.nqt, s.nkt_max, num_splits);
  if (S > 1) {
    const size_t need = splitkv_ws_bytes(s.BHkv, s.nqt, d, S);
    if (workspace == nullptr) return fail(FA_ERR_INVALID_ARG, "workspace is null (num_splits=%d)", S);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(FA_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    if (workspace_bytes < need)
      return fail(FA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  }
  CUtensorMap tq, tk, tv;
  // q [B,H,Nq,d] = [B*Hkv][R][d]: the rows of a key/value head's query heads are contiguous
  if ((r = make_tile_map(&tq, q, dtype, s.R, s.BHkv, d, "q", fa::DecCfg<64>::kQRows)) != FA_OK) return r;
  const long long pool = static_cast<long long>(num_pages) * Hkv;
  if ((r = make_tile_map(&tk, k_cache, dtype, page_size, pool, d, "k_cache", page_size)) != FA_OK) return r;
  if ((r = make_tile_map(&tv, v_cache, dtype, page_size, pool, d, "v_cache", page_size)) != FA_OK) return r;
  fa::FwdArgs a{};
  a.o = o;
  a.o_res = nullptr;
  a.lse = lse;
  a.kv_len = seq_len;
  a.block_mask = nullptr;
  a.H = Hkv;  // the grid runs over (batch, key/value head) blocks of R rows
  a.N = s.R;
  a.nqt = s.nqt;
  a.nkt = s.nkt_max;
  a.hgroup = 1;
  a.Hkv = Hkv;
  a.kv_group = 1;
  a.num_splits = S;
  a.o_part = S > 1 ? static_cast<float *>(workspace) : nullptr;
  a.lse_part = S > 1 ? a.o_part + static_cast<size_t>(S) * s.BHkv * s.nqt * 128 * d : nullptr;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.o_scale = 1.f;
  a.block_table = block_table;
  a.page_size = page_size;
  a.pages_per_seq = pages_per_seq;
  a.dec_nq = Nq;
  const int grid = static_cast<int>(s.BHkv * s.nqt);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 64)
    r = dtype == FA_BF16 ? launch_decode<64, true>(tq, tk, tv, a, grid, st)
                         : launch_decode<64, false>(tq, tk, tv, a, grid, st);
  else
    r = dtype == FA_BF16 ? launch_decode<128, true>(tq, tk, tv, a, grid, st)
                         : launch_decode<128, false>(tq, tk, tv, a, grid, st);
  if (r != FA_OK) return r;
  if (S > 1) {
    const long long rows = s.BHkv * s.R;
    r = dtype == FA_BF16 ? launch_merge<true>(a, rows, d, st) : launch_merge<false>(a, rows, d, st);
    if (r != FA_OK) return r;
  }
  return ok();
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  return fa_bwd_ws_bytes(B, H, N, d);
}

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, const int32_t *kv_len, const void *o_res,
                 void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, dtype, kv_len,
                  nullptr, false, o_res, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const float *lse,
                     const void *dout, void *dq, void *dk, void *dv, int B, int H, int Hkv, int N,
                     int d, float scale, int causal, fa_dtype dtype, const int32_t *kv_len,
                     const void *o_res, void *workspace, size_t workspace_bytes, void *stream) {
  if (Hkv < 1) return fail(FA_ERR_INVALID_ARG, "Hkv=%d must be >= 1", Hkv);
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, dtype, kv_len,
                  nullptr, false, o_res, workspace, workspace_bytes, stream, kAll, Hkv);
}

fa_status fa_bwd_blocksparse(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, void *dq, void *dk, void *dv,
                             int B, int H, int N, int d, float scale, fa_dtype dtype,
                             const uint8_t *block_mask, const void *o_res, void *workspace,
                             size_t workspace_bytes, void *stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, 0, dtype, nullptr,
                  block_mask, true, o_res, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_prepare(const void *q, const void *v, const void *o, const void *o_res,
                         const float *lse, const void *dout, int B, int H, int N, int d, fa_dtype dtype,
                         void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_impl(q, nullptr, v, o, lse, dout, nullptr, nullptr, nullptr, B, H, N, d, 1.0f, 0,
                  dtype, nullptr, nullptr, false, o_res, workspace, workspace_bytes, stream, kPrepare);
}

fa_status fa_bwd_main(const void *q, const void *k, const void *v, const void *dout, void *dk,
                      void *dv, int B, int H, int N, int d, float scale, int causal,
                      fa_dtype dtype, const int32_t *kv_len, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_impl(q, k, v, nullptr, nullptr, dout, nullptr, dk, dv, B, H, N, d, scale,
                  block_mask ? 0 : causal, dtype, kv_len, block_mask, block_mask != nullptr,
                  nullptr, workspace, workspace_bytes, stream, kMain);
}

fa_status fa_bwd_finish(void *dq, int B, int H, int N, int d, fa_dtype dtype, void *workspace,
                        size_t workspace_bytes, void *stream) {
  return bwd_impl(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr, B, H,
                  N, d, 1.0f, 0, dtype, nullptr, nullptr, false, nullptr, workspace,
                  workspace_bytes, stream, kFinish);
}

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                         int H, int N, int d, float scale, int causal, fa_dtype dtype,
                         const int32_t *kv_len, const uint8_t *block_mask, const void *o_res,
                         void *stream) {
  Shape s;
  fa_status r = check_common(B, H, N, d, scale, dtype, &s);
  if (r != FA_OK) return r;
  const size_t need = fa_bwd_ws_bytes(B, H, N, d);
  if (need > kNoAllocScratchBytes)
    return fail(FA_ERR_INVALID_ARG,
                "fa_bwd_noalloc: these sizes need %zu bytes of scratch, more than the %zu bytes "
                "built into the library; use fa_bwd with a caller-owned workspace",
                need, kNoAllocScratchBytes);
  if (block_mask != nullptr && kv_len != nullptr)
    return fail(FA_ERR_INVALID_ARG, "kv_len cannot be combined with a block mask");
  void *ws = nullptr;
  if ((r = noalloc_scratch(&ws)) != FA_OK) return r;
  const bool sparse = block_mask != nullptr;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, sparse ? 0 : causal, dtype,
                  kv_len, block_mask, sparse, o_res, ws, kNoAllocScratchBytes, stream);
}

size_t fa_bwd_noalloc_max_workspace(void) { return kNoAllocScratchBytes; }

fa_status fa_get_device_error(void *stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, fa::g_fa_device_error, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read device error flag");
  if (v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(fa::g_fa_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clear device error flag");
    if (v & fa::kDevErrTimeout)
      return fail(FA_ERR_TIMEOUT, "a kernel pipeline wait timed out (flag 0x%x)", v);
    if (v & fa::kDevErrSmemAlign)
      return fail(FA_ERR_CUDA, "a kernel's shared-memory base was not 1 KB aligned; it did no work (flag 0x%x)", v);
    return fail(FA_ERR_RANGE, "a bf16 input of the backward exceeds 65504 in magnitude and was clamped (flag 0x%x)", v);
  }
  return ok();
}

fa_status fa_set_wait_limit_ns(unsigned long long ns) {
  const unsigned long long v = ns == 0 ? fa::kWaitLimitNs : ns;
  const cudaError_t e = cudaMemcpyToSymbol(fa::g_fa_wait_limit_ns, &v, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "set the wait limit");
  return ok();
}

fa_status fa_debug_starve_pipelines(int enable) {
  const unsigned int v = enable ? 1u : 0u;
  const cudaError_t e = cudaMemcpyToSymbol(fa::g_fa_starve_pipelines, &v, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "set the pipeline starvation switch");
  return ok();
}

const char *fa_status_str(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_RANGE: return "FA_ERR_RANGE";
  }
  return "FA_ERR_UNKNOWN";
}

const char *fa_last_error_message(void) { return g_last_error.c_str(); }

const char *fa_version(void) { return "0.1.0"; }

}  // extern "C"
