/*
 * fa.h -- C ABI of the exact IO-aware attention library (libfa.so).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T + M) V
 *
 * ("Flash Attention: revolutionizing transformer efficiency", standard
 * attention listing, and the FlashAttention abstract on the Tri Dao author
 * page, which describes the method as exact attention computed in tiles to
 * save memory traffic), tile by
 * tile on the GPU with the online-softmax rescaling of the same page (section
 * "The Math Behind Flash Attention": softmax decomposition and merger), so the
 * N x N score matrix never reaches device memory. The forward pass also writes
 * the per-row log-sum-exp; the backward pass recomputes the score tiles from
 * Q, K and that log-sum-exp (same page, key idea 2, "Recomputation").
 *
 * M is 0 where a key is visible and -inf where it is masked:
 *   causal       key j is masked for query i when j > i (top-left aligned);
 *   key padding  key j is masked for every query of batch b when
 *                j >= kv_len[b];
 *   block-sparse the 128 x 128 tile (i / 128, j / 128) is skipped entirely
 *                when block_mask[(i / 128) * nb + j / 128] == 0
 *                (block-sparse FlashAttention, same abstract).
 * A query row with no visible key gets O = 0 and LSE = -inf and contributes
 * nothing to any gradient.
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout    q, k, v, o, dout, dq, dk, dv are contiguous [B, H, N, d] arrays of
 *           16-bit floats (fp16 or bf16, chosen by `dtype`), d fastest; lse is
 *           a contiguous fp32 [B, H, N] array holding the NATURAL-log
 *           log-sum-exp of the scaled, masked scores of each row. Queries and
 *           keys have the same length N (self-attention).
 * Sizes     B >= 1, H >= 1, N >= 1, d in {64, 128}; B * H <= 65535 * 65535.
 * Memory    every pointer is a DEVICE pointer owned by the caller, 16-byte
 *           aligned, on the current CUDA device. The library allocates no
 *           device memory; the backward takes a caller-owned workspace.
 *           Outputs must not alias inputs.
 * Streams   `stream` is a cudaStream_t (NULL = legacy default stream). Every
 *           call is asynchronous on that stream and never synchronises, except
 *           fa_get_device_error.
 * Numerics  inputs are read as fp16/bf16; every product is accumulated in fp32;
 *           the softmax runs in fp32 with exp2. The forward rounds the
 *           probabilities to the input type before the P V product. The
 *           backward runs all five of its products on fp16 operands whatever
 *           the input type (P and dS rounded to fp16, 11 significant bits;
 *           bf16 Q, K, V converted to fp16, which is exact for
 *           2^-17 <= |x| <= 65504; bf16 dO converted after scaling by a
 *           power of two chosen from max |dO|), so sharp softmax does not
 *           lose its gradients to bf16's 8-bit significand.
 * Errors    argument checks run on the host before any launch and return
 *           FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED without touching memory.
 *           A failed launch returns FA_ERR_CUDA. A pipeline wait inside a
 *           kernel that exceeds its time limit (about two seconds; it cannot
 *           happen in a correct build) makes the kernel stop early and sets a
 *           device flag that fa_get_device_error reports as FA_ERR_TIMEOUT.
 *           A bf16 q, k or v value beyond +-65504 given to the backward is
 *           clamped and reported the same way as FA_ERR_RANGE.
 *           fa_last_error_message() gives the detail of the last failure on
 *           the calling thread.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer   */
    FA_ERR_UNSUPPORTED = 2,  /* valid but not built: d not in {64, 128}     */
    FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed           */
    FA_ERR_TIMEOUT = 4,      /* a kernel pipeline wait ran out (device flag) */
    FA_ERR_RANGE = 5         /* a bf16 input of the backward beyond +-65504 (device flag) */
} fa_status;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

#define FA_BLOCK 128 /* tile edge: rows of a query tile and keys of a key tile */

/*
 * Forward pass: O and LSE of exact attention, dense (causal = 0) or causal
 * (causal != 0). The block loop with running row max m and row sum l
 * ("Flash Attention: revolutionizing transformer efficiency", sections "The
 * Flash Attention Algorithm" and "Implementation Details"; corrected so the
 * output is normalised once, at the end).
 *   q, k, v  [B,H,N,d] in;   o [B,H,N,d] out;   lse [B,H,N] fp32 out.
 *   scale    multiplier of Q K^T (1/sqrt(d) for standard attention).
 */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int H, int N, int d, float scale, int causal,
                 fa_dtype dtype, void *stream);

/*
 * fa_fwd with key padding and an optional output residual.
 *   kv_len  DEVICE int32 [B] array, or NULL for none; keys j >= kv_len[b] are
 *           masked for all queries of batch b. Values above N act as N;
 *           values below 1 mask every key of that batch.
 *   o_res   DEVICE [B,H,N,d] array of the same 16-bit type, or NULL. When
 *           given, it receives the rounding residual of O: the fp32 result
 *           minus its 16-bit rounding, itself rounded to 16 bits, so that
 *           o + o_res carries about twice the precision of o. The backward
 *           uses it for D = rowsum(dO * O); with bf16 alone, the rounding of O
 *           moves D by up to ~0.05 at d = 128, which reaches dQ and dK.
 */
fa_status fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int H, int N, int d, float scale, int causal,
                    fa_dtype dtype, const int32_t *kv_len, void *o_res, void *stream);

/*
 * Block-sparse forward (the FlashAttention abstract names a block-sparse
 * extension of the method). block_mask is a DEVICE uint8
 * array [nb, nb], nb = ceil(N / 128), row = query tile, column = key tile,
 * nonzero = keep, shared by all (b, h). Masked tiles are neither loaded nor
 * multiplied; inside a kept tile attention is dense and non-causal.
 * o_res as in fa_fwd_ex (NULL for none).
 */
fa_status fa_fwd_blocksparse(const void *q, const void *k, const void *v, void *o,
                             float *lse, int B, int H, int N, int d, float scale,
                             fa_dtype dtype, const uint8_t *block_mask, void *o_res,
                             void *stream);

/*
 * Grouped-query (and multi-query) forward: Hkv key/value heads shared by
 * groups of H / Hkv query heads, query head h reading key/value head
 * h / (H / Hkv). The FlashAttention-2 page ("Flash Attention:
 * revolutionizing transformer efficiency", section FlashAttention-2) lists
 * multi-query and grouped-query attention among its additions; the
 * arithmetic per head is that of fa_fwd_ex.
 *   q, o [B,H,N,d]; k, v [B,Hkv,N,d]; lse [B,H,N]; kv_len, o_res as in
 *   fa_fwd_ex. 1 <= Hkv <= H and H % Hkv == 0, else FA_ERR_INVALID_ARG.
 *   Hkv == H is fa_fwd_ex.
 */
fa_status fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                     int B, int H, int Hkv, int N, int d, float scale, int causal,
                     fa_dtype dtype, const int32_t *kv_len, void *o_res, void *stream);

/*
 * Split-KV forward: the key tiles of every 128-row query tile are divided
 * into S contiguous shares, one CTA per (query tile, share), so that few
 * heads still fill the GPU. Each CTA writes its share's normalised fp32
 * O_s = (sum over its keys of p V) / l_s and LSE_s; a second kernel combines
 * the shares with the softmax merge identity ("Flash Attention:
 * revolutionizing transformer efficiency", section "The Math Behind Flash
 * Attention", softmax merger):
 *   LSE = M + log sum_s e^(LSE_s - M),  O = sum_s e^(LSE_s - LSE) O_s,
 *   M = max_s LSE_s; shares without keys (LSE_s = -inf) contribute nothing.
 * O, lse, o_res mean what they mean for fa_fwd_gqa (same layouts, q, k, v as
 * there); the result equals fa_fwd_gqa's up to fp32 rounding order.
 *   num_splits: S >= 1 as given (S may exceed the key tiles of a row; the
 *     surplus shares are empty); <= 0 lets the library choose S from the
 *     grid size and the SM count (fa_fwd_splitkv_num_splits). At most 256.
 *     S == 1 runs fa_fwd_gqa itself and needs no workspace.
 *   workspace: DEVICE memory of at least
 *     fa_fwd_splitkv_workspace_size(B, H, N, d, causal, num_splits) bytes,
 *     256-byte aligned, owned by the caller, contents ignored on entry; may
 *     be NULL when that size is 0.
 * Invalid sizes, pointers or a short workspace: FA_ERR_INVALID_ARG, nothing
 * launched.
 */
fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int H, int Hkv, int N, int d, float scale, int causal,
                         fa_dtype dtype, const int32_t *kv_len, void *o_res, int num_splits,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * 8-bit forward (the FlashAttention-3 section of "Flash Attention:
 * revolutionizing transformer efficiency" names low-precision FP8 attention;
 * the arithmetic is that of fa_fwd_gqa on the dequantised inputs):
 *   q [B,H,N,d], k, v [B,Hkv,N,d]: DEVICE e4m3 bytes (OCP FP8 E4M3, the
 *     layout of torch.float8_e4m3fn), 16-byte aligned; the real values are
 *     q_descale * q, k_descale * k, v_descale * v (per-tensor factors,
 *     finite and > 0).
 *   o [B,H,N,d] bf16 out; lse [B,H,N] fp32 out (natural log); scale,
 *     causal, Hkv, kv_len as in fa_fwd_gqa. d must be 128
 *     (FA_ERR_UNSUPPORTED otherwise).
 *   workspace: DEVICE memory of at least fa_fwd_fp8_workspace_size(B, Hkv,
 *     N, d) bytes, 256-byte aligned, owned by the caller, contents ignored
 *     on entry; receives V transposed per head ([d][N rounded up to 128]),
 *     the layout the 8-bit P V product reads.
 * Both products run on the tensor cores in e4m3 with fp32 accumulation;
 * P = softmax probabilities times 2^8 is rounded to e4m3 (relative error
 * <= 2^-4 per probability) before P V, the row sums use the unrounded
 * values, so LSE is as accurate as the 16-bit forward's and O carries the
 * rounding of P.
 */
fa_status fa_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int Hkv, int N, int d, float scale, int causal, float q_descale,
                     float k_descale, float v_descale, const int32_t *kv_len, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Workspace bytes of fa_fwd_fp8: B * Hkv * d * ceil(N / 128) * 128; 0 for invalid sizes. */
size_t fa_fwd_fp8_workspace_size(int B, int Hkv, int N, int d);

/*
 * Decode attention over a paged key/value cache ("Enhancing Transformer
 * Models: Innovations in Attention Mechanisms and Performance Optimization",
 * section "From FlashAttention to PagedAttention", which presents
 * PagedAttention as page-wise management of the data moved between HBM and
 * on-chip memory; the arithmetic per query row is exact attention as in
 * fa_fwd_gqa).
 *   q       [B,H,Nq,d] 16-bit: the Nq newest tokens of each of B sequences.
 *   k_cache, v_cache  [num_pages, Hkv, page_size, d] 16-bit page pools: page
 *           p holds page_size consecutive key (value) rows of every
 *           key/value head.
 *   block_table  DEVICE int32 [B, pages_per_seq]: logical page i of
 *           sequence b is pool page block_table[b * pages_per_seq + i].
 *           Entries must lie in [0, num_pages) for the pages that hold keys
 *           below seq_len[b]; entries past them are not read. An entry
 *           outside the pool reads as zero keys and values.
 *   seq_len DEVICE int32 [B]: keys of sequence b (the cached context,
 *           including the Nq new tokens); values above pages_per_seq *
 *           page_size act as that, values below 1 mask every key. Cache
 *           slots past seq_len may hold anything (they are never used).
 *   o [B,H,Nq,d] out (same 16-bit type); lse [B,H,Nq] fp32 out.
 *   Query i (0-based among the Nq) of sequence b sees keys
 *   j <= seq_len[b] - Nq + i (the new tokens attend causally to each other
 *   and to the whole cached prefix); query head h reads key/value head
 *   h / (H / Hkv). A query with no visible key gets O = 0, LSE = -inf.
 *   page_size in {16, 32, 64, 128}; d in {64, 128}; H % Hkv == 0.
 *   num_splits, workspace: as for fa_fwd_splitkv (the key tiles of each
 *   sequence are shared by S CTAs and merged); num_splits <= 0 picks S
 *   to fill one wave of CTAs (two per SM) when that gives at least two
 *   shares, else about two waves, with at least 16 key tiles of the
 *   longest sequence per share. The workspace size is
 *   fa_decode_paged_workspace_size.
 */
fa_status fa_decode_paged(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_table, const int32_t *seq_len, void *o, float *lse,
                          int B, int H, int Hkv, int Nq, int d, int page_size, int num_pages,
                          int pages_per_seq, float scale, fa_dtype dtype, int num_splits,
                          void *workspace, size_t workspace_bytes, void *stream);

/* The S fa_decode_paged uses (num_splits >= 1: itself; <= 0: the library's
 * choice for sequences of up to pages_per_seq * page_size keys); 0 for
 * invalid sizes. */
int fa_decode_paged_num_splits(int B, int H, int Hkv, int Nq, int d, int page_size,
                               int pages_per_seq, int num_splits);

/* Workspace bytes of fa_decode_paged: with T = ceil(H / Hkv * Nq / 64)
 * query tiles per (b, key/value head), S * B * Hkv * T * 128 * (d + 1) * 4;
 * 0 when S == 1 or for invalid sizes. */
size_t fa_decode_paged_workspace_size(int B, int H, int Hkv, int Nq, int d, int page_size,
                                      int pages_per_seq, int num_splits);

/*
 * The S fa_fwd_splitkv uses for these arguments (num_splits >= 1: itself;
 * <= 0: the library's choice for the current device), 0 for invalid sizes.
 */
int fa_fwd_splitkv_num_splits(int B, int H, int N, int d, int causal, int num_splits);

/*
 * Workspace bytes of fa_fwd_splitkv: with R = B * H * ceil(N / 128) * 128
 * padded query rows, fp32 O_s [S][R][d] then fp32 LSE_s [S][R];
 * 0 when S == 1 or for invalid sizes.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int causal, int num_splits);

/*
 * Bytes of device workspace fa_bwd / fa_bwd_blocksparse need for these
 * sizes. With R = B * H * ceil(N / 128) * 128 query rows padded to whole
 * tiles: fp32 LSE * log2(e) [R], fp32 D = rowsum(dO * O) [R] and an fp32 dQ
 * accumulator [R, d], each rounded up to 256 bytes; 256 bytes of statistics
 * (max |dO|, max |D|, max |V|, the dS exponent, the main kernel's work-item
 * counter); then room for fp16 copies of Q and of the scaled dO
 * ([B, H, N, d] each, rounded up to 256 bytes; used for bf16 inputs only).
 * Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass. The gradient of O = softmax(scale Q K^T + M) V with respect
 * to Q, K, V given dO, recomputing P tile by tile from Q, K and LSE instead of
 * storing it (key idea 2 of "Flash Attention: revolutionizing transformer
 * efficiency"):
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P o (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *   q, k, v, o, dout [B,H,N,d] in; lse [B,H,N] in (from the forward with the
 *   same arguments); dq, dk, dv [B,H,N,d] out; kv_len as in fa_fwd_ex.
 *   o_res: the residual fa_fwd_ex wrote for this O, or NULL (then D uses O
 *   alone).
 *   workspace: DEVICE memory of at least fa_bwd_workspace_size(B,H,N,d)
 *   bytes, 256-byte aligned, owned by the caller, contents ignored on entry.
 * dK and dV are deterministic; dQ sums the key tiles with fp32 atomics, so
 * its last bits may vary between runs.
 */
fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o,
                 const float *lse, const void *dout, void *dq, void *dk, void *dv,
                 int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                 const int32_t *kv_len, const void *o_res, void *workspace,
                 size_t workspace_bytes, void *stream);

/*
 * Grouped-query backward (the gradients of fa_fwd_gqa): dq [B,H,N,d] per
 * query head; dk, dv [B,Hkv,N,d], each the sum over the H / Hkv query heads
 * that read that key/value head. Each work item (batch, key/value head,
 * key tile) is walked by one CTA over every query head of its group, so dK
 * and dV are accumulated on chip and stay deterministic. Other arguments as in fa_bwd; the
 * workspace is fa_bwd_workspace_size(B, H, N, d) (query rows).
 */
fa_status fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv,
                     int B, int H, int Hkv, int N, int d, float scale, int causal,
                     fa_dtype dtype, const int32_t *kv_len, const void *o_res, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Block-sparse backward: fa_bwd with the block mask of fa_fwd_blocksparse. */
fa_status fa_bwd_blocksparse(const void *q, const void *k, const void *v, const void *o,
                             const float *lse, const void *dout, void *dq, void *dk,
                             void *dv, int B, int H, int N, int d, float scale,
                             fa_dtype dtype, const uint8_t *block_mask, const void *o_res,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * The three launches fa_bwd makes, in order, for callers that schedule or
 * time them separately (fa_bwd == prepare; main; finish on one stream, same
 * workspace). Arguments mean what they mean for fa_bwd / fa_bwd_blocksparse.
 *   fa_bwd_prepare  D = rowsum(dO * (O + o_res)) and LSE * log2(e) into the
 *                   workspace; zeroes the workspace's fp32 dQ accumulator;
 *                   records max |dO|, max |D| and max |V|; for bf16 inputs
 *                   writes the fp16 copies of Q and of the scaled dO into the
 *                   workspace.
 *   fa_bwd_main     zeroes the work-item counter in the workspace (a 4-byte
 *                   memset on the stream), then one persistent kernel (one
 *                   CTA per SM) takes the 128-key tiles of each key/value
 *                   head from it: dK and dV (written directly), dQ partials
 *                   added into the accumulator. Two fa_bwd_main calls that
 *                   share a workspace must not overlap. block_mask NULL
 *                   means dense/causal (causal applies only then); kv_len
 *                   must be NULL when block_mask is given
 *                   (FA_ERR_INVALID_ARG otherwise).
 *   fa_bwd_finish   dQ accumulator -> dq (fp16/bf16).
 */
fa_status fa_bwd_prepare(const void *q, const void *v, const void *o, const void *o_res,
                         const float *lse, const void *dout, int B, int H, int N, int d,
                         fa_dtype dtype, void *workspace, size_t workspace_bytes, void *stream);
fa_status fa_bwd_main(const void *q, const void *k, const void *v, const void *dout, void *dk,
                      void *dv, int B, int H, int N, int d, float scale, int causal,
                      fa_dtype dtype, const int32_t *kv_len, const uint8_t *block_mask,
                      void *workspace, size_t workspace_bytes, void *stream);
fa_status fa_bwd_finish(void *dq, int B, int H, int N, int d, fa_dtype dtype, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Backward pass for callers that cannot allocate device memory. (The paper
 * has no counterpart: this is a library convenience.) Some callers may not
 * call cudaMalloc or any allocator on the path that runs the backward: code
 * that executes inside another framework's or engine's enqueue/execute
 * callback, where device memory belongs to that host and allocating is
 * forbidden or unsafe, and code bound to a fixed memory budget that cannot
 * grow. They cannot supply fa_bwd's workspace, so this call uses a fixed
 * scratch array built into the library instead; everything else (inputs and
 * outputs) is still passed in, exactly as for fa_bwd / fa_bwd_blocksparse.
 *   block_mask  NULL: dense or causal (as fa_bwd); non-NULL: block-sparse
 *               (as fa_bwd_blocksparse; causal is ignored, and kv_len must
 *               be NULL: FA_ERR_INVALID_ARG otherwise).
 * Limits and behaviour:
 *   - the scratch holds fa_bwd_noalloc_max_workspace() bytes (32 MiB); sizes
 *     whose fa_bwd_workspace_size exceeds it are rejected with
 *     FA_ERR_INVALID_ARG before anything runs (for d = 128 that is about
 *     32K query rows: B * H * N <= 32512 when N is a multiple of 128);
 *   - the array is part of the library's device image: every GPU that loads
 *     the library holds it until the process exits;
 *   - the first call on a device looks up the array's device address (once
 *     per device and CUDA context, with that device current; a context that
 *     was reset and recreated is looked up again); make that first call
 *     before any stream capture;
 *   - all calls share the one array and it keeps the last call's contents;
 *     each call rewrites every part it reads (the dQ accumulator is zeroed
 *     by the call itself), but two calls that overlap on the GPU (different
 *     streams, or different host threads) race on it and must be ordered by
 *     the caller;
 *   - no cudaMalloc, cudaFree or other allocating routine is called.
 */
fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv,
                         int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                         const int32_t *kv_len, const uint8_t *block_mask, const void *o_res,
                         void *stream);

/* Bytes of the scratch array fa_bwd_noalloc uses (its size limit). */
size_t fa_bwd_noalloc_max_workspace(void);

/*
 * Synchronises `stream`, then reads and clears the device error word. Returns
 * FA_OK; FA_ERR_TIMEOUT when a kernel's pipeline wait timed out;
 * FA_ERR_CUDA when a kernel found its shared memory misaligned (it did no
 * work) or the synchronisation itself failed; FA_ERR_RANGE when the backward
 * clamped a bf16 input beyond +-65504. Several conditions: the first in
 * that order.
 */
fa_status fa_get_device_error(void *stream);

/*
 * Time limit of the kernels' pipeline waits on the current device, in
 * nanoseconds (0 restores the default of 2 s). A wait that runs out stops
 * its kernel early and sets the flag fa_get_device_error reports as
 * FA_ERR_TIMEOUT; a lower limit detects a stuck pipeline sooner. Waits for
 * copies already in flight after such a stop always allow the default, so
 * those copies land before the kernel exits. Synchronous; do not call while
 * kernels of this library run.
 */
fa_status fa_set_wait_limit_ns(unsigned long long ns);

/*
 * Test switch of the failure path (no counterpart in the pages). enable != 0
 * makes the load-issuing thread of every attention kernel on the current
 * device issue nothing, so each kernel's first pipeline wait can only run
 * out: the kernels then stop early, write zero outputs and set the
 * FA_ERR_TIMEOUT flag, which exercises the time limit, the abort of the
 * other roles and fa_get_device_error without any fault. Pair it with a low
 * fa_set_wait_limit_ns. enable == 0 restores normal operation. Synchronous.
 */
fa_status fa_debug_starve_pipelines(int enable);

/* Static string naming a status code. */
const char *fa_status_str(fa_status status);

/* Detail of the last failed call on this host thread ("" if none). */
const char *fa_last_error_message(void);

/* Library version string ("major.minor.patch"). */
const char *fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_H_ */
