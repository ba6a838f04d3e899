/*
 * sa.h -- C ABI of libsa27: DeepSeek-V4 style hybrid compressed attention
 * (CSA + HCA) on one NVIDIA B300 (sm_103a).
 *
 * The operations follow these web pages (cited by title and section):
 *  [P2]  "오픈소스 LLM의 새 이정표: DeepSeek-V4 시리즈" -- section
 *        "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)": CSA compresses every m
 *        consecutive KV entries into one, each query attends only its top-k
 *        compressed entries, and a sliding-window branch keeps local detail;
 *        HCA compresses m' (>> m) entries into one and attends densely.
 *  [P2q] same page, section "오픈소스 MoE 인프라: MegaMoE와 TileLang": the
 *        indexer QK path is stored as MXFP4 and dequantised to FP8 losslessly.
 *  [P3]  "DeepSeek-V4 논문 읽기: 백만 토큰 컨텍스트를 저렴하게" -- sections
 *        "Compressed Sparse Attention (CSA)" (1 compress blocks, 2 the indexer
 *        finds relevant blocks, 3 only the top candidates are attended, 4 recent
 *        tokens kept by a sliding window), "Heavily Compressed Attention (HCA)"
 *        and "KV Cache 관리: 저장 구조까지 변경" (compressed cache, sliding-window
 *        cache, tail of tokens not yet compressed).
 *  [P1]  "EP 95. DeepSeek-V4 논문 읽기 — 노정석" -- section IDEAS: KV cache
 *        compressed to 1/4, a lightning indexer selects the top-k, multi-query
 *        attention (one shared KV head).
 * Readings where the pages are silent: pooling = softmax over one fp32 logit
 * per raw token; indexer score s = sum_h w_h * ReLU(q_h . k); block j is
 * visible to a query at position t iff j < floor((t+1)/m); ties in top-k go
 * to the lower index; the CSA softmax runs over selected rows and window rows
 * together; HCA also attends the window.
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; dense,
 *    row-major, in the layouts given per call.  Bulk arrays must be 16-byte
 *    aligned.  Nothing is allocated, freed or synchronised inside a call;
 *    work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Scratch memory is the caller's `ws` of `ws_bytes` bytes, at least the
 *    size the matching *_workspace_bytes() query returns (256-byte aligned).
 *    The attention calls also keep a work counter there, zeroed by the call
 *    on its stream: calls that share a workspace must not overlap.
 *  - Return value: SA_OK, or an sa_status for a host-side rejection (bad
 *    argument, unsupported shape) or a CUDA launch error.  Problems found on
 *    the device (an index out of range, a NaN score, a wait that timed out) are
 *    OR-ed as (1 << status) into the optional device word `err` (may be NULL);
 *    the kernels never trap and leave the context usable.
 *  - Positions are 0-based.  q_pos[b*T + t] is the position of query t of
 *    sequence b; L = q_pos + 1 tokens are visible to it, including itself.
 *  - Raw (uncompressed) per-token arrays are rings of R rows: raw position p
 *    lives in row p mod R (R = sequence length gives the identity layout).
 *  - Calls are stateless and may be issued from several host threads.
 */
#ifndef SA27_H
#define SA27_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned array  */
  SA_ERR_UNSUPPORTED = 2,    /* valid but not implemented for this shape  */
  SA_ERR_CUDA = 3,           /* CUDA runtime/driver error at launch       */
  SA_ERR_DEVICE_TIMEOUT = 4, /* device: a bounded wait gave up            */
  SA_ERR_BOUNDS = 5,         /* device: index/position outside its range  */
  SA_ERR_NAN = 6             /* device: NaN candidate score in top-k      */
} sa_status;

typedef enum {
  SA_F32 = 0,   /* float32                                                  */
  SA_BF16 = 1,  /* bfloat16                                                 */
  SA_MXFP4 = 2  /* indexer path only: e2m1 codes, two per byte (element 2i in
                   the low nibble), plus one e8m0 scale byte per 32 elements */
} sa_dtype;

/* Text for a status code (static string). */
const char* sa_status_string(int status);

/* ---------------------------------------------------------------------------
 * csa_compress -- block compression ([P2], [P3] CSA step 1; KV cache layout
 * of [P3] "KV Cache 관리").
 * For each sequence b and each block j in [blk_lo[b], blk_hi[b]):
 *     a_i = softmax(z[p_i] : i < m)_i,   p_i = j*m + i,
 *     X_c[b, j, :] = sum_i a_i * X_raw[b, p_i mod R, :]
 * for X in {K, V} (width d) and, if ik_raw != NULL, the indexer keys
 * (width dI).  Results are rounded to the storage type (bf16: nearest-even).
 * The same call with m = m' builds the HCA cache (ik_raw = NULL).
 *  dtype     SA_F32 or SA_BF16: storage type of k_raw, v_raw, k_c, v_c
 *  ik_dtype  SA_F32 / SA_BF16 (ik_raw and ik_c share it) or SA_MXFP4
 *            (ik_raw bf16; ik_c receives codes [B,N_cap,dI/2] u8 and
 *            ik_c_scales [B,N_cap,dI/32] u8, quantised from the bf16-rounded
 *            pooled values by the OCP MX v1.0 rule)
 *  k_raw, v_raw [B,R,d]; ik_raw [B,R,dI] or NULL; z [B,R] f32 pooling logits
 *  blk_lo, blk_hi [B] int32 device; max_blocks = host bound on
 *            blk_hi[b]-blk_lo[b] (sizes the grid; larger ranges -> SA_ERR_BOUNDS)
 *  k_c, v_c [B,N_cap,d]; ik_c as above (NULL iff ik_raw is NULL)
 * Device errors: block outside [0, N_cap) -> SA_ERR_BOUNDS (block skipped).
 */
int csa_compress(int dtype, int ik_dtype, int B, int d, int dI, int m, const void* k_raw,
                 const void* v_raw, const void* ik_raw, const float* z, int R,
                 const int32_t* blk_lo, const int32_t* blk_hi, int max_blocks, void* k_c,
                 void* v_c, void* ik_c, void* ik_c_scales, int N_cap, int32_t* err,
                 void* stream);

/* ---------------------------------------------------------------------------
 * csa_index_topk -- lightning-indexer scores and per-query top-k ([P1] IDEAS;
 * [P3] CSA steps 2-3; [P2] "top-k compressed entries").
 * For query row r = b*T + t at position p = q_pos[r], n = floor((p+1)/m):
 *     s[r, j] = sum_h w[r,h] * max(0, q_I[r,h,:] . Ik_c[b,j,:]),  0 <= j < n
 * idx[r, :] = the min(k, n) indices j with the highest s (equal scores: lower
 * j first), written in ascending order, padded with -1.
 *  q_dtype   SA_F32, SA_BF16 or SA_MXFP4; ik_c has the same dtype
 *  q_idx     [B,T,HI,dI] (MXFP4: codes [B,T,HI,dI/2] + q_scales [B,T,HI,dI/32])
 *  w         [B,T,HI] f32 indexer head weights
 *  ik_c      [B,N_cap,dI] (MXFP4: codes + ik_scales as in csa_compress)
 *  q_pos     [B,T] int32
 *  idx       [B,T,k] int32 output
 *  scores_out  optional [B,T,N_cap] f32: receives s (entries j >= n untouched)
 *  scores_in   optional [B,T,N_cap] f32: if given, scoring is skipped and the
 *              top-k selects from these values (same n per row)
 *  k = 0 with scores_out given computes the scores only (idx untouched).
 *  ws          scratch of csa_index_topk_workspace_bytes() bytes when
 *              scores_out and scores_in are both NULL (holds the scores)
 * Kernels: bf16 with HI = 64, dI = 64 scores on the tensor cores (tcgen05);
 * other f32/bf16 shapes (HI*dI <= 12K) on CUDA cores.  SA_MXFP4 (HI = 64,
 * dI = 64, N_cap a multiple of 8, 16-byte aligned codes and key scales):
 * codes are dequantised in-kernel to e4m3 with each 64-wide row's larger
 * block exponent factored out -- exact while the row's two block exponents
 * differ by at most 8 -- contracted with tcgen05 kind::f8f6f4 into fp32, and
 * the row exponents applied in fp32 before the weighted ReLU head sum.
 * N_cap <= 524288 (a row's candidates split over at most 16 CTAs of one
 * thread-block cluster; SA_ERR_UNSUPPORTED if the device cannot run the
 * cluster size a row needs).
 * Device errors: NaN score -> SA_ERR_NAN (row written as all -1);
 * n > N_cap -> SA_ERR_BOUNDS (n clamped).
 */
int csa_index_topk(int q_dtype, int B, int T, int HI, int dI, int m, int k, const void* q_idx,
                   const void* q_scales, const float* w, const void* ik_c,
                   const void* ik_scales, int N_cap, const int32_t* q_pos, int32_t* idx,
                   float* scores_out, const float* scores_in, void* ws, size_t ws_bytes,
                   int32_t* err, void* stream);
size_t csa_index_topk_workspace_bytes(int B, int T, int N_cap, int k);

/* ---------------------------------------------------------------------------
 * csa_index_topk_noalloc -- csa_index_topk for callers that cannot give the
 * library any scratch memory.  The pages have no counterpart to this call;
 * it is a convenience of this library.
 *
 * Who needs it: a caller that owns every byte of device memory and hands a
 * kernel library only its inputs and outputs -- for example a serving engine
 * that reserved the whole GPU for its KV-cache pool at start-up, or a plugin
 * whose host framework forbids side allocations -- and a decode loop that
 * cannot afford cudaMalloc, which may synchronise the device and takes
 * unbounded time.
 *
 * Same operation, arguments, layouts, host-side and device errors as
 * csa_index_topk, without scores_out, scores_in and the workspace.  q_dtype
 * must be SA_F32 or SA_BF16 (SA_MXFP4 gives SA_ERR_UNSUPPORTED; an unknown
 * dtype SA_ERR_INVALID_ARG, as csa_index_topk).  The scores live in a fixed device array inside the library
 * (SA_NOALLOC_MAX_SCORES floats, 8 MiB), which every GPU that loads the
 * library holds until the process exits.  Limit: B * T * N_cap <=
 * SA_NOALLOC_MAX_SCORES, otherwise SA_ERR_UNSUPPORTED is returned before any
 * work is enqueued.  Nothing is allocated or freed (no cudaMalloc, cudaFree
 * or allocating library routine).
 *
 * First call on a device: it looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it; make that
 * first call before any stream capture.  Calls on the same device share the
 * one array and it keeps the last call's scores: two calls that overlap on
 * the GPU (different streams, no ordering between them) race and give wrong
 * results.  No part of the array needs to start at zero -- every score the
 * top-k reads is written by the same call first -- so nothing is cleared.
 */
#define SA_NOALLOC_MAX_SCORES 2097152
int csa_index_topk_noalloc(int q_dtype, int B, int T, int HI, int dI, int m, int k,
                           const void* q_idx, const void* q_scales, const float* w,
                           const void* ik_c, const void* ik_scales, int N_cap,
                           const int32_t* q_pos, int32_t* idx, int32_t* err, void* stream);

/* ---------------------------------------------------------------------------
 * csa_attend -- sparse multi-query attention over the selected compressed
 * rows plus the sliding window, in one softmax ([P2]; [P3] CSA steps 3-4).
 * For query row r (sequence b, position p), n = floor((p+1)/m),
 * S = { idx[r,i] : i < min(k,n), idx[r,i] >= 0 },  Wn = min(W, p+1):
 *     keys   = { K_c[b,j] : j in S }  (+)  { K_raw[b, u mod R] : p-Wn < u <= p }
 *     l      = sm_scale * q[r,h,:] . key
 *     lse[r,h] = log sum exp(l),   o[r,h,:] = sum softmax(l) * value
 * An empty key set gives o = 0, lse = -inf.
 *  dtype     SA_F32 or SA_BF16 for q, k_c, v_c, k_raw, v_raw
 *  q [B,T,H,d]; k_c, v_c [B,N_cap,d]; idx [B,T,k]; k_raw, v_raw [B,R,d]
 *  o [B,T,H,d] in o_dtype (SA_F32, or SA_BF16 rounded to nearest-even from
 *  the fp32 result); lse [B,T,H] f32 (natural log)
 * bf16 with H <= 64, d = 128 runs on the tensor cores; other shapes on CUDA
 * cores (d <= 256, d a multiple of 4, H * d <= 16384).  Requires R >= W.
 * Device errors: idx entry >= n or < -1 -> SA_ERR_BOUNDS (entry ignored).
 */
int csa_attend(int dtype, int B, int T, int H, int d, int m, int k, int W, float sm_scale,
               const void* q, const int32_t* q_pos, const void* k_c, const void* v_c,
               int N_cap, const int32_t* idx, const void* k_raw, const void* v_raw, int R,
               void* o, int o_dtype, float* lse, void* ws, size_t ws_bytes, int32_t* err,
               void* stream);
size_t csa_attend_workspace_bytes(int dtype, int B, int T, int H, int d, int k, int W);

/* ---------------------------------------------------------------------------
 * hca_compress_attend -- heavy compression then dense attention ([P2] HCA;
 * [P3] "Heavily Compressed Attention (HCA)").
 * First compresses blocks [blk_lo[b], blk_hi[b]) of m2 raw rows into
 * hk_c/hv_c exactly as csa_compress does (no indexer keys); then, for query
 * row r at position p, n2 = floor((p+1)/m2), Wn = min(W, p+1):
 *     keys = { hK_c[b,j] : j < n2 }  (+)  { K_raw[b, u mod R] : p-Wn < u <= p }
 * with the same softmax, o and lse definitions as csa_attend.
 *  q [B,T,H,d]; k_raw, v_raw [B,R,d]; z_hca [B,R] f32; hk_c, hv_c [B,N2_cap,d]
 *  o [B,T,H,d] in o_dtype (SA_F32 or SA_BF16, as csa_attend); lse [B,T,H] f32
 * Requires R >= W and, when compressing, R >= m2; d <= 256, a multiple of 4.
 */
int hca_compress_attend(int dtype, int B, int T, int H, int d, int m2, int W, float sm_scale,
                        const void* q, const int32_t* q_pos, const void* k_raw,
                        const void* v_raw, const float* z_hca, int R, const int32_t* blk_lo,
                        const int32_t* blk_hi, int max_blocks, void* hk_c, void* hv_c,
                        int N2_cap, void* o, int o_dtype, float* lse, void* ws,
                        size_t ws_bytes, int32_t* err, void* stream);
size_t hca_compress_attend_workspace_bytes(int dtype, int B, int T, int H, int d, int N2_cap,
                                           int W);

/* ---------------------------------------------------------------------------
 * csa_decode -- the whole CSA layer for one new token per sequence, in one
 * launch: csa_compress of the blocks [blk_lo[b], blk_hi[b]) this step closes,
 * csa_index_topk and csa_attend, fused ([P2]; [P3] CSA steps 1-4 and "KV
 * Cache 관리"; [P1] IDEAS: the mega-kernel direction).  Results are those of
 * the three calls in sequence on the same inputs: the cache rows written and
 * idx are bit-identical to theirs (same arithmetic, same order); o and lse
 * differ only by the fp32 rounding of a different split of the key list.
 * One query per sequence (T = 1): query b sits at position q_pos[b].
 *  q [B,H,128] bf16 (H <= 64); q_idx [B,64,64] bf16; w [B,64] f32
 *  k_raw, v_raw [B,R,128] bf16; ik_raw [B,R,64] bf16; z [B,R] f32 (R >= W, R >= m)
 *  blk_lo, blk_hi [B] int32 device; max_blocks host bound on blk_hi - blk_lo
 *  k_c, v_c [B,N_cap,128] bf16; ik_c [B,N_cap,64] bf16 (read, and the closed
 *            blocks written); m <= 128; N_cap <= 262144
 *  idx [B,k] int32 output; o [B,H,128] in o_dtype (SA_F32 or SA_BF16);
 *  lse [B,H] f32
 * No workspace: each sequence is one thread-block cluster of up to 16 CTAs
 * that keeps its scores, its selection and its partial results in shared
 * memory.  Fastest when B x (CTAs per cluster) fills the GPU (e.g. B = 32 at
 * 128K context); SA_ERR_UNSUPPORTED if the device cannot run the cluster.
 * Device errors as csa_compress, csa_index_topk and csa_attend.
 */
int csa_decode(int B, int H, int d, int HI, int dI, int m, int k, int W, float sm_scale,
               const void* q, const void* q_idx, const float* w, const int32_t* q_pos,
               const void* k_raw, const void* v_raw, const void* ik_raw, const float* z, int R,
               const int32_t* blk_lo, const int32_t* blk_hi, int max_blocks, void* k_c,
               void* v_c, void* ik_c, int N_cap, int32_t* idx, void* o, int o_dtype,
               float* lse, int32_t* err, void* stream);

/* ---------------------------------------------------------------------------
 * sa_decode_step -- the whole decode step of both layers for one new token
 * per sequence, in one launch ([P2] "압축 희소 어텐션(CSA)과 극압축 어텐션(HCA)";
 * [P3] CSA steps 1-4, HCA and "KV Cache 관리"; [P1] IDEAS: the mega-kernel
 * direction): what csa_compress, csa_index_topk, csa_attend and
 * hca_compress_attend compute for the same inputs, in one persistent kernel
 * whose CTAs take work items (pooling, 2048-entry score slices, a row's
 * top-k, shares of a row's key list) from a queue, so that one sequence's
 * top-k and attention run while others are still scored.  The cache rows
 * written and idx are bit-identical to the separate calls'; o, lse, ho and
 * hlse differ only by the fp32 rounding of a different split of the key
 * list.  One query per sequence (T = 1) at position q_pos[b].
 *  q, q_hca [B,H,128] bf16 (H <= 64): the CSA and the HCA layer's queries
 *  q_idx [B,64,64] bf16; w [B,64] f32: indexer queries and head weights
 *  k_raw, v_raw, hk_raw, hv_raw [B,R,128] bf16; ik_raw [B,R,64] bf16;
 *  z, hz [B,R] f32: each layer's ring of raw rows and pooling logits
 *  (R >= W, R >= m, R >= m2)
 *  blk_lo, blk_hi / hblk_lo, hblk_hi [B] int32 device: the CSA / HCA blocks
 *  this step closes; max_blocks / max_blocks2 host bounds on their lengths
 *  k_c, v_c [B,N_cap,128], ik_c [B,N_cap,64]; hk_c, hv_c [B,N2_cap,128]
 *  bf16: the caches (read; the closed blocks written); m, m2 <= 128;
 *  N_cap <= 32768 (a row's scores fit one CTA's shared memory), else
 *  SA_ERR_UNSUPPORTED -- longer rows take the separate calls or csa_decode
 *  idx [B,k] int32; o, ho [B,H,128] in o_dtype (SA_F32 or SA_BF16);
 *  lse, hlse [B,H] f32: outputs
 *  ws: sa_decode_step_workspace_bytes(B, H, N_cap, k, W, N2_cap) bytes,
 *  16-byte aligned, owned by the caller; the call zeroes its counters on
 *  `stream` first, so calls sharing a workspace must not overlap.  Too
 *  small -> SA_ERR_INVALID_ARG; 0 from the query means the shape is not
 *  taken (SA_ERR_UNSUPPORTED).
 * Device errors as the separate calls; a bounded wait that gives up raises
 * SA_ERR_DEVICE_TIMEOUT and every CTA stops taking work.
 */
size_t sa_decode_step_workspace_bytes(int B, int H, int N_cap, int k, int W, int N2_cap);
int sa_decode_step(int B, int H, int d, int HI, int dI, int m, int k, int W, int m2,
                   float sm_scale, const void* q, const void* q_idx, const float* w,
                   const void* q_hca, const int32_t* q_pos, const void* k_raw, const void* v_raw,
                   const void* ik_raw, const float* z, const void* hk_raw, const void* hv_raw,
                   const float* hz, int R, const int32_t* blk_lo, const int32_t* blk_hi,
                   int max_blocks, const int32_t* hblk_lo, const int32_t* hblk_hi,
                   int max_blocks2, void* k_c, void* v_c, void* ik_c, int N_cap, void* hk_c,
                   void* hv_c, int N2_cap, int32_t* idx, int o_dtype, void* o, float* lse,
                   void* ho, float* hlse, void* ws, size_t ws_bytes, int32_t* err,
                   void* stream);

/* ---------------------------------------------------------------------------
 * Backward pass.  The top-k selection is not differentiable ([P1] IDEAS), so
 * it is a constant mask: the gradient of a loss with dL/dO given reaches the
 * queries, the attended cache rows and window rows, and -- through the
 * pooling of the blocks a pass compressed -- the raw rows and their pooling
 * logits.  The indexer (q_idx, w, the indexer keys) gets no gradient.  The
 * caches' storage rounding is taken as the identity.  Every gradient output
 * is fp32 and is ADDED to (the caller zeroes it first, or accumulates over
 * layers and steps); several queries that attend the same row add their
 * parts with atomics, so the summation order is not fixed.
 *
 * csa_attend_backward -- gradient of csa_attend for the given idx:
 *   with P = exp(sm_scale q.k - lse) over the row's key list,
 *   dV += sum_h P dO_h; dS = P (dO_h.V - dO_h.O_h); dq += sm_scale sum dS K;
 *   dK += sm_scale sum_h dS q_h  (selected rows -> dk_c/dv_c, window rows ->
 *   dk_raw/dv_raw at ring row u mod R).
 *  arguments as csa_attend, plus o [B,T,H,d] f32 and lse [B,T,H] f32 (the
 *  forward's outputs, o_dtype SA_F32) and dout [B,T,H,d] f32;
 *  dq [B,T,H,d], dk_c, dv_c [B,N_cap,d], dk_raw, dv_raw [B,R,d]: f32, added to.
 *  CUDA cores, fp32 (H*d*12 + 33*(d+1)*8 bytes of shared memory <= 227 KB).
 */
int csa_attend_backward(int dtype, int B, int T, int H, int d, int m, int k, int W,
                        float sm_scale, const void* q, const int32_t* q_pos, const void* k_c,
                        const void* v_c, int N_cap, const int32_t* idx, const void* k_raw,
                        const void* v_raw, int R, const float* o, const float* lse,
                        const float* dout, float* dq, float* dk_c, float* dv_c, float* dk_raw,
                        float* dv_raw, int32_t* err, void* stream);

/* hca_attend_backward -- gradient of the attention of hca_compress_attend
 * (every visible HCA row plus the window): as csa_attend_backward with the
 * dense key list; dhk_c, dhv_c [B,N2_cap,d]. */
int hca_attend_backward(int dtype, int B, int T, int H, int d, int m2, int W, float sm_scale,
                        const void* q, const int32_t* q_pos, const void* hk_c, const void* hv_c,
                        int N2_cap, const void* k_raw, const void* v_raw, int R, const float* o,
                        const float* lse, const float* dout, float* dq, float* dhk_c,
                        float* dhv_c, float* dk_raw, float* dv_raw, int32_t* err, void* stream);

/* sa_compress_backward -- gradient of the K/V pooling of csa_compress (or of
 * hca_compress_attend's, with m = m') for the blocks [blk_lo[b], blk_hi[b]):
 * with a = softmax(z over the block) and the unrounded pooled row
 * Xc = sum_i a_i X_i, for X in {K, V}:
 *     dX_raw[p_i mod R] += a_i dXc;   dz[p_i mod R] += a_i (X_i - Xc) . dXc
 *  k_raw, v_raw [B,R,d] in dtype; z [B,R] f32; dk_c, dv_c [B,N_cap,d] f32
 *  (the cache-row gradients, e.g. from csa_attend_backward); dk_raw, dv_raw
 *  [B,R,d] and dz [B,R] f32, added to.  m <= 6144.
 */
int sa_compress_backward(int dtype, int B, int d, int m, const void* k_raw, const void* v_raw,
                         const float* z, int R, const int32_t* blk_lo, const int32_t* blk_hi,
                         int max_blocks, const float* dk_c, const float* dv_c, int N_cap,
                         float* dk_raw, float* dv_raw, float* dz, int32_t* err, void* stream);

/* ---------------------------------------------------------------------------
 * sa_mxfp4_quantize -- MXFP4 storage of bf16 rows for the low-precision
 * indexer path ([P2q]: the indexer QK path is stored in FP4 (MXFP4)).
 * Block rule of the OCP Microscaling Formats (MX) v1.0 specification: for
 * each block of 32 consecutive values, e = floor(log2(max |x|)) - 2 clamped to
 * [-127, 127] (an all-zero block gets -127); each element is x / 2^e rounded
 * to the nearest e2m1 value (0, .5, 1, 1.5, 2, 3, 4, 6; ties to the even
 * code), saturating at 6; a negative element that rounds to 0 is stored as +0.
 *  x       [nblk * 32] bf16 (device)
 *  codes   [nblk * 16] u8: element 2i in the low nibble of byte i
 *  scales  [nblk] u8: e + 127 (e8m0)
 * Used for the indexer queries of each step (the indexer key cache is written
 * in this format by csa_compress with ik_dtype = SA_MXFP4).
 */
int sa_mxfp4_quantize(const void* x, int64_t nblk, void* codes, void* scales, void* stream);

/* ---------------------------------------------------------------------------
 * sa_compress_channels -- the compressor variant with one pooling logit per
 * raw token AND channel ([P3] "Compressed Sparse Attention (CSA)" step 1: m
 * consecutive entries merged into one; here every channel has its own merge
 * weights):
 *     x_c[b, j, c] = sum_i softmax_i(z[b, p_i, c]) * x_raw[b, p_i, c],
 * p_i = (j*m + i) mod R, i < m, for the blocks [blk_lo[b], blk_hi[b]).  Pools
 * one array (K, V or the indexer key, each with its own logits); rounds to
 * the storage type.
 *  dtype      SA_F32 or SA_BF16: x_raw and x_c
 *  x_raw [B,R,d]; z [B,R,d] f32; x_c [B,N_cap,d]
 *  blk_lo, blk_hi [B] int32 device; max_blocks host bound on their lengths
 * fp32 evaluation, per channel in ascending i: the max logit, the sum of
 * exp(z_i - max), then sum_i (exp(z_i - max) / sum) * x_i by fused
 * multiply-adds.  Device errors: a block outside [0, N_cap) or a range
 * longer than max_blocks -> SA_ERR_BOUNDS (block skipped).
 */
int sa_compress_channels(int dtype, int B, int d, int m, const void* x_raw, const float* z, int R,
                         const int32_t* blk_lo, const int32_t* blk_hi, int max_blocks, void* x_c,
                         int N_cap, int32_t* err, void* stream);

/* ---------------------------------------------------------------------------
 * sa_ring_write -- writes each sequence's new token into the sliding-window
 * rings ([P3] "KV Cache 관리: 저장 구조까지 변경": the raw rows of a layer's
 * last tokens are kept per sequence in a ring of R rows, token t in row
 * t mod R, from which the window is attended and the next blocks pooled):
 *     ring_i[b, pos[b] mod R, :] = rows_i[b, :]   for each array i < n
 * One launch for all arrays (e.g. a step's K, V, indexer key and pooling
 * logit of both layers).
 *  n          number of arrays, 1..8
 *  rings      HOST array of n device pointers: ring i [B, R, row_bytes[i]]
 *  rows       HOST array of n device pointers: rows i [B, row_bytes[i]]
 *  row_bytes  HOST array of n sizes, each a positive multiple of 4
 *  pos        [B] int32 device: each sequence's new position
 * Errors: n outside 1..8, a size not a positive multiple of 4, a null or
 * misaligned (4-byte) pointer -> SA_ERR_INVALID_ARG.  Device errors:
 * pos[b] < 0 -> SA_ERR_BOUNDS (that sequence's rows are skipped).
 */
int sa_ring_write(int B, int R, const int32_t* pos, int n, void* const* rings,
                  const void* const* rows, const int* row_bytes, int32_t* err, void* stream);

/* ---------------------------------------------------------------------------
 * attn_merge -- exact log-sum-exp merge of attention partials computed over
 * disjoint key sets (the branches of the multi-branch design, [P2] and [P1]
 * IDEAS; also split-K partials):
 *     lse = log sum_i exp(lse_i),   o = sum_i exp(lse_i - lse) * o_i
 * Parts with lse_i = -inf contribute nothing; all -inf gives o = 0, lse = -inf.
 *  n         number of parts, 1..8
 *  o_parts   HOST array of n device pointers, each [rows, d] f32
 *  lse_parts HOST array of n device pointers, each [rows] f32
 *  o         [rows, d] in o_dtype (SA_F32 or SA_BF16); lse [rows] f32
 */
int attn_merge(int n, const float* const* o_parts, const float* const* lse_parts, int64_t rows,
               int d, void* o, int o_dtype, float* lse, int32_t* err, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SA27_H */
