/*
 * attn.h -- C ABI of the exact-attention library for NVIDIA GB300 (sm_103a).
 *
 * The library computes exact softmax attention
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V,     LSE_i = ln sum_j e^{s_ij},
 *
 * and its backward, with the tiled online-softmax method described in
 * "LLM 注意力与计算内核精读笔记 · 02 FlashAttention：IO 感知的精确注意力"
 * (§4 tiling, §5 online softmax merge, §6 recomputation) and in
 * "[Attention优化][2w字]原理&图解: 从Online-Softmax到FlashAttention V1/V2/V3"
 * (0x04 backward recomputation, 0x05 FlashAttention-2 loop order and the
 * deferred 1/l, 0x09 GQA indexing and causal tiles).  The result is exact up
 * to floating-point rounding: no approximation of the softmax is made.
 *
 * Data layout (all tensors): row-major [B, H, N, d], d contiguous.
 *   Q, O, dO, dQ : H = Hq            K, V, dK, dV : H = Hkv
 *   LSE          : [B, Hq, N] fp32, natural-log units of the scaled logits
 * Query head h reads key/value head h / (Hq / Hkv) (contiguous groups).
 * Causal masking keeps key j for query i when j <= i (Nq = Nk = N).
 *
 * Ownership: the caller owns every buffer; all pointers are device pointers
 * unless stated otherwise.  The library allocates no device memory: the
 * backward takes a caller-provided workspace.  Tensor pointers must be 16-byte
 * aligned and LSE 4-byte aligned.
 *
 * Streams: `stream` is a cudaStream_t passed as void*; NULL means the legacy
 * default stream.  Every call is asynchronous on that stream.  Argument and
 * launch errors are returned synchronously; a device-side failure (a bounded
 * wait inside a kernel that ran out) is recorded in a device status word and
 * reported by attn_last_device_status().  Calls on different streams may run
 * at the same time: the dense forward with more than 128 query rows runs
 * persistent CTAs that take work items from a pair of device counters, and
 * each stream has a pair of its own (64 per device; a 65th stream takes over
 * the pair of the stream seen longest ago, so keep at most 64 streams per
 * device issuing such forwards at once).  A captured graph holds its stream's
 * pair: do not replay it concurrently with itself or with calls on the
 * stream it was captured from.
 *
 * Errors: ATTN_ERR_INVALID_ARG for null or misaligned pointers, non-positive
 * sizes, Hq % Hkv != 0, a scale that is not finite and positive, or an
 * unknown dtype;
 * ATTN_ERR_UNSUPPORTED for combinations the kernels do not implement
 * (d other than 64 or 128, fp32 backward, fp32 input with bf16 output, the
 * FP8 forward with d other than 128, sizes past the grid or list limits);
 * ATTN_ERR_CUDA when a CUDA runtime call or launch fails.  There is no CPU
 * fallback.
 */
#ifndef EXACT_ATTENTION_GB300_ATTN_H
#define EXACT_ATTENTION_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,
  ATTN_ERR_UNSUPPORTED = 2,
  ATTN_ERR_CUDA = 3,
  ATTN_ERR_TIMEOUT = 4,
  ATTN_ERR_DEVICE = 5
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1 } attn_dtype;

/*
 * Forward.  Per (batch b, query head h, query row i):
 *   s_ij = scale * <Q[b,h,i,:], K[b,h/G,j,:]> for kept j,
 *   O[b,h,i,:] = sum_j softmax_j(s_i) V[b,h/G,j,:],  LSE[b,h,i] = ln sum_j e^{s_ij}
 * ("02 FlashAttention" §2 defines S, P, O; §5 the blockwise merge used).
 *
 *   Q [B,Hq,N,d], K and V [B,Hkv,N,d]   in_dtype (bf16: tensor-core path;
 *                                       fp32: CUDA-core path)
 *   O [B,Hq,N,d]                        out_dtype: bf16 or fp32 for bf16 input,
 *                                       fp32 for fp32 input
 *   LSE [B,Hq,N] fp32                   may not be NULL (the backward needs it)
 *   B, Hq, Hkv, N >= 1; Hq % Hkv == 0; d in {64, 128}; causal in {0, 1}.
 * O and LSE are fully overwritten.  Inputs are not modified.
 */
attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype in_dtype, attn_dtype out_dtype, void* stream);

/*
 * Forward with separate query and key lengths and an optional split of the
 * key range.  With Nq != Nk the causal mask is aligned to the bottom-right
 * corner ("从Online-Softmax…" 0x09): key j is kept for query i when
 * j <= i + (Nk - Nq); a query row with no kept key gets O = 0 and LSE = -inf.
 * The key range can be cut into num_splits contiguous parts (whole 128-key
 * tiles) that run in parallel and write partial (O, LSE) pairs, which a
 * merge kernel combines with the online-softmax merge ("02 FlashAttention"
 * §5; §12.1 applies it to key splits, FlashDecoding): LSE = ln sum_s e^{LSE_s},
 * O = sum_s e^{LSE_s - LSE} O_s.  This fills the GPU when B * Hq * ceil(Nq/256)
 * is small (decoding: Nq = 1 or a few rows against a long key range).  When
 * the G = Hq / Hkv query heads of a kv head have G * Nq <= 128 rows in all,
 * they share one 128-row tile (and one pass over K and V).
 *
 *   Q [B,Hq,Nq,d], K and V [B,Hkv,Nk,d]  bf16
 *   O [B,Hq,Nq,d]                        out_dtype: bf16 or fp32
 *   LSE [B,Hq,Nq] fp32
 *   B, Hq, Hkv, Nq, Nk >= 1; Hq % Hkv == 0; d in {64, 128}; causal in {0, 1}.
 *   num_splits: 0 chooses (1 when the unsplit grid fills the GPU, else the
 *     count that completes in the fewest waves of one CTA per SM), else
 *     1..256; it is capped
 *     at one split per 128-key tile and rounded so that no split is empty.
 *   workspace: attn_fwd_split_workspace_size(B, Hq, Hkv, Nq, Nk, d, num_splits)
 *     bytes, 256-byte aligned, owned by the caller, not shared with a
 *     concurrent call; NULL is allowed when that size is 0 (one split).
 * O and LSE are fully overwritten.  Inputs are not modified.  Errors as for
 * attn_fwd (a missing or short workspace: ATTN_ERR_INVALID_ARG).
 */
attn_status attn_fwd_split(const void* Q, const void* K, const void* V, void* O, float* LSE,
                           int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                           attn_dtype out_dtype, int num_splits, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Block-sparse forward: attn_fwd with a block mask on top of the causal rule
 * (Block-Sparse FlashAttention, "从Online-Softmax…" 0x04: the masked blocks
 * are skipped outright, i.e. their keys take no part in the softmax).
 *   block_mask: device pointer, uint8 [mask_heads][T][T] with T = ceil(N / 128)
 *     (query tile, key tile); mask_heads 1 (one mask for every head) or Hq;
 *     a zero entry removes the 128 x 128 block.  T <= 2048.
 *   A query row whose blocks are all removed gets O = 0 and LSE = -inf.
 * Other arguments as attn_fwd with bf16 input.
 */
attn_status attn_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, int mask_heads, attn_dtype out_dtype, void* stream);

/*
 * FP8 block quantization ("02 FlashAttention" §10: FlashAttention-3's FP8
 * path; §12.2: one scale per block).  Per head and per block of 128
 * consecutive rows (the last block may be shorter):
 *   scale = amax / 448 (fp32 division; 1 for an all-zero block),
 *   code  = e4m3(x / scale)  (fp32 quotient; OCP e4m3, round to nearest even,
 *           saturating to +-448).
 *   X      [BH, N, d] bf16 (device)
 *   codes  transpose = 0: [BH, N, d] uint8;
 *          transpose = 1: [BH, d, attn_fp8_vt_stride(N)] uint8, codes[b][c][i]
 *          = code of X[b][i][c], columns i >= N written as 0
 *   scales [BH, ceil(N / 128)] fp32
 *   BH, N >= 1; d in {64, 128}.  All outputs fully overwritten.
 */
int attn_fp8_vt_stride(int N); /* N rounded up to 16 (0 for N < 1) */
attn_status attn_quantize_fp8(const void* X, void* codes, float* scales, long long BH, int N, int d,
                              int transpose, void* stream);

/*
 * FP8 forward on block-quantized inputs: the function of attn_fwd evaluated
 * on the dequantized tensors Q = sq * Qc, K = sk * Kc, V = sv * Vc (the scale
 * of each element's 128-row block).  Both products run on e4m3 tensor cores
 * with fp32 accumulation; the probabilities P are rounded to e4m3 before P V
 * (scaled per key block so that P <= 256), the row sums use the unrounded P.
 *   Qc [B,Hq,N,128], Kc [B,Hkv,N,128] uint8 codes, q_scale [B,Hq,T],
 *   k_scale and v_scale [B,Hkv,T] fp32 with T = ceil(N / 128), Vtc the V
 *   codes transposed, [B,Hkv,128,attn_fp8_vt_stride(N)] (as written by
 *   attn_quantize_fp8 with transpose = 1); all scales > 0.
 *   O [B,Hq,N,128] out_dtype (bf16 or fp32), LSE [B,Hq,N] fp32.
 *   d must be 128 (else ATTN_ERR_UNSUPPORTED).  Other rules as attn_fwd.
 */
attn_status attn_fwd_fp8(const void* Qc, const float* q_scale, const void* Kc, const float* k_scale,
                         const void* Vtc, const float* v_scale, void* O, float* LSE, int B, int Hq, int Hkv,
                         int N, int d, float scale, int causal, attn_dtype out_dtype, void* stream);

/*
 * Block-sparse backward: attn_bwd with the block mask of attn_fwd_masked
 * (same layout and meaning); LSE must come from attn_fwd_masked with the same
 * mask.  Blocks the mask removes contribute nothing to dQ, dK, dV; a key row
 * that no kept block reaches gets dK = dV = 0.  (Hq / Hkv) * ceil(N / 128)
 * <= 4096.  Workspace and other arguments as attn_bwd (bf16).
 */
attn_status attn_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, int mask_heads, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Bytes of workspace attn_fwd_split needs for these sizes and num_splits
 * (0 when the key range is not split); 0 on bad sizes. */
size_t attn_fwd_split_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits);

/*
 * Backward of O with respect to Q, K, V given dO (no gradient through LSE).
 * The probabilities are recomputed per tile from the saved LSE
 * ("从Online-Softmax…" 0x04: recompute instead of storing S and P;
 * "02 FlashAttention" §6), with K/V tiles in the outer loop and dQ
 * accumulated across tiles (0x05).  With D_i = sum_k dO_ik O_ik:
 *   dP_ij = <dO_i, v_j>,  dS_ij = p_ij (dP_ij - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_{i, heads of group} dS_ij q_i,
 *   dV_j = sum_{i, heads of group} p_ij dO_i.
 *
 *   Q, O, dO [B,Hq,N,d] bf16; K, V [B,Hkv,N,d] bf16; LSE [B,Hq,N] fp32 as
 *   written by attn_fwd for the same Q, K, V, scale and causal.
 *   dQ [B,Hq,N,d], dK, dV [B,Hkv,N,d] bf16: fully overwritten.
 *   dtype must be ATTN_BF16 (fp32 backward: ATTN_ERR_UNSUPPORTED).
 *   workspace: device memory of at least attn_bwd_workspace_size() bytes,
 *   256-byte aligned, owned by the caller, contents need not be initialised;
 *   it must not be shared with a concurrent call.
 */
attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O,
                     const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* The three stages attn_bwd runs, in this order, as separate calls with the
 * same arguments (for callers that schedule or time them separately):
 *   attn_bwd_preprocess  D = rowsum(dO * O), LSE in log2 units, zeroed dQ
 *                        accumulator (all in the workspace);
 *   attn_bwd_main        the recompute-based tile loop: dK, dV written, dQ
 *                        accumulated in the workspace;
 *   attn_bwd_convert     dQ = bf16(scale * accumulator).
 * Each stage reads what the previous ones wrote to the workspace; running
 * them in order on one stream equals one attn_bwd call. */
attn_status attn_bwd_preprocess(const void* Q, const void* K, const void* V, const void* O,
                                const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                attn_dtype dtype, void* workspace, size_t workspace_bytes,
                                void* stream);
attn_status attn_bwd_main(const void* Q, const void* K, const void* V, const void* O,
                          const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                          int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                          attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);
attn_status attn_bwd_convert(const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                             int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                             attn_dtype dtype, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory where they run the backward: code hosted in a runtime that
 * owns every device allocation and hands out no workspace, and
 * latency-critical paths that must not call cudaMalloc (it can synchronise the
 * device, and it can fail).  The pages describe no such interface; it has no
 * counterpart there.
 *
 * Arguments and results are those of attn_bwd.  The scratch memory is a fixed
 * array of ATTN_NOALLOC_SCRATCH_BYTES bytes compiled into the library; every
 * GPU that loads the library holds it until the process exits.  Problems whose
 * attn_bwd_workspace_size() exceeds it return ATTN_ERR_UNSUPPORTED; null,
 * misaligned or mistyped arguments are reported first, with attn_bwd's
 * ATTN_ERR_INVALID_ARG, whatever the sizes.  The call
 * allocates nothing.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  All calls on a device share the array and
 * it keeps the last call's contents; the backward re-initialises what it
 * reads, so this does not affect results, but calls that overlap on the GPU
 * (other streams, other host threads) race on it: serialise them.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
attn_status attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                             int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                             attn_dtype dtype, void* stream);

/* Bytes of workspace attn_bwd needs: an fp32 dQ accumulator and two fp32
 * per-row vectors (D = rowsum(dO * O) and LSE in log2 units).  0 on bad sizes. */
size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d);

/* Static string naming a status code. */
const char* attn_status_string(attn_status s);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns ATTN_ERR_TIMEOUT if a kernel's bounded wait ran out
 * since the last call, ATTN_OK otherwise (ATTN_ERR_CUDA if the read fails). */
attn_status attn_last_device_status(void* stream);

/* Diagnostic: launches one CTA that waits, with the library's bounded-wait
 * routine and a limit of `limit_ns` nanoseconds (at most 1e9), on an mbarrier
 * that nothing will ever complete, then returns.  A working timeout path makes
 * the following attn_last_device_status() report ATTN_ERR_TIMEOUT. */
attn_status attn_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTENTION_GB300_ATTN_H */
