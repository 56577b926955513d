// kernels.h -- internal launch interface between the C-ABI host code (api.cu)
// and the kernels.  Not part of the public API.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

struct FwdParams {
  void* O;          // [B, Hq, N, d] bf16 or fp32
  float* LSE;       // [B, Hq, N] natural-log units
  int* status;      // device status word
  int B, Hq, Hkv, N;  // N: query rows per head
  int Nk;           // keys per head (N for the plain forward)
  int kv_off;       // causal: key j is kept for query i when j <= i + kv_off (Nk - N)
  int n_splits;     // key range cut into n_splits parts of tiles_per_split 128-key tiles
  int tiles_per_split;
  long long o_split_stride;    // elements between the O outputs of consecutive splits
  long long lse_split_stride;  // same for LSE
  // GQA packing: with packed = 1 the G = Hq / Hkv query heads of a kv head
  // share one tile, whose row r is query r % N of head r / N of the group
  // (the heads of a group are adjacent, so their rows are contiguous).
  int packed;
  // Block-sparse mask (NULL: dense): uint8 [bmask_heads][n_qtiles][ceil(Nk/128)],
  // bmask_heads 1 or Hq; zero entries skip the 128 x 128 tile.
  const uint8_t* bmask;
  int bmask_heads;
  int heads;        // grid heads: B * Hq, or B * Hkv when packed
  int rows;         // rows per grid head: N, or G * N when packed
  int n_qtiles;     // ceil(rows / 128)
  int n_pairs;      // ceil(n_qtiles / 2): each CTA owns two 128-row query tiles
  int head_group;   // heads whose CTAs are launched together (L2 reuse of K/V)
  float scale_log2; // scale * log2(e)
  int causal;
  int out_f32;
  unsigned long long wait_limit_ns;
  // Persistent launch: items = heads * n_pairs * n_splits handed out by the
  // counter pair sched[0] (next item) and sched[1] (CTAs finished), both 0
  // at launch and reset to 0 by the last CTA.
  unsigned* sched;
  int n_items;
};

// Counter pair for a persistent launch on `stream`: each stream has its own
// pair from a per-device pool of 64 (launches on one stream run in order and
// share it; launches on different streams may run at once and do not).
unsigned* sched_counter_pair(cudaStream_t stream);

// tcgen05 forward for bf16 inputs with one query tile (rows <= 128) or a
// block mask.  tmQ/tmK/tmV are 3-D maps over [B*H][N][d] with a (64, 128, 1)
// box and 128-byte swizzle.
cudaError_t launch_fwd_bf16(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const FwdParams& p, cudaStream_t stream);
size_t fwd_bf16_smem_bytes(int d);
// Persistent form of the dense two-tile forward (rows > 128, no block mask):
// `ctas` CTAs (at most one per SM) walk the p.n_items work items.
cudaError_t launch_fwd_persist(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const FwdParams& p, int ctas, cudaStream_t stream);
constexpr int kMaxMaskTiles = 2048;  // key tiles a block-sparse forward may list per CTA

// Merge of a split forward's partial results: Opart [n_splits][rows][d] fp32
// (each normalised over its part), Lpart [n_splits][rows] fp32 (natural log)
// -> O [rows][d] (bf16 or fp32) and LSE [rows].
cudaError_t launch_fwd_merge(int d, const float* Opart, const float* Lpart, void* O, float* LSE, long long rows,
                             int n_splits, int out_f32, cudaStream_t stream);

// FP8 (e4m3) forward, d = 128, Nq = Nk = N.  tmQ/tmK: 3-D uint8 maps over
// [B*H][N][128] codes; tmVt over the transposed V codes [B*Hkv][128][Npad];
// all with a (128, 128, 1) box and 128-byte swizzle.
struct Fp8FwdParams {
  const float* sq;  // [B*Hq][T] block scales of Q (T = ceil(N / 128))
  const float* sk;  // [B*Hkv][T]
  const float* sv;  // [B*Hkv][T]
  void* O;          // [B, Hq, N, 128] bf16 or fp32
  float* LSE;       // [B, Hq, N]
  int* status;
  int B, Hq, Hkv, N, T;
  int heads;        // B * Hq
  int n_pairs;      // ceil(T / 2)
  int head_group;
  float scale_log2;
  int causal;
  int out_f32;
  unsigned long long wait_limit_ns;
};
cudaError_t launch_fwd_fp8(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmVt,
                           const Fp8FwdParams& p, cudaStream_t stream);
// Block quantizer: X bf16 [BH][N][d] -> codes ([BH][N][d], or [BH][d][ldt]
// when transposed) and scales [BH][ceil(N / 128)].
cudaError_t launch_quantize_fp8(int d, const uint16_t* X, uint8_t* codes, float* scales, long long BH, int N,
                                int transpose, int ldt, cudaStream_t stream);

// fp32 SIMT forward (exact fp32 arithmetic, FFMA + ex2).
cudaError_t launch_fwd_f32(int d, const float* Q, const float* K, const float* V, float* O,
                           float* LSE, int B, int Hq, int Hkv, int N, float scale_log2,
                           int causal, cudaStream_t stream);

struct BwdParams {
  const uint16_t* Q;    // [B, Hq, N, d] bf16
  const uint16_t* K;    // [B, Hkv, N, d]
  const uint16_t* V;
  const uint16_t* O;    // [B, Hq, N, d]
  const uint16_t* dO;
  const float* LSE;     // [B, Hq, N]
  uint16_t* dQ;         // [B, Hq, N, d]
  uint16_t* dK;         // [B, Hkv, N, d]
  uint16_t* dV;
  float* dQacc;         // workspace [B, Hq, Npad, d] fp32 (Npad: N rounded up to 128)
  float* negD;          // workspace [B, Hq, Npad]  -rowsum(dO * O)
  float* negLSE2;       // workspace [B, Hq, Npad]  -LSE * log2(e)
  int* status;
  int B, Hq, Hkv, N, Npad;
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  int causal;
  int head_group;       // kv heads whose CTAs are launched together (L2 reuse)
  unsigned long long wait_limit_ns;
  // Block-sparse mask (NULL: dense), as FwdParams::bmask with Nk = N.
  const uint8_t* bmask;
  int bmask_heads;
};
constexpr int kMaxMaskIters = 4096;  // (query head, query tile) pairs a masked backward CTA may list

// Query rows are padded to a multiple of this in the backward workspace.
int bwd_row_padding();
// Workspace layout of the backward (bytes), all fp32: dQacc then D then LSE2.
size_t bwd_workspace_bytes(int B, int Hq, int N, int d);

// Stages of the backward, launched in this order.
enum : unsigned { kBwdPre = 1u, kBwdMain = 2u, kBwdConvert = 4u, kBwdAll = 7u };

// tmDQ is a 2-D fp32 map over the dQ accumulator [B*Hq*Npad][d] with a
// (d, 64) box and no swizzle (bulk reduce-add target).
cudaError_t launch_bwd_bf16(int d, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                            const CUtensorMap& tmV, const CUtensorMap& tmdO, const CUtensorMap& tmDQ,
                            const BwdParams& p, unsigned stages, cudaStream_t stream);

}  // namespace attn
