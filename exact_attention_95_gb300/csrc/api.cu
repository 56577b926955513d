// api.cu -- the C ABI declared in include/attn.h: argument checks, TMA
// tensor-map construction, kernel launches and the device status word.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {

// Device status word: kernels record the first failure of a launch here
// (atomicCAS from 0); attn_last_device_status reads and clears it.
__device__ int g_status = 0;

// Work counters of persistent launches: kSchedPairs pairs (next item, CTAs
// finished) per device, 0 between launches (each launch's last CTA resets its
// pair).  A pair belongs to a stream: launches on one stream run one after
// the other and reuse it; up to kSchedPairs streams per device get pairs of
// their own (a further stream takes over the pair of the stream seen longest
// ago).
constexpr int kSchedPairs = 64;
__device__ unsigned g_sched[2 * kSchedPairs];

namespace {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s per wait

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// cuTensorMapEncodeTiled through a small cache keyed by every argument that
// enters the encoding (a map holds the address and the geometry, nothing of
// the contents, so a hit is exactly the map a new encoding would give).
// Repeated calls on the same buffers -- a training or decoding loop -- skip
// the host-side encoding.  64 entries, replaced in turn; one mutex.
struct MapKey {
  int dtype, rank, swizzle;
  uintptr_t base;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3];
  bool operator==(const MapKey& o) const {
    if (dtype != o.dtype || rank != o.rank || swizzle != o.swizzle || base != o.base) return false;
    for (int i = 0; i < 3; ++i)
      if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
    return strides[0] == o.strides[0] && strides[1] == o.strides[1];
  }
};

bool encode_tiled(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  constexpr int kEntries = 64;
  static MapKey keys[kEntries];
  static CUtensorMap maps[kEntries];
  static bool used[kEntries] = {};
  static int next = 0;
  static std::mutex mu;
  MapKey k{};
  k.dtype = (int)dtype;
  k.rank = rank;
  k.swizzle = (int)swizzle;
  k.base = reinterpret_cast<uintptr_t>(base);
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < kEntries; ++i)
      if (used[i] && keys[i] == k) {
        *m = maps[i];
        return true;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(mu);
  keys[next] = k;
  maps[next] = *m;
  used[next] = true;
  next = (next + 1) % kEntries;
  return true;
}

// Device address of the status word on the current device.
int* status_ptr() {
  static int* ptrs[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

}  // namespace

unsigned* sched_counter_pair(cudaStream_t stream) {
  static unsigned* base[64] = {};
  static cudaStream_t owner[64][kSchedPairs] = {};
  static bool taken[64][kSchedPairs] = {};
  static unsigned next[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!base[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sched) != cudaSuccess) return nullptr;
    base[dev] = static_cast<unsigned*>(p);
  }
  for (int i = 0; i < kSchedPairs; ++i)
    if (taken[dev][i] && owner[dev][i] == stream) return base[dev] + 2 * i;
  const int i = (int)(next[dev]++ % kSchedPairs);
  owner[dev][i] = stream;
  taken[dev][i] = true;
  return base[dev] + 2 * i;
}

namespace {

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    sms[dev] = n;
  }
  return sms[dev];
}

// 3-D map over a bf16 [BH][N][d] tensor: box of 64 columns (128 bytes, the
// 128-byte swizzle width) x box_rows rows x 1 head.  Rows past N read as zero.
bool make_map(CUtensorMap* m, const void* base, long long BH, int N, int d, int box_rows) {
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 2-D fp32 map over the backward's dQ accumulator [rows][d]: box (d, 64), no
// swizzle; the target of bulk reduce-adds of 64-row tiles.
bool make_acc_map(CUtensorMap* m, const void* base, long long rows, int d) {
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  const cuuint32_t box[2] = {(cuuint32_t)d, 64};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// 3-D map over uint8 e4m3 codes [planes][rows][cols] (row stride `ld` bytes):
// box of 128 bytes x 128 rows x 1 plane, 128-byte swizzle.  Reads past the
// extents return zero.
bool make_map_u8(CUtensorMap* m, const void* base, long long planes, int rows, int cols, long long ld) {
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)ld, (cuuint64_t)ld * rows};
  const cuuint32_t box[3] = {128, 128, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks shared by forward and backward.  Returns ATTN_OK or an error.
attn_status check_shape(int B, int Hq, int Hkv, int N, int d, float scale, int causal) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  // Grid limits: query tiles on grid.y, (b, h) on grid.x; element counts fit int64.
  if ((N + 127) / 128 > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

unsigned long long wait_limit() { return kDefaultWaitLimitNs; }

// Number of heads whose CTAs are scheduled together so that the operands they
// share (about `bytes_per_head` each) stay resident in L2 (`budget` bytes of
// the 126 MiB L2).  Fewer, larger groups shorten the tail: the heaviest CTAs of
// the last group then start earlier.
int head_group_for(size_t bytes_per_head, long long heads, size_t budget) {
  long long g = bytes_per_head ? (long long)(budget / bytes_per_head) : 32;
  if (g < 1) g = 1;
  if (g > 32) g = 32;
  if (g > heads) g = heads;
  return (int)g;
}

// Diagnostic kernel: one thread waits on an mbarrier that is never completed.
__global__ void selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtx wc{&abort_flag, status, limit_ns};
    mbar_wait(smem_u32(&bar), 0, wc);
  }
}

}  // namespace
}  // namespace attn

namespace attn {
namespace {

constexpr int kMaxSplits = 256;

// Number of key splits: the caller's, or (num_splits == 0) one when the
// unsplit grid already fills the SMs, else the count that minimises the
// forward's span with one CTA per SM: waves (ceil of CTAs / SMs) times (tiles
// per split + one tile's worth of per-CTA prologue and epilogue), preferring
// fewer splits on ties; at most 64 and one split per 128-key tile.  The result
// never leaves a split without a tile.  -1 for an invalid request.
int fwd_splits(int B, int Hq, int Hkv, int Nq, int Nk, int num_splits) {
  if (num_splits < 0 || num_splits > kMaxSplits) return -1;
  const int ktiles = (Nk + 127) / 128;
  auto rounded = [&](int want) {
    want = std::max(1, std::min(want, ktiles));
    const int per = (ktiles + want - 1) / want;
    return (ktiles + per - 1) / per;
  };
  if (num_splits > 0) return rounded(num_splits);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int G = Hq / Hkv;
  const bool packed = G > 1 && (long long)G * Nq <= 128;  // as in fwd_bf16_run
  const long long ctas = packed ? (long long)B * Hkv : (long long)B * Hq * (((Nq + 127) / 128 + 1) / 2);
  if (ctas >= sms) return 1;
  int best = 1;
  long long best_cost = -1;
  for (int want = 1; want <= std::min(64, ktiles); ++want) {
    const int s = rounded(want);
    const long long per = (ktiles + s - 1) / s;
    const long long waves = (ctas * s + sms - 1) / sms;
    const long long cost = waves * (per + 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

size_t fwd_split_lse_offset(long long rows, int d, int splits) {
  return ((size_t)splits * rows * d * 4 + 255) / 256 * 256;
}

size_t fwd_split_workspace_bytes(int B, int Hq, int Nq, int d, int splits) {
  const long long rows = (long long)B * Hq * Nq;
  return fwd_split_lse_offset(rows, d, splits) + ((size_t)splits * rows * 4 + 255) / 256 * 256;
}

// The tcgen05 forward over key splits: splits == 1 writes O (bf16 or fp32)
// and LSE; otherwise O and LSE are the fp32 partial arrays with the given
// strides between splits.
attn_status fwd_bf16_run(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq,
                         int Hkv, int Nq, int Nk, int d, float sl2, int causal, int out_f32, int splits,
                         long long o_stride, long long lse_stride, cudaStream_t s,
                         const uint8_t* bmask = nullptr, int bmask_heads = 1) {
  int* status = status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  // GQA packing when the whole group fits one 128-row tile (decoding).
  const int G = Hq / Hkv;
  const bool packed = G > 1 && (long long)G * Nq <= 128 && !bmask;  // masks may differ per head
  const long long heads = packed ? (long long)B * Hkv : (long long)B * Hq;
  const int rows = packed ? G * Nq : Nq;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, Q, heads, rows, d, 128) || !make_map(&tk, K, (long long)B * Hkv, Nk, d, 128) ||
      !make_map(&tv, V, (long long)B * Hkv, Nk, d, 128))
    return ATTN_ERR_CUDA;
  FwdParams p{};
  p.packed = packed ? 1 : 0;
  p.bmask = bmask;
  p.bmask_heads = bmask_heads;
  p.heads = (int)heads;
  p.rows = rows;
  p.O = O;
  p.LSE = LSE;
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = Nq;
  p.Nk = Nk;
  p.kv_off = causal ? Nk - Nq : 0;
  const int ktiles = (Nk + 127) / 128;
  p.n_splits = splits;
  p.tiles_per_split = (ktiles + splits - 1) / splits;
  p.o_split_stride = o_stride;
  p.lse_split_stride = lse_stride;
  p.n_qtiles = (rows + 127) / 128;
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.head_group = head_group_for((size_t)Nk * d * 2 * 2, heads, size_t(64) << 20);
  if (heads * p.n_pairs * splits > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  p.scale_log2 = sl2;
  p.causal = causal;
  p.out_f32 = out_f32;
  p.wait_limit_ns = wait_limit();
  cudaError_t e;
  if (rows > 128 && !bmask) {
    // Dense two-tile forward: persistent, one CTA per SM (its shared memory
    // and TMEM allow one) over the items.
    const int sms = sm_count();
    p.sched = sched_counter_pair(s);
    if (sms < 1 || !p.sched) return ATTN_ERR_CUDA;
    p.n_items = (int)(heads * p.n_pairs * splits);
    e = launch_fwd_persist(d, tq, tk, tv, p, std::min(p.n_items, sms), s);
  } else {
    e = launch_fwd_bf16(d, tq, tk, tv, p, s);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
  }
  return "ATTN_UNKNOWN_STATUS";
}

attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype in_dtype, attn_dtype out_dtype, void* stream) {
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if ((in_dtype != ATTN_BF16 && in_dtype != ATTN_F32) ||
      (out_dtype != ATTN_BF16 && out_dtype != ATTN_F32))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
    return ATTN_ERR_INVALID_ARG;
  attn_status st = check_shape(B, Hq, Hkv, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float sl2 = scale * 1.4426950408889634f;
  if (in_dtype == ATTN_F32) {
    if (out_dtype != ATTN_F32) return ATTN_ERR_UNSUPPORTED;
    cudaError_t e = launch_fwd_f32(d, static_cast<const float*>(Q), static_cast<const float*>(K),
                                   static_cast<const float*>(V), static_cast<float*>(O), LSE, B, Hq,
                                   Hkv, N, sl2, causal, s);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  return fwd_bf16_run(Q, K, V, O, LSE, B, Hq, Hkv, N, N, d, sl2, causal, out_dtype == ATTN_F32, 1, 0, 0, s);
}

attn_status attn_fwd_split(const void* Q, const void* K, const void* V, void* O, float* LSE,
                           int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                           attn_dtype out_dtype, int num_splits, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_BF16 && out_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
    return ATTN_ERR_INVALID_ARG;
  attn_status st = check_shape(B, Hq, Hkv, Nq, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (Nk < 1) return ATTN_ERR_INVALID_ARG;
  if ((Nk + 127) / 128 > 65535) return ATTN_ERR_UNSUPPORTED;
  const int splits = fwd_splits(B, Hq, Hkv, Nq, Nk, num_splits);
  if (splits < 1) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float sl2 = scale * 1.4426950408889634f;
  if (splits == 1)
    return fwd_bf16_run(Q, K, V, O, LSE, B, Hq, Hkv, Nq, Nk, d, sl2, causal, out_dtype == ATTN_F32, 1, 0, 0, s);
  const size_t need = fwd_split_workspace_bytes(B, Hq, Nq, d, splits);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const long long rows = (long long)B * Hq * Nq;
  float* Opart = static_cast<float*>(workspace);
  float* Lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + fwd_split_lse_offset(rows, d, splits));
  st = fwd_bf16_run(Q, K, V, Opart, Lpart, B, Hq, Hkv, Nq, Nk, d, sl2, causal, 1, splits, rows * d, rows, s);
  if (st != ATTN_OK) return st;
  cudaError_t e = launch_fwd_merge(d, Opart, Lpart, O, LSE, rows, splits, out_dtype == ATTN_F32 ? 1 : 0, s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_fwd_masked(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, int mask_heads, attn_dtype out_dtype, void* stream) {
  if (!Q || !K || !V || !O || !LSE || !block_mask) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_BF16 && out_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
    return ATTN_ERR_INVALID_ARG;
  attn_status st = check_shape(B, Hq, Hkv, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (mask_heads != 1 && mask_heads != Hq) return ATTN_ERR_INVALID_ARG;
  if ((N + 127) / 128 > kMaxMaskTiles) return ATTN_ERR_UNSUPPORTED;
  return fwd_bf16_run(Q, K, V, O, LSE, B, Hq, Hkv, N, N, d, scale * 1.4426950408889634f, causal,
                      out_dtype == ATTN_F32, 1, 0, 0, static_cast<cudaStream_t>(stream), block_mask, mask_heads);
}

int attn_fp8_vt_stride(int N) { return N < 1 ? 0 : (N + 15) / 16 * 16; }

attn_status attn_quantize_fp8(const void* X, void* codes, float* scales, long long BH, int N, int d,
                              int transpose, void* stream) {
  if (!X || !codes || !scales) return ATTN_ERR_INVALID_ARG;
  if (BH < 1 || N < 1 || (transpose != 0 && transpose != 1)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(X, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = launch_quantize_fp8(d, static_cast<const uint16_t*>(X), static_cast<uint8_t*>(codes), scales, BH,
                                      N, transpose, attn_fp8_vt_stride(N), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue) return ATTN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_fwd_fp8(const void* Qc, const float* q_scale, const void* Kc, const float* k_scale,
                         const void* Vtc, const float* v_scale, void* O, float* LSE, int B, int Hq, int Hkv,
                         int N, int d, float scale, int causal, attn_dtype out_dtype, void* stream) {
  if (!Qc || !q_scale || !Kc || !k_scale || !Vtc || !v_scale || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_BF16 && out_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (!aligned(Qc, 16) || !aligned(Kc, 16) || !aligned(Vtc, 16) || !aligned(O, 16) || !aligned(LSE, 4) ||
      !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
    return ATTN_ERR_INVALID_ARG;
  attn_status st = check_shape(B, Hq, Hkv, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  int* status = status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  const int ldt = attn_fp8_vt_stride(N);
  CUtensorMap tq, tk, tv;
  if (!make_map_u8(&tq, Qc, (long long)B * Hq, N, 128, 128) || !make_map_u8(&tk, Kc, (long long)B * Hkv, N, 128, 128) ||
      !make_map_u8(&tv, Vtc, (long long)B * Hkv, 128, ldt, ldt))
    return ATTN_ERR_CUDA;
  Fp8FwdParams p{};
  p.sq = q_scale;
  p.sk = k_scale;
  p.sv = v_scale;
  p.O = O;
  p.LSE = LSE;
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.T = (N + 127) / 128;
  p.heads = B * Hq;
  p.n_pairs = (p.T + 1) / 2;
  if ((long long)p.heads * p.n_pairs > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  p.head_group = head_group_for((size_t)N * 128 * 2, p.heads, size_t(64) << 20);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal;
  p.out_f32 = out_dtype == ATTN_F32;
  p.wait_limit_ns = wait_limit();
  cudaError_t e = launch_fwd_fp8(tq, tk, tv, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_fwd_split_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int num_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nq < 1 || Nk < 1 || (d != 64 && d != 128)) return 0;
  const int splits = fwd_splits(B, Hq, Hkv, Nq, Nk, num_splits);
  if (splits < 1) return 0;
  return splits == 1 ? 0 : fwd_split_workspace_bytes(B, Hq, Nq, d, splits);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d) {
  if (check_shape(B, Hq, Hkv, N, d, 1.0f, 0) != ATTN_OK) return 0;
  return bwd_workspace_bytes(B, Hq, N, d);
}

}  // extern "C"

namespace {

attn_status bwd_stages(unsigned stages, const void* Q, const void* K, const void* V,
                       const void* O, const void* dO, const float* LSE, void* dQ, void* dK,
                       void* dV, int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                       attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream,
                       const uint8_t* bmask = nullptr, int bmask_heads = 1) {
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
    return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!aligned(q, 16)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(LSE, 4) || !aligned(workspace, 256)) return ATTN_ERR_INVALID_ARG;
  attn_status st = check_shape(B, Hq, Hkv, N, d, scale, causal);
  if (st != ATTN_OK) return st;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < bwd_workspace_bytes(B, Hq, N, d)) return ATTN_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk, tv, tdo;
  // Query-side tiles of the backward are 128 rows, like the key-side tiles.
  if (!make_map(&tq, Q, (long long)B * Hq, N, d, 128) || !make_map(&tdo, dO, (long long)B * Hq, N, d, 128) ||
      !make_map(&tk, K, (long long)B * Hkv, N, d, 128) || !make_map(&tv, V, (long long)B * Hkv, N, d, 128))
    return ATTN_ERR_CUDA;
  const int Npad = (N + bwd_row_padding() - 1) / bwd_row_padding() * bwd_row_padding();
  BwdParams p{};
  p.Q = static_cast<const uint16_t*>(Q);
  p.K = static_cast<const uint16_t*>(K);
  p.V = static_cast<const uint16_t*>(V);
  p.O = static_cast<const uint16_t*>(O);
  p.dO = static_cast<const uint16_t*>(dO);
  p.LSE = LSE;
  p.dQ = static_cast<uint16_t*>(dQ);
  p.dK = static_cast<uint16_t*>(dK);
  p.dV = static_cast<uint16_t*>(dV);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t rows = (size_t)B * Hq * Npad;
  const size_t acc_bytes = (rows * d * 4 + 255) / 256 * 256;
  const size_t vec_bytes = (rows * 4 + 255) / 256 * 256;
  p.dQacc = reinterpret_cast<float*>(ws);
  p.negD = reinterpret_cast<float*>(ws + acc_bytes);
  p.negLSE2 = reinterpret_cast<float*>(ws + acc_bytes + vec_bytes);
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.Npad = Npad;
  p.bmask = bmask;
  p.bmask_heads = bmask_heads;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal;
  // Per kv head the CTAs share Q and dO (bf16) and the dQ accumulator (fp32) of its group.
  p.head_group = head_group_for((size_t)(Hq / Hkv) * N * d * (2 + 2 + 4), (long long)B * Hkv,
                                size_t(32) << 20);
  if ((long long)B * Hkv * ((N + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  p.wait_limit_ns = wait_limit();
  CUtensorMap tacc;
  if (!make_acc_map(&tacc, p.dQacc, (long long)rows, d)) return ATTN_ERR_CUDA;
  cudaError_t e = launch_bwd_bf16(d, tq, tk, tv, tdo, tacc, p, stages, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

attn_status attn_bwd_masked(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, int mask_heads, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (!block_mask || (mask_heads != 1 && mask_heads != Hq)) return ATTN_ERR_INVALID_ARG;
  if (check_shape(B, Hq, Hkv, N, d, scale, causal) == ATTN_OK &&
      (long long)(Hq / Hkv) * ((N + 127) / 128) > kMaxMaskIters)
    return ATTN_ERR_UNSUPPORTED;
  return bwd_stages(kBwdAll, Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, scale, causal, ATTN_BF16,
                    workspace, workspace_bytes, stream, block_mask, mask_heads);
}

attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O,
                     const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_stages(kBwdAll, Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, scale, causal,
                    dtype, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_preprocess(const void* Q, const void* K, const void* V, const void* O,
                                const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                attn_dtype dtype, void* workspace, size_t workspace_bytes,
                                void* stream) {
  return bwd_stages(kBwdPre, Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, scale, causal,
                    dtype, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_main(const void* Q, const void* K, const void* V, const void* O,
                          const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                          int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                          attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_stages(kBwdMain, Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, scale, causal,
                    dtype, workspace, workspace_bytes, stream);
}

attn_status attn_bwd_convert(const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                             int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                             attn_dtype dtype, void* workspace, size_t workspace_bytes,
                             void* stream) {
  return bwd_stages(kBwdConvert, Q, K, V, O, dO, LSE, dQ, dK, dV, B, Hq, Hkv, N, d, scale, causal,
                    dtype, workspace, workspace_bytes, stream);
}

attn_status attn_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int* p = status_ptr();
  if (!p) return ATTN_ERR_CUDA;
  int v = 0, zero = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0 && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (v == kDevTimeout) return ATTN_ERR_TIMEOUT;
  return v == 0 ? ATTN_OK : ATTN_ERR_DEVICE;
}

attn_status attn_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return ATTN_ERR_INVALID_ARG;
  int* status = status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
