// fwd_merge.cu -- combine the partial results of a forward split over keys.
//
// A forward whose key range is cut into S parts produces, per query row, S
// partial results (O_s normalised over the keys of part s, LSE_s = ln of that
// part's sum of e^{s_ij}).  They merge exactly as two blocks of the online
// softmax do ("LLM 注意力与计算内核精读笔记 · 02 FlashAttention" §5, the (m, l)
// merge; §12.1, FlashDecoding, applies it to key splits):
//     LSE = ln sum_s e^{LSE_s},    O = sum_s e^{LSE_s - LSE} O_s.
// Parts with no kept key carry LSE_s = -inf and O_s = 0 and get weight 0; a
// row with no kept key at all gets O = 0 and LSE = -inf.
#include <algorithm>

#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

template <int EPL>
struct MergeVec;  // the EPL floats of one lane, loaded as one vector
template <>
struct MergeVec<4> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ void zero() { v = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ float operator[](int k) const {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
  }
};
template <>
struct MergeVec<2> {
  float2 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float2*>(p); }
  __device__ __forceinline__ void zero() { v = make_float2(0.f, 0.f); }
  __device__ __forceinline__ float operator[](int k) const { return k == 0 ? v.x : v.y; }
};

// One warp per query row; lane c holds columns [c*D/32, (c+1)*D/32).  Lane s
// reads part s's LSE and computes its weight; the parts' O rows are read in
// batches of 16 with every load of a batch issued before the batch is summed,
// so a row costs a few memory latencies instead of one per part.
template <int D>
__global__ void __launch_bounds__(256, 1) fwd_merge_kernel(const float* __restrict__ Opart,
                                                        const float* __restrict__ Lpart, void* O, float* LSE,
                                                        long long rows, int n_splits, int out_f32) {
  constexpr int EPL = D / 32;
  constexpr int BATCH = 16;
  const int lane = threadIdx.x & 31;
  // Launched behind the split forward: its partial results must be complete.
  griddep_wait();
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((long long)gridDim.x * blockDim.x) >> 5) {
    // Largest partial LSE (natural-log units), then the weights in base 2.
    float mx = -INFINITY;
    float ls_first = -INFINITY;  // this lane's part among the first 32
    for (int s = lane; s < n_splits; s += 32) {
      const float v = Lpart[(long long)s * rows + r];
      if (s < 32) ls_first = v;
      mx = fmaxf(mx, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
      for (int s0 = 0; s0 < n_splits; s0 += 32) {
        const int s = s0 + lane;
        const float ls = s0 == 0 ? ls_first : (s < n_splits ? Lpart[(long long)s * rows + r] : -INFINITY);
        const float w = ex2((ls - mx) * 1.4426950408889634f);  // 0 for an empty part or past the last
        wsum += w;
        const int cnt = min(32, n_splits - s0);
        for (int b = 0; b < cnt; b += BATCH) {
          MergeVec<EPL> v[BATCH];
#pragma unroll
          for (int u = 0; u < BATCH; ++u) {
            if (b + u < cnt)
              v[u].load(Opart + ((long long)(s0 + b + u) * rows + r) * D + lane * EPL);
            else
              v[u].zero();
          }
#pragma unroll
          for (int u = 0; u < BATCH; ++u) {
            const float wu = __shfl_sync(0xffffffffu, w, b + u);  // b + u < 32
#pragma unroll
            for (int k = 0; k < EPL; ++k) acc[k] = fmaf(wu, v[u][k], acc[k]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (out_f32) {
      float* dst = static_cast<float*>(O) + r * D + lane * EPL;
#pragma unroll
      for (int k = 0; k < EPL; ++k) dst[k] = acc[k] * inv;
    } else {
      uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(O) + r * D + lane * EPL);
#pragma unroll
      for (int k = 0; k < EPL / 2; ++k) dst[k] = pack_bf16(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    }
    if (lane == 0) LSE[r] = wsum > 0.f ? mx + lg2(wsum) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_fwd_merge(int d, const float* Opart, const float* Lpart, void* O, float* LSE, long long rows,
                             int n_splits, int out_f32, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = (int)std::min<long long>((rows + 7) / 8, (long long)sms * 8);
  // Programmatic stream serialization: the merge may be scheduled while the
  // split forward drains, and waits for it on the device (griddep_wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (d == 128)
    e = cudaLaunchKernelEx(&cfg, fwd_merge_kernel<128>, Opart, Lpart, O, LSE, rows, n_splits, out_f32);
  else if (d == 64)
    e = cudaLaunchKernelEx(&cfg, fwd_merge_kernel<64>, Opart, Lpart, O, LSE, rows, n_splits, out_f32);
  else
    return cudaErrorInvalidValue;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn
