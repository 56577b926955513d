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

// One warp per query row; lane c holds columns [c*D/32, (c+1)*D/32).
template <int D>
__global__ void __launch_bounds__(256) fwd_merge_kernel(const float* __restrict__ Opart,
                                                        const float* __restrict__ Lpart, void* O, float* LSE,
                                                        long long rows, int n_splits, int out_f32) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += ((long long)gridDim.x * blockDim.x) >> 5) {
    // Largest partial LSE (natural-log units), then the weights in base 2.
    float mx = -INFINITY;
    for (int s = lane; s < n_splits; s += 32) mx = fmaxf(mx, Lpart[(long long)s * rows + r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float acc[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
      for (int s = 0; s < n_splits; ++s) {
        const float ls = Lpart[(long long)s * rows + r];
        const float w = ex2((ls - mx) * 1.4426950408889634f);  // 0 for an empty part
        wsum += w;
        const float* src = Opart + ((long long)s * rows + r) * D + lane * EPL;
#pragma unroll
        for (int k = 0; k < EPL; ++k) acc[k] = fmaf(w, src[k], acc[k]);
      }
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
  if (d == 128)
    fwd_merge_kernel<128><<<blocks, 256, 0, stream>>>(Opart, Lpart, O, LSE, rows, n_splits, out_f32);
  else if (d == 64)
    fwd_merge_kernel<64><<<blocks, 256, 0, stream>>>(Opart, Lpart, O, LSE, rows, n_splits, out_f32);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace attn
