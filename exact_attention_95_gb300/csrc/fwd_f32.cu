// fwd_f32.cu -- exact attention forward in fp32 on CUDA cores.
//
// Same mathematics as the tensor-core forward (online max / sum merge of
// "LLM 注意力与计算内核精读笔记 · 02 FlashAttention" §5, 1/l applied once),
// carried out entirely in fp32 FFMA so that fp32 inputs keep fp32 accuracy.
// The work is small (latency-bound); the kernel favours simplicity.
//
// Block: 256 threads in two groups of 128 that take alternate key tiles of
// the same query rows (a row's work is a chain over its keys; two chains per
// row halve it) and merge their (m, l, O) at the end as two blocks of the
// online softmax.  In a group, TPR = d/32 consecutive threads share one query
// row, each holding 32 of its d components of q and of the output
// accumulator.  Keys are streamed in tiles of 32 through the group's shared
// memory (the next tile's loads are in flight in registers while the current
// one is used) and read back as float4: the threads of a warp read at most
// TPR distinct addresses at a time (broadcasts), so rows need no padding.
// The partial dot products of a row's TPR threads are combined with warp
// shuffles.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kKT = 32;      // keys per shared-memory tile
constexpr int kGroups = 2;   // key-tile groups per block
constexpr int kF32Threads = 128 * kGroups;

template <int D>
constexpr int f32_smem_bytes() {
  return kGroups * 2 * kKT * D * 4;  // K and V tiles per group
}

__device__ __forceinline__ void group_sync(int grp) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(128) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kF32Threads)
    fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                   const float* __restrict__ V, float* __restrict__ O, float* __restrict__ LSE,
                   int Hq, int Hkv, int N, float sl2, int causal) {
  constexpr int TPR = D / 32;
  constexpr int RPB = 128 / TPR;           // rows per block
  constexpr int PER = kKT * D / 4 / 128;   // float4 of K (and of V) per thread and tile
  extern __shared__ float4 f32_smem[];
  const int grp = threadIdx.x >> 7;
  const int tid = threadIdx.x & 127;
  float* const Ks = reinterpret_cast<float*>(f32_smem) + grp * 2 * kKT * D;  // [kKT][D]
  float* const Vs = Ks + kKT * D;

  const int bh = blockIdx.y;
  const int b = bh / Hq, h = bh - (bh / Hq) * Hq;
  const int bh_kv = b * Hkv + h / (Hq / Hkv);
  const int sub = tid % TPR;
  const int r = tid / TPR;
  const int q = blockIdx.x * RPB + r;
  const bool valid = q < N;
  const size_t qrow = (size_t)bh * N + (valid ? q : 0);

  float qv[32], acc[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    qv[k] = Q[qrow * D + sub * 32 + k];
    acc[k] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int q_last = min(N - 1, blockIdx.x * RPB + RPB - 1);
  const int kend = causal ? q_last + 1 : N;
  const float4* Kh = reinterpret_cast<const float4*>(K + (size_t)bh_kv * N * D);
  const float4* Vh = reinterpret_cast<const float4*>(V + (size_t)bh_kv * N * D);
  float4 pk[PER], pv[PER];
  auto load_tile = [&](int k0) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = tid + i * 128;  // float4 index within the tile
      const int kr = idx / (D / 4);
      const bool in = k0 + kr < N;
      const size_t g = (size_t)k0 * (D / 4) + idx;
      pk[i] = in ? Kh[g] : make_float4(0.f, 0.f, 0.f, 0.f);
      pv[i] = in ? Vh[g] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  const int k_first = grp * kKT;
  if (k_first < kend) load_tile(k_first);
  for (int k0 = k_first; k0 < kend; k0 += kGroups * kKT) {
    group_sync(grp);  // the previous tile has been read
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = tid + i * 128;
      reinterpret_cast<float4*>(Ks)[idx] = pk[i];
      reinterpret_cast<float4*>(Vs)[idx] = pv[i];
    }
    group_sync(grp);
    if (k0 + kGroups * kKT < kend) load_tile(k0 + kGroups * kKT);  // lands while this tile is used
    float s[kKT];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kKT; ++j) {
      const float4* kr4 = reinterpret_cast<const float4*>(Ks + j * D + sub * 32);
      float part = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 8; ++k4) {
        const float4 kv = kr4[k4];
        part = fmaf(qv[4 * k4 + 0], kv.x, part);
        part = fmaf(qv[4 * k4 + 1], kv.y, part);
        part = fmaf(qv[4 * k4 + 2], kv.z, part);
        part = fmaf(qv[4 * k4 + 3], kv.w, part);
      }
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      const int key = k0 + j;
      const bool keep = key < N && (!causal || key <= q);
      s[j] = keep ? part * sl2 : -INFINITY;
      mx = fmaxf(mx, s[j]);
    }
    const float m_new = fmaxf(m, mx);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2(m - m_use);
    float rs = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] *= alpha;
#pragma unroll
    for (int j = 0; j < kKT; ++j) {
      const float pj = ex2(s[j] - m_use);
      rs += pj;
      const float4* vr4 = reinterpret_cast<const float4*>(Vs + j * D + sub * 32);
#pragma unroll
      for (int k4 = 0; k4 < 8; ++k4) {
        const float4 vv = vr4[k4];
        acc[4 * k4 + 0] = fmaf(pj, vv.x, acc[4 * k4 + 0]);
        acc[4 * k4 + 1] = fmaf(pj, vv.y, acc[4 * k4 + 1]);
        acc[4 * k4 + 2] = fmaf(pj, vv.z, acc[4 * k4 + 2]);
        acc[4 * k4 + 3] = fmaf(pj, vv.w, acc[4 * k4 + 3]);
      }
    }
    l = l * alpha + rs;
    m = m_new;
  }
  // Merge the two groups' (m, l, O) per row ("LLM 注意力与计算内核精读笔记 ·
  // 02 FlashAttention" §5): group 1 hands its partial results to group 0
  // through shared memory (the tiles are no longer needed).
  __syncthreads();
  float* const part = reinterpret_cast<float*>(f32_smem);  // [128 threads][34]
  if (grp == 1) {
    float* dst = part + tid * 34;
    dst[0] = m;
    dst[1] = l;
#pragma unroll
    for (int k = 0; k < 32; ++k) dst[2 + k] = acc[k];
  }
  __syncthreads();
  if (grp == 0) {
    const float* src = part + tid * 34;
    const float m1 = src[0], l1 = src[1];
    const float mt = fmaxf(m, m1);
    const float mu = mt == -INFINITY ? 0.f : mt;
    const float a0 = ex2(m - mu), a1 = ex2(m1 - mu);
    const float lt = a0 * l + a1 * l1;
    if (valid) {
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) O[qrow * D + sub * 32 + k] = (a0 * acc[k] + a1 * src[2 + k]) * inv;
      if (sub == 0) LSE[qrow] = lt > 0.f ? (mt + lg2(lt)) * 0.69314718055994531f : -INFINITY;
    }
  }
}

}  // namespace

cudaError_t launch_fwd_f32(int d, const float* Q, const float* K, const float* V, float* O,
                           float* LSE, int B, int Hq, int Hkv, int N, float scale_log2,
                           int causal, cudaStream_t stream) {
  const int rpb = 128 / (d / 32);
  dim3 grid((N + rpb - 1) / rpb, B * Hq);
  cudaError_t e;
  if (d == 64) {
    constexpr int smem = f32_smem_bytes<64>();
    static_assert(smem >= 128 * 34 * 4, "merge buffer");
    e = cudaFuncSetAttribute(fwd_f32_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fwd_f32_kernel<64><<<grid, kF32Threads, smem, stream>>>(Q, K, V, O, LSE, Hq, Hkv, N, scale_log2, causal);
  } else if (d == 128) {
    constexpr int smem = f32_smem_bytes<128>();
    static_assert(smem >= 128 * 34 * 4, "merge buffer");
    e = cudaFuncSetAttribute(fwd_f32_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fwd_f32_kernel<128><<<grid, kF32Threads, smem, stream>>>(Q, K, V, O, LSE, Hq, Hkv, N, scale_log2, causal);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace attn
